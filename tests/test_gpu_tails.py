"""bf16 fused forward and backward when 128 does not divide N (and N < 128), through the
C ABI, against the oracle with the tolerances of the other bf16 tests.

The definition on the first page ('Attention as a mathematical problem') puts no
condition on N.  The last 128-row tile of every head is then partial: its loads bring
in rows past N (the next head's, or zeros past the end of the arrays), which must get
no weight, and nothing may be written past row N of any head.  Several heads are used
so that a row of one head leaking into another shows up against the oracle, and the
outputs sit between canaries (a write past the last head's rows breaks them; a row
left unwritten keeps its NaN fill and fails the comparison)."""
import math

import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16_GRAD_RL2, TOL_BF16_LSE_REL, TOL_BF16_O_ABS, Guarded, lse_rel, max_abs, rel_l2
from optimal_tiling_gb300 import attn, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _fwd(x, scale, mask=None, block=128):
    B, H, N, d = x["q"].shape
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    dm = mask.to(DEV) if mask is not None else None
    O = Guarded((B, H, N, d), torch.bfloat16, DEV)
    L = Guarded((B, H, N), torch.float32, DEV)
    attn.attn_fwd_masked(q, k, v, scale, mask=dm, block=block, out=O.t, lse=L.t)
    assert attn.attn_device_status() == attn.ATTN_OK
    assert O.intact() and L.intact(), "write outside an output tensor"
    return O.t, L.t


def _bwd(x, scale, o, lse, mask=None, block=128):
    B, H, N, d = x["q"].shape
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    dm = mask.to(DEV) if mask is not None else None
    g = [Guarded((B, H, N, d), torch.bfloat16, DEV) for _ in range(3)]
    attn.attn_bwd_masked(q, k, v, o, do, lse, scale, mask=dm, block=block, dq=g[0].t, dk=g[1].t, dv=g[2].t)
    assert attn.attn_device_status() == attn.ATTN_OK
    assert all(t.intact() for t in g), "write outside an output tensor"
    return [t.t.float().cpu().numpy() for t in g]


def _per_head_masks(nh, N, block, seed):
    nb = (N + block - 1) // block
    ms = [inputs.random_block_mask(nb * 128, seed=seed + h, p=0.5)[:nb, :nb].clone() for h in range(nh)]
    return torch.stack(ms).contiguous()


@pytest.mark.parametrize("N", [1, 5, 64, 100, 129, 192, 200, 383, 1000])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_forward_tails(oracle_mod, N, d):
    B, H = 1, 3
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=N + d, with_do=False)
    s = 1.0 / math.sqrt(d)
    o, lse = _fwd(x, s)
    Or, Lr = oracle_mod.fwd_naive(x["q"], x["k"], x["v"], s)
    assert max_abs(o.float().cpu().numpy(), Or) <= TOL_BF16_O_ABS
    assert lse_rel(lse.cpu().numpy(), Lr) <= TOL_BF16_LSE_REL


@pytest.mark.parametrize("N,d,block,shared", [(200, 128, 128, True), (300, 64, 128, True), (300, 128, 64, False),
                                              (150, 64, 64, False), (450, 256, 64, False), (333, 256, 128, True)])
def test_forward_tails_masked(oracle_mod, N, d, block, shared):
    """Block masks over ceil(N / block) blocks: with 64-blocks the last 128-row tile may cover
    one mask row and the last key block one mask column (N % 128 <= 64)."""
    B, H = 2, 1
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=3 * N + d, with_do=False)
    s = 1.0 / math.sqrt(d)
    nb = (N + block - 1) // block
    mask = (inputs.random_block_mask(nb * 128, seed=N, p=0.5)[:nb, :nb].contiguous() if shared
            else _per_head_masks(B * H, N, block, seed=N))
    o, lse = _fwd(x, s, mask, block)
    om = np.broadcast_to(mask.numpy(), (B * H, nb, nb)).copy()
    Or, Lr = oracle_mod.fwd_naive_m(x["q"], x["k"], x["v"], s, om, block)
    assert max_abs(o.float().cpu().numpy(), Or) <= TOL_BF16_O_ABS
    assert lse_rel(lse.cpu().numpy(), Lr) <= TOL_BF16_LSE_REL


@pytest.mark.parametrize("N", [1, 37, 64, 100, 129, 192, 200, 383])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_backward_tails(oracle_mod, N, d):
    """The backward's row terms and dQ accumulator have N rounded up to 64 rows per head;
    the rows past N are padding with zero weight."""
    B, H = 1, 3
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=5 * N + d)
    s = 1.0 / math.sqrt(d)
    o, lse = _fwd(x, s)
    dq, dk, dv = _bwd(x, s, o, lse)
    gQ, gK, gV, _, _ = oracle_mod.bwd_naive(x["q"], x["k"], x["v"], x["do"], s)
    for name, got, ref in (("dQ", dq, gQ), ("dK", dk, gK), ("dV", dv, gV)):
        assert rel_l2(got, ref) <= TOL_BF16_GRAD_RL2, name


@pytest.mark.parametrize("N,d,block", [(200, 128, 128), (300, 64, 64), (150, 128, 64), (383, 64, 128),
                                         (200, 256, 64), (330, 256, 128)])
def test_backward_tails_masked(oracle_mod, N, d, block):
    B, H = 1, 2
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=7 * N + block)
    s = 1.0 / math.sqrt(d)
    mask = _per_head_masks(B * H, N, block, seed=2 * N)
    o, lse = _fwd(x, s, mask, block)
    dq, dk, dv = _bwd(x, s, o, lse, mask, block)
    om = mask.numpy()
    gQ, gK, gV = oracle_mod.bwd_naive_m(x["q"], x["k"], x["v"], x["do"], s, om, block)
    for name, got, ref in (("dQ", dq, gQ), ("dK", dk, gK), ("dV", dv, gV)):
        assert rel_l2(got, ref) <= TOL_BF16_GRAD_RL2, name

