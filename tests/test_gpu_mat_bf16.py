"""Materialising two-GEMM forward (the small-cache comparison schedule) against
the oracle, through the C ABI, with the same tolerances as the fused forward:
O max-abs <= 1e-2, LSE relative <= 1e-3."""
import math

import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16_LSE_REL, TOL_BF16_O_ABS, Guarded, lse_rel, max_abs
from optimal_tiling_gb300 import attn, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _mat(x, scale, mask=None):
    B, H, N, d = x["q"].shape
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    dm = mask.to(DEV) if mask is not None else None
    O = Guarded((B, H, N, d), torch.bfloat16, DEV)
    L = Guarded((B, H, N), torch.float32, DEV)
    attn.attn_fwd_materialized(q, k, v, scale, block_mask=dm, out=O.t, lse=L.t)
    assert attn.attn_device_status() == attn.ATTN_OK
    assert O.intact() and L.intact(), "write outside an output tensor"
    return O.t.float().cpu().numpy(), L.t.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N,BH", [(128, (1, 1)), (384, (1, 3))])
def test_small_shapes(oracle_mod, d, N, BH):
    x = inputs.make_inputs(*BH, N, d, torch.bfloat16, seed=N * 3 + d, with_do=False)
    s = 1.0 / math.sqrt(d)
    O, L = _mat(x, s)
    Or, Lr = oracle_mod.fwd_naive(x["q"], x["k"], x["v"], s)
    assert max_abs(O, Or) <= TOL_BF16_O_ABS
    assert lse_rel(L, Lr) <= TOL_BF16_LSE_REL


def test_block_mask_and_empty_rows(oracle_mod):
    N, d = 768, 128
    x = inputs.make_inputs(2, 1, N, d, torch.bfloat16, seed=31, with_do=False)
    m = inputs.random_block_mask(N, seed=8, p=0.3)
    m[2, :] = 0
    O, L = _mat(x, 0.09, m)
    Or, Lr = oracle_mod.fwd_naive(x["q"], x["k"], x["v"], 0.09, m.numpy())
    assert max_abs(O, Or) <= TOL_BF16_O_ABS
    assert lse_rel(L, Lr) <= TOL_BF16_LSE_REL
    assert np.all(O[:, :, 256:384] == 0) and np.all(np.isneginf(L[:, :, 256:384]))


@pytest.mark.parametrize("name", ["dsweep_d64", "dsweep_d128", "dsweep_d256"])
def test_dsweep_workloads_sampled_and_against_fused(oracle_mod, name):
    """The d-sweep workloads, full size: sampled rows against the oracle, and the
    whole output against the fused kernel's (both evaluate the same function)."""
    w = inputs.WORKLOADS[name]
    x, _ = inputs.workload_inputs(w, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    om, lm = attn.attn_fwd_materialized(q, k, v, w.scale)
    of, lf = attn.attn_fwd(q, k, v, w.scale)
    assert attn.attn_device_status() == attn.ATTN_OK
    B, H, N, d = w.shape
    r = np.random.default_rng(d)
    heads = np.concatenate([[0, B * H - 1], r.integers(0, B * H, 30)]).astype(np.int32)
    rows = np.concatenate([[0, N - 1], r.integers(0, N, 30)]).astype(np.int32)
    Or, Lr = oracle_mod.fwd_rows(x["q"], x["k"], x["v"], w.scale, heads, rows)
    Om = om.float().cpu().numpy().reshape(B * H, N, d)
    Lm = lm.cpu().numpy().reshape(B * H, N)
    assert max_abs(Om[heads, rows], Or) <= TOL_BF16_O_ABS
    assert lse_rel(Lm[heads, rows], Lr) <= TOL_BF16_LSE_REL
    assert float((om.float() - of.float()).abs().max()) <= 2 * TOL_BF16_O_ABS
    assert float(((lm - lf).abs() / lf.abs()).max()) <= 2 * TOL_BF16_LSE_REL


@pytest.mark.parametrize("d", [64, 128, 256])
def test_negative_scale(oracle_mod, d):
    """s < 0: the row bound c_i = |s| |q_i| max_j |k_j| still bounds every score s q_i . k_j
    from above, so the stored exponentials stay <= 1 and O, LSE match the oracle."""
    N = 384
    x = inputs.make_inputs(1, 2, N, d, torch.bfloat16, seed=N + d + 5, with_do=False)
    s = -1.0 / math.sqrt(d)
    O, L = _mat(x, s)
    Or, Lr = oracle_mod.fwd_naive(x["q"], x["k"], x["v"], s)
    assert max_abs(O, Or) <= TOL_BF16_O_ABS
    assert lse_rel(L, Lr) <= TOL_BF16_LSE_REL
