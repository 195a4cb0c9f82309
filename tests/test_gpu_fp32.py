"""fp32 SIMT path (true fp32 arithmetic) against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from gpu_util import TOL_F32_ABS, Guarded, max_abs
from optimal_tiling_gb300 import attn, inputs

pytestmark = pytest.mark.gpu


def _run(B, H, N, d, scale, mask, seed=0, oracle_mod=None):
    dev = torch.device("cuda")
    x = inputs.make_inputs(B, H, N, d, torch.float32, seed=seed)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    dmask = mask.to(dev) if mask is not None else None
    O = Guarded((B, H, N, d), torch.float32, dev)
    L = Guarded((B, H, N), torch.float32, dev)
    attn.attn_fwd(q, k, v, scale, block_mask=dmask, out=O.t, lse=L.t)
    dQ, dK, dV = (Guarded((B, H, N, d), torch.float32, dev) for _ in range(3))
    attn.attn_bwd(q, k, v, O.t, do, L.t, scale, block_mask=dmask, dq=dQ.t, dk=dK.t, dv=dV.t)
    assert attn.attn_device_status() == attn.ATTN_OK
    for g in (O, L, dQ, dK, dV):
        assert g.intact(), "write outside an output tensor"
    m = mask.numpy() if mask is not None else None
    Or, Lr = oracle_mod.fwd_naive(x["q"], x["k"], x["v"], scale, m)
    gQ, gK, gV, _, _ = oracle_mod.bwd_naive(x["q"], x["k"], x["v"], x["do"], scale, m)
    return (O.t.cpu().numpy(), L.t.cpu().numpy(), dQ.t.cpu().numpy(), dK.t.cpu().numpy(),
            dV.t.cpu().numpy()), (Or, Lr, gQ, gK, gV)


def _check(got, ref):
    O, L, dQ, dK, dV = got
    Or, Lr, gQ, gK, gV = ref
    assert max_abs(O, Or) <= TOL_F32_ABS
    fin = np.isfinite(Lr)
    assert np.array_equal(np.isneginf(L), np.isneginf(Lr))
    assert max_abs(L[fin], Lr[fin]) <= TOL_F32_ABS
    for g, r in ((dQ, gQ), (dK, gK), (dV, gV)):
        assert max_abs(g, r) <= TOL_F32_ABS * max(1.0, float(np.max(np.abs(r))))


def test_fp32_small_workload(oracle_mod):
    """B=1 H=1 N=256 d=64, s=1, no mask, seed 0."""
    w = inputs.WORKLOADS["fp32_small"]
    got, ref = _run(w.B, w.H, w.N, w.d, w.scale, None, oracle_mod=oracle_mod)
    _check(got, ref)


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 1, 8), (2, 3, 7, 24), (1, 2, 300, 64), (1, 1, 130, 256),
                                     (2, 1, 129, 33)])
def test_fp32_ragged_shapes(oracle_mod, B, H, N, d):
    got, ref = _run(B, H, N, d, 1.0 / np.sqrt(d), None, seed=N + d, oracle_mod=oracle_mod)
    _check(got, ref)


def test_fp32_block_mask_and_empty_rows(oracle_mod):
    N = 384
    mask = torch.tensor([[0, 0, 0], [1, 0, 1], [0, 1, 1]], dtype=torch.uint8)  # query block 0 sees nothing
    got, ref = _run(1, 2, N, 32, 0.3, mask, seed=3, oracle_mod=oracle_mod)
    _check(got, ref)
    O, L = got[0], got[1]
    assert np.all(O[:, :, :128] == 0) and np.all(np.isneginf(L[:, :, :128]))
    assert np.all(got[2][:, :, :128] == 0)
