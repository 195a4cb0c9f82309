"""Materialising backward (P and dS stored in HBM, then three GEMMs) against the
oracle and against the fused backward, through the C ABI.  Tolerance: the
backward's relative-L2 <= 2e-2 on dQ, dK and dV."""
import math

import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16_GRAD_RL2, Guarded, rel_l2
from optimal_tiling_gb300 import attn, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _run(x, scale, mask=None):
    B, H, N, d = x["q"].shape
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    dm = mask.to(DEV) if mask is not None else None
    o, lse = attn.attn_fwd(q, k, v, scale, block_mask=dm)
    g = [Guarded((B, H, N, d), torch.bfloat16, DEV) for _ in range(3)]
    attn.attn_bwd_materialized(q, k, v, o, do, lse, scale, block_mask=dm, dq=g[0].t, dk=g[1].t, dv=g[2].t)
    assert attn.attn_device_status() == attn.ATTN_OK
    assert all(t.intact() for t in g), "write outside an output tensor"
    return [t.t.float().cpu().numpy() for t in g], (q, k, v, o, do, lse, dm)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,BH", [(128, (1, 1)), (384, (1, 3))])
def test_small_shapes(oracle_mod, d, N, BH):
    x = inputs.make_inputs(*BH, N, d, torch.bfloat16, seed=N + 7 * d)
    s = 1.0 / math.sqrt(d)
    got, _ = _run(x, s)
    ref = oracle_mod.bwd_naive(x["q"], x["k"], x["v"], x["do"], s)[:3]
    for name, a, r in zip(("dQ", "dK", "dV"), got, ref):
        assert rel_l2(a, r) <= TOL_BF16_GRAD_RL2, name


def test_block_mask_and_empty_rows(oracle_mod):
    N, d = 768, 128
    x = inputs.make_inputs(1, 2, N, d, torch.bfloat16, seed=71)
    m = inputs.random_block_mask(N, seed=9, p=0.3)
    m[1, :] = 0
    got, _ = _run(x, 0.09, m)
    ref = oracle_mod.bwd_naive(x["q"], x["k"], x["v"], x["do"], 0.09, m.numpy())[:3]
    for name, a, r in zip(("dQ", "dK", "dV"), got, ref):
        assert rel_l2(a, r) <= TOL_BF16_GRAD_RL2, name
    assert np.all(got[0][:, :, 128:256] == 0)


def test_full_size_backward_workload_against_oracle_and_fused(oracle_mod):
    """B=4 H=16 N=4096 d=128: sampled rows against the oracle; whole tensors against
    the fused backward (both evaluate the same gradients)."""
    w = inputs.WORKLOADS["bwd_d128"]
    x, _ = inputs.workload_inputs(w)
    got, (q, k, v, o, do, lse, dm) = _run(x, w.scale)
    fused = [t.float().cpu().numpy() for t in attn.attn_bwd(q, k, v, o, do, lse, w.scale)]
    for a, f in zip(got, fused):
        assert rel_l2(a, f) <= TOL_BF16_GRAD_RL2
    B, H, N, d = w.shape
    r = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, N - 1], r.integers(0, N, 14)])).astype(np.int32)
    gQ, gK, gV = oracle_mod.bwd_rows(x["q"][1, 3], x["k"][1, 3], x["v"][1, 3], x["do"][1, 3], w.scale, rows, rows)
    assert rel_l2(got[0][1, 3][rows], gQ) <= TOL_BF16_GRAD_RL2
    assert rel_l2(got[1][1, 3][rows], gK) <= TOL_BF16_GRAD_RL2
    assert rel_l2(got[2][1, 3][rows], gV) <= TOL_BF16_GRAD_RL2
