"""Decode-shaped attention (Nq <= 16 queries against Nk keys) against the
rectangular oracle, through the C ABI.  Tolerances as the bf16 forward:
O max-abs <= 1e-2, LSE relative <= 1e-3."""
import math

import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16_LSE_REL, TOL_BF16_O_ABS, Guarded, lse_rel, max_abs
from optimal_tiling_gb300 import attn, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _decode(x, scale):
    B, H, Nq, d = x["q"].shape
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    O = Guarded((B, H, Nq, d), torch.bfloat16, DEV)
    L = Guarded((B, H, Nq), torch.float32, DEV)
    attn.attn_decode(q, k, v, scale, out=O.t, lse=L.t)
    assert attn.attn_device_status() == attn.ATTN_OK
    assert O.intact() and L.intact(), "write outside an output tensor"
    return O.t.float().cpu().numpy(), L.t.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 31), (3, 200), (8, 4096), (16, 1000), (5, 129)])
def test_shapes_against_oracle(oracle_mod, d, Nq, Nk):
    x = inputs.make_decode_inputs(2, 3, Nq, Nk, d, seed=Nq * 1000 + Nk + d)
    s = 1.0 / math.sqrt(d)
    O, L = _decode(x, s)
    Or, Lr = oracle_mod.fwd_rect(x["q"], x["k"], x["v"], s)
    assert max_abs(O, Or) <= TOL_BF16_O_ABS
    assert lse_rel(L, Lr) <= TOL_BF16_LSE_REL


def test_matches_rows_of_the_fused_forward():
    """A query row of a square problem against the same keys: the decode path
    and the fused forward evaluate the same function."""
    N, d = 1024, 128
    x = inputs.make_inputs(1, 2, N, d, torch.bfloat16, seed=5, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    of, lf = attn.attn_fwd(q, k, v, 0.1)
    rows = [0, 3, 511, 1023]
    od, ld = attn.attn_decode(q[:, :, rows].contiguous(), k, v, 0.1)
    assert float((od.float() - of[:, :, rows].float()).abs().max()) <= TOL_BF16_O_ABS
    assert float(((ld - lf[:, :, rows]).abs() / lf[:, :, rows].abs()).max()) <= TOL_BF16_LSE_REL


def test_decode_workload_sampled(oracle_mod):
    """B=8 H=32, one query against 32768 keys: sampled heads against the oracle."""
    w = inputs.DECODE_WORKLOAD
    x = inputs.make_decode_inputs(w["B"], w["H"], w["Nq"], w["Nk"], w["d"], seed=0)
    s = 1.0 / math.sqrt(w["d"])
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, l = attn.attn_decode(q, k, v, s)
    assert attn.attn_device_status() == attn.ATTN_OK
    for b, h in ((0, 0), (7, 31), (3, 17)):
        Or, Lr = oracle_mod.fwd_rect(x["q"][b, h], x["k"][b, h], x["v"][b, h], s)
        assert max_abs(o[b, h].float().cpu().numpy(), Or) <= TOL_BF16_O_ABS
        assert lse_rel(l[b, h].cpu().numpy(), Lr) <= TOL_BF16_LSE_REL
