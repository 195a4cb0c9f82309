"""The largest head count the ABI takes (B * H = 65535, one grid row per head) through the bf16
kernels, against the oracle on sampled heads.

Every kernel indexes heads by its grid's y coordinate, whose limit this is; the rows of the last
heads sit furthest into every array.  N = 64 with d = 64 takes the partial-tile kernels (128 does
not divide N), N = 128 with d = 256 the full-tile forward and the two-pass backward; the
materialising schedules and decode are checked at the same head count.  The inputs (seeded) are
drawn on the device: 65535 heads are slow to draw on the host."""
import math

import pytest
import torch

from gpu_util import TOL_BF16_GRAD_RL2, TOL_BF16_LSE_REL, TOL_BF16_O_ABS, lse_rel, max_abs, rel_l2
from optimal_tiling_gb300 import attn

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.mark.parametrize("N,d", [(64, 64), (128, 256)])
def test_most_heads(oracle_mod, N, d):
    BH = 65535
    g = torch.Generator(device=DEV)
    g.manual_seed(N + d)
    q, k, v, do = (torch.randn((1, BH, N, d), generator=g, device=DEV).to(torch.bfloat16) for _ in range(4))
    s = 1.0 / math.sqrt(d)
    o, lse = attn.attn_fwd(q, k, v, s)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, do, lse, s)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    for h in (0, 1, BH // 2, BH - 2, BH - 1):
        x = {n: t[:, h:h + 1].cpu() for n, t in (("q", q), ("k", k), ("v", v), ("do", do))}
        Or, Lr = oracle_mod.fwd_naive(x["q"], x["k"], x["v"], s)
        assert max_abs(o[:, h:h + 1].float().cpu().numpy(), Or) <= TOL_BF16_O_ABS, h
        assert lse_rel(lse[:, h:h + 1].cpu().numpy(), Lr) <= TOL_BF16_LSE_REL, h
        gQ, gK, gV, _, _ = oracle_mod.bwd_naive(x["q"], x["k"], x["v"], x["do"], s)
        for name, got, ref in (("dQ", dq, gQ), ("dK", dk, gK), ("dV", dv, gV)):
            assert rel_l2(got[:, h:h + 1].float().cpu().numpy(), ref) <= TOL_BF16_GRAD_RL2, (name, h)
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t).all()
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


def test_most_heads_materialised_and_decode(oracle_mod):
    """The materialising forward and backward (N = 128, d = 64) and decode (one query against
    256 keys, d = 128) at B * H = 65535, on sampled heads against the oracle."""
    BH, N, d = 65535, 128, 64
    g = torch.Generator(device=DEV)
    g.manual_seed(7)
    q, k, v, do = (torch.randn((1, BH, N, d), generator=g, device=DEV).to(torch.bfloat16) for _ in range(4))
    s = 1.0 / math.sqrt(d)
    o, lse = attn.attn_fwd_materialized(q, k, v, s)
    dq, dk, dv = attn.attn_bwd_materialized(q, k, v, o, do, lse, s)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    for h in (0, BH // 2, BH - 1):
        x = {n: t[:, h:h + 1].cpu() for n, t in (("q", q), ("k", k), ("v", v), ("do", do))}
        Or, Lr = oracle_mod.fwd_naive(x["q"], x["k"], x["v"], s)
        assert max_abs(o[:, h:h + 1].float().cpu().numpy(), Or) <= TOL_BF16_O_ABS, h
        assert lse_rel(lse[:, h:h + 1].cpu().numpy(), Lr) <= TOL_BF16_LSE_REL, h
        gQ, gK, gV, _, _ = oracle_mod.bwd_naive(x["q"], x["k"], x["v"], x["do"], s)
        for name, got, ref in (("dQ", dq, gQ), ("dK", dk, gK), ("dV", dv, gV)):
            assert rel_l2(got[:, h:h + 1].float().cpu().numpy(), ref) <= TOL_BF16_GRAD_RL2, (name, h)
    del q, k, v, do, o, lse, dq, dk, dv
    Nk, dd = 256, 128
    qd = torch.randn((1, BH, 1, dd), generator=g, device=DEV).to(torch.bfloat16)
    kd, vd = (torch.randn((1, BH, Nk, dd), generator=g, device=DEV).to(torch.bfloat16) for _ in range(2))
    sd = 1.0 / math.sqrt(dd)
    od, ld = attn.attn_decode(qd, kd, vd, sd)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    for h in (0, BH // 2, BH - 1):
        Or, Lr = oracle_mod.fwd_rect(qd[:, h:h + 1].cpu(), kd[:, h:h + 1].cpu(), vd[:, h:h + 1].cpu(), sd)
        assert max_abs(od[:, h:h + 1].float().cpu().numpy(), Or) <= TOL_BF16_O_ABS, h
        assert lse_rel(ld[:, h:h + 1].cpu().numpy(), Lr) <= TOL_BF16_LSE_REL, h
    torch.cuda.empty_cache()
