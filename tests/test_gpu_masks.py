"""General block masks (64- or 128-blocks, one shared mask or one per head)
through attn_fwd_masked / attn_bwd_masked, against the oracle's masked forward
and backward, with the tolerances of the unmasked tests.

Masks are drawn with some rows and columns of blocks left empty, so that rows
with no kept score (O = 0, LSE = -inf, zero dQ) and keys that no query sees
(zero dK, dV) occur; with 64-blocks, 128-key blocks that a 128-row query tile
visits with only one key half, or only one row half, kept occur too."""
import math

import numpy as np
import pytest
import torch

from gpu_util import (TOL_BF16_GRAD_RL2, TOL_BF16_LSE_REL, TOL_BF16_O_ABS, TOL_F32_ABS, Guarded, lse_rel,
                      max_abs, rel_l2)
from optimal_tiling_gb300 import attn, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _masks(nh, N, block, seed, p=0.35):
    """[nh, nb, nb] uint8: random blocks plus the diagonal, then one empty block row
    and one empty block column per head (different ones per head)."""
    nb = (N + block - 1) // block
    ms = []
    for h in range(nh):
        m = inputs.random_block_mask(nb * 128, seed=seed + h, p=p)[:nb, :nb].clone()
        m[(h + 1) % nb, :] = 0
        m[:, (2 * h + 3) % nb] = 0
        ms.append(m)
    return torch.stack(ms).contiguous()


def _fwd(x, scale, mask, block, guarded=True):
    B, H, N, d = x["q"].shape
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    dm = mask.to(DEV) if mask is not None else None
    O = Guarded((B, H, N, d), x["q"].dtype, DEV)
    L = Guarded((B, H, N), torch.float32, DEV)
    attn.attn_fwd_masked(q, k, v, scale, mask=dm, block=block, out=O.t, lse=L.t)
    assert attn.attn_device_status() == attn.ATTN_OK
    assert O.intact() and L.intact(), "write outside an output tensor"
    return O.t, L.t


def _bwd(x, scale, mask, block, o, lse):
    B, H, N, d = x["q"].shape
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    dm = mask.to(DEV) if mask is not None else None
    g = [Guarded((B, H, N, d), x["q"].dtype, DEV) for _ in range(3)]
    attn.attn_bwd_masked(q, k, v, o, do, lse, scale, mask=dm, block=block, dq=g[0].t, dk=g[1].t, dv=g[2].t)
    assert attn.attn_device_status() == attn.ATTN_OK
    assert all(t.intact() for t in g), "write outside an output tensor"
    return [t.t.float().cpu().numpy() for t in g]


def _oracle_mask(mask, B, H):
    return None if mask is None else mask.reshape(B * H, mask.shape[-2], mask.shape[-1]).numpy()


@pytest.mark.parametrize("N,block", [(300, 64), (320, 128), (200, 64)])
def test_fp32_per_head_masks(oracle_mod, N, block):
    B, H, d = 2, 2, 64
    x = inputs.make_inputs(B, H, N, d, torch.float32, seed=N + block)
    mask = _masks(B * H, N, block, seed=N).view(B, H, -1, (N + block - 1) // block)
    scale = 1.0 / math.sqrt(d)
    o, lse = _fwd(x, scale, mask, block)
    dq, dk, dv = _bwd(x, scale, mask, block, o, lse)
    om = _oracle_mask(mask, B, H)
    Or, Lr = oracle_mod.fwd_naive_m(x["q"], x["k"], x["v"], scale, om, block)
    gQ, gK, gV = oracle_mod.bwd_naive_m(x["q"], x["k"], x["v"], x["do"], scale, om, block)
    O, L = o.cpu().numpy(), lse.cpu().numpy()
    assert max_abs(O, Or) <= TOL_F32_ABS
    assert np.array_equal(np.isneginf(L), np.isneginf(Lr)) and np.isneginf(Lr).any()
    fin = np.isfinite(Lr)
    assert max_abs(L[fin], Lr[fin]) <= TOL_F32_ABS
    for g, r in ((dq, gQ), (dk, gK), (dv, gV)):
        assert max_abs(g, r) <= TOL_F32_ABS * max(1.0, float(np.max(np.abs(r))))


@pytest.mark.parametrize("N,d,block", [(512, 64, 64), (512, 128, 64), (384, 256, 64), (640, 128, 128)])
def test_bf16_forward_per_head_masks(oracle_mod, N, d, block):
    B, H = 1, 3
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=7 * N + d, with_do=False)
    mask = _masks(B * H, N, block, seed=d + block)
    scale = 1.0 / math.sqrt(d)
    o, lse = _fwd(x, scale, mask, block)
    Or, Lr = oracle_mod.fwd_naive_m(x["q"], x["k"], x["v"], scale, _oracle_mask(mask, B, H), block)
    O, L = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isneginf(Lr).any()
    assert max_abs(O, Or) <= TOL_BF16_O_ABS
    assert lse_rel(L, Lr) <= TOL_BF16_LSE_REL
    assert np.all(O[np.isneginf(Lr)] == 0)


@pytest.mark.parametrize("N,block,d", [(512, 64, 128), (768, 128, 128), (384, 64, 128), (512, 64, 64),
                                       (768, 128, 64), (384, 64, 256), (512, 128, 256)])
def test_bf16_backward_per_head_masks(oracle_mod, N, block, d):
    B, H = 1, 2
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=3 * N + block + d)
    mask = _masks(B * H, N, block, seed=5 * block)
    scale = 1.0 / math.sqrt(d)
    o, lse = _fwd(x, scale, mask, block)
    dq, dk, dv = _bwd(x, scale, mask, block, o, lse)
    om = _oracle_mask(mask, B, H)
    gQ, gK, gV = oracle_mod.bwd_naive_m(x["q"], x["k"], x["v"], x["do"], scale, om, block)
    for name, got, ref in (("dQ", dq, gQ), ("dK", dk, gK), ("dV", dv, gV)):
        assert rel_l2(got, ref) <= TOL_BF16_GRAD_RL2, name
    # removed rows and never-seen keys get exactly zero
    for h in range(H):
        rows = np.repeat(om[h].any(axis=1), block)[:N]
        cols = np.repeat(om[h].any(axis=0), block)[:N]
        assert np.all(dq[0, h][~rows] == 0)
        assert np.all(dk[0, h][~cols] == 0) and np.all(dv[0, h][~cols] == 0)


def test_bf16_backward_fine_masks_many_blocks_d256(oracle_mod):
    """64-row per-head masks on the two-pass d = 256 backward with many query blocks per key tile
    (N = 2048: 32 blocks of 64 rows, 16 key tiles a head), whole tensors against the oracle."""
    B, H, N, d, block = 1, 2, 2048, 256, 64
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=91)
    mask = _masks(B * H, N, block, seed=13)
    scale = 1.0 / math.sqrt(d)
    o, lse = _fwd(x, scale, mask, block)
    dq, dk, dv = _bwd(x, scale, mask, block, o, lse)
    gQ, gK, gV = oracle_mod.bwd_naive_m(x["q"], x["k"], x["v"], x["do"], scale, _oracle_mask(mask, B, H), block)
    for name, got, ref in (("dQ", dq, gQ), ("dK", dk, gK), ("dV", dv, gV)):
        assert rel_l2(got, ref) <= TOL_BF16_GRAD_RL2, name


def _same_grads(g1, g2):
    """dK and dV come out of one CTA each: bit-identical.  dQ is summed over key
    tiles by fp32 reductions whose order is not fixed, so two runs may differ in
    the last bits before the bf16 rounding."""
    dq1, dk1, dv1 = g1
    dq2, dk2, dv2 = g2
    assert np.array_equal(dk1, dk2) and np.array_equal(dv1, dv2)
    assert rel_l2(dq1, dq2) <= 1e-3


@pytest.mark.parametrize("d", [128, 256])
def test_fine_mask_equal_to_coarse_gives_identical_results(d):
    """A 64-block mask that repeats each entry of a 128-block mask 2 x 2 removes the
    same scores: both give bit-identical O, LSE, dK, dV (and dQ up to the order of its
    fp32 reductions).  The 128-block mask is given per head, so that both take the
    kernel with one query tile per CTA (one mask for both heads would pair the heads'
    tiles in one CTA, which rounds differently)."""
    B, H, N = 1, 2, 768
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=31)
    shared = inputs.random_block_mask(N, seed=9, p=0.4)
    coarse = shared.expand(B, H, -1, -1).contiguous()
    fine = shared.repeat_interleave(2, dim=0).repeat_interleave(2, dim=1).contiguous()
    scale = 1.0 / math.sqrt(d)
    o1, l1 = _fwd(x, scale, coarse, 128)
    o2, l2 = _fwd(x, scale, fine, 64)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    _same_grads(_bwd(x, scale, coarse, 128, o1, l1), _bwd(x, scale, fine, 64, o2, l2))


def test_per_head_copies_equal_shared_mask():
    """One mask shared by every head (stride 0) and a copy per head (stride nb*nb) keep
    the same scores.  The forward pairs the heads' query tiles under the shared mask and
    not under the copies: the two agree within the rounding bound, and attn_fwd with the
    same 128-block mask takes the paired kernel too (bit for bit).  The backward takes
    one kernel for both: bit-identical dK, dV from the same O and LSE."""
    B, H, N, d = 2, 2, 512, 128
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=41)
    shared = inputs.random_block_mask(N, seed=4, p=0.5)
    per_head = shared.expand(B, H, -1, -1).contiguous()
    scale = 1.0 / math.sqrt(d)
    o1, l1 = _fwd(x, scale, shared, 128)
    o2, l2 = _fwd(x, scale, per_head, 128)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o3, l3 = attn.attn_fwd(q, k, v, scale, block_mask=shared.to(DEV))
    assert max_abs(o1.float().cpu().numpy(), o2.float().cpu().numpy()) <= TOL_BF16_O_ABS
    assert lse_rel(l1.cpu().numpy(), l2.cpu().numpy()) <= TOL_BF16_LSE_REL
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
    _same_grads(_bwd(x, scale, shared, 128, o1, l1), _bwd(x, scale, per_head, 128, o1, l1))


def test_no_mask_through_masked_entry_points():
    B, H, N, d = 1, 2, 512, 128
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=51)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o1, l1 = attn.attn_fwd(q, k, v, scale)
    o2, l2 = _fwd(x, scale, None, 64)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [128, 256])
def test_all_removed_mask(d):
    """Every block removed: O = 0, LSE = -inf, every gradient zero."""
    B, H, N = 1, 1, 256
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=61)
    mask = torch.zeros((4, 4), dtype=torch.uint8)
    o, lse = _fwd(x, 0.1, mask, 64)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    for g in _bwd(x, 0.1, mask, 64, o, lse):
        assert np.all(g == 0)


@pytest.mark.parametrize("N,H,with_bwd", [(133120, 1, True), (131072, 1, True), (1052672, 1, False),
                                          (1052672, 2, False)])
def test_long_mask_rows(oracle_mod, N, H, with_bwd):
    """Block-diagonal masks on long rows.  The kernels keep the blocks a CTA visits as
    a bit set in shared memory up to 131072 rows (backward) and 1048576 rows
    (forward) and read the mask directly beyond: 133120 and 1052672 take the direct
    path, 131072 the largest bit set; with two heads the forward pairs their query
    tiles.  With only the diagonal kept, every 128-row block is an independent
    problem: sampled blocks are checked against the oracle on that block alone."""
    d, scale = 128, 1.0 / math.sqrt(128)
    x = inputs.make_inputs(1, H, N, d, torch.bfloat16, seed=N % 1000, with_do=with_bwd)
    nb = N // 128
    mask = torch.eye(nb, dtype=torch.uint8)
    o, lse = _fwd(x, scale, mask, 128)
    grads = _bwd(x, scale, mask, 128, o, lse) if with_bwd else None
    for h in range(H):
        O, L = o.float().cpu().numpy()[0, h], lse.cpu().numpy()[0, h]
        for blk in (0, nb // 2 + 1, nb - 1):
            sl = slice(blk * 128, (blk + 1) * 128)
            sub = {k: v[:, h:h + 1, sl] for k, v in x.items()}
            Or, Lr = oracle_mod.fwd_naive(sub["q"], sub["k"], sub["v"], scale)
            assert max_abs(O[sl], Or[0, 0]) <= TOL_BF16_O_ABS
            assert lse_rel(L[sl], Lr[0, 0]) <= TOL_BF16_LSE_REL
            if with_bwd:
                gQ, gK, gV, _, _ = oracle_mod.bwd_naive(sub["q"], sub["k"], sub["v"], sub["do"], scale)
                for g, r in zip(grads, (gQ, gK, gV)):
                    assert rel_l2(g[0, h][sl], r[0, 0]) <= TOL_BF16_GRAD_RL2


def _kept_keys(mask_row, N):
    """Key indices of the kept 64-blocks of one mask row."""
    cols = np.nonzero(np.asarray(mask_row))[0]
    return np.concatenate([np.arange(64 * c, min(64 * c + 64, N)) for c in cols]) if cols.size else np.zeros(0, int)


def test_fine_mask_full_size_sampled(oracle_mod):
    """The 64-row-block workload at full size in the bench's launch configuration (B=1 H=16
    N=16384 d=128, one band-plus-random mask per head): sampled 64-row blocks against the
    oracle's forward of those rows over the keys their mask row keeps (a removed score has
    no weight, so the row's softmax is the one over the kept keys alone)."""
    B, H, N, d = 1, 16, 16384, 128
    scale = 1.0 / math.sqrt(d)
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=0, with_do=False)
    mask = inputs.band_random_mask_fine(N, B * H, seed=0)
    o, lse = _fwd(x, scale, mask, 64, guarded=False)
    O, L = o.float().cpu().numpy()[0], lse.cpu().numpy()[0]
    nb = N // 64
    for h, blk in ((0, 0), (3, 1), (7, 100), (11, 201), (15, nb - 1), (5, nb // 2)):
        keys = _kept_keys(mask[h, blk], N)
        rows = slice(64 * blk, 64 * blk + 64)
        q = x["q"][0, h, rows][None, None]
        kk = torch.from_numpy(keys)
        k, v = x["k"][0, h, kk][None, None], x["v"][0, h, kk][None, None]
        Or, Lr = oracle_mod.fwd_rect(q, k, v, scale)
        assert max_abs(O[h, rows], Or[0, 0]) <= TOL_BF16_O_ABS
        assert lse_rel(L[h, rows], Lr[0, 0]) <= TOL_BF16_LSE_REL


@pytest.mark.parametrize("N", [524288, 532480])
def test_long_fine_mask_rows(oracle_mod, N):
    """64-row blocks on long rows, the diagonal kept: the forward keeps the visited 64-key
    columns as a bit set up to 8192 columns (N = 524288) and reads the mask directly beyond.
    Each 64-row block is an independent problem; sampled blocks against the oracle."""
    d, scale = 128, 1.0 / math.sqrt(128)
    x = inputs.make_inputs(1, 1, N, d, torch.bfloat16, seed=N % 997, with_do=False)
    nb = N // 64
    mask = torch.eye(nb, dtype=torch.uint8)
    o, lse = _fwd(x, scale, mask, 64, guarded=False)
    O, L = o.float().cpu().numpy()[0, 0], lse.cpu().numpy()[0, 0]
    for blk in (0, 1, nb // 2 + 1, nb - 2, nb - 1):
        sl = slice(blk * 64, (blk + 1) * 64)
        sub = {k: v[:, :, sl] for k, v in x.items()}
        Or, Lr = oracle_mod.fwd_naive(sub["q"], sub["k"], sub["v"], scale)
        assert max_abs(O[sl], Or[0, 0]) <= TOL_BF16_O_ABS
        assert lse_rel(L[sl], Lr[0, 0]) <= TOL_BF16_LSE_REL
