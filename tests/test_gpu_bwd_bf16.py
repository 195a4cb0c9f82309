"""bf16 recompute backward (tcgen05) against the oracle, through the C ABI.

Tolerance: relative-L2 <= 2e-2 on dQ, dK and dV (bf16 inputs, fp32
accumulation; the kernel rounds P and dS to bf16 before its products, the oracle
does not).  The kernel's backward takes O and LSE from the kernel's forward; the
oracle recomputes everything from Q, K, V and dO in double."""
import math

import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16_GRAD_RL2, Guarded, rel_l2
from optimal_tiling_gb300 import attn, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _fwd_bwd(x, scale, mask=None, guarded=True):
    B, H, N, d = x["q"].shape
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    dm = mask.to(DEV) if mask is not None else None
    o, lse = attn.attn_fwd(q, k, v, scale, block_mask=dm)
    if guarded:
        g = [Guarded((B, H, N, d), torch.bfloat16, DEV) for _ in range(3)]
        attn.attn_bwd(q, k, v, o, do, lse, scale, block_mask=dm, dq=g[0].t, dk=g[1].t, dv=g[2].t)
        assert attn.attn_device_status() == attn.ATTN_OK
        assert all(x.intact() for x in g), "write outside an output tensor"
        outs = [x.t for x in g]
    else:
        outs = attn.attn_bwd(q, k, v, o, do, lse, scale, block_mask=dm)
        assert attn.attn_device_status() == attn.ATTN_OK
    return [t.float().cpu().numpy() for t in outs]


def _check_full(x, scale, oracle_mod, mask=None):
    dq, dk, dv = _fwd_bwd(x, scale, mask)
    gQ, gK, gV, _, _ = oracle_mod.bwd_naive(x["q"], x["k"], x["v"], x["do"], scale,
                                            None if mask is None else mask.numpy())
    for name, got, ref in (("dQ", dq, gQ), ("dK", dk, gK), ("dV", dv, gV)):
        assert rel_l2(got, ref) <= TOL_BF16_GRAD_RL2, name
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N,BH", [(128, (1, 1)), (256, (1, 3)), (384, (3, 1)), (1024, (1, 2))])
def test_small_shapes(oracle_mod, N, BH, d):
    B, H = BH
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=N + d + 1)
    _check_full(x, 1.0 / math.sqrt(d), oracle_mod)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_block_masks_and_empty_rows(oracle_mod, d):
    N = 768
    x = inputs.make_inputs(1, 2, N, d, torch.bfloat16, seed=21 + d)
    s = 1.0 / math.sqrt(d)
    _check_full(x, s, oracle_mod, inputs.block_diagonal_mask(N))
    _check_full(x, s, oracle_mod, inputs.random_block_mask(N, seed=6, p=0.3))
    m = torch.zeros((6, 6), dtype=torch.uint8)
    m[3, 1] = 1
    m[5, 1] = 1
    m[5, 4] = 1
    dq, dk, dv = _check_full(x, s, oracle_mod, m)
    # rows of query blocks with nothing kept get no gradient; keys never kept get none
    assert np.all(dq[:, :, 0:384] == 0) and np.all(dq[:, :, 512:640] == 0)
    assert np.all(dk[:, :, 0:128] == 0) and np.all(dv[:, :, 256:512] == 0)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_gradient_invariants(d):
    """Rows of P sum to one: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i."""
    N = 1024
    x = inputs.make_inputs(1, 1, N, d, torch.bfloat16, seed=22 + d)
    dq, dk, dv = _fwd_bwd(x, 1.0 / math.sqrt(d))
    dO = x["do"].double().numpy()[0, 0]
    sk = np.abs(dk[0, 0].sum(axis=0))
    assert np.max(sk) <= 2e-2 * np.sqrt(N) * np.sqrt(np.mean(dk ** 2))
    assert np.linalg.norm(dv[0, 0].sum(axis=0) - dO.sum(axis=0)) <= 2e-2 * np.linalg.norm(dO.sum(axis=0))


@pytest.mark.parametrize("d", [128, 256])
def test_deterministic_inputs_repeat(d):
    """Two calls on the same inputs agree to the rounding of fp32 additions
    (the dQ accumulation order between key tiles is not fixed)."""
    x = inputs.make_inputs(1, 2, 512, d, torch.bfloat16, seed=23)
    a = _fwd_bwd(x, 0.09, guarded=False)
    b = _fwd_bwd(x, 0.09, guarded=False)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])   # dK, dV: fixed order
    assert rel_l2(a[0], b[0]) <= 1e-3


def _sample(n, N, seed):
    r = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, N - 1], r.integers(0, N, n - 2)])).astype(np.int32)


@pytest.mark.parametrize("name", ["teaching", "bwd_d128", "sparse_16k", "dense_16k", "dsweep_d256"])
def test_full_size_workloads_sampled(oracle_mod, name):
    """Full-size workloads in the bench's launch configuration; the oracle computes
    sampled gradient rows of the first and the last head: dQ rows (one query row each)
    and dK, dV rows (which need every query row's LSE and D of that head).  On the
    N = 16384 shapes the last head holds tiles of the split last wave (2048 key tiles
    on 152 SMs leave 72 in the last wave), each accumulating 128 query blocks per
    half; the key rows sampled there include the head's last one.  The d-sweep's
    d = 256 shape (2 x 16 x 8192) takes the two-pass backward."""
    w = inputs.WORKLOADS[name]
    x, mask = inputs.workload_inputs(w)
    dq, dk, dv = _fwd_bwd(x, w.scale, mask, guarded=False)
    B, H, N, d = w.shape
    m = None if mask is None else mask.numpy()
    for head in (0, B * H - 1):
        b, h = divmod(head, H)
        qr = _sample(24, N, head)
        kr = _sample(16, N, head + 100)
        gQ, gK, gV = oracle_mod.bwd_rows(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["do"][b, h], w.scale,
                                         qr, kr, m)
        assert rel_l2(dq[b, h][qr], gQ) <= TOL_BF16_GRAD_RL2
        assert rel_l2(dk[b, h][kr], gK) <= TOL_BF16_GRAD_RL2
        assert rel_l2(dv[b, h][kr], gV) <= TOL_BF16_GRAD_RL2
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


@pytest.mark.parametrize("d", [64, 128])
def test_last_wave_split_matches_unsplit(oracle_mod, d):
    """A dense shape whose last wave is split into query halves (the SM count does not
    divide the 128-key tiles and the remainder is at most half the SMs).  With r tiles
    per head and r dividing the SM count, the split tiles are exactly the last head.
    dK and dV of the other heads are bit-identical to the masked path, which never
    splits; the split head, whose two fp32 partials are added in either order, agrees
    to a few bf16 roundings, and with the oracle on sampled rows."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    r = max(t for t in range(1, sms // 4 + 1) if sms % t == 0)
    H, N = sms // r + 1, 128 * r
    s = 1.0 / math.sqrt(d)
    x = inputs.make_inputs(1, H, N, d, torch.bfloat16, seed=31 + d)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = attn.attn_fwd(q, k, v, s)
    lib = attn.load()
    rows = H * N
    base = -(-rows * 8 // 256) * 256 + -(-rows * d * 4 // 256) * 256
    assert lib.attn_bwd_workspace_size(1, H, N, d, attn.ATTN_DTYPE_BF16) == base + r * 2 * 128 * d * 4
    split = attn.attn_bwd(q, k, v, o, do, lse, s)
    ones = torch.ones((r, r), dtype=torch.uint8, device=DEV)
    whole = attn.attn_bwd_masked(q, k, v, o, do, lse, s, ones)
    assert attn.attn_device_status() == attn.ATTN_OK
    dq_s, dk_s, dv_s = (t.float().cpu().numpy()[0] for t in split)
    dq_w, dk_w, dv_w = (t.float().cpu().numpy()[0] for t in whole)
    assert np.array_equal(dk_s[:-1], dk_w[:-1]) and np.array_equal(dv_s[:-1], dv_w[:-1])
    assert rel_l2(dk_s[-1], dk_w[-1]) <= 2e-3 and rel_l2(dv_s[-1], dv_w[-1]) <= 2e-3
    assert rel_l2(dq_s, dq_w) <= 1e-3
    kr = _sample(16, N, 7)
    qr = _sample(8, N, 8)
    gQ, gK, gV = oracle_mod.bwd_rows(x["q"][0, -1], x["k"][0, -1], x["v"][0, -1], x["do"][0, -1], s, qr, kr, None)
    assert rel_l2(dk_s[-1][kr], gK) <= TOL_BF16_GRAD_RL2 and rel_l2(dv_s[-1][kr], gV) <= TOL_BF16_GRAD_RL2
    assert rel_l2(dq_s[-1][qr], gQ) <= TOL_BF16_GRAD_RL2


@pytest.mark.parametrize("d", [64, 128, 256])
def test_negative_scale_forward_and_backward(oracle_mod, d):
    """s < 0 through the whole step: the forward's O and LSE feed the backward, whose
    gradients match the oracle's chain rule for the same negative scale."""
    N = 512
    x = inputs.make_inputs(1, 2, N, d, torch.bfloat16, seed=33)
    _check_full(x, -1.0 / math.sqrt(d), oracle_mod)


def test_side_stream_without_workspace(oracle_mod):
    """A call on a stream other than the current one, with no workspace or outputs given:
    the binding allocates them for that stream, so the caching allocator does not reuse
    their memory while the kernels run.  Results equal the current-stream call's."""
    N, d = 1024, 128
    s = 1.0 / math.sqrt(d)
    x = inputs.make_inputs(1, 2, N, d, torch.bfloat16, seed=34)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    o, lse = attn.attn_fwd(q, k, v, s, stream=side)
    got = attn.attn_bwd(q, k, v, o, do, lse, s, stream=side)
    # allocations on the current stream meanwhile must not land in the side stream's buffers
    junk = [torch.full((1 << 20,), 7.0, device=DEV) for _ in range(8)]
    side.synchronize()
    ref = attn.attn_bwd(q, k, v, o, do, lse, s)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    assert rel_l2(got[0].float().cpu().numpy(), ref[0].float().cpu().numpy()) <= 1e-3
    del junk


def test_masked_with_empty_key_tiles(oracle_mod):
    """A block mask over more 128-key tiles than the GPU has SMs, with whole key-tile columns
    removed: dK and dV of the removed columns are exactly zero (their tiles visit no query
    block), sampled rows of two heads agree with the oracle, and a second call gives the same
    dK and dV."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H, d = 1, 2, 128
    N = 128 * (sms // 2 + 40)  # H * N / 128 tiles > SMs
    nb = N // 128
    s = 1.0 / math.sqrt(d)
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=77)
    mask = inputs.random_block_mask(N, seed=12, p=0.2)
    empty = [3, nb // 2, nb - 1]
    mask[:, empty] = 0
    dm = mask.to(DEV)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = attn.attn_fwd(q, k, v, s, block_mask=dm)
    dq, dk, dv = (t.float().cpu().numpy() for t in attn.attn_bwd(q, k, v, o, do, lse, s, block_mask=dm))
    dq2, dk2, dv2 = (t.float().cpu().numpy() for t in attn.attn_bwd(q, k, v, o, do, lse, s, block_mask=dm))
    assert np.array_equal(dk, dk2) and np.array_equal(dv, dv2)
    for c in empty:
        assert np.all(dk[0, :, 128 * c:128 * (c + 1)] == 0) and np.all(dv[0, :, 128 * c:128 * (c + 1)] == 0)
    m = mask.numpy()
    for h in range(H):
        qr = _sample(16, N, h)
        kr = np.concatenate([_sample(12, N, h + 50), [128 * empty[0] + 5]]).astype(np.int32)
        gQ, gK, gV = oracle_mod.bwd_rows(x["q"][0, h], x["k"][0, h], x["v"][0, h], x["do"][0, h], s, qr, kr, m)
        assert rel_l2(dq[0, h][qr], gQ) <= TOL_BF16_GRAD_RL2
        assert rel_l2(dk[0, h][kr], gK) <= TOL_BF16_GRAD_RL2
        assert rel_l2(dv[0, h][kr], gV) <= TOL_BF16_GRAD_RL2


@pytest.mark.parametrize("d", [64, 128])
def test_persistent_tiles_match_one_cta_per_tile(d):
    """Dense problems run their 128-key tiles in a persistent grid (one CTA per SM, a fixed set
    of tiles each); an all-ones block mask takes the one-CTA-per-tile kernel, which computes
    every tile the same way.  Tile counts equal to the SM count, and above it with an uneven
    share per CTA and no split of the last wave (remainder above half the SMs): dK and dV
    bit-identical, dQ equal up to the order of its fp32 reductions."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s = 1.0 / math.sqrt(d)
    for tiles, N in ((sms, 128), (sms + sms // 2 + 1, 128), (2 * sms + sms // 2 + 3, 256)):
        H = -(-tiles // (N // 128))
        x = inputs.make_inputs(1, H, N, d, torch.bfloat16, seed=tiles + d)
        q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
        o, lse = attn.attn_fwd(q, k, v, s)
        dq1, dk1, dv1 = attn.attn_bwd(q, k, v, o, do, lse, s)
        ones = torch.ones((N // 128, N // 128), dtype=torch.uint8, device=DEV)
        dq2, dk2, dv2 = attn.attn_bwd_masked(q, k, v, o, do, lse, s, ones)
        assert attn.attn_device_status() == attn.ATTN_OK
        assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2), tiles
        assert rel_l2(dq1.float().cpu().numpy(), dq2.float().cpu().numpy()) <= 1e-3


def test_d256_mask_columns_longer_than_the_bit_set(oracle_mod):
    """At d = 256 a key tile's visited query blocks are held as a bit set of up to 1024 64-row
    blocks (N <= 65536); longer mask columns are read entry by entry.  N = 65664 (1026 query
    blocks) with a tridiagonal 128-block mask: sampled dQ, dK and dV rows of the last blocks,
    which only the entry-by-entry walk reaches, against the oracle."""
    N, d = 65664, 256
    s = 1.0 / math.sqrt(d)
    nb = N // 128
    x = inputs.make_inputs(1, 1, N, d, torch.bfloat16, seed=41)
    i = torch.arange(nb)
    mask = ((i[:, None] - i[None, :]).abs() <= 1).to(torch.uint8)
    dq, dk, dv = _fwd_bwd(x, s, mask)
    qr = np.array([0, 5, N // 2, N - 200, N - 65, N - 1], dtype=np.int32)
    kr = np.array([3, N // 2 + 7, N - 300, N - 129, N - 2], dtype=np.int32)
    gQ, gK, gV = oracle_mod.bwd_rows(x["q"][0, 0], x["k"][0, 0], x["v"][0, 0], x["do"][0, 0], s, qr, kr,
                                     mask.numpy())
    assert rel_l2(dq[0, 0][qr], gQ) <= TOL_BF16_GRAD_RL2
    assert rel_l2(dk[0, 0][kr], gK) <= TOL_BF16_GRAD_RL2
    assert rel_l2(dv[0, 0][kr], gV) <= TOL_BF16_GRAD_RL2
