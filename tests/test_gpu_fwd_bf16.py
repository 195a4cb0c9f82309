"""bf16 fused forward (tcgen05) against the oracle, through the C ABI.

Tolerances: O max-abs <= 1e-2, LSE relative <= 1e-3 (bf16 inputs, fp32
accumulation; the kernel rounds P to bf16 before the second product, the oracle
does not).  Inputs are the exact bf16 values handed to the GPU, widened to
double for the oracle."""
import math

import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16_LSE_REL, TOL_BF16_O_ABS, Guarded, lse_rel, max_abs
from optimal_tiling_gb300 import attn, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _fwd(x, scale, mask=None, guarded=True):
    B, H, N, d = x["q"].shape
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    dm = mask.to(DEV) if mask is not None else None
    if guarded:
        O = Guarded((B, H, N, d), torch.bfloat16, DEV)
        L = Guarded((B, H, N), torch.float32, DEV)
        attn.attn_fwd(q, k, v, scale, block_mask=dm, out=O.t, lse=L.t)
        assert attn.attn_device_status() == attn.ATTN_OK
        assert O.intact() and L.intact(), "write outside an output tensor"
        return O.t.float().cpu().numpy(), L.t.cpu().numpy()
    o, l = attn.attn_fwd(q, k, v, scale, block_mask=dm)
    assert attn.attn_device_status() == attn.ATTN_OK
    return o.float().cpu().numpy(), l.cpu().numpy()


def _check_full(x, scale, oracle_mod, mask=None, o_scale=False):
    """o_scale: outside the target workloads |O| can exceed 1, where bf16's own
    output rounding (relative 2^-9) plus the rounding of P (relative 2^-9 per
    weight) approach 1e-2; those stress cases scale the bound by max(1, |O|)."""
    O, L = _fwd(x, scale, mask)
    Or, Lr = oracle_mod.fwd_naive(x["q"], x["k"], x["v"], scale, None if mask is None else mask.numpy())
    tol = TOL_BF16_O_ABS * (max(1.0, float(np.max(np.abs(Or)))) if o_scale else 1.0)
    assert max_abs(O, Or) <= tol
    assert lse_rel(L, Lr) <= TOL_BF16_LSE_REL
    return O, L


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N,BH", [(128, (1, 1)), (256, (1, 3)), (384, (3, 1))])
def test_small_shapes(oracle_mod, d, N, BH):
    B, H = BH
    x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=N + d, with_do=False)
    _check_full(x, 1.0 / math.sqrt(d), oracle_mod)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_many_key_blocks_and_large_scale(oracle_mod, d):
    """Sixteen key blocks and a large score scale: the running max moves often,
    which exercises the conditional O rescale."""
    x = inputs.make_inputs(1, 2, 2048, d, torch.bfloat16, seed=7, with_do=False)
    _check_full(x, 2.0 / math.sqrt(d), oracle_mod, o_scale=True)


@pytest.mark.parametrize("d", [64, 128])
def test_all_ones_mask_matches_no_mask(oracle_mod, d):
    """An all-ones mask removes nothing.  Without a mask (N % 256 == 0) two query tiles
    of one head share a CTA; with one 128-block mask for both heads, the same query tile
    of the two heads shares one; with 64-blocks, each tile has a CTA of its own.  The
    three differ only in rounding: each against the oracle, and against each other
    within the same bound.  A 64-block mask and a per-head copy of the 128-block mask
    keep the same scores and take the same kernel: they agree bit for bit."""
    x = inputs.make_inputs(1, 2, 512, d, torch.bfloat16, seed=11 + d, with_do=False)
    O1, L1 = _check_full(x, 0.1, oracle_mod)
    ones = torch.ones((4, 4), dtype=torch.uint8)
    O2, L2 = _check_full(x, 0.1, oracle_mod, ones)
    assert max_abs(O1, O2) <= TOL_BF16_O_ABS and lse_rel(L1, L2) <= TOL_BF16_LSE_REL
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o3, l3 = attn.attn_fwd_masked(q, k, v, 0.1, mask=torch.ones((8, 8), dtype=torch.uint8, device=DEV), block=64)
    O3, L3 = o3.float().cpu().numpy(), l3.cpu().numpy()
    assert max_abs(O2, O3) <= TOL_BF16_O_ABS and lse_rel(L2, L3) <= TOL_BF16_LSE_REL
    o4, l4 = attn.attn_fwd_masked(q, k, v, 0.1, mask=torch.ones((1, 2, 4, 4), dtype=torch.uint8, device=DEV),
                                  block=128)
    assert np.array_equal(O3, o4.float().cpu().numpy()) and np.array_equal(L3, l4.cpu().numpy())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("blocks", [1, 2, 3, 5])
def test_few_visited_key_blocks(oracle_mod, d, blocks):
    """Query tiles that visit 1, 2, 3 or 5 key blocks under a mask, so that the double
    buffered S and the K/V ring run with fewer blocks than buffers and stages."""
    N = 128 * 6
    x = inputs.make_inputs(1, 2, N, d, torch.bfloat16, seed=100 + blocks + d, with_do=False)
    m = torch.zeros((6, 6), dtype=torch.uint8)
    for i in range(6):
        for t in range(blocks):
            m[i, (i + t) % 6] = 1
    _check_full(x, 1.0 / math.sqrt(d), oracle_mod, m)


@pytest.mark.parametrize("BH", [(2, 1), (1, 3)])
@pytest.mark.parametrize("d", [64, 128])
def test_block_masks(oracle_mod, d, BH):
    """One mask for every head: with an even number of heads the same query tile of two
    heads shares a CTA, with an odd number each tile has its own.  Block-diagonal, random,
    and a single kept block (every other query tile visits nothing: O = 0, LSE = -inf)."""
    N = 768
    x = inputs.make_inputs(*BH, N, d, torch.bfloat16, seed=12, with_do=False)
    s = 1.0 / math.sqrt(d)
    _check_full(x, s, oracle_mod, inputs.block_diagonal_mask(N))
    _check_full(x, s, oracle_mod, inputs.random_block_mask(N, seed=4, p=0.3))
    single = torch.zeros((6, 6), dtype=torch.uint8)
    single[3, 1] = 1
    O, L = _check_full(x, s, oracle_mod, single)
    rows = np.r_[0:384, 512:768]
    assert np.all(O[:, :, rows] == 0) and np.all(np.isneginf(L[:, :, rows]))


def test_zero_queries_give_column_mean():
    """Q = 0: O is the column mean of V over the kept keys, LSE = ln(#kept)."""
    N, d = 512, 128
    x = inputs.make_inputs(1, 1, N, d, torch.bfloat16, seed=13, with_do=False)
    x["q"] = torch.zeros_like(x["q"])
    mask = torch.tensor([[1, 0, 0, 0], [1, 1, 0, 0], [1, 1, 1, 0], [1, 1, 1, 1]], dtype=torch.uint8)
    O, L = _fwd(x, 0.3, mask)
    V = x["v"].double().numpy()[0, 0]
    for bi in range(4):
        kept = (bi + 1) * 128
        rows = slice(128 * bi, 128 * (bi + 1))
        assert np.max(np.abs(O[0, 0, rows] - V[:kept].mean(axis=0))) <= TOL_BF16_O_ABS
        assert np.max(np.abs(L[0, 0, rows] - math.log(kept))) <= 1e-3 * math.log(kept)


def test_dominant_score_selects_value_row():
    N, d = 256, 64
    x = inputs.make_inputs(1, 1, N, d, torch.bfloat16, seed=14, with_do=False)
    k = x["k"][0, 0].float()
    k = k / k.norm(dim=1, keepdim=True) * 4.0
    x["k"] = k.to(torch.bfloat16).view(1, 1, N, d)
    jstar = torch.arange(N) * 7 % N        # query i aligned with key jstar[i]
    x["q"] = (x["k"][0, 0, jstar].float() * 8.0).to(torch.bfloat16).view(1, 1, N, d)
    O, _ = _fwd(x, 1.0)
    V = x["v"].float().numpy()[0, 0]
    assert np.max(np.abs(O[0, 0] - V[jstar.numpy()])) <= TOL_BF16_O_ABS


# ----------------------------------------------------------------- full-size workloads

def _sampled_rows(B, H, N, n, seed):
    r = np.random.default_rng(seed)
    heads = np.concatenate([[0, B * H - 1], r.integers(0, B * H, n - 2)])
    rows = np.concatenate([[0, N - 1], r.integers(0, N, n - 2)])
    return heads.astype(np.int32), rows.astype(np.int32)


@pytest.mark.parametrize("name", ["teaching", "dsweep_d64", "dsweep_d128", "dsweep_d256", "sparse_16k",
                                  "dense_16k"])
def test_full_size_workloads_sampled(oracle_mod, name):
    """Full-size workloads in the bench's launch configuration; the oracle
    checks sampled rows one by one (first and last row of the tensor included)."""
    w = inputs.WORKLOADS[name]
    x, mask = inputs.workload_inputs(w, with_do=False)
    O, L = _fwd(x, w.scale, mask, guarded=False)
    B, H, N, d = w.shape
    heads, rows = _sampled_rows(B, H, N, 48, seed=len(name))
    Or, Lr = oracle_mod.fwd_rows(x["q"], x["k"], x["v"], w.scale, heads, rows,
                                 None if mask is None else mask.numpy())
    Of = O.reshape(B * H, N, d)[heads, rows]
    Lf = L.reshape(B * H, N)[heads, rows]
    assert max_abs(Of, Or) <= TOL_BF16_O_ABS
    assert lse_rel(Lf, Lr) <= TOL_BF16_LSE_REL
    assert np.all(np.isfinite(O))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_negative_scale(oracle_mod, d):
    """A negative score scale (the softmax of the first page's definition takes any real
    scores): the two-tile kernel (no mask, N % 256 == 0), the single-tile kernel (N = 384,
    and under a block mask with an odd number of heads), the head-pair kernel (one block
    mask, two heads) against the oracle; and s Q K^T = |s| (-Q) K^T exactly, so the call
    with -s equals the call with -Q and +s bit for bit."""
    s = -1.0 / math.sqrt(d)
    m = inputs.random_block_mask(512, seed=3, p=0.5)
    for N, H, mask in ((512, 2, None), (384, 2, None), (512, 2, m), (512, 3, m)):
        x = inputs.make_inputs(1, H, N, d, torch.bfloat16, seed=N + d + H, with_do=False)
        O, L = _check_full(x, s, oracle_mod, mask)
        flipped = dict(x, q=-x["q"])
        O2, L2 = _fwd(flipped, -s, mask)
        assert np.array_equal(O, O2) and np.array_equal(L, L2)
