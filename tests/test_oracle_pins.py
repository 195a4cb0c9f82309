"""Pins for the CPU oracle: it is checked against facts other than itself.

Each test names the passage or mathematical fact it relies on.  Pages cited:
  [p1] "The I/O Complexity of Attention" exposition (blog.aeilot.top,
       attention-io-complexity);
  [p3] "On Fine-Grained I/O Complexity of Attention Backward Passes" summary
       (gist.science 2410.09397).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from optimal_tiling_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng_global = np.random.default_rng(1234)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _torch_attention(Q, K, V, s, mask=None):
    """Independent evaluation with torch's float64 library softmax/logsumexp."""
    Qt, Kt, Vt = (torch.tensor(x, dtype=torch.float64) for x in (Q, K, V))
    S = s * (Qt @ Kt.transpose(-1, -2))
    if mask is not None:
        N = Q.shape[-2]
        keep = torch.tensor(np.kron(mask, np.ones((128, 128)))[:N, :N] > 0)
        S = S.masked_fill(~keep, float("-inf"))
    P = torch.softmax(S, dim=-1)
    return (P @ Vt).numpy(), torch.logsumexp(S, dim=-1).numpy()


def _torch_attention_block(Q, K, V, s, mask, block):
    Qt, Kt, Vt = (torch.tensor(x, dtype=torch.float64) for x in (Q, K, V))
    N = Q.shape[-2]
    keep = torch.tensor(np.kron(mask, np.ones((block, block)))[:N, :N] > 0)
    S = (s * (Qt @ Kt.transpose(-1, -2))).masked_fill(~keep, float("-inf"))
    return (torch.softmax(S, dim=-1) @ Vt).numpy(), torch.logsumexp(S, dim=-1).numpy()


# --------------------------------------------------------------------------- forward

@pytest.mark.parametrize("N,d", [(7, 3), (130, 16), (300, 8)])
def test_stream_equals_naive_random_blocks(oracle_mod, N, d):
    """[p1] 'Softmax without storing the score matrix': the block-streamed
    online update computes the same function; only rounding differs."""
    Q, K, V = _rand((2, N, d), 1), _rand((2, N, d), 2), _rand((2, N, d), 3)
    O1, L1 = oracle_mod.fwd_naive(Q, K, V, 0.7)
    r = np.random.default_rng(N)
    for trial in range(4):
        cuts = np.sort(r.choice(np.arange(1, N), size=min(N - 1, r.integers(1, 9)), replace=False))
        ends = list(cuts) + [N]
        O2, L2 = oracle_mod.fwd_stream(Q, K, V, 0.7, ends)
        assert np.max(np.abs(O1 - O2)) < 1e-12
        assert np.max(np.abs(L1 - L2)) < 1e-12
    # one key per block and one block for everything
    for ends in (list(range(1, N + 1)), [N]):
        O2, L2 = oracle_mod.fwd_stream(Q, K, V, 0.7, ends)
        assert np.max(np.abs(O1 - O2)) < 1e-12


def test_stream_equals_naive_with_mask(oracle_mod):
    N, d = 384, 4
    Q, K, V = _rand((N, d), 4), _rand((N, d), 5), _rand((N, d), 6)
    mask = inputs.random_block_mask(N, seed=3, p=0.4).numpy()
    O1, L1 = oracle_mod.fwd_naive(Q, K, V, 1.3, mask)
    O2, L2 = oracle_mod.fwd_stream(Q, K, V, 1.3, [50, 128, 129, 300, 384], mask)
    assert np.max(np.abs(O1 - O2)) < 1e-12 and np.max(np.abs(L1 - L2)) < 1e-12


def test_identity_values_give_weights_rows_sum_to_one(oracle_mod):
    """[p1] 'Attention as a mathematical problem': softmax turns each score row into
    weights.  With V = I (d = N) the output rows ARE the weights; they match the
    library softmax and each row sums to 1."""
    N = 24
    Q, K = _rand((N, N), 7) * 2, _rand((N, N), 8)
    O, L = oracle_mod.fwd_naive(Q, K, np.eye(N), 0.3)
    ref = scipy.special.softmax(0.3 * Q @ K.T, axis=1)
    assert np.all(O >= 0)
    assert np.max(np.abs(O.sum(axis=1) - 1.0)) < 1e-12
    assert np.max(np.abs(O - ref)) < 1e-13
    assert np.max(np.abs(L - scipy.special.logsumexp(0.3 * Q @ K.T, axis=1))) < 1e-12


@pytest.mark.parametrize("masked", [False, True])
def test_zero_queries_give_column_mean(oracle_mod, masked):
    """Q = 0 makes every score 0: uniform weights over the kept keys, so
    o_i is the column mean of V over those keys and LSE_i = ln(#kept)."""
    N, d = 256, 5
    K, V = _rand((N, d), 9), _rand((N, d), 10)
    mask = np.array([[1, 0], [1, 1]], dtype=np.uint8) if masked else None
    O, L = oracle_mod.fwd_naive(np.zeros((N, d)), K, V, 2.0, mask)
    if not masked:
        assert np.max(np.abs(O - V.mean(axis=0))) < 1e-13
        assert np.max(np.abs(L - math.log(N))) < 1e-13
    else:
        assert np.max(np.abs(O[:128] - V[:128].mean(axis=0))) < 1e-13
        assert np.max(np.abs(L[:128] - math.log(128))) < 1e-13
        assert np.max(np.abs(O[128:] - V.mean(axis=0))) < 1e-13
        assert np.max(np.abs(L[128:] - math.log(256))) < 1e-13


def test_single_key(oracle_mod):
    """N = 1: the only weight is 1, so O = V and LSE = s q.k."""
    q, k, v = _rand((1, 6), 11), _rand((1, 6), 12), _rand((1, 6), 13)
    O, L = oracle_mod.fwd_naive(q, k, v, 0.9)
    assert np.max(np.abs(O - v)) < 1e-15
    assert abs(L[0] - 0.9 * float(q[0] @ k[0])) < 1e-14


def test_two_keys_logistic(oracle_mod):
    """N = 2: the first weight is the logistic function of the score difference."""
    Q, K, V = _rand((2, 3), 14), _rand((2, 3), 15), _rand((2, 3), 16)
    s = 1.7
    O, L = oracle_mod.fwd_naive(Q, K, V, s)
    for i in range(2):
        a, b = s * Q[i] @ K[0], s * Q[i] @ K[1]
        p0 = 1.0 / (1.0 + math.exp(b - a))
        assert np.max(np.abs(O[i] - (p0 * V[0] + (1 - p0) * V[1]))) < 1e-14
        assert abs(L[i] - (max(a, b) + math.log1p(math.exp(-abs(a - b))))) < 1e-14


def test_golden_two_key_example(oracle_mod):
    """Hand-derived worked example (tests/golden/two_key_example.json)."""
    g = json.load(open(os.path.join(GOLDEN, "two_key_example.json")))
    Q, K, V, dO = (np.array(g[k]) for k in ("Q", "K", "V", "dO"))
    O, L = oracle_mod.fwd_naive(Q, K, V, g["scale"])
    assert np.max(np.abs(O - np.array(g["O"]))) < 1e-14
    assert np.max(np.abs(L - np.array(g["LSE"]))) < 1e-14
    dQ, dK, dV, D, L2 = oracle_mod.bwd_naive(Q, K, V, dO, g["scale"])
    for name, got in (("dQ", dQ), ("dK", dK), ("dV", dV), ("D", D)):
        assert np.max(np.abs(got - np.array(g[name]))) < 1e-14, name


def test_dominant_score_selects_value_row(oracle_mod):
    """A query aligned with one key far more than with the others puts almost all
    weight on that key: |o - v_j*| <= sum_{j != j*} P_j |v_j - v_j*| (closed bound)."""
    N, d = 64, 8
    K, V = _rand((N, d), 17), _rand((N, d), 18)
    K /= np.linalg.norm(K, axis=1, keepdims=True)   # unit keys: k_j*.k_j < 1 for j != j*
    jstar = 37
    Q = _rand((N, d), 19)
    Q[0] = 400.0 * K[jstar]
    O, _ = oracle_mod.fwd_naive(Q, K, V, 1.0)
    S = Q[0] @ K.T
    P = scipy.special.softmax(S)
    bound = sum(P[j] * np.linalg.norm(V[j] - V[jstar]) for j in range(N) if j != jstar)
    assert np.linalg.norm(O[0] - V[jstar]) <= bound + 1e-12
    assert np.linalg.norm(O[0] - V[jstar]) < 1e-6


def test_key_shift_invariance(oracle_mod):
    """Adding one vector c to every key adds s q_i.c to every score of row i:
    the weights do not change, LSE_i grows by s q_i.c."""
    N, d = 50, 6
    Q, K, V = _rand((N, d), 19), _rand((N, d), 20), _rand((N, d), 21)
    c = _rand((d,), 22)
    O1, L1 = oracle_mod.fwd_naive(Q, K, V, 0.6)
    O2, L2 = oracle_mod.fwd_naive(Q, K + c, V, 0.6)
    assert np.max(np.abs(O1 - O2)) < 1e-12
    assert np.max(np.abs(L2 - L1 - 0.6 * Q @ c)) < 1e-12


def test_value_shift_and_permutation(oracle_mod):
    """Weights sum to one, so V + 1 b^T shifts every output row by b; permuting
    key and value rows together leaves the output unchanged."""
    N, d = 40, 5
    Q, K, V = _rand((N, d), 23), _rand((N, d), 24), _rand((N, d), 25)
    b = _rand((d,), 26)
    O1, L1 = oracle_mod.fwd_naive(Q, K, V, 0.8)
    O2, _ = oracle_mod.fwd_naive(Q, K, V + b, 0.8)
    assert np.max(np.abs(O2 - O1 - b)) < 1e-12
    perm = np.random.default_rng(27).permutation(N)
    O3, L3 = oracle_mod.fwd_naive(Q, K[perm], V[perm], 0.8)
    assert np.max(np.abs(O3 - O1)) < 1e-12 and np.max(np.abs(L3 - L1)) < 1e-12


def test_scale_folds_into_queries(oracle_mod):
    """(s, Q) and (1, sQ) give the same scores."""
    N, d = 33, 7
    Q, K, V = _rand((N, d), 28), _rand((N, d), 29), _rand((N, d), 30)
    O1, L1 = oracle_mod.fwd_naive(Q, K, V, 0.37)
    O2, L2 = oracle_mod.fwd_naive(0.37 * Q, K, V, 1.0)
    assert np.max(np.abs(O1 - O2)) < 1e-12 and np.max(np.abs(L1 - L2)) < 1e-12


def test_mask_all_ones_and_block_diagonal(oracle_mod):
    """An all-ones block mask changes nothing; a block-diagonal mask splits the
    sequence into independent 128-row attentions."""
    N, d = 384, 4
    Q, K, V = _rand((N, d), 31), _rand((N, d), 32), _rand((N, d), 33)
    O0, L0 = oracle_mod.fwd_naive(Q, K, V, 0.5)
    O1, L1 = oracle_mod.fwd_naive(Q, K, V, 0.5, np.ones((3, 3), np.uint8))
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)
    Ob, Lb = oracle_mod.fwd_naive(Q, K, V, 0.5, inputs.block_diagonal_mask(N).numpy())
    for t in range(3):
        sl = slice(128 * t, 128 * (t + 1))
        Ot, Lt = oracle_mod.fwd_naive(Q[sl], K[sl], V[sl], 0.5)
        assert np.max(np.abs(Ob[sl] - Ot)) < 1e-13 and np.max(np.abs(Lb[sl] - Lt)) < 1e-13


def test_fully_masked_row(oracle_mod):
    """A query block with no kept key block gets O = 0, LSE = -inf and no gradient."""
    N, d = 256, 3
    Q, K, V, dO = (_rand((N, d), 34 + i) for i in range(4))
    mask = np.array([[0, 0], [1, 1]], dtype=np.uint8)
    O, L = oracle_mod.fwd_naive(Q, K, V, 1.0, mask)
    assert np.all(O[:128] == 0) and np.all(np.isneginf(L[:128]))
    O2, L2 = oracle_mod.fwd_stream(Q, K, V, 1.0, [100, 256], mask)
    assert np.all(O2[:128] == 0) and np.all(np.isneginf(L2[:128]))
    dQ, dK, dV, D, _ = oracle_mod.bwd_naive(Q, K, V, dO, 1.0, mask)
    assert np.all(dQ[:128] == 0)
    # keys only receive gradient from the kept rows 128..255: the same as an
    # unmasked pass whose upstream gradient is zero on rows 0..127
    dO0 = dO.copy()
    dO0[:128] = 0.0
    dQr, dKr, dVr, _, _ = oracle_mod.bwd_naive(Q, K, V, dO0, 1.0)
    assert np.max(np.abs(dK - dKr)) < 1e-12 and np.max(np.abs(dV - dVr)) < 1e-12
    assert np.max(np.abs(dQ[128:] - dQr[128:])) < 1e-12


def test_large_scores_stay_finite(oracle_mod):
    """Scores around 1e3 would overflow e^x without the max; LSE matches the library."""
    N, d = 20, 4
    Q, K, V = 30 * _rand((N, d), 38), 30 * _rand((N, d), 39), _rand((N, d), 40)
    O, L = oracle_mod.fwd_naive(Q, K, V, 1.0)
    assert np.all(np.isfinite(O))
    assert np.max(np.abs(L - scipy.special.logsumexp(Q @ K.T, axis=1))) < 1e-9


@pytest.mark.parametrize("masked", [False, True])
def test_forward_matches_library_evaluation(oracle_mod, masked):
    """Independent evaluation: torch float64 softmax / logsumexp / matmul."""
    N, d = 256, 16
    Q, K, V = _rand((2, N, d), 41), _rand((2, N, d), 42), _rand((2, N, d), 43)
    mask = np.array([[1, 0], [1, 1]], dtype=np.uint8) if masked else None
    O, L = oracle_mod.fwd_naive(Q, K, V, 0.25, mask)
    Or, Lr = _torch_attention(Q, K, V, 0.25, mask)
    assert np.max(np.abs(O - Or)) < 1e-12 and np.max(np.abs(L - Lr)) < 1e-12


def test_fwd_rows_matches_full(oracle_mod):
    N, d = 200, 8
    Q, K, V = _rand((3, N, d), 44), _rand((3, N, d), 45), _rand((3, N, d), 46)
    mask = inputs.random_block_mask(N, seed=5, p=0.5).numpy()
    O, L = oracle_mod.fwd_naive(Q, K, V, 0.4, mask)
    heads, rows = [0, 2, 1, 2], [0, 199, 130, 5]
    Or, Lr = oracle_mod.fwd_rows(Q, K, V, 0.4, heads, rows, mask)
    for n, (h, i) in enumerate(zip(heads, rows)):
        assert np.array_equal(Or[n], O[h, i]) and Lr[n] == L[h, i]


# --------------------------------------------------------------------------- general block masks

def _kron_mask(mask, block, N):
    return np.kron(mask, np.ones((block, block)))[:N, :N] > 0


def test_general_mask_against_library(oracle_mod):
    """64-granular per-head masks: forward and backward equal torch float64
    autograd of softmax attention with the expanded element mask."""
    N, d, s = 256, 8, 0.4
    Q, K, V, dO = (_rand((3, N, d), 300 + i) for i in range(4))
    r = np.random.default_rng(301)
    masks = (r.random((3, 4, 4)) < 0.5).astype(np.uint8)
    masks[:, np.arange(4), np.arange(4)] = 1          # every query row keeps its diagonal block
    O, L = oracle_mod.fwd_naive_m(Q, K, V, s, masks, block=64)
    dQ, dK, dV = oracle_mod.bwd_naive_m(Q, K, V, dO, s, masks, block=64)
    Qt, Kt, Vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    keep = torch.tensor(np.stack([_kron_mask(m, 64, N) for m in masks]))
    S = (s * Qt @ Kt.transpose(-1, -2)).masked_fill(~keep, float("-inf"))
    Ot = torch.softmax(S, dim=-1) @ Vt
    Ot.backward(torch.tensor(dO))
    assert np.max(np.abs(O - Ot.detach().numpy())) < 1e-12
    assert np.max(np.abs(L - torch.logsumexp(S, dim=-1).detach().numpy())) < 1e-12
    for got, t in ((dQ, Qt), (dK, Kt), (dV, Vt)):
        assert np.max(np.abs(got - t.grad.numpy())) < 1e-12


def test_general_mask_special_cases(oracle_mod):
    """A 64-granular refinement of a 128 mask equals the 128 mask; shared masks
    equal per-head copies; a 64-block-diagonal mask splits into 64-row attentions."""
    N, d = 384, 4
    Q, K, V, dO = (_rand((2, N, d), 310 + i) for i in range(4))
    m128 = inputs.random_block_mask(N, seed=11, p=0.5).numpy()
    m64 = np.kron(m128, np.ones((2, 2), np.uint8))
    O1, L1 = oracle_mod.fwd_naive(Q, K, V, 0.7, m128)
    O2, L2 = oracle_mod.fwd_naive_m(Q, K, V, 0.7, m64, block=64)
    O3, L3 = oracle_mod.fwd_naive_m(Q, K, V, 0.7, np.stack([m64, m64]), block=64)
    assert np.max(np.abs(O1 - O2)) < 1e-13 and np.max(np.abs(O1 - O3)) < 1e-13
    assert np.array_equal(np.isneginf(L1), np.isneginf(L2))
    g1 = oracle_mod.bwd_naive(Q, K, V, dO, 0.7, m128)[:3]
    g2 = oracle_mod.bwd_naive_m(Q, K, V, dO, 0.7, m64, block=64)
    for a, b in zip(g1, g2):
        assert np.max(np.abs(a - b)) < 1e-12
    eye = np.eye(N // 64, dtype=np.uint8)
    Ob, Lb = oracle_mod.fwd_naive_m(Q, K, V, 0.7, eye, block=64)
    for t in range(N // 64):
        sl = slice(64 * t, 64 * (t + 1))
        Ot, Lt = oracle_mod.fwd_naive(Q[:, sl], K[:, sl], V[:, sl], 0.7)
        assert np.max(np.abs(Ob[:, sl] - Ot)) < 1e-13 and np.max(np.abs(Lb[:, sl] - Lt)) < 1e-13


# --------------------------------------------------------------------------- rectangular (decode)

def test_rect_matches_library_and_square_rows(oracle_mod):
    """Nq queries against Nk keys: equals the library evaluation, and each query
    row equals the same row of a square problem that shares the keys."""
    Nq, Nk, d = 5, 300, 16
    Q, K, V = _rand((2, Nq, d), 90), _rand((2, Nk, d), 91), _rand((2, Nk, d), 92)
    O, L = oracle_mod.fwd_rect(Q, K, V, 0.3)
    Or, Lr = _torch_attention(Q, K, V, 0.3)
    assert np.max(np.abs(O - Or)) < 1e-12 and np.max(np.abs(L - Lr)) < 1e-12
    Qsq = _rand((2, Nk, d), 93)
    Qsq[:, 17:17 + Nq] = Q
    Osq, Lsq = oracle_mod.fwd_naive(Qsq, K, V, 0.3)
    assert np.max(np.abs(O - Osq[:, 17:17 + Nq])) < 1e-13 and np.max(np.abs(L - Lsq[:, 17:17 + Nq])) < 1e-13


def test_rect_single_key_and_zero_query(oracle_mod):
    """Nk = 1 gives O = v and LSE = s q.k; q = 0 gives the column mean and ln Nk."""
    q, k, v = _rand((3, 2, 6), 94), _rand((3, 1, 6), 95), _rand((3, 1, 6), 96)
    O, L = oracle_mod.fwd_rect(q, k, v, 0.7)
    assert np.max(np.abs(O - v)) < 1e-15
    assert np.max(np.abs(L - 0.7 * np.einsum("hqd,hkd->hq", q, k))) < 1e-14
    K, V = _rand((1, 77, 4), 97), _rand((1, 77, 4), 98)
    O, L = oracle_mod.fwd_rect(np.zeros((1, 3, 4)), K, V, 1.0)
    assert np.max(np.abs(O - V.mean(axis=1, keepdims=True))) < 1e-14
    assert np.max(np.abs(L - math.log(77))) < 1e-14


# --------------------------------------------------------------------------- backward

def _loss(oracle_mod, Q, K, V, G, s, mask):
    O, _ = oracle_mod.fwd_naive(Q, K, V, s, mask)
    return float(np.sum(O * G))


@pytest.mark.parametrize("N,d,masked", [(5, 3, False), (8, 4, False), (2, 2, False), (6, 4, True)])
def test_backward_finite_differences(oracle_mod, N, d, masked):
    """[p3] backward pass of the same attention: gradients of L = sum(O o G)
    against central finite differences (h = 1e-6) of the forward oracle."""
    r = np.random.default_rng(N * 10 + d)
    Q, K, V, G = (r.standard_normal((N, d)) for _ in range(4))
    s = 0.8
    mask = None
    if masked:
        # N < 128 puts every entry in block (0, 0); a zero mask there removes all
        # scores, so check the kept case here and the removed case elsewhere.
        mask = np.ones((1, 1), np.uint8)
    dQ, dK, dV, _, _ = oracle_mod.bwd_naive(Q, K, V, G, s, mask)
    h = 1e-6
    for name, X, dX in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"Q": Q, "K": K, "V": V}
            args_m = {"Q": Q, "K": K, "V": V}
            args_p[name], args_m[name] = Xp, Xm
            num[idx] = (_loss(oracle_mod, args_p["Q"], args_p["K"], args_p["V"], G, s, mask)
                        - _loss(oracle_mod, args_m["Q"], args_m["K"], args_m["V"], G, s, mask)) / (2 * h)
        assert np.max(np.abs(num - dX)) < 1e-8, name


def test_backward_matches_library_autograd(oracle_mod):
    """Independent evaluation: torch float64 autograd of softmax attention."""
    N, d = 256, 8
    Q, K, V, dO = (_rand((2, N, d), 50 + i) for i in range(4))
    mask = np.array([[1, 0], [1, 1]], dtype=np.uint8)
    s = 0.35
    dQ, dK, dV, D, L = oracle_mod.bwd_naive(Q, K, V, dO, s, mask)
    Qt, Kt, Vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    S = s * (Qt @ Kt.transpose(-1, -2))
    keep = torch.tensor(np.kron(mask, np.ones((128, 128))) > 0)
    P = torch.softmax(S.masked_fill(~keep, float("-inf")), dim=-1)
    (P @ Vt).backward(torch.tensor(dO))
    for got, t in ((dQ, Qt), (dK, Kt), (dV, Vt)):
        assert np.max(np.abs(got - t.grad.numpy())) < 1e-12


def test_backward_invariants(oracle_mod):
    """Each weight row sums to one, so: sum_j dK_j = 0 (the scores of a row are
    shift-invariant in the keys), sum_j dV_j = sum_i dO_i, and
    D_i = sum_j P_ij dP_ij equals dO_i . o_i."""
    N, d = 300, 6
    Q, K, V, dO = (_rand((N, d), 60 + i) for i in range(4))
    dQ, dK, dV, D, L = oracle_mod.bwd_naive(Q, K, V, dO, 0.5)
    O, L2 = oracle_mod.fwd_naive(Q, K, V, 0.5)
    assert np.max(np.abs(dK.sum(axis=0))) < 1e-11
    assert np.max(np.abs(dV.sum(axis=0) - dO.sum(axis=0))) < 1e-11
    assert np.max(np.abs(D - np.sum(dO * O, axis=1))) < 1e-12
    assert np.max(np.abs(L - L2)) < 1e-12


def test_bwd_rows_matches_full(oracle_mod):
    N, d = 260, 5
    Q, K, V, dO = (_rand((N, d), 70 + i) for i in range(4))
    mask = inputs.random_block_mask(N, seed=9, p=0.5).numpy()
    dQ, dK, dV, _, _ = oracle_mod.bwd_naive(Q, K, V, dO, 0.45, mask)
    qr, kr = [0, 259, 131], [3, 200, 259, 128]
    a, b, c = oracle_mod.bwd_rows(Q, K, V, dO, 0.45, qr, kr, mask)
    assert np.max(np.abs(a - dQ[qr])) < 1e-13
    assert np.max(np.abs(b - dK[kr])) < 1e-13
    assert np.max(np.abs(c - dV[kr])) < 1e-13


# --------------------------------------------------------------------------- planted mistakes

# (description, exact text in the oracle source, planted replacement)
MUTATIONS = [
    ("scale dropped from the scores",
     "srow[j] = s * dot(Q + (size_t)i * d, K + (size_t)j * d, d);",
     "srow[j] = dot(Q + (size_t)i * d, K + (size_t)j * d, d);"),
    ("query and key indices swapped",
     "srow[j] = s * dot(Q + (size_t)i * d, K + (size_t)j * d, d);",
     "srow[j] = s * dot(Q + (size_t)j * d, K + (size_t)i * d, d);"),
    ("weights not normalised",
     "double p = exp(srow[j] - L);",
     "double p = exp(srow[j] - mx);"),
    ("online rescale of l dropped",
     "l *= alpha;",
     ";"),
    ("sign of D flipped in dS",
     "double dS = prow[j] * (dprow[j] - D);",
     "double dS = prow[j] * (dprow[j] + D);"),
    ("scale dropped from dK",
     "dk[t] += s * dS * qi[t];",
     "dk[t] += dS * qi[t];"),
    ("dV takes dS instead of P",
     "dv[t] += P * doi[t];",
     "dv[t] += dS * doi[t];"),
    ("general mask: row and column block swapped",
     "return mv->mask[(size_t)(i / mv->block) * mv->nb + (j / mv->block)] != 0;",
     "return mv->mask[(size_t)(j / mv->block) * mv->nb + (i / mv->block)] != 0;"),
    ("rectangular: scale dropped",
     "srow[j] = s * dot(q, Kh + (size_t)j * d, d);",
     "srow[j] = dot(q, Kh + (size_t)j * d, d);"),
    ("rectangular: weights not normalised",
     "double p = exp(srow[j] - L);\n                    const double *vj = Vh",
     "double p = exp(srow[j] - mx);\n                    const double *vj = Vh"),
]


def _pins_pass(oracle_mod, handle) -> bool:
    """The library comparisons and the streaming identity, run against one build."""
    N, d = 130, 4
    Q, K, V, dO = (_rand((N, d), 80 + i) for i in range(4))
    s = 0.6
    O, L = oracle_mod.fwd_naive(Q, K, V, s, _oracle=handle)
    Or, Lr = _torch_attention(Q, K, V, s)
    if not (np.max(np.abs(O - Or)) < 1e-12 and np.max(np.abs(L - Lr)) < 1e-12):
        return False
    O2, L2 = oracle_mod.fwd_stream(Q, K, V, s, [17, 64, 130], _oracle=handle)
    if not (np.max(np.abs(O - O2)) < 1e-12):
        return False
    Qr, Kr, Vr = _rand((3, d), 88), _rand((N, d), 86), _rand((N, d), 87)
    Orr, Lrr = oracle_mod.fwd_rect(Qr[None], Kr[None], Vr[None], s, _oracle=handle)
    Ort, Lrt = _torch_attention(Qr, Kr, Vr, s)
    if not (np.max(np.abs(Orr[0] - Ort)) < 1e-12 and np.max(np.abs(Lrr[0] - Lrt)) < 1e-12):
        return False
    mg = np.array([[1, 0, 0], [1, 1, 0], [1, 1, 1]], dtype=np.uint8)   # not symmetric
    Om, _ = oracle_mod.fwd_naive_m(_rand((192, 4), 89), _rand((192, 4), 90), _rand((192, 4), 91), s, mg,
                                   block=64, _oracle=handle)
    Omr, _ = _torch_attention_block(_rand((192, 4), 89), _rand((192, 4), 90), _rand((192, 4), 91), s, mg, 64)
    if not np.max(np.abs(Om - Omr)) < 1e-12:
        return False
    dQ, dK, dV, _, _ = oracle_mod.bwd_naive(Q, K, V, dO, s, _oracle=handle)
    Qt, Kt, Vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    (torch.softmax(s * Qt @ Kt.T, dim=-1) @ Vt).backward(torch.tensor(dO))
    return all(np.max(np.abs(a - t.grad.numpy())) < 1e-12 for a, t in ((dQ, Qt), (dK, Kt), (dV, Vt)))


def test_pins_reject_planted_mistakes(oracle_mod, tmp_path):
    """Plant each plausible mistake in a copy of the oracle source, build it on the
    CPU, and check that the pins above reject it (while the real oracle passes)."""
    assert _pins_pass(oracle_mod, None)
    src = open(oracle_mod.SOURCE_PATH).read()
    for n, (what, old, new) in enumerate(MUTATIONS):
        assert src.count(old) >= 1, f"mutation site missing: {what}"
        c = tmp_path / f"mut{n}.c"
        c.write_text(src.replace(old, new, 1))
        so = oracle_mod.compile_source(str(c), str(tmp_path / f"libmut{n}.so"))
        assert not _pins_pass(oracle_mod, oracle_mod.Oracle(so)), f"pins missed: {what}"
