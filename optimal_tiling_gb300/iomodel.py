"""The pages' two-level memory model, evaluated for reporting.

Sources (all in element counts unless a name says bytes):

* "The I/O Complexity of Attention" exposition (blog.aeilot.top,
  attention-io-complexity):
  - "Attention as a mathematical problem": the two products cost about 4 N^2 d
    FLOPs (multiply and add counted separately);
  - "Two memory levels": fast memory holds M elements; C bytes of w-byte
    elements give M = C / w, and L elements moved are w L bytes;
  - "Large caches": query blocks of B = Theta(M / d) rows, leading movement
    term N^2 d^2 / M, regime M >= d^2;
  - "Small caches": square tiles of side b = Theta(sqrt M), leading term
    N^2 d / sqrt(M), regime M < d^2;
  - "Putting the regimes together" (Theorem 3.1): min(N^2 d^2 / M, N^2 d / sqrt M),
    read with the compulsory input/output term N d added;
  - "From a movement lower bound to a performance upper bound":
    T >= max(w L / beta, F / P).
* "On Fine-Grained I/O Complexity of Attention Backward Passes" summary
  (gist.science 2410.09397): Theorem 1.1, min((n^2 d^2 + n d^3)/M,
  (n^2 d + n d^2)/sqrt M); Theorem 4.5, sparse bound
  min(Z_in^2 / M, Z_in sqrt(Z_QK) / sqrt M).

These are asymptotic leading terms without constants; the bench prints them
beside the measured counters, never in place of them.
"""
from __future__ import annotations

import math


def fwd_flops(N: int, d: int, heads: int = 1) -> float:
    """Two products QK^T and PV: 2 N^2 d each."""
    return 4.0 * N * N * d * heads


def bwd_flops(N: int, d: int, heads: int = 1) -> float:
    """Five products of the recompute backward (S, dP, dV, dK, dQ): 2 N^2 d each."""
    return 10.0 * N * N * d * heads


def elements_in_fast_memory(capacity_bytes: float, elem_bytes: int) -> float:
    """M = C / w."""
    return capacity_bytes / elem_bytes


def query_block_rows(M: float, d: int) -> float:
    """B = M / d (large-cache schedule, constants ignored)."""
    return M / d


def square_tile_side(M: float) -> float:
    """b = sqrt(M) (small-cache schedule)."""
    return math.sqrt(M)


def is_large_cache(M: float, d: int) -> bool:
    return M >= d * d


def fused_stream_io(N: int, d: int, M: float) -> float:
    """Leading term of the fused streaming schedule: N^2 d^2 / M."""
    return N * N * d * d / M


def square_tile_io(N: int, d: int, M: float) -> float:
    """Leading term of the square-tile schedule: N^2 d / sqrt(M)."""
    return N * N * d / math.sqrt(M)


def compulsory_io(N: int, d: int) -> float:
    """The N d term (reading inputs, writing the output)."""
    return float(N * d)


def fwd_io_bound(N: int, d: int, M: float) -> float:
    """Theorem 3.1 read with the compulsory term: min(N^2 d^2/M, N^2 d/sqrt M) + N d."""
    return min(fused_stream_io(N, d, M), square_tile_io(N, d, M)) + compulsory_io(N, d)


def bwd_io_large(n: int, d: int, M: float) -> float:
    return (n * n * d * d + n * d ** 3) / M


def bwd_io_small(n: int, d: int, M: float) -> float:
    return (n * n * d + n * d * d) / math.sqrt(M)


def bwd_io_bound(n: int, d: int, M: float) -> float:
    """Theorem 1.1 of the backward paper: the smaller of the two branches."""
    return min(bwd_io_large(n, d, M), bwd_io_small(n, d, M))


def sparse_io_bound(z_input: float, z_qk: float, M: float) -> float:
    """Theorem 4.5: min(Z_in^2 / M, Z_in sqrt(Z_QK) / sqrt(M))."""
    return min(z_input * z_input / M, z_input * math.sqrt(z_qk) / math.sqrt(M))


def sparse_regime_split(z_input: float, z_qk: float) -> float:
    """Cache size where the two sparse branches meet: M = Z_in^2 / Z_QK."""
    return z_input * z_input / z_qk


def time_lower_bound(L_elems: float, elem_bytes: int, bw_bytes_per_s: float,
                     flops: float, flops_per_s: float) -> float:
    """T >= max(w L / beta, F / P), ideal overlap assumed."""
    return max(elem_bytes * L_elems / bw_bytes_per_s, flops / flops_per_s)


# --- the same model evaluated at a kernel's actual tile -------------------

def fwd_dram_compulsory_bytes(N: int, d: int, heads: int, w: int) -> float:
    """Q, K, V read once, O written once (w bytes each), LSE written (4 bytes)."""
    return heads * (4.0 * N * d * w + 4.0 * N)


def bwd_dram_compulsory_bytes(N: int, d: int, heads: int, w: int) -> float:
    """Q, K, V, O, dO read; dQ, dK, dV written; LSE read; D written and read (fp32)."""
    return heads * (8.0 * N * d * w + 4.0 * N * 3)


def fwd_kv_rescan_bytes(N: int, d: int, heads: int, w: int, rows_per_query_tile: int,
                        kept_fraction: float = 1.0) -> float:
    """K and V re-read once per query tile: 2 N d w * (N / Br), times the kept-block share."""
    return heads * 2.0 * N * d * w * (N / rows_per_query_tile) * kept_fraction


def materialized_extra_bytes(N: int, heads: int, w: int) -> float:
    """The stored exp-score matrix: N^2 elements written and read back once."""
    return heads * 2.0 * N * N * w


def materialized_bwd_extra_bytes(N: int, heads: int, w: int) -> float:
    """The small-cache backward's stored N x N matrices: P written and read once (dV = P^T dO),
    dS written once and read twice (dK = s dS^T Q, dQ = s dS K)."""
    return heads * 5.0 * N * N * w


def report(N: int, d: int, heads: int, elem_bytes: int, M: float, hbm_bytes_per_s: float,
           flops_per_s: float, kept_fraction: float = 1.0) -> dict:
    """The pages' bounds for one workload, per GPU, as a flat dict.

    M is the fast-memory capacity in elements (the pages' model); the leading
    terms are per head and multiplied by the head count.  For a block-sparse
    workload the sparse bound of Theorem 4.5 is evaluated with Z_input = N d
    (the non-zeros of one dense input matrix: the reading under which the bound
    reduces to the dense N^2 d^2 / M and its split M = Z_input^2 / Z_QK to the
    dense d^2, as the page says it does) and Z_QK = kept * N^2; the dense forms
    are scaled by the kept-block fraction.  Time bounds use
    T >= max(w L / beta, F / P) with L the compulsory elements plus the leading
    term (ideal overlap; no constant is known for the Theta forms).
    """
    fwd_lead = fused_stream_io(N, d, M) if is_large_cache(M, d) else square_tile_io(N, d, M)
    bwd_lead = bwd_io_bound(N, d, M)
    out = {
        "M_elements": M,
        "large_cache_regime": is_large_cache(M, d),
        "fwd_leading_elements": heads * fwd_lead * kept_fraction,
        "fwd_bound_elements": heads * (fwd_lead * kept_fraction + compulsory_io(N, d)),
        "bwd_leading_elements": heads * bwd_lead * kept_fraction,
        "fwd_flops": fwd_flops(N, d, heads) * kept_fraction,
        "bwd_flops": bwd_flops(N, d, heads) * kept_fraction,
    }
    out["fwd_time_lower_bound_s"] = time_lower_bound(out["fwd_bound_elements"], elem_bytes, hbm_bytes_per_s,
                                                     out["fwd_flops"], flops_per_s)
    out["bwd_time_lower_bound_s"] = time_lower_bound(out["bwd_leading_elements"] + heads * 2 * compulsory_io(N, d),
                                                     elem_bytes, hbm_bytes_per_s, out["bwd_flops"], flops_per_s)
    if kept_fraction < 1.0:
        z_in, z_qk = float(N * d), kept_fraction * N * N
        out["sparse_bound_elements"] = heads * sparse_io_bound(z_in, z_qk, M)
        out["sparse_regime_split_M"] = sparse_regime_split(z_in, z_qk)
    return out
