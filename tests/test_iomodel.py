"""The pages' I/O model as the bench reports it, pinned at the teaching example.

'The I/O Complexity of Attention' exposition (blog.aeilot.top,
attention-io-complexity): 'Large caches' (teaching example N=4096, d=64,
M=65536; doubling M roughly halves the leading term), 'Small caches',
'Putting the regimes together' (the regime table), 'From a movement lower
bound to a performance upper bound'.  Backward: 'On Fine-Grained I/O Complexity
of Attention Backward Passes' summary (gist.science 2410.09397), Theorem 1.1.
"""
import json
import os

from optimal_tiling_gb300 import iomodel

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "teaching_example.json")))


def test_teaching_example_values():
    N, d, M = G["N"], G["d"], G["M"]
    assert iomodel.fused_stream_io(N, d, M) == G["fused_stream_io"]
    assert iomodel.compulsory_io(N, d) == G["compulsory_io"]
    assert iomodel.query_block_rows(M, d) == G["query_block_rows"]
    assert iomodel.is_large_cache(M, d) is G["large_cache"] and d * d == G["d_squared"]
    assert iomodel.square_tile_io(N, d, M) == G["square_tile_io"]
    assert iomodel.square_tile_side(M) == G["square_tile_side"]
    assert iomodel.fused_stream_io(N, d, 2 * M) == G["fused_stream_io_at_2M"]
    assert iomodel.bwd_io_large(N, d, M) == G["bwd_io_large"]
    assert iomodel.bwd_io_small(N, d, M) == G["bwd_io_small"]
    assert iomodel.fwd_flops(N, d) == G["fwd_flops"]


def test_regime_table_picks_the_smaller_term():
    """M >= d^2: the fused streaming term is the smaller one; M < d^2: the square-tile one."""
    N, d = 4096, 64
    for M in (d * d, 2 * d * d, 65536, 10 ** 6):
        assert iomodel.fused_stream_io(N, d, M) <= iomodel.square_tile_io(N, d, M)
        assert iomodel.fwd_io_bound(N, d, M) == iomodel.fused_stream_io(N, d, M) + N * d
    for M in (16, 256, d * d - 1):
        assert iomodel.square_tile_io(N, d, M) < iomodel.fused_stream_io(N, d, M)
    # the two branches meet at M = d^2 (forward) and at M = d^2 for the backward too
    assert abs(iomodel.fused_stream_io(N, d, d * d) - iomodel.square_tile_io(N, d, d * d)) < 1e-6
    assert abs(iomodel.bwd_io_large(N, d, d * d) - iomodel.bwd_io_small(N, d, d * d)) < 1e-3


def test_doubling_fast_memory_halves_leading_term():
    for N, d, M in ((4096, 64, 65536), (16384, 128, 116736)):
        assert iomodel.fused_stream_io(N, d, 2 * M) * 2 == iomodel.fused_stream_io(N, d, M)


def test_sparse_bound_reduces_to_dense():
    """Theorem 4.5 with the dense counts Z_in = N d, Z_QK = N^2 gives the dense forms
    N^2 d^2 / M and N^2 d / sqrt(M); the split sits at M = Z_in^2 / Z_QK = d^2."""
    N, d = 2048, 64
    zin, zqk = N * d, N * N
    assert iomodel.sparse_regime_split(zin, zqk) == d * d
    for M in (1024, 65536):
        assert abs(iomodel.sparse_io_bound(zin, zqk, M)
                   - min(iomodel.fused_stream_io(N, d, M), iomodel.square_tile_io(N, d, M))) < 1e-6


def test_time_bound_is_max_of_memory_and_compute():
    t = iomodel.time_lower_bound(1e9, 2, 1e12, 1e12, 1e15)
    assert t == max(2e9 / 1e12, 1e12 / 1e15)
    assert iomodel.elements_in_fast_memory(65536 * 2, 2) == 65536


def test_report_at_teaching_example():
    r = iomodel.report(4096, 64, 1, 2, 65536, 1e12, 1e15)
    assert r["large_cache_regime"] and r["fwd_leading_elements"] == G["fused_stream_io"]
    assert r["fwd_bound_elements"] == G["fused_stream_io"] + G["compulsory_io"]
    assert r["bwd_leading_elements"] == G["bwd_io_large"]
    assert r["fwd_time_lower_bound_s"] == max(2 * r["fwd_bound_elements"] / 1e12, G["fwd_flops"] / 1e15)
    s = iomodel.report(4096, 64, 1, 2, 65536, 1e12, 1e15, kept_fraction=0.25)
    assert s["sparse_bound_elements"] == iomodel.sparse_io_bound(4096 * 64, 0.25 * 4096 ** 2, 65536)


def test_byte_counts_match_the_buffers_they_describe():
    """The bench's byte helpers against the sizes of the buffers each pass must move once:
    counted from tensors of those shapes, not from the helpers' formulas."""
    import torch

    N, d, heads = 384, 64, 3
    nb = lambda *shape, dt=torch.bfloat16: torch.empty(shape, dtype=dt).nbytes
    x = nb(heads, N, d)            # one of Q, K, V, O, dO, dQ, dK, dV
    row = nb(heads, N, dt=torch.float32)  # one of LSE, D
    nn = nb(heads, N, N)           # one N x N bf16 matrix per head
    # forward: Q, K, V read, O written, LSE written
    assert iomodel.fwd_dram_compulsory_bytes(N, d, heads, 2) == 4 * x + row
    # backward: Q, K, V, O, dO read, dQ, dK, dV written, LSE read, D written and read back
    assert iomodel.bwd_dram_compulsory_bytes(N, d, heads, 2) == 8 * x + 3 * row
    # materialising forward: the exp-score matrix written, then read by the E V product
    assert iomodel.materialized_extra_bytes(N, heads, 2) == 2 * nn
    # materialising backward: P written and read by dV; dS written, read by dK and by dQ
    assert iomodel.materialized_bwd_extra_bytes(N, heads, 2) == (1 + 1) * nn + (1 + 2) * nn
    # K and V re-read once per 128-row query tile (N / 128 tiles), scaled by the kept share
    kv = 2 * x
    assert iomodel.fwd_kv_rescan_bytes(N, d, heads, 2, 128) == kv * (N // 128)
    assert iomodel.fwd_kv_rescan_bytes(N, d, heads, 2, 128, 0.25) == kv * (N // 128) * 0.25


def test_report_sparse_bound_uses_the_dense_reduction():
    """report() evaluates Theorem 4.5 with Z_input = N d and Z_QK = kept N^2: at kept = 1
    (a mask that keeps everything, still passed as sparse) it equals the dense leading
    term, and its split sits at d^2 whatever N is."""
    for N, d, M in ((4096, 64, 65536.0), (16384, 128, 116736.0)):
        almost_all = 1.0 - 1e-12
        r = iomodel.report(N, d, 1, 2, M, 1e12, 1e15, almost_all)
        dense = min(iomodel.fused_stream_io(N, d, M), iomodel.square_tile_io(N, d, M))
        assert abs(r["sparse_bound_elements"] - dense) <= 1e-6 * dense
        assert abs(r["sparse_regime_split_M"] - d * d) <= 1e-6 * d * d
