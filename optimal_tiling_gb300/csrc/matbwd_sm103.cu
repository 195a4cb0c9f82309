// Materialising backward for sm_103a: the backward twin of the materialising
// forward, after the small-cache backward algorithm ("Algorithm 6") of "On
// Fine-Grained I/O Complexity of Attention Backward Passes" (gist.science
// 2410.09397), which explicitly writes the n x n attention matrices and reads
// them back in tiles instead of recomputing them.  The page gives no listing;
// the plainest reading, with the chain rule of O = softmax(s Q K^T) V:
//
//   D  = rowsum(dO o O)                                   (n x 1, fp32)
//   P  = exp(s Q K^T - LSE),  dP = dO V^T,  dS = P o (dP - D)   -> P, dS to HBM (bf16)
//   dV = P^T dO,   dK = s dS^T Q,   dQ = s dS K          (three GEMMs over the stored matrices)
//
// Kernels: matbwd_rowdot (D), matbwd_scores (one CTA per 128-row query tile
// streaming the kept key tiles: S and dP on tcgen05 into tensor memory, P and dS
// staged in shared memory and TMA-stored), and three launches of the shared
// block GEMM (gemm_sm103.cuh).
// Blocks removed by the block mask are neither written nor read.
#include <cuda_bf16.h>

#include "gemm_sm103.cuh"
#include "internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int BT = 128;

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Every bulk group this thread committed has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(256) matbwd_rowdot_kernel(const __nv_bfloat16 *__restrict__ O,
                                                            const __nv_bfloat16 *__restrict__ dO,
                                                            float *__restrict__ Dv, size_t rows) {
    const size_t row = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float acc = 0.f;
    for (int c = lane * 2; c < D; c += 64) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(O + row * D + c));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(dO + row * D + c));
        acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
    }
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) Dv[row] = acc;
}

template <int D>
struct ScoresCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = BT * D * 2;   // a Q, K, dO or V tile
    static constexpr int kSlab = BT * 128;     // one 64-column slab of a 128-row tile
    static constexpr int kStages = D == 64 ? 3 : 1;  // K/V ring depth (as deep as shared memory allows)
    static constexpr int kStage = BT * BT * 2; // one bf16 P or dS tile: two 64-column slabs
    static constexpr int kQOff = 0, kdOOff = kTile, kKVOff = 2 * kTile;   // a K/V stage: K tile, V tile
    static constexpr int kPOff = kKVOff + kStages * 2 * kTile;
    static constexpr int kdSOff = kPOff + kStage;
    static constexpr int kBarOff = kdSOff + kStage;
    // q, kvfull[S], kvempty[S], sfull[2], sfree[2], drain
    static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kMaxMaskWords = 256;
    static constexpr int kBitsOff = kMiscOff + 64;
    static constexpr int kSmemBytes = kBitsOff + 4 * kMaxMaskWords + 1024;  // + slack to align the base
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

// One CTA per (query tile, head), 320 threads: warps 0-7 epilogue (warp w: rows of tensor memory
// lane quarter w % 4, score columns 64 (w / 4) .. + 63), warp 8 TMA, warp 9 MMA.  Q and dO stay
// in shared memory while the kept key tiles' K and V stream through a ring; S = Q K^T and
// dP = dO V^T of a key tile go to one of two tensor-memory buffer pairs (S in columns 256 b ..,
// dP in 256 b + 128 ..), so the next tile's products run while the epilogue turns this one into
// P = exp(s S - LSE) and dS = P o (dP - D) (bf16) and stores them with tensor stores from two
// staging tiles.  (One CTA per score tile, the earlier form, fit one CTA per SM at d = 128, whose
// loads, products, exps and stores then ran one after another.)
template <int D>
__global__ void __launch_bounds__(320, 1) matbwd_scores_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
    const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmdS, const Problem p,
    const float *__restrict__ LSE, const float *__restrict__ Dv) {
    using C = ScoresCfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t bar0 = smem_addr(sm + C::kBarOff);
    auto kvfull = [&](int s) { return bar0 + 8u * (1 + s); };
    auto kvempty = [&](int s) { return bar0 + 8u * (1 + S + s); };
    auto sfull = [&](int b) { return bar0 + 8u * (1 + 2 * S + b); };
    auto sfree = [&](int b) { return bar0 + 8u * (3 + 2 * S + b); };
    const uint32_t bar_q = bar0, bar_drain = bar0 + 8u * (5 + 2 * S);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qt = blockIdx.x, head = blockIdx.y;
    const int nb = p.N / BT;
    const int q0 = head * p.N + qt * BT;
    uint32_t *vwords = reinterpret_cast<uint32_t *>(sm + C::kBitsOff);
    const int nwords = (nb + 31) >> 5;
    const bool use_bits = p.mask != nullptr && nwords <= C::kMaxMaskWords;
    auto kept = [&](int k) { return p.mask == nullptr || p.mask[(size_t)qt * nb + k] != 0; };
    const uint32_t sQ = smem_addr(sm + C::kQOff), sdO = smem_addr(sm + C::kdOOff), sKV = smem_addr(sm + C::kKVOff);
    const uint32_t sP = smem_addr(sm + C::kPOff), sdS = smem_addr(sm + C::kdSOff);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(kvfull(s), 1);
            mbar_init(kvempty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sfull(b), 1);
            mbar_init(sfree(b), 256);
        }
        mbar_init(bar_drain, 1);
        fence_barrier_init();
        // Q and dO are needed whatever the mask says: start their loads before the mask is read
        mbar_arrive_expect_tx(bar_q, 2 * C::kTile);
        for (int c = 0; c < C::kChunks; ++c) {
            tma_load_2d(sQ + c * C::kSlab, &tmQ, c * 64, q0, bar_q);
            tma_load_2d(sdO + c * C::kSlab, &tmdO, c * 64, q0, bar_q);
        }
    }
    if (use_bits) build_visit_bits(vwords, nb, kept);
    if (warp == 9) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const VisitBits vb{vwords, nwords};
    int n = nb;  // kept key tiles of this query tile
    if (use_bits) {
        n = vb.count();
    } else if (p.mask != nullptr) {  // rows longer than the bit set: read the mask directly
        n = 0;
        for (int k = 0; k < nb; ++k) n += kept(k) ? 1 : 0;
    }
    auto next_block = [&](int k) -> int {
        if (p.mask == nullptr) return k + 1;
        if (use_bits) return vb.next(k);
        do {
            ++k;
        } while (!kept(k));
        return k;
    };

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int k = -1;
            for (int it = 0; it < n; ++it) {
                k = next_block(k);
                const int s = it % S;
                if (it >= S && !mbar_wait(kvempty(s), ((uint32_t)(it / S) & 1u) ^ 1u, abort_flag, p.dev_status)) break;
                const uint32_t kb = sKV + s * 2 * C::kTile, vb_ = kb + C::kTile;
                mbar_arrive_expect_tx(kvfull(s), 2 * C::kTile);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_2d(kb + c * C::kSlab, &tmK, c * 64, head * p.N + k * BT, kvfull(s));
                    tma_load_2d(vb_ + c * C::kSlab, &tmV, c * 64, head * p.N + k * BT, kvfull(s));
                }
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n > 0) {
            constexpr uint32_t id = idesc_bf16_f32(BT, BT, false, false);
            bool ok = mbar_wait(bar_q, 0, abort_flag, p.dev_status);
            for (int it = 0; it < n && ok; ++it) {
                const int s = it % S, b = it & 1;
                if (!(ok = mbar_wait(kvfull(s), (uint32_t)(it / S) & 1u, abort_flag, p.dev_status))) break;
                // the epilogue has read S and dP of tile it - 2 out of this buffer pair
                if (it >= 2 && !(ok = mbar_wait(sfree(b), (uint32_t)((it - 2) >> 1) & 1u, abort_flag, p.dev_status)))
                    break;
                tc_fence_after();
                const uint32_t kb = sKV + s * 2 * C::kTile, vb_ = kb + C::kTile;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::kSlab + (ks & 3) * 32;
                    mma_ss(tmem + 256 * b, smem_desc_sw128(sQ + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024), id,
                           ks > 0);
                    mma_ss(tmem + 256 * b + 128, smem_desc_sw128(sdO + off, 16, 1024),
                           smem_desc_sw128(vb_ + off, 16, 1024), id, ks > 0);
                }
                mma_commit(kvempty(s));
                mma_commit(sfull(b));
            }
            if (!ok) {
                // let every MMA already issued finish before tensor memory is released
                mma_commit(bar_drain);
                mbar_wait(bar_drain, 0, abort_flag, p.dev_status);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue warps 0-7
        // Every epilogue thread meets the named barriers of every tile whatever happens: after a
        // failed (timed-out) wait the work is skipped but the barriers are kept.
        const int hc = warp >> 2, row = tid & 127;  // score columns 64 hc .. 64 hc + 63 of this row
        const float sl2 = p.scale * kLog2e;
        const float l2 = LSE[q0 + row] * kLog2e;
        const float dd = Dv[q0 + row];
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        bool ok = true;
        int k = -1;
        for (int it = 0; it < n; ++it) {
            k = next_block(k);
            const int b = it & 1;
            ok = ok && mbar_wait(sfull(b), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            // the staging tiles are free once the previous tile's tensor stores have read them
            if (tid == 0) bulk_wait_read_all();
            named_bar_sync(1, 256);
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 64 * hc; c0 < 64 * hc + 64; c0 += 32) {
                    uint32_t sr[32], pr[32];
                    tmem_ld32(lane_base + 256 * b + c0, sr);
                    tmem_ld32(lane_base + 256 * b + 128 + c0, pr);
                    tmem_wait_ld();
                    reg_fence(sr);
                    reg_fence(pr);
                    uint32_t pk[16], dk[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const float p0 = ex2(fmaf(__uint_as_float(sr[2 * t]), sl2, -l2));
                        const float p1 = ex2(fmaf(__uint_as_float(sr[2 * t + 1]), sl2, -l2));
                        pk[t] = pack_bf16(p0, p1);
                        dk[t] = pack_bf16(p0 * (__uint_as_float(pr[2 * t]) - dd), p1 * (__uint_as_float(pr[2 * t + 1]) - dd));
                    }
                    const int slab = c0 / 64;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int chunk = ((c0 % 64) / 8) + v;  // 16-byte chunk within the 128-byte row
                        const uint32_t off = slab * C::kSlab + row * 128 + ((chunk ^ (row & 7)) * 16);
                        *reinterpret_cast<uint4 *>(sm + C::kPOff + off) =
                            make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                        *reinterpret_cast<uint4 *>(sm + C::kdSOff + off) =
                            make_uint4(dk[4 * v], dk[4 * v + 1], dk[4 * v + 2], dk[4 * v + 3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(sfree(b));
                fence_proxy_async_smem();
            }
            named_bar_sync(1, 256);
            if (tid == 0 && ok) {
                tma_store_2d(&tmP, k * BT, q0, sP);
                tma_store_2d(&tmP, k * BT + 64, q0, sP + C::kSlab);
                tma_store_2d(&tmdS, k * BT, q0, sdS);
                tma_store_2d(&tmdS, k * BT + 64, q0, sdS + C::kSlab);
                bulk_commit();
            }
        }
        if (tid == 0) bulk_wait_all();
    }

    // a tile that visits no key tile still received its Q and dO tiles: let those copies land first
    if (n == 0 && tid == 0) mbar_wait(bar_q, 0, abort_flag, p.dev_status);
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Epilogue of the three gradient GEMMs: out = mul * acc in bf16; removed rows are zero.
template <int D>
struct ScaledStore {
    __nv_bfloat16 *out;
    float mul;
    __device__ void operator()(size_t grow, const uint32_t (&r)[32], int c0) const {
        gemm::store_row_chunk<D>(out, grow, r, c0, mul);
    }
    __device__ void finish(size_t) const {}
    __device__ void empty(size_t grow) const { gemm::zero_row<D>(out, grow); }
};

template <int D>
cudaError_t launch_d(const Problem &p, const MatBwdMaps &m, const void *O, const void *dO, const float *LSE,
                     float *Dv, void *dQ, void *dK, void *dV, cudaStream_t st) {
    const size_t rows = (size_t)p.B * p.H * p.N;
    {
        ProfScope prof_("matbwd_rowdot", st);
        matbwd_rowdot_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(O), static_cast<const __nv_bfloat16 *>(dO), Dv, rows);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto ks = matbwd_scores_kernel<D>;
    if ((e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, ScoresCfg<D>::kSmemBytes)) !=
        cudaSuccess)
        return e;
    {
        ProfScope prof_("matbwd_scores", st);
        ks<<<dim3(p.N / BT, p.B * p.H), 320, ScoresCfg<D>::kSmemBytes, st>>>(m.q, m.k, m.v, m.dO, m.p, m.ds, p,
                                                                            LSE, Dv);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // dV = P^T dO and dK = s dS^T Q (A transposed: one output block per key tile)
    if ((e = gemm::launch_block_gemm<D, true>("matbwd_dv", p, m.p, m.dO,
                                              ScaledStore<D>{static_cast<__nv_bfloat16 *>(dV), 1.f}, st)) !=
        cudaSuccess)
        return e;
    if ((e = gemm::launch_block_gemm<D, true>("matbwd_dk", p, m.ds, m.q,
                                              ScaledStore<D>{static_cast<__nv_bfloat16 *>(dK), p.scale}, st)) !=
        cudaSuccess)
        return e;
    // dQ = s dS K (one output block per query tile)
    return gemm::launch_block_gemm<D, false>("matbwd_dq", p, m.ds, m.k,
                                             ScaledStore<D>{static_cast<__nv_bfloat16 *>(dQ), p.scale}, st);
}

}  // namespace

cudaError_t launch_bwd_materialized_bf16(const Problem &p, const MatBwdMaps &maps, const void *O, const void *dO,
                                         const float *LSE, float *Dv, void *dQ, void *dK, void *dV, cudaStream_t st) {
    if (p.B * p.H > 65535 || p.N / BT > 65535) return cudaErrorNotSupported;
    switch (p.d) {
        case 64: return launch_d<64>(p, maps, O, dO, LSE, Dv, dQ, dK, dV, st);
        case 128: return launch_d<128>(p, maps, O, dO, LSE, Dv, dQ, dK, dV, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace attn
