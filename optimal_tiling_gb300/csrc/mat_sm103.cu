// Materialising two-GEMM attention forward for sm_103a: the comparison point.
//
// Method: "The I/O Complexity of Attention" exposition (blog.aeilot.top,
// attention-io-complexity), section "Small caches: when storing an intermediate
// matrix helps": the exponentiated score matrix (N^2 elements per head) is
// written to slow memory, then multiplied by V.  The page's schedule targets a
// cache with M < d^2; every supported d has d^2 below a GB300 SM's shared
// memory, so this variant shows the cost of the extra N^2 traffic that the fused
// kernel avoids.  The page leaves the exponent unstabilised; here each row i is
// shifted by c_i = s |q_i| max_j |k_j|, an upper bound of every score in the
// row (Cauchy-Schwarz), so E never overflows and the result is the same
// function:  E = exp(s Q K^T - c),  l = rowsum E,  O = E V / l,  LSE = c + ln l.
//
// Kernels (caller's stream): mat_init (zero l and the per-head key-norm max),
// mat_norms (|q_i| and the per-head max |k_j|), mat_scores (per query tile, the
// kept key tiles' S on tcgen05 -> E tiles, bf16, TMA-stored; l = the row sums of
// the stored values),
// mat_output (the shared block GEMM of gemm_sm103.cuh: O = E V over the kept
// key blocks, then O / l and LSE).
// Key blocks removed by the block mask are neither written nor read.
#include <cuda_bf16.h>

#include "gemm_sm103.cuh"
#include "internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int BT = 128;  // tile rows / columns

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Every bulk group this thread committed has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__global__ void mat_init_kernel(float *__restrict__ rowl, float *__restrict__ kmax, size_t rows, int heads) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows; i += (size_t)gridDim.x * blockDim.x)
        rowl[i] = 0.f;
    if (blockIdx.x == 0)
        for (int h = threadIdx.x; h < heads; h += blockDim.x) kmax[h] = 0.f;
}

// |q_row| into qnorm and the max over the head's |k_row| into kmax.  A block of 8 warps takes
// kNormRows consecutive rows of one head (N is a multiple of 128), a warp one row at a time; the
// block's maximum goes into kmax with one atomic (one atomic per row put all rows of a head on
// one address, and those atomics, not the reads, set the kernel's time).
constexpr int kNormRows = 128;

template <int D>
__global__ void __launch_bounds__(256) mat_norms_kernel(const __nv_bfloat16 *__restrict__ Q,
                                                        const __nv_bfloat16 *__restrict__ K,
                                                        float *__restrict__ qnorm, float *__restrict__ kmax,
                                                        size_t rows, int N) {
    __shared__ float wmax[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t row0 = (size_t)blockIdx.x * kNormRows;
    float kmx = 0.f;
    for (int rr = warp; rr < kNormRows; rr += 8) {
        const size_t row = row0 + rr;
        if (row >= rows) break;
        float aq = 0.f, ak = 0.f;
        for (int c = lane * 2; c < D; c += 64) {
            const float2 q = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(Q + row * D + c));
            const float2 k = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(K + row * D + c));
            aq = fmaf(q.x, q.x, fmaf(q.y, q.y, aq));
            ak = fmaf(k.x, k.x, fmaf(k.y, k.y, ak));
        }
        for (int off = 16; off > 0; off >>= 1) {
            aq += __shfl_xor_sync(0xffffffffu, aq, off);
            ak += __shfl_xor_sync(0xffffffffu, ak, off);
        }
        if (lane == 0) qnorm[row] = sqrtf(aq);
        kmx = fmaxf(kmx, sqrtf(ak));
    }
    if (lane == 0) wmax[warp] = kmx;
    __syncthreads();
    if (threadIdx.x == 0 && row0 < rows) {
        float m = wmax[0];
        for (int w = 1; w < 8; ++w) m = fmaxf(m, wmax[w]);
        // norms are non-negative, so their bit patterns order like the values
        atomicMax(reinterpret_cast<int *>(kmax) + row0 / N, __float_as_int(m));
    }
}

template <int D>
struct ScoreCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = BT * D * 2;           // a Q or K tile
    static constexpr int kSlab = BT * 128;             // one 64-column slab of a 128-row tile
    static constexpr int kStages = D == 256 ? 2 : 3;   // K ring depth (as deep as shared memory allows at d = 256)
    static constexpr int kETile = BT * BT * 2;         // one bf16 E tile: two 64-column slabs
    // staging tiles for E: two where they fit beside Q and the K ring without costing a CTA per
    // SM (d = 128), so that a tile's epilogue need not wait for the previous tile's store to read
    static constexpr int kEStages = D == 128 ? 2 : 1;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kTile;
    static constexpr int kEOff = kKOff + kStages * kTile;
    static constexpr int kBarOff = kEOff + kEStages * kETile;
    // q, kfull[S], kempty[S], sfull[2], sfree[2], drain
    static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    // kept key blocks of the CTA's mask row as a bit set, up to 32 * kMaxMaskWords blocks
    static constexpr int kMaxMaskWords = 256;
    static constexpr int kBitsOff = kMiscOff + 64;
    static constexpr int kSmemBytes = kBitsOff + 4 * kMaxMaskWords + 1024;  // + slack to align the base
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

// One CTA per (query tile, head), 320 threads: warps 0-7 epilogue (warp w: rows of tensor memory
// lane quarter w % 4, score columns 64 (w / 4) .. + 63), warp 8 TMA, warp 9 MMA.  The Q tile stays in shared memory while the kept key tiles stream
// through a K ring; S = Q K^T alternates between two 128-column tensor-memory buffers, so the
// next tile's product runs while the epilogue turns this one into E = exp(s S - c) (bf16) and
// stores it with tensor stores from one staging tile.  Each thread keeps its half of a row's sum
// of the stored values in a register and adds it into l once.  (With one CTA per SM at d >= 128,
// four epilogue warps, one thread per row, set the pace.)  (One CTA per score tile, the earlier form, left one CTA
// per SM at d = 256, whose loads, product, exps and store then ran one after another.)
template <int D>
__global__ void __launch_bounds__(320, D == 64 ? 2 : 1) mat_scores_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                            const __grid_constant__ CUtensorMap tmK,
                                                            const __grid_constant__ CUtensorMap tmE, const Problem p,
                                                            const float *__restrict__ qnorm,
                                                            const float *__restrict__ kmax, float *__restrict__ rowl) {
    using C = ScoreCfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t bar0 = smem_addr(sm + C::kBarOff);
    auto kfull = [&](int s) { return bar0 + 8u * (1 + s); };
    auto kempty = [&](int s) { return bar0 + 8u * (1 + S + s); };
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
    const uint32_t sQ = smem_addr(sm + C::kQOff), sK = smem_addr(sm + C::kKOff), sE = smem_addr(sm + C::kEOff);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(kfull(s), 1);
            mbar_init(kempty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sfull(b), 1);
            mbar_init(sfree(b), 256);
        }
        mbar_init(bar_drain, 1);
        fence_barrier_init();
        // the Q tile is needed whatever the mask says: start its load before the mask is read
        mbar_arrive_expect_tx(bar_q, C::kTile);
        for (int c = 0; c < C::kChunks; ++c) tma_load_2d(sQ + c * C::kSlab, &tmQ, c * 64, q0, bar_q);
    }
    if (use_bits) build_visit_bits(vwords, nb, kept);
    if (warp == 9) {
        tmem_alloc(smem_addr(tmem_slot), 256);
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
            int k = -1;
            for (int it = 0; it < n; ++it) {
                k = next_block(k);
                const int s = it % S;
                if (it >= S && !mbar_wait(kempty(s), ((uint32_t)(it / S) & 1u) ^ 1u, abort_flag, p.dev_status)) break;
                mbar_arrive_expect_tx(kfull(s), C::kTile);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_2d(sK + s * C::kTile + c * C::kSlab, &tmK, c * 64, head * p.N + k * BT, kfull(s));
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n > 0) {
            constexpr uint32_t id = idesc_bf16_f32(BT, BT, false, false);
            bool ok = mbar_wait(bar_q, 0, abort_flag, p.dev_status);
            for (int it = 0; it < n && ok; ++it) {
                const int s = it % S, b = it & 1;
                // the epilogue has read S of tile it - 2 out of this buffer.  At d <= 128 that is what
                // the product usually waits for, so it is waited for first (d = 128: 0.824 -> 0.806 ms
                // on 2 x 16 x 8192; at d = 256, where the K tile arrives later, 1.258 -> 1.276 ms).
                if constexpr (D == 256) {
                    if (!(ok = mbar_wait(kfull(s), (uint32_t)(it / S) & 1u, abort_flag, p.dev_status))) break;
                }
                if (it >= 2 && !(ok = mbar_wait(sfree(b), (uint32_t)((it - 2) >> 1) & 1u, abort_flag, p.dev_status)))
                    break;
                if constexpr (D != 256) {
                    if (!(ok = mbar_wait(kfull(s), (uint32_t)(it / S) & 1u, abort_flag, p.dev_status))) break;
                }
                tc_fence_after();
                const uint32_t kb = sK + s * C::kTile;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::kSlab + (ks & 3) * 32;
                    mma_ss(tmem + b * BT, smem_desc_sw128(sQ + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024), id,
                           ks > 0);
                }
                mma_commit(kempty(s));
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
        const float c2 = fabsf(p.scale) * qnorm[q0 + row] * kmax[head] * kLog2e;  // row bound, log2 domain
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        float rs = 0.f;
        bool ok = true;
        int k = -1;
        for (int it = 0; it < n; ++it) {
            k = next_block(k);
            const int b = it & 1;
            ok = ok && mbar_wait(sfull(b), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            // this tile's staging tile is free once the stores issued from it kEStages tiles ago
            // have read it
            uint8_t *stage = sm + C::kEOff + (it % C::kEStages) * C::kETile;
            const uint32_t sEs = sE + (it % C::kEStages) * C::kETile;
            if (tid == 0) {
                if (C::kEStages == 2) bulk_wait_read_but_one();
                else bulk_wait_read_all();
            }
            named_bar_sync(1, 256);
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 64 * hc; c0 < 64 * hc + 64; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + b * BT + c0, r);
                    tmem_wait_ld();
                    reg_fence(r);
                    uint32_t pk[16];
                    // two scores per step on the packed fp32 path; the row sum adds the values
                    // actually stored (bf16 widened by a shift), in an even and an odd chain
                    const uint64_t sl2x2 = f2_pack(sl2, sl2), nc2 = f2_pack(-c2, -c2);
                    uint64_t rs2 = f2_pack(0.f, 0.f);
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * t]), __uint_as_float(r[2 * t + 1])), sl2x2, nc2),
                                  x0, x1);
                        pk[t] = pack_bf16(ex2(x0), ex2(x1));
                        rs2 = f2_add(rs2, f2_pack(__uint_as_float(pk[t] << 16), __uint_as_float(pk[t] & 0xffff0000u)));
                    }
                    float rs0, rs1;
                    f2_unpack(rs2, rs0, rs1);
                    rs += rs0 + rs1;
                    const int slab = c0 / 64;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int chunk = ((c0 % 64) / 8) + v;  // 16-byte chunk within the 128-byte row
                        const uint32_t off = slab * C::kSlab + row * 128 + ((chunk ^ (row & 7)) * 16);
                        *reinterpret_cast<uint4 *>(stage + off) =
                            make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(sfree(b));
                fence_proxy_async_smem();
            }
            named_bar_sync(1, 256);
            if (tid == 0 && ok) {
                tma_store_2d(&tmE, k * BT, q0, sEs);
                tma_store_2d(&tmE, k * BT + 64, q0, sEs + C::kSlab);
                bulk_commit();
            }
        }
        if (ok && n > 0) atomicAdd(rowl + q0 + row, rs);  // l stays 0 for a row whose every key tile is removed
        if (tid == 0) bulk_wait_all();
    }

    // a tile that visits no key tile still received its Q tile: let that copy land first
    if (n == 0 && tid == 0) mbar_wait(bar_q, 0, abort_flag, p.dev_status);
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// O = E V / l and LSE = c + ln l, as the epilogue of the shared block GEMM
// (one CTA per 128-row query tile, E blocks in K-major orientation).
template <int D>
struct MatOutEpi {
    __nv_bfloat16 *O;
    float *LSE;
    const float *rowl, *qnorm, *kmax;
    float scale;
    int N;
    __device__ void operator()(size_t grow, const uint32_t (&r)[32], int c0) const {
        gemm::store_row_chunk<D>(O, grow, r, c0, 1.f / rowl[grow]);
    }
    __device__ void finish(size_t grow) const {
        LSE[grow] = fabsf(scale) * qnorm[grow] * kmax[grow / N] + __log2f(rowl[grow]) * kLn2;
    }
    __device__ void empty(size_t grow) const {
        gemm::zero_row<D>(O, grow);
        LSE[grow] = -INFINITY;
    }
};

template <int D>
cudaError_t launch_d(const Problem &p, const MatMaps &m, const void *Q, const void *K, float *qnorm, float *rowl,
                     float *kmax, void *O, float *LSE, cudaStream_t st) {
    const size_t rows = (size_t)p.B * p.H * p.N;
    const int heads = p.B * p.H;
    {
        ProfScope prof_("mat_init", st);
        mat_init_kernel<<<152 * 4, 256, 0, st>>>(rowl, kmax, rows, heads);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    {
        ProfScope prof_("mat_norms", st);
        mat_norms_kernel<D><<<(unsigned)((rows + kNormRows - 1) / kNormRows), 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(Q), static_cast<const __nv_bfloat16 *>(K), qnorm, kmax, rows, p.N);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    auto ks = mat_scores_kernel<D>;
    if ((e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, ScoreCfg<D>::kSmemBytes)) !=
        cudaSuccess)
        return e;
    {
        ProfScope prof_("mat_scores", st);
        ks<<<dim3(p.N / BT, heads), 320, ScoreCfg<D>::kSmemBytes, st>>>(m.q, m.k, m.e, p, qnorm, kmax, rowl);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return gemm::launch_block_gemm<D, false>(
        "mat_output", p, m.e, m.v,
        MatOutEpi<D>{static_cast<__nv_bfloat16 *>(O), LSE, rowl, qnorm, kmax, p.scale, p.N}, st);
}

}  // namespace

cudaError_t launch_fwd_materialized_bf16(const Problem &p, const MatMaps &maps, const void *Q, const void *K,
                                         void *E, float *rowc, float *rowl, float *kmax, void *O, float *LSE,
                                         cudaStream_t st) {
    (void)E;
    if (p.B * p.H > 65535 || p.N / BT > 65535) return cudaErrorNotSupported;
    switch (p.d) {
        case 64: return launch_d<64>(p, maps, Q, K, rowc, rowl, kmax, O, LSE, st);
        case 128: return launch_d<128>(p, maps, Q, K, rowc, rowl, kmax, O, LSE, st);
        case 256: return launch_d<256>(p, maps, Q, K, rowc, rowl, kmax, O, LSE, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace attn
