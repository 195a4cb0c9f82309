// One pipelined tcgen05 GEMM shape shared by the materialising schedules:
//
//     C_t = sum over kept 128-blocks k of  A(t, k) * B_k          (128 x D, fp32 in TMEM)
//
// where A is a 128 x 128 bf16 block of an N x N matrix per head (the stored
// exp-scores E, or P, or dS) and B_k is the 128 x D block k of an [rows, D]
// bf16 matrix (V, dO, Q or K).  Two orientations of A:
//   kTransA = false: A(t, k) = M[t-block rows, k-block cols]   (K-major operand),
//                    block kept when mask[t][k] != 0;
//   kTransA = true:  A(t, k) = M[k-block rows, t-block cols]^T (MN-major operand),
//                    block kept when mask[k][t] != 0.
// B_k is always [k-block rows][D] with D contiguous: an MN-major operand.
// One CTA per (output block t, head), 192 threads: warps 0-3 epilogue (row =
// tensor memory lane), warp 4 TMA, warp 5 MMA; a ring of (A, B) stages.
// The epilogue is the caller's functor: epi(row_global, acc_row_pointer_in_regs...).
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "visit_bits.cuh"

namespace attn {
namespace gemm {

using namespace ptx;

constexpr int BT = 128;

template <int D>
struct Cfg {
    static constexpr int kATile = BT * BT * 2;   // 32 KB
    static constexpr int kBTile = BT * D * 2;
    static constexpr int kSlab = BT * 128;       // 16 KB
    static constexpr int kStages = D == 64 ? 4 : (D == 128 ? 3 : 2);
    static constexpr int kAOff = 0;
    static constexpr int kBOff = kStages * kATile;
    static constexpr int kBarOff = kBOff + kStages * kBTile;
    static constexpr int kNumBars = 2 * kStages + 2;  // full[S], empty[S], done, drain
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    // kept blocks of the CTA's row (or column) of the mask as a bit set, up to 32 * kMaxMaskWords
    static constexpr int kMaxMaskWords = 256;
    static constexpr int kBitsOff = kMiscOff + 64;
    static constexpr int kSmemBytes = kBitsOff + 4 * kMaxMaskWords + 1024;
    static constexpr uint32_t kTmemCols = D < 32 ? 32 : D;
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

__device__ __forceinline__ bool kept_block(const uint8_t *mask, int nb, int t, int k, bool trans) {
    if (mask == nullptr) return true;
    return trans ? mask[(size_t)k * nb + t] != 0 : mask[(size_t)t * nb + k] != 0;
}

// Epi: struct with  __device__ void operator()(size_t grow, const uint32_t (&acc)[32], int c0)
// called for each 32-column chunk of row grow, and  __device__ void empty(size_t grow)  for a
// row whose every block was removed; plus  __device__ void finish(size_t grow)  after the chunks.
template <int D, bool kTransA, class Epi>
__global__ void __launch_bounds__(192, 1)
block_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Problem p,
                  Epi epi) {
    using C = Cfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t bar0 = smem_addr(sm + C::kBarOff);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };
    const uint32_t bar_done = bar0 + 8u * (2 * S), bar_drain = bar0 + 8u * (2 * S + 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = blockIdx.x, head = blockIdx.y;
    const int nb = p.N / BT;
    uint32_t *vwords = reinterpret_cast<uint32_t *>(sm + C::kBitsOff);
    const int nwords = (nb + 31) >> 5;
    const bool use_bits = p.mask != nullptr && nwords <= C::kMaxMaskWords;
    if (use_bits) build_visit_bits(vwords, nb, [&](int k) { return kept_block(p.mask, nb, t, k, kTransA); });
    const int hrow = head * p.N;
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_drain, 1);
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sA = smem_addr(sm + C::kAOff), sB = smem_addr(sm + C::kBOff);
    const VisitBits vb{vwords, nwords};
    int n = nb;  // kept blocks
    if (use_bits) {
        n = vb.count();
    } else if (p.mask != nullptr) {  // rows longer than the bit set: read the mask directly
        n = 0;
        for (int k = 0; k < nb; ++k) n += kept_block(p.mask, nb, t, k, kTransA) ? 1 : 0;
    }
    auto next_block = [&](int k) -> int {
        if (p.mask == nullptr) return k + 1;
        if (use_bits) return vb.next(k);
        do {
            ++k;
        } while (!kept_block(p.mask, nb, t, k, kTransA));
        return k;
    };
    if (warp == 4) {
        if (lane == 0 && n > 0) {
            int k = -1;
            for (int it = 0; it < n; ++it) {
                k = next_block(k);
                const int s = it % S;
                if (it >= S && !mbar_wait(empty(s), ((uint32_t)(it / S) & 1u) ^ 1u, abort_flag, p.dev_status)) break;
                mbar_arrive_expect_tx(full(s), C::kATile + C::kBTile);
                // A block: two 64-column slabs of a 128 x 128 block
                const int ax = kTransA ? t * BT : k * BT;
                const int ay = hrow + (kTransA ? k * BT : t * BT);
                tma_load_2d(sA + s * C::kATile, &tmA, ax, ay, full(s));
                tma_load_2d(sA + s * C::kATile + C::kSlab, &tmA, ax + 64, ay, full(s));
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d(sB + s * C::kBTile + c * C::kSlab, &tmB, c * 64, hrow + k * BT, full(s));
            }
        }
    } else if (warp == 5) {
        if (lane == 0 && n > 0) {
            constexpr uint32_t id = idesc_bf16_f32(BT, D, kTransA, true);
            bool ok = true;
            for (int it = 0; it < n; ++it) {
                const int s = it % S;
                if (!(ok = mbar_wait(full(s), (uint32_t)(it / S) & 1u, abort_flag, p.dev_status))) break;
                tc_fence_after();
                const uint32_t ab = sA + s * C::kATile, bb = sB + s * C::kBTile;
#pragma unroll
                for (int ks = 0; ks < BT / 16; ++ks) {
                    // K-major A: 16 contraction elements = 32 bytes inside a 64-column slab;
                    // MN-major A: 16 contraction rows = 2 groups of 8 rows of 128 bytes
                    const uint64_t ad = kTransA ? smem_desc_sw128(ab + ks * 2048, C::kSlab, 1024)
                                                : smem_desc_sw128(ab + (ks >> 2) * C::kSlab + (ks & 3) * 32, 16, 1024);
                    mma_ss(tmem, ad, smem_desc_sw128(bb + ks * 2048, C::kSlab, 1024), id, (it > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(empty(s));
            }
            if (ok) {
                mma_commit(bar_done);
            } else {
                mma_commit(bar_drain);
                mbar_wait(bar_drain, 0, abort_flag, p.dev_status);
            }
        }
    } else {
        bool ok = true;
        if (n > 0) {
            ok = mbar_wait(bar_done, 0, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        const size_t grow = (size_t)hrow + (size_t)t * BT + tid;
        if (ok && n > 0) {
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_base + c0, r);
                tmem_wait_ld();
                reg_fence(r);
                epi(grow, r, c0);
            }
            epi.finish(grow);
        } else if (n == 0) {
            epi.empty(grow);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Scaled bf16 store of a 32-column chunk of one output row.
template <int D>
__device__ __forceinline__ void store_row_chunk(__nv_bfloat16 *out, size_t grow, const uint32_t (&r)[32], int c0,
                                                float mul) {
    uint32_t pk[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) pk[t] = pack_bf16(__uint_as_float(r[2 * t]) * mul, __uint_as_float(r[2 * t + 1]) * mul);
    uint4 *o = reinterpret_cast<uint4 *>(out + grow * D + c0);
#pragma unroll
    for (int v = 0; v < 4; ++v) o[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
}

template <int D>
__device__ __forceinline__ void zero_row(__nv_bfloat16 *out, size_t grow) {
    uint4 *o = reinterpret_cast<uint4 *>(out + grow * D);
    for (int v = 0; v < D / 8; ++v) o[v] = make_uint4(0, 0, 0, 0);
}

template <int D, bool kTransA, class Epi>
cudaError_t launch_block_gemm(const char *name, const Problem &p, const CUtensorMap &a, const CUtensorMap &b, Epi epi,
                              cudaStream_t st) {
    auto kern = block_gemm_kernel<D, kTransA, Epi>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    {
        ProfScope prof_(name, st);
        kern<<<dim3(p.N / BT, p.B * p.H), 192, Cfg<D>::kSmemBytes, st>>>(a, b, p, epi);
    }
    return cudaGetLastError();
}

}  // namespace gemm
}  // namespace attn
