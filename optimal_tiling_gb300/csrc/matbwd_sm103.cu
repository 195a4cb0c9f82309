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
// Kernels: matbwd_rowdot (D), matbwd_scores (one CTA per 128 x 128 tile: S and
// dP on tcgen05 into tensor memory, P and dS staged in shared memory and
// TMA-stored), and three launches of the shared block GEMM (gemm_sm103.cuh).
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
    static constexpr int kTile = BT * D * 2;   // Q, K, dO or V tile
    static constexpr int kSlab = BT * 128;
    static constexpr int kQOff = 0, kKOff = kTile, kdOOff = 2 * kTile, kVOff = 3 * kTile;
    static constexpr int kPStage = 0;          // P staging (32 KB) over Q (and K when d = 64)
    static constexpr int kdSStage = 2 * kTile; // dS staging (32 KB) over dO (and V when d = 64)
    static constexpr int kBarOff = 4 * kTile;
    // at least 80 KB: at most two CTAs per SM, so their 256 tensor-memory columns always fit
    static constexpr int kSmemBytes = (kBarOff + 64 + 1024) > 80 * 1024 ? (kBarOff + 64 + 1024) : 80 * 1024;
    static_assert(2 * kTile >= BT * BT * 2, "staging fits in the freed operand tiles");
};

// One CTA per (key tile kt, query tile qt, head): S = Q K^T and dP = dO V^T
// (tensor memory columns 0-127 and 128-255), then P and dS as bf16 tiles.
template <int D>
__global__ void __launch_bounds__(128) matbwd_scores_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
    const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmdS, const Problem p,
    const float *__restrict__ LSE, const float *__restrict__ Dv) {
    using C = ScoresCfg<D>;
    const int kt = blockIdx.x, qt = blockIdx.y, head = blockIdx.z;
    const int nb = p.N / BT;
    if (p.mask && p.mask[(size_t)qt * nb + kt] == 0) return;  // removed block: never written, never read
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t bar_ld = smem_addr(sm + C::kBarOff), bar_mma = bar_ld + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kBarOff + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kBarOff + 24);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t sQ = smem_addr(sm + C::kQOff), sK = smem_addr(sm + C::kKOff);
    const uint32_t sdO = smem_addr(sm + C::kdOOff), sV = smem_addr(sm + C::kVOff);
    const int q0 = head * p.N + qt * BT, k0 = head * p.N + kt * BT;
    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_ld, 4 * C::kTile);
        for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(sQ + c * C::kSlab, &tmQ, c * 64, q0, bar_ld);
            tma_load_2d(sK + c * C::kSlab, &tmK, c * 64, k0, bar_ld);
            tma_load_2d(sdO + c * C::kSlab, &tmdO, c * 64, q0, bar_ld);
            tma_load_2d(sV + c * C::kSlab, &tmV, c * 64, k0, bar_ld);
        }
    }
    bool ok = mbar_wait(bar_ld, 0, abort_flag, p.dev_status);
    if (tid == 0 && ok) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16_f32(BT, BT, false, false);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * C::kSlab + (ks & 3) * 32;
            mma_ss(tmem, smem_desc_sw128(sQ + off, 16, 1024), smem_desc_sw128(sK + off, 16, 1024), id, ks > 0);
            mma_ss(tmem + 128, smem_desc_sw128(sdO + off, 16, 1024), smem_desc_sw128(sV + off, 16, 1024), id, ks > 0);
        }
        mma_commit(bar_mma);
    }
    ok = ok && mbar_wait(bar_mma, 0, abort_flag, p.dev_status);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
        const float sl2 = p.scale * kLog2e;
        const float l2 = LSE[q0 + tid] * kLog2e;
        const float dd = Dv[q0 + tid];
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
        for (int c0 = 0; c0 < BT; c0 += 32) {
            uint32_t sr[32], pr[32];
            tmem_ld32(lane_base + c0, sr);
            tmem_ld32(lane_base + 128 + c0, pr);
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
                const int chunk = ((c0 % 64) / 8) + v;
                const uint32_t off = slab * C::kSlab + tid * 128 + ((chunk ^ (tid & 7)) * 16);
                *reinterpret_cast<uint4 *>(sm + C::kPStage + off) = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                *reinterpret_cast<uint4 *>(sm + C::kdSStage + off) = make_uint4(dk[4 * v], dk[4 * v + 1], dk[4 * v + 2], dk[4 * v + 3]);
            }
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        const uint32_t ps = smem_addr(sm + C::kPStage), ds = smem_addr(sm + C::kdSStage);
        tma_store_2d(&tmP, kt * BT, q0, ps);
        tma_store_2d(&tmP, kt * BT + 64, q0, ps + C::kSlab);
        tma_store_2d(&tmdS, kt * BT, q0, ds);
        tma_store_2d(&tmdS, kt * BT + 64, q0, ds + C::kSlab);
        bulk_commit();
        bulk_wait_all();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
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
        ks<<<dim3(p.N / BT, p.N / BT, p.B * p.H), 128, ScoresCfg<D>::kSmemBytes, st>>>(m.q, m.k, m.v, m.dO, m.p,
                                                                                      m.ds, p, LSE, Dv);
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
