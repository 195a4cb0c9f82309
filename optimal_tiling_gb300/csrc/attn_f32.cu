// fp32 SIMT attention (true fp32 FFMA, no tensor cores): forward and recompute
// backward for any N and 1 <= d <= 256.
//
// Forward follows the stabilised online update of "The I/O Complexity of
// Attention" exposition (blog.aeilot.top, attention-io-complexity), section
// "Softmax without storing the score matrix": keys are visited in blocks of 32,
// each row keeps its running max m, sum l and accumulator u, and o = u / l.
// Backward is the chain rule of the same definition (the pass studied by "On
// Fine-Grained I/O Complexity of Attention Backward Passes"), split into a
// query-row kernel (dQ) and a key-row kernel (dK, dV) so that no two threads
// ever add into the same output.
//
// One warp owns one output row; lane t holds dimensions t, t+32, ... of it.
// Blocks of 4 warps stage 32 rows of the streamed operand in shared memory
// (padded by one float so that the per-lane dot products hit distinct banks).
#include <math.h>

#include "internal.h"

namespace attn {
namespace {

constexpr int kWarps = 4;       // output rows per block
constexpr int kChunk = 32;      // streamed rows per stage (one per lane)
constexpr int kMaxDPL = 8;      // dimensions per lane: d <= 256

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Mask entry of (query qi, key kj) in one head's [nb][nb] block mask.  Every
// 32-key chunk and every 4-row query group lies inside one block (64 or 128).
__device__ __forceinline__ bool block_kept(const uint8_t *mask, int nb, int block, int qi, int kj) {
    return mask == nullptr || mask[(size_t)(qi / block) * nb + kj / block] != 0;
}

// Stage rows [r0, r0+32) of X (one head, [N][d]) into S[32][ld]; rows past N are zero.
__device__ __forceinline__ void stage_rows(float *S, int ld, const float *X, int r0, int N, int d) {
    for (int t = threadIdx.x; t < kChunk * d; t += blockDim.x) {
        int rr = t / d, c = t - rr * d;
        int r = r0 + rr;
        S[rr * ld + c] = r < N ? X[(size_t)r * d + c] : 0.f;
    }
}

__global__ void __launch_bounds__(kWarps * 32)
fwd_f32_kernel(Problem p, const float *__restrict__ Q, const float *__restrict__ K,
               const float *__restrict__ V, float *__restrict__ O, float *__restrict__ LSE) {
    extern __shared__ float sm[];
    const int N = p.N, d = p.d, ld = d + 1;
    float *Ks = sm;                  // [32][d+1]
    float *Vs = Ks + kChunk * ld;    // [32][d+1]
    float *Qs = Vs + kChunk * ld;    // [4][d]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * kWarps, i = row0 + warp;
    const size_t hb = (size_t)blockIdx.y * N * d;
    const int nb = p.mask_nb();
    const uint8_t *hmask = p.head_mask(blockIdx.y);

    for (int t = threadIdx.x; t < kWarps * d; t += blockDim.x) {
        int r = row0 + t / d;
        Qs[t] = r < N ? Q[hb + (size_t)r * d + t % d] : 0.f;
    }
    float u[kMaxDPL];
#pragma unroll
    for (int r = 0; r < kMaxDPL; ++r) u[r] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int j0 = 0; j0 < N; j0 += kChunk) {
        if (!block_kept(hmask, nb, p.mask_block, row0, j0)) continue;  // same for the whole block
        __syncthreads();
        stage_rows(Ks, ld, K + hb, j0, N, d);
        stage_rows(Vs, ld, V + hb, j0, N, d);
        __syncthreads();
        const int j = j0 + lane;
        float sj = -INFINITY;
        if (j < N && i < N) {
            float acc = 0.f;
            for (int c = 0; c < d; ++c) acc = fmaf(Qs[warp * d + c], Ks[lane * ld + c], acc);
            sj = p.scale * acc;
        }
        const float mnew = fmaxf(m, warp_max(sj));
        if (mnew == -INFINITY) continue;
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - mnew);
        const float pj = (sj == -INFINITY) ? 0.f : expf(sj - mnew);
        l = alpha * l + warp_sum(pj);
#pragma unroll
        for (int r = 0; r < kMaxDPL; ++r) u[r] *= alpha;
        for (int jj = 0; jj < kChunk; ++jj) {
            const float pjj = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
            for (int r = 0; r < kMaxDPL; ++r) {
                const int c = lane + 32 * r;
                if (c < d) u[r] = fmaf(pjj, Vs[jj * ld + c], u[r]);
            }
        }
        m = mnew;
    }
    if (i < N) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int r = 0; r < kMaxDPL; ++r) {
            const int c = lane + 32 * r;
            if (c < d) O[hb + (size_t)i * d + c] = u[r] * inv;
        }
        if (lane == 0) LSE[(size_t)blockIdx.y * N + i] = l > 0.f ? m + logf(l) : -INFINITY;
    }
}

// D_i = sum_t dO_it O_it (one warp per row).
__global__ void __launch_bounds__(kWarps * 32)
bwd_f32_rowdot_kernel(Problem p, const float *__restrict__ O, const float *__restrict__ dO,
                      float *__restrict__ D) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * kWarps + warp;
    if (i >= p.N) return;
    const size_t base = ((size_t)blockIdx.y * p.N + i) * p.d;
    float acc = 0.f;
    for (int c = lane; c < p.d; c += 32) acc = fmaf(dO[base + c], O[base + c], acc);
    acc = warp_sum(acc);
    if (lane == 0) D[(size_t)blockIdx.y * p.N + i] = acc;
}

// dQ_i = s sum_j P_ij (dP_ij - D_i) k_j, one warp per query row.
__global__ void __launch_bounds__(kWarps * 32)
bwd_f32_dq_kernel(Problem p, const float *__restrict__ Q, const float *__restrict__ K,
                  const float *__restrict__ V, const float *__restrict__ dO,
                  const float *__restrict__ LSE, const float *__restrict__ D,
                  float *__restrict__ dQ) {
    extern __shared__ float sm[];
    const int N = p.N, d = p.d, ld = d + 1;
    float *Ks = sm;                   // [32][d+1]
    float *Vs = Ks + kChunk * ld;     // [32][d+1]
    float *Qs = Vs + kChunk * ld;     // [4][d]
    float *dOs = Qs + kWarps * d;     // [4][d]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * kWarps, i = row0 + warp;
    const size_t hb = (size_t)blockIdx.y * N * d;
    const int nb = p.mask_nb();
    const uint8_t *hmask = p.head_mask(blockIdx.y);
    for (int t = threadIdx.x; t < kWarps * d; t += blockDim.x) {
        int r = row0 + t / d;
        Qs[t] = r < N ? Q[hb + (size_t)r * d + t % d] : 0.f;
        dOs[t] = r < N ? dO[hb + (size_t)r * d + t % d] : 0.f;
    }
    const float Li = i < N ? LSE[(size_t)blockIdx.y * N + i] : -INFINITY;
    const float Di = i < N ? D[(size_t)blockIdx.y * N + i] : 0.f;
    float acc[kMaxDPL];
#pragma unroll
    for (int r = 0; r < kMaxDPL; ++r) acc[r] = 0.f;
    for (int j0 = 0; j0 < N; j0 += kChunk) {
        if (!block_kept(hmask, nb, p.mask_block, row0, j0)) continue;
        __syncthreads();
        stage_rows(Ks, ld, K + hb, j0, N, d);
        stage_rows(Vs, ld, V + hb, j0, N, d);
        __syncthreads();
        const int j = j0 + lane;
        float dS = 0.f;
        if (j < N && Li != -INFINITY) {
            float s = 0.f, dp = 0.f;
            for (int c = 0; c < d; ++c) {
                s = fmaf(Qs[warp * d + c], Ks[lane * ld + c], s);
                dp = fmaf(dOs[warp * d + c], Vs[lane * ld + c], dp);
            }
            const float P = expf(p.scale * s - Li);
            dS = P * (dp - Di);
        }
        for (int jj = 0; jj < kChunk; ++jj) {
            const float w = __shfl_sync(0xffffffffu, dS, jj);
#pragma unroll
            for (int r = 0; r < kMaxDPL; ++r) {
                const int c = lane + 32 * r;
                if (c < d) acc[r] = fmaf(w, Ks[jj * ld + c], acc[r]);
            }
        }
    }
    if (i < N) {
#pragma unroll
        for (int r = 0; r < kMaxDPL; ++r) {
            const int c = lane + 32 * r;
            if (c < d) dQ[hb + (size_t)i * d + c] = p.scale * acc[r];
        }
    }
}

// dV_j = sum_i P_ij dO_i and dK_j = s sum_i dS_ij q_i, one warp per key row.
__global__ void __launch_bounds__(kWarps * 32)
bwd_f32_dkv_kernel(Problem p, const float *__restrict__ Q, const float *__restrict__ K,
                   const float *__restrict__ V, const float *__restrict__ dO,
                   const float *__restrict__ LSE, const float *__restrict__ D,
                   float *__restrict__ dK, float *__restrict__ dV) {
    extern __shared__ float sm[];
    const int N = p.N, d = p.d, ld = d + 1;
    float *Qs = sm;                    // [32][d+1]
    float *dOs = Qs + kChunk * ld;     // [32][d+1]
    float *Ks = dOs + kChunk * ld;     // [4][d]
    float *Vs = Ks + kWarps * d;       // [4][d]
    float *Ls = Vs + kWarps * d;       // [32]
    float *Ds = Ls + kChunk;           // [32]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = blockIdx.x * kWarps, j = col0 + warp;
    const size_t hb = (size_t)blockIdx.y * N * d;
    const int nb = p.mask_nb();
    const uint8_t *hmask = p.head_mask(blockIdx.y);
    for (int t = threadIdx.x; t < kWarps * d; t += blockDim.x) {
        int r = col0 + t / d;
        Ks[t] = r < N ? K[hb + (size_t)r * d + t % d] : 0.f;
        Vs[t] = r < N ? V[hb + (size_t)r * d + t % d] : 0.f;
    }
    float ak[kMaxDPL], av[kMaxDPL];
#pragma unroll
    for (int r = 0; r < kMaxDPL; ++r) { ak[r] = 0.f; av[r] = 0.f; }
    for (int i0 = 0; i0 < N; i0 += kChunk) {
        if (!block_kept(hmask, nb, p.mask_block, i0, col0)) continue;
        __syncthreads();
        stage_rows(Qs, ld, Q + hb, i0, N, d);
        stage_rows(dOs, ld, dO + hb, i0, N, d);
        if (threadIdx.x < kChunk) {
            const int ii = i0 + threadIdx.x;
            Ls[threadIdx.x] = ii < N ? LSE[(size_t)blockIdx.y * N + ii] : -INFINITY;
            Ds[threadIdx.x] = ii < N ? D[(size_t)blockIdx.y * N + ii] : 0.f;
        }
        __syncthreads();
        float P = 0.f, dS = 0.f;
        if (j < N && Ls[lane] != -INFINITY) {
            float s = 0.f, dp = 0.f;
            for (int c = 0; c < d; ++c) {
                s = fmaf(Qs[lane * ld + c], Ks[warp * d + c], s);
                dp = fmaf(dOs[lane * ld + c], Vs[warp * d + c], dp);
            }
            P = expf(p.scale * s - Ls[lane]);
            dS = P * (dp - Ds[lane]);
        }
        for (int ii = 0; ii < kChunk; ++ii) {
            const float wp = __shfl_sync(0xffffffffu, P, ii);
            const float ws = __shfl_sync(0xffffffffu, dS, ii);
#pragma unroll
            for (int r = 0; r < kMaxDPL; ++r) {
                const int c = lane + 32 * r;
                if (c < d) {
                    av[r] = fmaf(wp, dOs[ii * ld + c], av[r]);
                    ak[r] = fmaf(ws, Qs[ii * ld + c], ak[r]);
                }
            }
        }
    }
    if (j < N) {
#pragma unroll
        for (int r = 0; r < kMaxDPL; ++r) {
            const int c = lane + 32 * r;
            if (c < d) {
                dK[hb + (size_t)j * d + c] = p.scale * ak[r];
                dV[hb + (size_t)j * d + c] = av[r];
            }
        }
    }
}

}  // namespace

cudaError_t launch_fwd_f32(const Problem &p, const float *Q, const float *K, const float *V,
                           float *O, float *LSE, cudaStream_t st) {
    const size_t smem = (size_t)(2 * kChunk * (p.d + 1) + kWarps * p.d) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(fwd_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + kWarps - 1) / kWarps, p.B * p.H);
    {
        ProfScope prof_("fwd_f32", st);
        fwd_f32_kernel<<<grid, kWarps * 32, smem, st>>>(p, Q, K, V, O, LSE);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_f32(const Problem &p, const float *Q, const float *K, const float *V,
                           const float *O, const float *dO, const float *LSE, float *dQ,
                           float *dK, float *dV, float *D, cudaStream_t st) {
    dim3 grid((p.N + kWarps - 1) / kWarps, p.B * p.H);
    {
        ProfScope prof_("bwd_f32_rowdot", st);
        bwd_f32_rowdot_kernel<<<grid, kWarps * 32, 0, st>>>(p, O, dO, D);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem_q = (size_t)(2 * kChunk * (p.d + 1) + 2 * kWarps * p.d) * sizeof(float);
    e = cudaFuncSetAttribute(bwd_f32_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q);
    if (e != cudaSuccess) return e;
    {
        ProfScope prof_("bwd_f32_dq", st);
        bwd_f32_dq_kernel<<<grid, kWarps * 32, smem_q, st>>>(p, Q, K, V, dO, LSE, D, dQ);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem_k = (size_t)(2 * kChunk * (p.d + 1) + 2 * kWarps * p.d + 2 * kChunk) * sizeof(float);
    e = cudaFuncSetAttribute(bwd_f32_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_k);
    if (e != cudaSuccess) return e;
    {
        ProfScope prof_("bwd_f32_dkv", st);
        bwd_f32_dkv_kernel<<<grid, kWarps * 32, smem_k, st>>>(p, Q, K, V, dO, LSE, D, dK, dV);
    }
    return cudaGetLastError();
}

}  // namespace attn
