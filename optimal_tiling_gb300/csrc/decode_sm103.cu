// Decode-shaped attention: Nq (1..16) queries against Nk keys per head, no mask.
//
// "The I/O Complexity of Attention" exposition (blog.aeilot.top,
// attention-io-complexity), end of "From a movement lower bound to a
// performance upper bound": single-token decoding has query length one, so its
// cost is not an N^2 formula; it needs a rectangular account and the location
// of the existing K/V state.  Here K and V live in HBM and every element of
// them is read exactly once, so the pass is bound by HBM bandwidth
// (2 Nk d w bytes per head against 4 Nq Nk d FLOPs: ~Nq FLOP per byte), and
// it runs on the CUDA cores, not the tensor cores.
//
// Two kernels:
//   decode_split: the key range of each head is cut into splits (enough CTAs to
//     fill the GPU); a CTA streams its split in groups of 32 keys per warp, each
//     lane scoring one key against all queries (q pre-scaled by s log2 e, fp32
//     accumulation), and keeps per query the running max m, sum l and
//     unnormalised output u (lane t owns output columns t, t+32, ...) -- the
//     online update of the page's section "Softmax without storing the score
//     matrix".  The four warps' states are merged in shared memory and the
//     CTA writes (u, m, l) of its split.
//   decode_merge: for each (head, query) the splits are merged with the same
//     rule (m' = max m_s, l' = sum e^{m_s - m'} l_s, u' likewise), o = u'/l',
//     LSE = (m' + log2 l') ln 2.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kWarps = 4;
constexpr int kGroup = 32;  // keys per warp step (one per lane)

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Partial state layout per (head, split, query): [u_0 .. u_{D-1}, m, l] fp32.
template <int D>
__device__ __forceinline__ size_t part_index(int head, int split, int q, int splits, int nq) {
    return (((size_t)head * splits + split) * nq + q) * (D + 2);
}

template <int D, int NQ>
__global__ void __launch_bounds__(kWarps * 32)
decode_split_kernel(const __nv_bfloat16 *__restrict__ Q, const __nv_bfloat16 *__restrict__ K,
                    const __nv_bfloat16 *__restrict__ V, float *__restrict__ part, int Nq, int Nk, float scale,
                    int keys_per_split, int splits) {
    constexpr int DPL = D / 32;  // output columns per lane
    extern __shared__ float dsm[];
    float(*qs)[D] = reinterpret_cast<float(*)[D]>(dsm);                      // [NQ][D]
    float(*st_u)[NQ][D] = reinterpret_cast<float(*)[NQ][D]>(dsm + NQ * D);   // [kWarps][NQ][D]
    float(*st_m)[NQ] = reinterpret_cast<float(*)[NQ]>(dsm + (1 + kWarps) * NQ * D);
    float(*st_l)[NQ] = reinterpret_cast<float(*)[NQ]>(dsm + (1 + kWarps) * NQ * D + kWarps * NQ);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, head = blockIdx.y;
    const float sl2 = scale * kLog2e;
    for (int t = threadIdx.x; t < NQ * D; t += blockDim.x) {
        const int q = t / D, c = t % D;
        qs[q][c] = q < Nq ? __bfloat162float(Q[((size_t)head * Nq + q) * D + c]) * sl2 : 0.f;
    }
    __syncthreads();

    float m[NQ], l[NQ], u[NQ][DPL];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        m[q] = -INFINITY;
        l[q] = 0.f;
#pragma unroll
        for (int c = 0; c < DPL; ++c) u[q][c] = 0.f;
    }
    const int k_begin = split * keys_per_split;
    const int k_end = min(Nk, k_begin + keys_per_split);
    const __nv_bfloat16 *Kh = K + (size_t)head * Nk * D;
    const __nv_bfloat16 *Vh = V + (size_t)head * Nk * D;
    for (int g0 = k_begin + warp * kGroup; g0 < k_end; g0 += kWarps * kGroup) {
        const int j = g0 + lane;
        const bool valid = j < k_end;
        // scores of key j against every query, 8 columns (16 bytes) at a time
        float sc[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) sc[q] = 0.f;
        if (valid) {
            const uint4 *krow = reinterpret_cast<const uint4 *>(Kh + (size_t)j * D);
#pragma unroll 4
            for (int c8 = 0; c8 < D / 8; ++c8) {
                // every lane reads the same q columns (a shared-memory broadcast) and its own
                // key row; the row's remaining bytes are L1 hits for the next column blocks
                const uint4 kv = __ldg(krow + c8);
                const __nv_bfloat162 *kp = reinterpret_cast<const __nv_bfloat162 *>(&kv);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 kf = __bfloat1622float2(kp[e]);
#pragma unroll
                    for (int q = 0; q < NQ; ++q)
                        sc[q] = fmaf(qs[q][c8 * 8 + 2 * e], kf.x, fmaf(qs[q][c8 * 8 + 2 * e + 1], kf.y, sc[q]));
                }
            }
        }
        float pj[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const float s = valid ? sc[q] : -INFINITY;
            const float m_new = fmaxf(m[q], warp_max(s));  // finite: the group has at least one valid key
            const float alpha = ex2(m[q] - m_new);         // 0 while m was -inf
            pj[q] = valid ? ex2(s - m_new) : 0.f;
            l[q] = l[q] * alpha + warp_sum(pj[q]);
#pragma unroll
            for (int c = 0; c < DPL; ++c) u[q][c] *= alpha;
            m[q] = m_new;
        }
        // u_q += sum over the group's keys of p_qj v_j (lane owns columns lane, lane+32, ...)
        const int nvalid = min(kGroup, k_end - g0);
        for (int jj = 0; jj < nvalid; ++jj) {
            const __nv_bfloat16 *vrow = Vh + (size_t)(g0 + jj) * D;
            float vv[DPL];
#pragma unroll
            for (int c = 0; c < DPL; ++c) vv[c] = __bfloat162float(vrow[lane + 32 * c]);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float w = __shfl_sync(0xffffffffu, pj[q], jj);
#pragma unroll
                for (int c = 0; c < DPL; ++c) u[q][c] = fmaf(w, vv[c], u[q][c]);
            }
        }
    }
    // merge the four warps' states
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
#pragma unroll
        for (int c = 0; c < DPL; ++c) st_u[warp][q][lane + 32 * c] = u[q][c];
        if (lane == 0) {
            st_m[warp][q] = m[q];
            st_l[warp][q] = l[q];
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < NQ * D; t += blockDim.x) {
        const int q = t / D, c = t % D;
        if (q >= Nq) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, st_m[w][q]);
        float uu = 0.f, ll = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float a = ex2(st_m[w][q] - M);
                uu = fmaf(a, st_u[w][q][c], uu);
                ll = fmaf(a, st_l[w][q], ll);
            }
        }
        float *dst = part + part_index<D>(head, split, q, splits, Nq);
        dst[c] = uu;
        if (c == 0) {
            dst[D] = M;
            dst[D + 1] = ll;
        }
    }
}

// One warp per (head, query): merge the splits, normalise, store O (bf16) and LSE.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const float *__restrict__ part,
                                                           __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE,
                                                           int heads, int Nq, int splits) {
    constexpr int DPL = D / 32;
    const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= heads * Nq) return;
    const int head = gw / Nq, q = gw % Nq;
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, part[part_index<D>(head, s, q, splits, Nq) + D]);
    float uu[DPL], L = 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) uu[c] = 0.f;
    for (int s = 0; s < splits; ++s) {
        const float *src = part + part_index<D>(head, s, q, splits, Nq);
        const float a = ex2(src[D] - M);  // 0 for an empty split (m = -inf)
        L = fmaf(a, src[D + 1], L);
#pragma unroll
        for (int c = 0; c < DPL; ++c) uu[c] = fmaf(a, src[lane + 32 * c], uu[c]);
    }
    const float inv = 1.f / L;
    __nv_bfloat16 *orow = O + ((size_t)head * Nq + q) * D;
#pragma unroll
    for (int c = 0; c < DPL; ++c) orow[lane + 32 * c] = __float2bfloat16_rn(uu[c] * inv);
    if (lane == 0) LSE[(size_t)head * Nq + q] = (M + __log2f(L)) * kLn2;
}

template <int D, int NQ>
cudaError_t launch_dq(const DecodeShape &sh, const void *Q, const void *K, const void *V, void *O, float *LSE,
                      float *part, cudaStream_t st) {
    const int heads = sh.B * sh.H;
    const size_t smem = ((size_t)(1 + kWarps) * NQ * D + 2 * kWarps * NQ) * sizeof(float);
    auto kern = decode_split_kernel<D, NQ>;
    cudaError_t e0 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e0 != cudaSuccess) return e0;
    {
        ProfScope prof_("decode_split", st);
        kern<<<dim3(sh.splits, heads), kWarps * 32, smem, st>>>(
            static_cast<const __nv_bfloat16 *>(Q), static_cast<const __nv_bfloat16 *>(K),
            static_cast<const __nv_bfloat16 *>(V), part, sh.Nq, sh.Nk, sh.scale, sh.keys_per_split, sh.splits);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    {
        ProfScope prof_("decode_merge", st);
        decode_merge_kernel<D><<<(heads * sh.Nq + 3) / 4, 128, 0, st>>>(part, static_cast<__nv_bfloat16 *>(O), LSE,
                                                                      heads, sh.Nq, sh.splits);
    }
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeShape &sh, const void *Q, const void *K, const void *V, void *O, float *LSE,
                     float *part, cudaStream_t st) {
    if (sh.Nq <= 1) return launch_dq<D, 1>(sh, Q, K, V, O, LSE, part, st);
    if (sh.Nq <= 2) return launch_dq<D, 2>(sh, Q, K, V, O, LSE, part, st);
    if (sh.Nq <= 4) return launch_dq<D, 4>(sh, Q, K, V, O, LSE, part, st);
    if (sh.Nq <= 8) return launch_dq<D, 8>(sh, Q, K, V, O, LSE, part, st);
    return launch_dq<D, 16>(sh, Q, K, V, O, LSE, part, st);
}

}  // namespace

DecodeShape decode_shape(int B, int H, int Nq, int Nk, int d, float scale) {
    DecodeShape sh{B, H, Nq, Nk, d, scale, 1, Nk};
    const int heads = B * H;
    // enough CTAs to fill the GPU four times over, each split at least one group per warp
    const int want = std::max(1, (4 * 152 + heads - 1) / heads);
    const int max_splits = std::max(1, (Nk + kWarps * kGroup - 1) / (kWarps * kGroup));
    sh.splits = std::min(want, max_splits);
    const int per = (Nk + sh.splits - 1) / sh.splits;
    sh.keys_per_split = (per + kGroup - 1) / kGroup * kGroup;
    sh.splits = (Nk + sh.keys_per_split - 1) / sh.keys_per_split;
    return sh;
}

size_t decode_workspace_bytes(const DecodeShape &sh) {
    return (size_t)sh.B * sh.H * sh.splits * sh.Nq * (sh.d + 2) * sizeof(float);
}

cudaError_t launch_decode_bf16(const DecodeShape &sh, const void *Q, const void *K, const void *V, void *O,
                               float *LSE, float *part, cudaStream_t st) {
    switch (sh.d) {
        case 64: return launch_d<64>(sh, Q, K, V, O, LSE, part, st);
        case 128: return launch_d<128>(sh, Q, K, V, O, LSE, part, st);
        case 256: return launch_d<256>(sh, Q, K, V, O, LSE, part, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace attn
