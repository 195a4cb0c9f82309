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
//   decode_split: one persistent CTA per SM.  The 32-key steps of all heads,
//     taken in order (head by head), are cut into one contiguous equal range
//     per CTA, so every SM streams the same number of bytes and there is no
//     partial last wave; a range can start and end inside a head.  A producer
//     warp streams the range's K and V rows with TMA, step by step, into a ring
//     of shared-memory stages per consumer warp (~190 KB in flight per SM),
//     running on across head boundaries; six consumer warps (three at d = 256)
//     keep up with HBM.  Each consumer warp scores its step with one lane per
//     key against all queries (q pre-scaled by s log2 e, fp32 accumulation) and
//     keeps per query the running max m, sum l and unnormalised output u (lane t
//     owns output columns [t*d/32, (t+1)*d/32)) -- the online update of the
//     page's section "Softmax without storing the score matrix".  The 128-byte
//     TMA swizzle makes both the per-key row reads and the per-column V reads
//     conflict-free.  At the end of each head segment of its range the CTA
//     merges the warps' states in shared memory and writes (u, m, l) of the
//     segment.
//   decode_merge: for each (head, query) the segments of the CTAs whose ranges
//     meet the head are merged with the same rule (m' = max m_s,
//     l' = sum e^{m_s - m'} l_s, u' likewise), o = u'/l', LSE = (m' + log2 l') ln 2.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kGroup = 32;  // keys per warp step (one per lane)

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Partial state layout per (CTA, segment, query): [u_0 .. u_{D-1}, m, l] fp32.
template <int D>
__device__ __forceinline__ size_t part_index(int cta, int seg, int q, int max_seg, int nq) {
    return (((size_t)cta * max_seg + seg) * nq + q) * (D + 2);
}

// First global step of CTA c when S steps are cut into C equal contiguous ranges.
__host__ __device__ __forceinline__ long long range_begin(int c, long long S, int C) {
    return (long long)c * S / C;
}

// Shared-memory plan of decode_split: per consumer warp a ring of NS stages, each
// stage one 32-key step: the K rows and V rows of the step as 64-column slabs of
// 32 rows x 128 bytes in the 128-byte-swizzled TMA layout (16-byte chunk c of row
// r at chunk c ^ (r % 8)), then q (fp32, pre-scaled), the warps' final states and
// the barriers.
template <int D, int NQ>
struct DecCfg {
    // consumer warps: as many as leave two ring stages each.  Measured on the 8 x 32 x 32768
    // workload: the per-step scoring and V accumulation of a warp, not the bytes in flight,
    // set the pace (4 -> 6 warps at d = 128: 0.749 -> 0.632 ms; 2 -> 3 at d = 256:
    // 1.149 -> 0.765 ms).  More queries per step need the registers and shared memory of
    // the narrower configuration.
    static constexpr int kConsumers = NQ > 4 ? (D == 256 ? 2 : 4) : (D == 256 ? 3 : 6);
    static constexpr int kSlab = kGroup * 128;                        // 4 KB: 32 rows x 64 columns
    static constexpr int kTile = kGroup * D * 2;                      // K (or V) rows of one step
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kRest = NQ * D * 4 + kConsumers * NQ * (D + 2) * 4 + 4096;  // q, states, barriers
    static constexpr int kRingBudget = 220 * 1024 - kRest;
    static constexpr int kStages = kRingBudget / (kConsumers * kStageBytes) > 6 ? 6
                                                                                : kRingBudget / (kConsumers * kStageBytes);
    static constexpr int kRingOff = 0;
    static constexpr int kQOff = kConsumers * kStages * kStageBytes;
    static constexpr int kStOff = kQOff + NQ * D * 4;                 // [warps][NQ][D] u, then m, l
    static constexpr int kBarOff = kStOff + (kConsumers * NQ * (D + 2)) * 4;
    static constexpr int kBarBytes = 2 * kConsumers * kStages * 8;
    static constexpr int kSmemBytes = ((kBarOff + kBarBytes + 64) + 1023) / 1024 * 1024 + 1024;
    static constexpr int kThreads = (kConsumers + 1) * 32;            // + one producer warp
    static_assert(kStages >= 2, "at least double buffering");
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

template <int D, int NQ>
__global__ void __launch_bounds__(DecCfg<D, NQ>::kThreads, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __nv_bfloat16 *__restrict__ Q, float *__restrict__ part, int Nq, int Nk, float scale,
                    int sph, long long S, int max_seg, int *dev_status) {
    using C = DecCfg<D, NQ>;
    constexpr int W = C::kConsumers, NS = C::kStages;
    constexpr int DPL = D / 32;  // output columns per lane: lane owns [lane*DPL, lane*DPL + DPL)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float(*qs)[D] = reinterpret_cast<float(*)[D]>(sm + C::kQOff);
    float *st = reinterpret_cast<float *>(sm + C::kStOff);
    const uint32_t bar0 = smem_addr(sm + C::kBarOff);
    auto full = [&](int w, int s) { return bar0 + 8u * (w * NS + s); };
    auto empty = [&](int w, int s) { return bar0 + 8u * (W * NS + w * NS + s); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kBarOff + C::kBarBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const float sl2 = scale * kLog2e;
    const long long sb = range_begin(cta, S, gridDim.x), se = range_begin(cta + 1, S, gridDim.x);
    const int nloc = (int)(se - sb);             // steps of this CTA's range
    const int first_head = (int)(sb / sph);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < W * NS; ++i) {
            mbar_init(bar0 + 8u * i, 1);             // full: the producer's expect_tx
            mbar_init(bar0 + 8u * (W * NS + i), 1);  // empty: lane 0 of the consumer warp
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == W) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            for (int t = 0; t < nloc; ++t) {
                const int w = t % W, s = (t / W) % NS, use = t / (W * NS);
                if (use > 0 && !mbar_wait(empty(w, s), (uint32_t)(use - 1) & 1u, abort_flag, dev_status)) break;
                const uint32_t kb = smem_addr(sm + C::kRingOff) + (uint32_t)((w * NS + s) * C::kStageBytes);
                const long long g = sb + t;
                // rows past this head's keys (a ragged last step) belong to the next head or lie
                // past the tensor (zero fill); the consumers give them no weight
                const int row = (int)(g / sph) * Nk + (int)(g % sph) * kGroup;
                mbar_arrive_expect_tx(full(w, s), C::kStageBytes);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_2d(kb + c * C::kSlab, &tmK, c * 64, row, full(w, s));
                    tma_load_2d(kb + C::kTile + c * C::kSlab, &tmV, c * 64, row, full(w, s));
                }
            }
        }
        return;  // the consumers' named barriers do not include this warp
    }
    // ---------------------------------------------------------------- consumers
    // Every consumer thread runs the same sequence of named barriers (the head segments of
    // the range are fixed); after a failed wait the work is skipped but the barriers kept.
    bool alive = true;
    int t = warp;  // next local step of this warp
    for (long long g0 = sb; g0 < se;) {
        const int head = (int)(g0 / sph);
        const long long g1 = min(se, (long long)(head + 1) * sph);
        for (int i = threadIdx.x; i < NQ * D; i += W * 32) {
            const int q = i / D, c = i % D;
            qs[q][c] = q < Nq ? __bfloat162float(Q[((size_t)head * Nq + q) * D + c]) * sl2 : 0.f;
        }
        named_bar_sync(1, W * 32);
        float m[NQ], l[NQ], u[NQ][DPL];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            m[q] = -INFINITY;
            l[q] = 0.f;
#pragma unroll
            for (int c = 0; c < DPL; ++c) u[q][c] = 0.f;
        }
        for (; sb + t < g1; t += W) {
            const int s = (t / W) % NS, use = t / (W * NS);
            bool ok = alive && mbar_wait(full(warp, s), (uint32_t)use & 1u, abort_flag, dev_status);
            alive = __all_sync(0xffffffffu, ok);
            if (!alive) continue;
            const uint8_t *kt = sm + C::kRingOff + (warp * NS + s) * C::kStageBytes;
            const uint8_t *vt = kt + C::kTile;
            const int key0 = (int)((sb + t) % sph) * kGroup;  // first key of the step within the head
            const bool valid = key0 + lane < Nk;
            // scores: lane = key (row `lane` of the step); q columns are a broadcast
            float sc[NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) sc[q] = 0.f;
#pragma unroll 2
            for (int c8 = 0; c8 < D / 8; ++c8) {
                const int slab = c8 >> 3, chunk = c8 & 7;
                const uint4 kv = *reinterpret_cast<const uint4 *>(kt + slab * C::kSlab + lane * 128 +
                                                                  ((chunk ^ (lane & 7)) << 4));
                const __nv_bfloat162 *kp = reinterpret_cast<const __nv_bfloat162 *>(&kv);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 kf = __bfloat1622float2(kp[e]);
#pragma unroll
                    for (int q = 0; q < NQ; ++q)
                        sc[q] = fmaf(qs[q][c8 * 8 + 2 * e], kf.x, fmaf(qs[q][c8 * 8 + 2 * e + 1], kf.y, sc[q]));
                }
            }
            float pj[NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float sv = valid ? sc[q] : -INFINITY;
                const float m_new = fmaxf(m[q], warp_max(sv));  // finite: the step holds a valid key
                const float alpha = ex2(m[q] - m_new);
                pj[q] = valid ? ex2(sv - m_new) : 0.f;
                l[q] = l[q] * alpha + warp_sum(pj[q]);
#pragma unroll
                for (int c = 0; c < DPL; ++c) u[q][c] *= alpha;
                m[q] = m_new;
            }
            // u_q += sum_j p_qj v_j: lane reads its DPL columns of row j (2*DPL bytes)
            const int nvalid = min(kGroup, Nk - key0);
            const int byte0 = lane * DPL * 2;                 // byte offset of the lane's columns in a row
            const int vslab = byte0 >> 7, vin = byte0 & 127;  // 64-column slab, offset inside its 128 B
            auto accumulate_row = [&](int jj) {
                const int pos = (((vin >> 4) ^ (jj & 7)) << 4) | (vin & 15);
                const uint8_t *vp = vt + vslab * C::kSlab + jj * 128 + pos;
                float vv[DPL];
                if constexpr (DPL == 2) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(vp));
                    vv[0] = f.x;
                    vv[1] = f.y;
                } else if constexpr (DPL == 4) {
                    const uint2 r = *reinterpret_cast<const uint2 *>(vp);
                    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
                    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
                    vv[0] = a.x; vv[1] = a.y; vv[2] = b.x; vv[3] = b.y;
                } else {
                    const uint4 r = *reinterpret_cast<const uint4 *>(vp);
                    const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                        vv[2 * e] = a.x;
                        vv[2 * e + 1] = a.y;
                    }
                }
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const float w = __shfl_sync(0xffffffffu, pj[q], jj);
#pragma unroll
                    for (int c = 0; c < DPL; ++c) u[q][c] = fmaf(w, vv[c], u[q][c]);
                }
            };
            if (nvalid == kGroup) {
#pragma unroll 8
                for (int jj = 0; jj < kGroup; ++jj) accumulate_row(jj);
            } else {
                for (int jj = 0; jj < nvalid; ++jj) accumulate_row(jj);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(warp, s));
        }
        // this warp's state for the merge: u at [warp][q][D], then m, l at [W][NQ][D] + ...
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
#pragma unroll
            for (int c = 0; c < DPL; ++c) st[((size_t)warp * NQ + q) * D + lane * DPL + c] = u[q][c];
            if (lane == 0) {
                st[(size_t)W * NQ * D + warp * NQ + q] = m[q];
                st[(size_t)W * NQ * D + W * NQ + warp * NQ + q] = l[q];
            }
        }
        named_bar_sync(1, W * 32);
        const int seg = head - first_head;
        for (int i = threadIdx.x; i < NQ * D; i += W * 32) {
            const int q = i / D, c = i % D;
            if (q >= Nq) continue;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < W; ++w) M = fmaxf(M, st[(size_t)W * NQ * D + w * NQ + q]);
            float uu = 0.f, ll = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    const float a = ex2(st[(size_t)W * NQ * D + w * NQ + q] - M);
                    uu = fmaf(a, st[((size_t)w * NQ + q) * D + c], uu);
                    ll = fmaf(a, st[(size_t)W * NQ * D + W * NQ + w * NQ + q], ll);
                }
            }
            float *dst = part + part_index<D>(cta, seg, q, max_seg, Nq);
            dst[c] = uu;
            if (c == 0) {
                dst[D] = M;
                dst[D + 1] = ll;
            }
        }
        named_bar_sync(1, W * 32);  // qs and st are rewritten by the next segment
        g0 = g1;
    }
}

// One warp per (head, query): merge the segments of the CTAs whose step ranges meet
// the head, normalise, store O (bf16) and LSE.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const float *__restrict__ part,
                                                           __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE,
                                                           int heads, int Nq, int sph, long long S, int ctas,
                                                           int max_seg) {
    constexpr int DPL = D / 32;
    const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= heads * Nq) return;
    const int head = gw / Nq, q = gw % Nq;
    // CTAs holding the head's first and last steps
    auto owner = [&](long long g) {
        int c = (int)(g * ctas / S);
        while (c + 1 < ctas && range_begin(c + 1, S, ctas) <= g) ++c;
        while (c > 0 && range_begin(c, S, ctas) > g) --c;
        return c;
    };
    const int c_lo = owner((long long)head * sph), c_hi = owner((long long)(head + 1) * sph - 1);
    auto src_of = [&](int c) {
        const int seg = head - (int)(range_begin(c, S, ctas) / sph);
        return part + part_index<D>(c, seg, q, max_seg, Nq);
    };
    float M = -INFINITY;
    for (int c = c_lo; c <= c_hi; ++c) M = fmaxf(M, src_of(c)[D]);
    float uu[DPL], L = 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) uu[c] = 0.f;
    for (int c = c_lo; c <= c_hi; ++c) {
        const float *src = src_of(c);
        const float a = ex2(src[D] - M);
        L = fmaf(a, src[D + 1], L);
#pragma unroll
        for (int k = 0; k < DPL; ++k) uu[k] = fmaf(a, src[lane + 32 * k], uu[k]);
    }
    const float inv = 1.f / L;
    __nv_bfloat16 *orow = O + ((size_t)head * Nq + q) * D;
#pragma unroll
    for (int k = 0; k < DPL; ++k) orow[lane + 32 * k] = __float2bfloat16_rn(uu[k] * inv);
    if (lane == 0) LSE[(size_t)head * Nq + q] = (M + __log2f(L)) * kLn2;
}

template <int D, int NQ>
cudaError_t launch_dq(const DecodeShape &sh, const DecodeMaps &maps, const void *Q, void *O, float *LSE, float *part,
                      int *dev_status, cudaStream_t st) {
    using C = DecCfg<D, NQ>;
    const int heads = sh.B * sh.H;
    auto kern = decode_split_kernel<D, NQ>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    {
        ProfScope prof_("decode_split", st);
        kern<<<sh.ctas, C::kThreads, C::kSmemBytes, st>>>(maps.k, maps.v, static_cast<const __nv_bfloat16 *>(Q),
                                                         part, sh.Nq, sh.Nk, sh.scale, sh.sph, sh.steps, sh.max_seg,
                                                         dev_status);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {
        ProfScope prof_("decode_merge", st);
        decode_merge_kernel<D><<<(heads * sh.Nq + 3) / 4, 128, 0, st>>>(
            part, static_cast<__nv_bfloat16 *>(O), LSE, heads, sh.Nq, sh.sph, sh.steps, sh.ctas, sh.max_seg);
    }
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeShape &sh, const DecodeMaps &m, const void *Q, void *O, float *LSE, float *part,
                     int *dev_status, cudaStream_t st) {
    if (sh.Nq <= 1) return launch_dq<D, 1>(sh, m, Q, O, LSE, part, dev_status, st);
    if (sh.Nq <= 2) return launch_dq<D, 2>(sh, m, Q, O, LSE, part, dev_status, st);
    if (sh.Nq <= 4) return launch_dq<D, 4>(sh, m, Q, O, LSE, part, dev_status, st);
    if (sh.Nq <= 8) return launch_dq<D, 8>(sh, m, Q, O, LSE, part, dev_status, st);
    return launch_dq<D, 16>(sh, m, Q, O, LSE, part, dev_status, st);
}

}  // namespace

DecodeShape decode_shape(int B, int H, int Nq, int Nk, int d, float scale) {
    DecodeShape sh{};
    sh.B = B;
    sh.H = H;
    sh.Nq = Nq;
    sh.Nk = Nk;
    sh.d = d;
    sh.scale = scale;
    // one persistent CTA per SM of the current device
    const int sms = device_sm_count();
    sh.sph = (Nk + kGroup - 1) / kGroup;
    sh.steps = (long long)B * H * sh.sph;
    sh.ctas = (int)std::min<long long>(sms, sh.steps);
    // a range of ceil(steps / ctas) steps meets at most this many heads
    const long long per = (sh.steps + sh.ctas - 1) / sh.ctas;
    sh.max_seg = (int)((per + sh.sph - 1) / sh.sph) + 1;
    return sh;
}

size_t decode_workspace_bytes(const DecodeShape &sh) {
    return (size_t)sh.ctas * sh.max_seg * sh.Nq * (sh.d + 2) * sizeof(float);
}

cudaError_t launch_decode_bf16(const DecodeShape &sh, const DecodeMaps &maps, const void *Q, void *O, float *LSE,
                               float *part, int *dev_status, cudaStream_t st) {
    switch (sh.d) {
        case 64: return launch_d<64>(sh, maps, Q, O, LSE, part, dev_status, st);
        case 128: return launch_d<128>(sh, maps, Q, O, LSE, part, dev_status, st);
        case 256: return launch_d<256>(sh, maps, Q, O, LSE, part, dev_status, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace attn
