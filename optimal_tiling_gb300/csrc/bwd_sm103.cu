// Recompute backward of the fused attention for sm_103a (bf16 in, fp32
// accumulation): the pass whose I/O "On Fine-Grained I/O Complexity of
// Attention Backward Passes" (gist.science 2410.09397) bounds by
// Theta((n^2 d^2 + n d^3) / M) in the large-cache regime M >= d^2, which is
// where a GB300 SM sits for every supported d.
//
// The page prints no gradient formulas; this is the chain rule of
// O = softmax(s Q K^T) V with upstream gradient dO:
//   P = exp(s Q K^T - LSE),  dV = P^T dO,  dP = dO V^T,  D_i = sum_t dO_it O_it,
//   dS = P o (dP - D),  dQ = s dS K,  dK = s dS^T Q.
//
// Kernels on the caller's stream:
//   1. bwd_pre:     D = rowsum(dO o O) and L2 = LSE log2(e) in fp32 (so that P is
//                   one FMA and one exp2 per score), the fp32 dQ accumulator zeroed
//                   (and the split tiles' fp32 dK, dV scratch, see 2);
//   2. bwd_main:    per 128-row K/V tile of one head (one CTA per tile under a
//                   mask or with partial tiles; without a mask bwd_persist, one CTA
//                   per SM taking a fixed set of tiles in turn), looping over the
//                   64-row query blocks that the block mask keeps (with 64-row
//                   mask blocks one half of the tile's keys can be removed for a
//                   visited query block: those keys get P = dS = 0).  Five tcgen05
//                   products per block, all accumulating in tensor memory:
//                     S^T  = K Q_i^T         (128 x 64, into S buffer)
//                     dP^T = V dO_i^T        (128 x 64, into dP buffer)
//                     dV  += P^T dO_i        (A = P^T from tensor memory)
//                     dK  += dS^T Q_i        (A = dS^T from shared memory)
//                     dQ_i^T = K^T dS_i^T    (M = d: into a buffer of its own)
//                   P and dS come from eight warps (thread = key; warps 0-3 take
//                   queries 0-31 of a block, warps 4-7 queries 32-63): a clock trace
//                   of one CTA showed the elementwise work of four warps, ~1,560
//                   cycles per block, to be the longest stage of the loop.
//                   The MMAs come from three warps, each waiting only for what its
//                   own products need (one thread issuing all five stalls every
//                   product behind each wait on another role): warp 13 issues S^T
//                   then dV (so that S^T of block i+2 follows, in one thread's issue
//                   order, the dV that read P of block i from the same columns),
//                   warp 14 dP^T then dK, warp 15 dQ^T; warps 8-11 drain dQ^T,
//                   warp 12 loads.
//                   dQ_i^T is drained by its own warpgroup into shared memory as
//                   [q][d] fp32 and added into the accumulator by two bulk
//                   reductions (cp.reduce.async.bulk .add.f32), one per 32-query
//                   half, so that rewriting a half waits only for the reduction
//                   of the same half one block back.  S is double
//                   buffered (it holds P until dV has read it); dP has one buffer,
//                   released as soon as the P/dS warps have loaded it, so dP^T of
//                   the next block overlaps this block's elementwise work and no
//                   longer waits for the dQ^T drain (when dQ^T shared the dP
//                   buffers, the chain P/dS -> dQ^T -> drain -> dP^T of block
//                   i+2 set the pace of the loop).  dK and dV leave tensor memory
//                   once, at the end, through shared memory and tensor stores.
//                   When the SM count does not divide the tiles and the last wave
//                   would be at most half full, the tiles of that wave run as a
//                   second grid (a programmatic dependent launch) of two CTAs per
//                   tile, each over half of the query blocks, adding fp32 dK and dV
//                   into scratch;
//   3. bwd_kv_finish (split tiles only): dK, dV = bf16 of that scratch;
//   4. bwd_dq_convert: dQ = bf16(s * accumulator).
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "visit_bits.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int BKV = 128;   // key/value rows per CTA
constexpr int BQ = 64;     // query rows per inner block
constexpr int kThreads = 512;
constexpr int kDqWarp0 = 8;     // warps 0-7 P/dS, warps 8-11 drain dQ
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;    // warps 13, 14, 15 issue MMAs (see the kernel comment)
constexpr int kStages = 3;      // Q/dO/L2/D ring depth (loads run two blocks ahead of the MMAs)
constexpr uint32_t kTmemCols = 512;

template <int D>
struct BwdCfg {
    static_assert(D == 64 || D == 128, "tcgen05 backward is built for d = 64 and d = 128");
    static constexpr int kKVTile = BKV * D * 2;          // 16 / 32 KB
    static constexpr int kKVSlab = BKV * 128;            // 16 KB: 64 columns of the K/V tile
    static constexpr int kQTile = BQ * D * 2;            // 8 / 16 KB
    static constexpr int kQSlab = BQ * 128;              // 8 KB
    static constexpr int kDsTile = BKV * BQ * 2;         // 16 KB: dS^T, 128 rows x 128 B
    static constexpr int kDqTile = BQ * D * 4;           // 16 / 32 KB fp32
    // dQ^T = K^T dS^T has M = d.  At d = 64 it runs as an M = 128 product whose A rows 64..127
    // (the second 64-element M chunk of the MN-major K^T, one leading byte offset past the
    // first) are a zeroed region of shared memory: the accumulator then has the known M = 128
    // layout (lane = row), rows 0..63 holding dQ^T and rows 64..127 zeros.
    static constexpr int kZeroBytes = D == 64 ? BKV * 128 : 0;
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKOff + kKVTile;
    static constexpr int kQOff = kVOff + kKVTile;
    static constexpr int kdOOff = kQOff + kStages * kQTile;
    static constexpr int kDsOff = kdOOff + kStages * kQTile;
    static constexpr int kDqOff = kDsOff + 2 * kDsTile;
    static constexpr int kZeroOff = kDqOff + kDqTile;
    static constexpr int kLdOff = kZeroOff + kZeroBytes; // per stage: L2[64], D[64]
    // leading byte offset of K^T's second M chunk: the next 64 columns of K, or the zeros
    static constexpr uint32_t kDqALbo = D == 64 ? (uint32_t)(kZeroOff - kKOff) : (uint32_t)kKVSlab;
    static constexpr int kDqM = 128;                     // M of the dQ^T product
    static constexpr int kBarOff = kLdOff + kStages * 2 * BQ * 4;
    // kv, qfull[S], qempty[S], sfull[2], pfull[2], dsfree[2], dqfull, dqfree, dpfree, kvdone, drain[3],
    // stagefree (the persistent kernel), kread[2]
    static constexpr int kNumBars = 1 + 2 * kStages + 2 * 3 + 3 + 1 + 3 + 1 + 2;
    // The persistent kernel at d = 128: dK's A operand, dS^T, comes from tensor memory (bf16 pairs
    // in the 16 columns of each query half of an S buffer that P leaves free) instead of the dS tile
    // in shared memory: the products' operand reads from shared memory pace its loop, and this
    // removes 16 KB of them per block (dense_16k 4.09 -> 4.02 ms).  At d = 64, and in bwd_main
    // (masked and partial tiles: 1.6-2.0% slower there), dK reads the shared-memory tile.
    static constexpr bool kDsInTmem = D == 128;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    // visited query blocks as a bit set: up to 32 * kMaxMaskWords 64-row blocks (N <= 131072)
    static constexpr int kMaxMaskWords = 64;
    static constexpr int kBitsOff = kMiscOff + 64;
    static constexpr int kSmemBytes = kBitsOff + 4 * kMaxMaskWords + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
    // tensor memory columns
    // dV, dK accumulators; S^T twice (it holds P until dV has read it); dP^T once (read into
    // registers at the start of a block's elementwise work); dQ^T of one block
    static constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 2 * BQ, kColQ = kColDP + BQ;
    static_assert(kColQ + BQ <= kTmemCols, "tensor memory budget");
    static_assert(kDqALbo % 16 == 0 && (kDqALbo >> 4) < (1u << 14), "leading byte offset field");
};

struct BwdBars {
    uint32_t base;
    __device__ uint32_t kv() const { return base; }
    __device__ uint32_t qfull(int s) const { return base + 8u * (1 + s); }
    __device__ uint32_t qempty(int s) const { return base + 8u * (1 + kStages + s); }
    __device__ uint32_t sfull(int b) const { return base + 8u * (1 + 2 * kStages + b); }
    __device__ uint32_t pfull(int b) const { return base + 8u * (3 + 2 * kStages + b); }
    __device__ uint32_t dsfree(int b) const { return base + 8u * (5 + 2 * kStages + b); }
    __device__ uint32_t dqfull() const { return base + 8u * (7 + 2 * kStages); }
    __device__ uint32_t dqfree() const { return base + 8u * (8 + 2 * kStages); }
    __device__ uint32_t dpfree() const { return base + 8u * (9 + 2 * kStages); }
    __device__ uint32_t kvdone() const { return base + 8u * (10 + 2 * kStages); }
    __device__ uint32_t drain(int role) const { return base + 8u * (11 + 2 * kStages + role); }
    __device__ uint32_t stagefree() const { return base + 8u * (14 + 2 * kStages); }
    // dK has read dS^T of S buffer b (tensor memory), so S^T two blocks on may overwrite it
    __device__ uint32_t kread(int b) const { return base + 8u * (15 + 2 * kStages + b); }
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Bounded wait whose polls may sleep up to 2 us each (the thread resumes when the phase
// completes), for the producer and the MMA issuers at d = 64: fewer polls from threads that share
// an SMSP with the elementwise warps (teaching shape 0.856 -> 0.840 ms; at d = 128 it measured 1%
// slower, so there the plain bounded wait stays).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(2000u)
        : "memory");
    return ok != 0;
}
template <int D>
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *status) {
    if constexpr (D != 64) {
        return mbar_wait(bar, parity, abort_flag, status);
    } else {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        const unsigned long long t0 = global_timer_ns();
        for (;;) {
            if (mbar_try_wait_sleep(bar, parity)) return true;
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicExch(status, 1);
                return false;
            }
        }
    }
}

// Product of two packed fp32 pairs (one instruction, round to nearest).
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ------------------------------------------------------------------------- 1
// D_i = sum_t dO_it O_it and L2_i = LSE_i log2(e) (the row's log-sum-exp in the base-2 units of
// the exponentials below), both stored negated (-D, -L2: the main kernel adds them in packed
// pairs); the dQ accumulator row is zeroed.  d / 8 threads per row, each with 16-byte loads of O
// and dO and two 16-byte zero stores (a warp takes 2 rows at d = 128, 4 at d = 64; 8 warps a block).
// The split tiles' partial dK, dV (kv4: kv_n4 float4) are zeroed grid-stride.
// D, L2 and the accumulator hold npad rows per head (N rounded up to the 64-row query block;
// npad = N when 64 divides N, PAD = false): the rows from N on get D = 0 and L2 = +inf, so that
// their probabilities, and with them their dS, are exactly zero in the main kernel.
template <int D>
constexpr int kPreRowsPerBlock = 8 * (32 / (D / 8));
template <int D, bool PAD>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16 *__restrict__ O,
                                                      const __nv_bfloat16 *__restrict__ dO,
                                                      float *__restrict__ Dv, float *__restrict__ dQacc,
                                                      size_t rows, float4 *__restrict__ kv4, size_t kv_n4,
                                                      const float *__restrict__ LSE, float *__restrict__ L2, int N,
                                                      int npad) {
    constexpr int TPR = D / 8;  // threads per row
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < kv_n4; i += (size_t)gridDim.x * blockDim.x)
        kv4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int sub = threadIdx.x % TPR;
    const size_t prow = (size_t)blockIdx.x * kPreRowsPerBlock<D> + threadIdx.x / TPR;  // row of the padded layout
    const bool in = prow < rows;
    size_t row = prow;  // row of O, dO and LSE
    bool pad = !in;
    if constexpr (PAD) {
        const size_t hh = prow / (size_t)npad, q = prow - hh * (size_t)npad;
        pad = pad || q >= (size_t)N;
        row = hh * (size_t)N + q;
    }
    float acc = 0.f;
    if (!pad) {
        const uint4 a = *reinterpret_cast<const uint4 *>(O + row * D + sub * 8);
        const uint4 b = *reinterpret_cast<const uint4 *>(dO + row * D + sub * 8);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&aw[e]));
            const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&bw[e]));
            acc = fmaf(x.x, y.x, acc);
            acc = fmaf(x.y, y.y, acc);
        }
    }
    // the TPR lanes of a row are aligned groups of a warp: xor offsets below TPR stay inside one
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (!in) return;
    if (sub == 0) {
        Dv[prow] = -acc;
        L2[prow] = pad ? -INFINITY : -(LSE[row] * kLog2e);
    }
    float4 *z = reinterpret_cast<float4 *>(dQacc + prow * D) + sub * 2;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------------- 2
// HALVES = false: grid (N / 128, B * H), CTA (x, y) takes key tile x of head y; a tile at or
// after split_from (in the order head * (N / 128) + x) belongs to the split last wave and its
// CTA returns at once.  HALVES = true: grid 2 * (tiles - split_from), two CTAs per split tile,
// each taking one half of the query blocks and adding fp32 partial dK, dV into kvacc.
// TAIL (N % 128 != 0, never split): grid (ceil(N / 128), B * H).  The last key tile and query
// block of a head are partial, and the rows past N that their loads bring in belong to the next
// head (or read as zeros past the end).  Keys from N on get P = dS = 0 here; queries from N on
// get P = 0 from L2 = +inf (bwd_pre), so their dQ rows are zero and land in the padding rows of
// the accumulator; dK and dV rows from N on are not stored.
template <int D, bool HALVES, bool TAIL>
__global__ void __launch_bounds__(kThreads, 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                const Problem p, const float *__restrict__ L2, const float *__restrict__ Dv,
                float *__restrict__ dQacc, __nv_bfloat16 *__restrict__ dK, __nv_bfloat16 *__restrict__ dV,
                const int split_from, float *__restrict__ kvacc) {
    using C = BwdCfg<D>;
    static_assert(!(HALVES && TAIL), "a partial tile is never split");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const BwdBars bars{smem_addr(sm + C::kBarOff)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nq = TAIL ? (p.N + BQ - 1) / BQ : p.N / BQ;  // 64-row query blocks
    const int npad = TAIL ? nq * BQ : p.N;     // rows per head of D, L2 and the dQ accumulator
    int kvt, head, q_lo;                       // key tile, head, first query block
    if constexpr (HALVES) {
        const int tile = split_from + (int)(blockIdx.x >> 1);
        kvt = tile % (p.N / BKV);
        head = tile / (p.N / BKV);
        q_lo = (blockIdx.x & 1) * (nq / 2);
    } else {
        // The HALVES grid reads nothing this grid writes (both only add into accumulators),
        // so it may start on SMs this grid frees: allow that as soon as every CTA is running.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        kvt = blockIdx.x;
        head = blockIdx.y;
        q_lo = 0;
        if (head * (int)gridDim.x + kvt >= split_from) return;  // run by the HALVES launch
    }
    const int kv0 = head * p.N + kvt * BKV;    // first K/V row of this CTA in the [B*H*N, D] view
    const uint8_t *hm = p.head_mask(head);
    const int mb = p.mask_block, mnb = p.mask_nb();
    // query block iq is visited when a mask entry covering (its 64 rows, this tile's 128 keys) is kept
    auto qvisited = [&](int iq) -> bool {
        if (hm == nullptr) return true;
        if (mb == 128) return hm[(size_t)(iq >> 1) * mnb + kvt] != 0;
        const uint8_t *r = hm + (size_t)iq * mnb + 2 * kvt;
        if constexpr (TAIL) return (r[0] | (2 * kvt + 1 < mnb ? r[1] : 0)) != 0;  // last column may be absent
        return (r[0] | r[1]) != 0;
    };
    uint32_t *vwords = reinterpret_cast<uint32_t *>(sm + C::kBitsOff);
    const int nwords = (nq + 31) >> 5;
    const bool use_bits = hm != nullptr && nwords <= C::kMaxMaskWords;
    const uint32_t sK = smem_addr(sm + C::kKOff), sV = smem_addr(sm + C::kVOff);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bars.kv(), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bars.qfull(s), 1);
            mbar_init(bars.qempty(s), 2);   // dV (warp 13) and dK (warp 14) are the last readers
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.sfull(b), 2);    // S^T (warp 13) and dP^T (warp 14)
            mbar_init(bars.pfull(b), 8);    // one lane of each P/dS warp
            mbar_init(bars.dsfree(b), 2);   // dK (warp 14) and dQ^T (warp 15) read dS
        }
        mbar_init(bars.dqfull(), 1);
        mbar_init(bars.dqfree(), 4);        // the drain warps have read dQ^T (one lane each)
        mbar_init(bars.dpfree(), 8);        // the P/dS warps have read dP^T (one lane each)
        mbar_init(bars.kvdone(), 2);        // dV and dK complete
        for (int r = 0; r < 3; ++r) mbar_init(bars.drain(r), 1);
        fence_barrier_init();
        // the K/V tile is needed whatever the mask says: start its load before the mask is read
        mbar_arrive_expect_tx(bars.kv(), 2 * C::kKVTile);
        for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(sK + c * C::kKVSlab, &tmK, c * 64, kv0, bars.kv());
            tma_load_2d(sV + c * C::kKVSlab, &tmV, c * 64, kv0, bars.kv());
        }
    }
    if (use_bits) build_visit_bits(vwords, nq, qvisited);
    if constexpr (C::kZeroBytes > 0) {
        // the zero rows of the padded K^T operand (read by the tensor core: async proxy)
        uint4 *z = reinterpret_cast<uint4 *>(sm + C::kZeroOff);
        for (int i = tid; i < C::kZeroBytes / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const VisitBits vb{vwords, nwords};
    int n = HALVES ? nq / 2 : nq;  // query blocks this CTA visits
    if (use_bits) {
        n = vb.count();
    } else if (hm != nullptr) {  // columns longer than the bit set: read the mask directly
        n = 0;
        for (int iq = 0; iq < nq; ++iq) n += qvisited(iq) ? 1 : 0;
    }
    // the visited query block after iq (callers ask only while one remains)
    auto next_q = [&](int iq) -> int {
        if (hm == nullptr) return iq + 1;
        if (use_bits) return vb.next(iq);
        do {
            ++iq;
        } while (!qvisited(iq));
        return iq;
    };
    const uint32_t tmem = *tmem_slot;
    const uint32_t sQ = smem_addr(sm + C::kQOff), sdO = smem_addr(sm + C::kdOOff);
    const uint32_t sDs = smem_addr(sm + C::kDsOff), sDq = smem_addr(sm + C::kDqOff);
    const uint32_t sLd = smem_addr(sm + C::kLdOff);
    const float *ld_f = reinterpret_cast<const float *>(sm + C::kLdOff);

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmdO);
            int iq = q_lo - 1;
            for (int it = 0; it < n; ++it) {
                const int s = it % kStages;
                iq = next_q(iq);
                if (it >= kStages &&
                    !role_wait<D>(bars.qempty(s), ((uint32_t)(it / kStages) & 1u) ^ 1u, abort_flag, p.dev_status))
                    break;
                const int q0 = head * p.N + iq * BQ;
                const int ql = TAIL ? head * npad + iq * BQ : q0;  // the block's rows of L2 and D
                mbar_arrive_expect_tx(bars.qfull(s), 2 * C::kQTile + 2 * BQ * 4);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_2d(sQ + s * C::kQTile + c * C::kQSlab, &tmQ, c * 64, q0, bars.qfull(s));
                    tma_load_2d(sdO + s * C::kQTile + c * C::kQSlab, &tmdO, c * 64, q0, bars.qfull(s));
                }
                bulk_load(sLd + s * 2 * BQ * 4, L2 + ql, BQ * 4, bars.qfull(s));
                bulk_load(sLd + s * 2 * BQ * 4 + BQ * 4, Dv + ql, BQ * 4, bars.qfull(s));
            }
        }
    } else if (warp >= kMmaWarp) {
        // ------------------------------------------------------------ MMA issuers
        const int role = warp - kMmaWarp;  // 0: S^T then dV, 1: dP^T then dK, 2: dQ^T
        if (lane == 0 && n > 0) {
            constexpr uint32_t idSP = idesc_bf16_f32(BKV, BQ, false, false);  // S^T, dP^T
            constexpr uint32_t idKV = idesc_bf16_f32(BKV, D, false, true);    // dV, dK
            constexpr uint32_t idQ = idesc_bf16_f32(C::kDqM, BQ, true, true); // dQ^T (M padded to 128)
            bool ok = role_wait<D>(bars.kv(), 0, abort_flag, p.dev_status);
            if (role < 2) {
                // S^T_it (role 0) or dP^T_it (role 1) into buffer it & 1
                auto issue_first = [&](int it) -> bool {
                    const int s = it % kStages, b = it & 1;
                    if (!role_wait<D>(bars.qfull(s), (uint32_t)(it / kStages) & 1u, abort_flag, p.dev_status))
                        return false;
                    // one dP buffer: the P/dS warps must have read dP^T of block it-1
                    if (role == 1 && it >= 1 &&
                        !role_wait<D>(bars.dpfree(), (uint32_t)(it - 1) & 1u, abort_flag, p.dev_status))
                        return false;
                    tc_fence_after();
                    const uint32_t xb = (role == 0 ? sQ : sdO) + s * C::kQTile;
                    const uint32_t kb = role == 0 ? sK : sV;
                    const uint32_t dcol = tmem + (role == 0 ? C::kColS + b * BQ : C::kColDP);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t ko = (ks >> 2) * C::kKVSlab + (ks & 3) * 32;
                        const uint32_t qo = (ks >> 2) * C::kQSlab + (ks & 3) * 32;
                        mma_ss(dcol, smem_desc_sw128(kb + ko, 16, 1024), smem_desc_sw128(xb + qo, 16, 1024), idSP,
                               ks > 0);
                    }
                    mma_commit(bars.sfull(b));
                    return true;
                };
                if (ok) ok = issue_first(0);
                for (int it = 0; it < n && ok; ++it) {
                    const int s = it % kStages, b = it & 1;
                    if (it + 1 < n && !(ok = issue_first(it + 1))) break;
                    if (!(ok = role_wait<D>(bars.pfull(b), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status))) break;
                    tc_fence_after();
                    const uint32_t qb = sQ + s * C::kQTile, gb = sdO + s * C::kQTile, dsb = sDs + b * C::kDsTile;
                    if (role == 0) {
                        // dV += P^T dO_i : A = P^T (bf16 pairs; queries 32h.. at S column 32h),
                        // B = dO_i (d contiguous)
#pragma unroll
                        for (int ks = 0; ks < BQ / 16; ++ks)
                            mma_ts(tmem + C::kColDV, tmem + C::kColS + b * BQ + (ks >> 1) * 32 + (ks & 1) * 8,
                                   smem_desc_sw128(gb + ks * 2048, C::kQSlab, 1024), idKV,
                                   (it > 0 || ks > 0) ? 1u : 0u);
                    } else {
                        // dK += dS^T Q_i : A = dS^T (K-major, 64 q per row), B = Q_i (d contiguous)
#pragma unroll
                        for (int ks = 0; ks < BQ / 16; ++ks)
                            mma_ss(tmem + C::kColDK, smem_desc_sw128(dsb + ks * 32, 16, 1024),
                                   smem_desc_sw128(qb + ks * 2048, C::kQSlab, 1024), idKV,
                                   (it > 0 || ks > 0) ? 1u : 0u);
                        mma_commit(bars.dsfree(b));
                    }
                    mma_commit(bars.qempty(s));
                }
                if (ok) mma_commit(bars.kvdone());
            } else {
                // 64-row mask blocks: the key halves of this tile kept for query block iq (bit 0:
                // keys 0-63, bit 1: keys 64-127).  dS is zero over a removed half, so dQ^T skips the
                // k-steps that contract over it.  Read one block ahead, off the issue path.
                const bool fine = hm != nullptr && mb == 64;
                auto halves = [&](int iq) -> uint32_t {
                    if (!fine) return 3u;
                    const uint8_t *r = hm + (size_t)iq * mnb + 2 * kvt;
                    const bool has1 = !TAIL || 2 * kvt + 1 < mnb;
                    return (uint32_t)(r[0] != 0) | ((uint32_t)(has1 && r[1] != 0) << 1);
                };
                int iq_next = (fine && n > 0) ? next_q(q_lo - 1) : 0;
                uint32_t h_next = halves(iq_next);
                for (int it = 0; it < n && ok; ++it) {
                    const int b = it & 1;
                    const uint32_t h_cur = h_next;
                    if (fine && it + 1 < n) {
                        iq_next = next_q(iq_next);
                        h_next = halves(iq_next);
                    }
                    if (!(ok = role_wait<D>(bars.pfull(b), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status))) break;
                    // one dQ^T buffer: the drain warps must have read dQ^T of block it-1
                    if (it >= 1 && !(ok = role_wait<D>(bars.dqfree(), (uint32_t)(it - 1) & 1u, abort_flag, p.dev_status)))
                        break;
                    tc_fence_after();
                    const uint32_t dsb = sDs + b * C::kDsTile;
                    // dQ_i^T = K^T dS_i^T : A = K^T (d contiguous), B = dS (q contiguous)
                    if (h_cur == 3u) {
#pragma unroll
                        for (int ks = 0; ks < BKV / 16; ++ks)
                            mma_ss(tmem + C::kColQ, smem_desc_sw128(sK + ks * 2048, C::kDqALbo, 1024),
                                   smem_desc_sw128(dsb + ks * 2048, C::kDsTile, 1024), idQ, ks > 0);
                    } else {  // one key half kept for this query block: its four k-steps only
                        const int k0 = h_cur == 1u ? 0 : 4;
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
                            mma_ss(tmem + C::kColQ, smem_desc_sw128(sK + (k0 + k4) * 2048, C::kDqALbo, 1024),
                                   smem_desc_sw128(dsb + (k0 + k4) * 2048, C::kDsTile, 1024), idQ, k4 > 0);
                    }
                    mma_commit(bars.dsfree(b));
                    mma_commit(bars.dqfull());
                }
            }
            if (!ok) {
                // let every MMA this thread issued finish before tensor memory is released
                mma_commit(bars.drain(role));
                mbar_wait(bars.drain(role), 0, abort_flag, p.dev_status);
            }
        }
    } else if (warp < kDqWarp0) {
        // ------------------------------------------------------------ P / dS warps 0-7
        // Thread = key (tensor memory lane 32 (warp % 4) + lane); warps 0-3 take queries 0-31 of
        // each block, warps 4-7 queries 32-63: the work is elementwise given LSE and D, so the
        // two halves of a key row need nothing from each other.
        const int h = warp >> 2;
        const int key = (warp & 3) * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const float sl2 = p.scale * kLog2e;
        const uint32_t my_ds_row = (uint32_t)key * 128u;  // byte offset of dS^T row `key` in a dS tile
        uint8_t *ds_gen = sm + C::kDsOff;
        // 64-row mask blocks: this warp's 32 keys lie in one key half of the tile
        const bool fine = hm != nullptr && mb == 64;
        // TAIL: keys from N on (rows of the next head) get P = dS = 0
        const bool key_ok = !TAIL || kvt * BKV + key < p.N;
        int iq = q_lo - 1;
        bool ok = true;
        for (int it = 0; it < n; ++it) {
            const int s = it % kStages, b = it & 1;
            bool row_kept = true;
            if (fine) {
                iq = next_q(iq);
                if constexpr (TAIL) {  // the tile's second key half may have no mask column
                    const int kcol = 2 * kvt + ((warp & 3) >> 1);
                    row_kept = kcol < mnb && hm[(size_t)iq * mnb + kcol] != 0;
                } else {
                    row_kept = hm[(size_t)iq * mnb + 2 * kvt + ((warp & 3) >> 1)] != 0;
                }
            }
            ok = mbar_wait(bars.sfull(b), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status);
            if (ok && it >= 2)
                ok = mbar_wait(bars.dsfree(b), (uint32_t)((it - 2) >> 1) & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const float *nl2 = ld_f + s * 2 * BQ;  // -LSE log2(e) of the 64 queries, then -D
            const float *ndv = nl2 + BQ;
            uint32_t pk[16], dk[16];
            uint32_t sr[32], pr[32];
            if (row_kept) {
                tmem_ld32(lane_base + C::kColS + b * BQ + h * 32, sr);
                tmem_ld32(lane_base + C::kColDP + h * 32, pr);
                tmem_wait_ld();
                reg_fence(sr);
                reg_fence(pr);
            }
            // dP^T is in registers: the single dP buffer may take the next block's product.
            // A warp signals through one lane after a warp sync (256 single-thread arrivals on
            // one barrier per block made the backward ~1.5% slower).
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.dpfree());
            if (!row_kept) {
                // keys removed for this query block: P = dS = 0 (warp-uniform)
#pragma unroll
                for (int t = 0; t < 16; ++t) pk[t] = dk[t] = 0u;
            } else {
                // two queries per step on the packed fp32 path: x = s log2(e) S - L2, p = 2^x,
                // dS = p (dP - D); the same roundings as one query at a time
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int q = h * 32 + 2 * t;
                    // the row terms of four queries per 16-byte load, two of them per step
                    float4 nl, nd;
                    if ((t & 1) == 0) {
                        nl = *reinterpret_cast<const float4 *>(nl2 + q);
                        nd = *reinterpret_cast<const float4 *>(ndv + q);
                    }
                    const uint64_t l2p = (t & 1) ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y);
                    const uint64_t dvp = (t & 1) ? f2_pack(nd.z, nd.w) : f2_pack(nd.x, nd.y);
                    const uint64_t x2 =
                        f2_fma(f2_pack(__uint_as_float(sr[2 * t]), __uint_as_float(sr[2 * t + 1])), sl2x2, l2p);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    const uint64_t g2 =
                        f2_add(f2_pack(__uint_as_float(pr[2 * t]), __uint_as_float(pr[2 * t + 1])), dvp);
                    float d0, d1;
                    f2_unpack(f2_mul(f2_pack(p0, p1), g2), d0, d1);
                    pk[t] = pack_bf16(p0, p1);
                    dk[t] = pack_bf16(d0, d1);
                }
                if constexpr (TAIL) {
                    if (!key_ok) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) pk[t] = dk[t] = 0u;
                    }
                }
            }
            // P^T as bf16 pairs over the first 16 of this half's own 32 S columns
            tmem_st16(lane_base + C::kColS + b * BQ + h * 32, pk);
            // dS^T row into shared memory, 128-byte swizzle: 16-byte chunk c at c ^ (row % 8)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int chunk = h * 4 + c;
                const uint32_t off = my_ds_row + (uint32_t)((chunk ^ (key & 7)) * 16);
                *reinterpret_cast<uint4 *>(ds_gen + b * C::kDsTile + off) =
                    make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.pfull(b));
        }
        // ------------------------------------------------------------ dK (warps 0-3), dV (warps 4-7)
        if (ok && n > 0) {
            ok = mbar_wait(bars.kvdone(), 0, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        const size_t grow = (size_t)kv0 + key;
        uint4 *orow = reinterpret_cast<uint4 *>((h == 0 ? dK : dV) + grow * D);
        const uint32_t acc = lane_base + (h == 0 ? C::kColDK : C::kColDV);
        const float mul = h == 0 ? p.scale : 1.f;
        if (HALVES && ok && n > 0) {
            // one query half of a split tile: add this row's partial dK or dV in fp32
            float4 *prow = reinterpret_cast<float4 *>(kvacc + ((size_t)(blockIdx.x >> 1) * 2 + h) * BKV * D +
                                                      (size_t)key * D);
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t a[32];
                tmem_ld32(acc + c0, a);
                tmem_wait_ld();
                reg_fence(a);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    atomicAdd(prow + c0 / 4 + q,
                              make_float4(__uint_as_float(a[4 * q]) * mul, __uint_as_float(a[4 * q + 1]) * mul,
                                          __uint_as_float(a[4 * q + 2]) * mul, __uint_as_float(a[4 * q + 3]) * mul));
            }
        } else if (TAIL && n > 0 && (kvt + 1) * BKV > p.N) {
            // the last tile of a head with N % 128 != 0: the rows past N belong to the next head,
            // so each thread stores its own row, if it exists, instead of one tensor store
            if (ok) {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t a[32];
                    tmem_ld32(acc + c0, a);
                    tmem_wait_ld();
                    reg_fence(a);
                    uint32_t pa[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        pa[t] = pack_bf16(__uint_as_float(a[2 * t]) * mul, __uint_as_float(a[2 * t + 1]) * mul);
                    if (key_ok) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            orow[c0 / 8 + q] = make_uint4(pa[4 * q], pa[4 * q + 1], pa[4 * q + 2], pa[4 * q + 3]);
                    }
                }
            }
        } else if (!HALVES && n > 0) {
            // Stage the bf16 tile (dK in the Q ring, dV in the dO ring: every MMA that reads them
            // completed before kvdone) in the 128-byte-swizzled layout of a 64-column TMA box, then
            // one thread of the four warps stores it with two tensor stores.  The four warps meet
            // at the named barrier whatever `ok` says (a warp that gave up after a timed-out wait
            // still arrives), so that no warp waits there for one that skipped it.
            uint8_t *stage = sm + (h == 0 ? C::kQOff : C::kdOOff);
            if (ok) {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t a[32];
                    tmem_ld32(acc + c0, a);
                    tmem_wait_ld();
                    reg_fence(a);
                    uint32_t pa[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        pa[t] = pack_bf16(__uint_as_float(a[2 * t]) * mul, __uint_as_float(a[2 * t + 1]) * mul);
                    uint8_t *slab = stage + (c0 >> 6) * C::kKVSlab + key * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int u = ((c0 & 63) >> 3) + q;  // 16-byte unit within the 128-byte row
                        *reinterpret_cast<uint4 *>(slab + ((u ^ (key & 7)) << 4)) =
                            make_uint4(pa[4 * q], pa[4 * q + 1], pa[4 * q + 2], pa[4 * q + 3]);
                    }
                }
                fence_proxy_async_smem();
            }
            named_bar_sync(2 + h, 128);
            if ((tid & 127) == 0 && ok) {
                const CUtensorMap *tm = h == 0 ? &tmdK : &tmdV;
                const uint32_t src = smem_addr(stage);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) tma_store_2d(tm, c * 64, kv0, src + c * C::kKVSlab);
                bulk_commit();
                bulk_wait_all();
            }
        } else if (n == 0 && key_ok) {
            for (int q = 0; q < D / 8; ++q) orow[q] = make_uint4(0, 0, 0, 0);
        }
    } else if (warp < kTmaWarp) {
        // ------------------------------------------------------------ dQ drain warps 8-11
        // Every drain thread runs the same sequence of named barriers whatever happens:
        // after a failed (timed-out) wait the work is skipped but the barriers are kept,
        // and the CTA abort flag makes every later wait return at once.
        const int t = tid - kDqWarp0 * 32;  // 0..127 = d index (tensor memory lane); rows >= D are padding
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        float *dq_gen = reinterpret_cast<float *>(sm + C::kDqOff);
        bool alive = true;
        int iq = q_lo - 1;
        for (int it = 0; it < n; ++it) {
            iq = next_q(iq);
            bool ok = alive && mbar_wait(bars.dqfull(), (uint32_t)it & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            uint32_t r0[32], r1[32];
            if (ok) {
                tc_fence_after();
                tmem_ld32(lane_base + C::kColQ, r0);
                tmem_ld32(lane_base + C::kColQ + 32, r1);
                tmem_wait_ld();
                reg_fence(r0);
                reg_fence(r1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.dqfree());
            }
            // Two halves (queries 0-31 from r0, 32-63 from r1), each with its own 16 KB of the
            // staging tile and its own bulk reduction: before a half is rewritten only the
            // reduction of the same half one block back must have read it, not the one just issued.
            const size_t q0 = (size_t)head * npad + (size_t)iq * BQ;  // the block's accumulator rows
            auto stage = [&](const uint32_t(&r)[32], int hq) {
                if (t == 0) bulk_wait_read_but_one();
                named_bar_sync(1, 128);
                if (ok && t < D) {
                    float *dst = dq_gen + hq * 32 * D;
#pragma unroll
                    for (int q = 0; q < 32; ++q) dst[q * D + t] = __uint_as_float(r[q]);
                    fence_proxy_async_smem();
                }
                named_bar_sync(1, 128);
                if (t == 0 && ok) {
                    bulk_reduce_add_f32(dQacc + (q0 + 32 * hq) * D, sDq + hq * (C::kDqTile / 2), C::kDqTile / 2);
                    bulk_commit();
                }
            };
            stage(r0, 0);
            stage(r1, 1);
            alive = alive && ok;
        }
        if (t == 0) bulk_wait_all();
    }

    // a tile that visits no query block still received its K/V tile: let that copy land first
    if (n == 0 && tid == 0) mbar_wait(bars.kv(), 0, abort_flag, p.dev_status);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // The HALVES grid may run beside the full-tile grid. Each of its CTAs ends by waiting for
    // that grid to complete (its last tiles are done or nearly so by then), so that later work
    // on the stream, which reads the dQ accumulator both grids add into, follows both.
    if constexpr (HALVES) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------------- 2b
// Every bulk group this thread committed has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Persistent form of bwd_main for dense problems (no mask, 128 | N): a grid of at most one CTA per
// SM, CTA c taking key tiles c, c + P, c + 2P, ... (P = gridDim.x) below split_from.  Every tile
// has the same n query blocks, so each role's block counter g = T n + it (T = the CTA's tile
// number) runs on across tiles, and the ring, S, dP, dS and dQ^T barriers keep one phase sequence.
// Between tiles:
//   - kvdone counts three commits, one per issuing thread after a tile's last products: then K, V
//     and dS are no longer read and dK, dV are final.  The producer then loads the next K/V tile,
//     which overlaps the epilogue; the Q/dO ring runs on without a break.
//   - The epilogue reads dK and dV into registers before its warps signal pfull for the next tile's
//     first block, and the next dV and dK products wait for that pfull, so they cannot overwrite
//     the accumulators early.
//   - dK is staged in the two dS tiles, dV in the dQ staging tile once the drain's reductions of the
//     tile have read it (stagefree); all eight P/dS warps meet after the stores have read both, so
//     that no dS or dQ of the next tile is written there before.
// Within a block, at d = 128 dK's A operand (dS^T) is read from tensor memory beside P (kDsInTmem),
// and S^T two blocks on waits for dK's release of those columns (kread); at d = 64 the dQ drain
// adds straight from registers instead of through the staging tile.
// One CTA per SM also removes the per-CTA start (barrier set-up, tensor-memory allocation, the
// first loads) from all tiles but the first.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                   const Problem p, const float *__restrict__ L2, const float *__restrict__ Dv,
                   float *__restrict__ dQacc, const int split_from) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const BwdBars bars{smem_addr(sm + C::kBarOff)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);
    // the grid of split tiles reads nothing this grid writes (both only add into accumulators)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = p.N / BQ;        // query blocks of every tile
    const int tph = p.N / BKV;     // key tiles per head
    const int cta = (int)blockIdx.x, P = (int)gridDim.x;
    const int ntile = cta < split_from ? (split_from - 1 - cta) / P + 1 : 0;
    auto tile_head = [&](int T) -> int { return (cta + T * P) / tph; };
    auto tile_kv0 = [&](int T) -> int {  // first K/V row of the CTA's tile T in the [B*H*N, D] view
        const int tile = cta + T * P;
        return (tile / tph) * p.N + (tile % tph) * BKV;
    };
    const uint32_t sK = smem_addr(sm + C::kKOff), sV = smem_addr(sm + C::kVOff);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bars.kv(), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bars.qfull(s), 1);
            mbar_init(bars.qempty(s), 2);   // dV (warp 13) and dK (warp 14) are the last readers
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.sfull(b), 2);    // S^T (warp 13) and dP^T (warp 14)
            mbar_init(bars.pfull(b), 8);    // one lane of each P/dS warp
            mbar_init(bars.dsfree(b), 2);   // dK (warp 14) and dQ^T (warp 15) read dS
        }
        mbar_init(bars.dqfull(), 1);
        for (int b = 0; b < 2; ++b) mbar_init(bars.kread(b), 1);  // dK (warp 14) read dS^T of S buffer b
        mbar_init(bars.dqfree(), 4);        // the drain warps have read dQ^T (one lane each)
        mbar_init(bars.dpfree(), 8);        // the P/dS warps have read dP^T (one lane each)
        mbar_init(bars.kvdone(), 3);        // a tile's products complete: one commit per issuer
        mbar_init(bars.stagefree(), 1);     // the drain's reductions of a tile have read its staging
        for (int r = 0; r < 3; ++r) mbar_init(bars.drain(r), 1);
        fence_barrier_init();
        if (ntile > 0) {
            mbar_arrive_expect_tx(bars.kv(), 2 * C::kKVTile);
            const int kv0 = tile_kv0(0);
            for (int c = 0; c < D / 64; ++c) {
                tma_load_2d(sK + c * C::kKVSlab, &tmK, c * 64, kv0, bars.kv());
                tma_load_2d(sV + c * C::kKVSlab, &tmV, c * 64, kv0, bars.kv());
            }
        }
    }
    if constexpr (C::kZeroBytes > 0) {
        // the zero rows of the padded K^T operand (read by the tensor core: async proxy)
        uint4 *z = reinterpret_cast<uint4 *>(sm + C::kZeroOff);
        for (int i = tid; i < C::kZeroBytes / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sQ = smem_addr(sm + C::kQOff), sdO = smem_addr(sm + C::kdOOff);
    const uint32_t sDs = smem_addr(sm + C::kDsOff), sDq = smem_addr(sm + C::kDqOff);
    const uint32_t sLd = smem_addr(sm + C::kLdOff);
    const float *ld_f = reinterpret_cast<const float *>(sm + C::kLdOff);

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && ntile > 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmdO);
            bool ok = true;
            for (int T = 0; T < ntile && ok; ++T) {
                const int head = tile_head(T);
                if (T > 0) {
                    // every product of the previous tile is complete: K and V may be reloaded
                    if (!(ok = role_wait<D>(bars.kvdone(), (uint32_t)(T - 1) & 1u, abort_flag, p.dev_status)))
                        break;
                    const int kv0 = tile_kv0(T);
                    mbar_arrive_expect_tx(bars.kv(), 2 * C::kKVTile);
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_2d(sK + c * C::kKVSlab, &tmK, c * 64, kv0, bars.kv());
                        tma_load_2d(sV + c * C::kKVSlab, &tmV, c * 64, kv0, bars.kv());
                    }
                }
                for (int it = 0; it < n; ++it) {
                    const int g = T * n + it, s = g % kStages;
                    if (g >= kStages &&
                        !(ok = role_wait<D>(bars.qempty(s), ((uint32_t)(g / kStages) & 1u) ^ 1u, abort_flag,
                                            p.dev_status)))
                        break;
                    const int q0 = head * p.N + it * BQ;
                    mbar_arrive_expect_tx(bars.qfull(s), 2 * C::kQTile + 2 * BQ * 4);
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_2d(sQ + s * C::kQTile + c * C::kQSlab, &tmQ, c * 64, q0, bars.qfull(s));
                        tma_load_2d(sdO + s * C::kQTile + c * C::kQSlab, &tmdO, c * 64, q0, bars.qfull(s));
                    }
                    bulk_load(sLd + s * 2 * BQ * 4, L2 + q0, BQ * 4, bars.qfull(s));
                    bulk_load(sLd + s * 2 * BQ * 4 + BQ * 4, Dv + q0, BQ * 4, bars.qfull(s));
                }
            }
        }
    } else if (warp >= kMmaWarp) {
        // ------------------------------------------------------------ MMA issuers
        const int role = warp - kMmaWarp;  // 0: S^T then dV, 1: dP^T then dK, 2: dQ^T
        if (lane == 0 && ntile > 0) {
            constexpr uint32_t idSP = idesc_bf16_f32(BKV, BQ, false, false);  // S^T, dP^T
            constexpr uint32_t idKV = idesc_bf16_f32(BKV, D, false, true);    // dV, dK
            constexpr uint32_t idQ = idesc_bf16_f32(C::kDqM, BQ, true, true); // dQ^T (M padded to 128)
            bool ok = true;
            // S^T_g (role 0) or dP^T_g (role 1) into buffer g & 1
            auto issue_first = [&](int g) -> bool {
                const int s = g % kStages, b = g & 1;
                if (!role_wait<D>(bars.qfull(s), (uint32_t)(g / kStages) & 1u, abort_flag, p.dev_status))
                    return false;
                // one dP buffer: the P/dS warps must have read dP^T of block g-1
                if (role == 1 && g >= 1 &&
                    !role_wait<D>(bars.dpfree(), (uint32_t)(g - 1) & 1u, abort_flag, p.dev_status))
                    return false;
                // d = 128: S buffer g & 1 holds dS^T of block g-2 until dK (warp 14) has read it
                if (C::kDsInTmem && role == 0 && g >= 2 &&
                    !role_wait<D>(bars.kread(b), (uint32_t)((g - 2) >> 1) & 1u, abort_flag, p.dev_status))
                    return false;
                tc_fence_after();
                const uint32_t xb = (role == 0 ? sQ : sdO) + s * C::kQTile;
                const uint32_t kb = role == 0 ? sK : sV;
                const uint32_t dcol = tmem + (role == 0 ? C::kColS + b * BQ : C::kColDP);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t ko = (ks >> 2) * C::kKVSlab + (ks & 3) * 32;
                    const uint32_t qo = (ks >> 2) * C::kQSlab + (ks & 3) * 32;
                    mma_ss(dcol, smem_desc_sw128(kb + ko, 16, 1024), smem_desc_sw128(xb + qo, 16, 1024), idSP,
                           ks > 0);
                }
                mma_commit(bars.sfull(b));
                return true;
            };
            for (int T = 0; T < ntile && ok; ++T) {
                // K and V of tile T are in shared memory
                if (!(ok = role_wait<D>(bars.kv(), (uint32_t)T & 1u, abort_flag, p.dev_status))) break;
                const int g0 = T * n;
                if (role < 2) {
                    if (!(ok = issue_first(g0))) break;
                    for (int it = 0; it < n && ok; ++it) {
                        const int g = g0 + it, s = g % kStages, b = g & 1;
                        if (it + 1 < n && !(ok = issue_first(g + 1))) break;
                        if (!(ok = role_wait<D>(bars.pfull(b), (uint32_t)(g >> 1) & 1u, abort_flag, p.dev_status)))
                            break;
                        tc_fence_after();
                        const uint32_t qb = sQ + s * C::kQTile, gb = sdO + s * C::kQTile, dsb = sDs + b * C::kDsTile;
                        if (role == 0) {
                            // dV += P^T dO_i : A = P^T (bf16 pairs in the S columns), B = dO_i
#pragma unroll
                            for (int ks = 0; ks < BQ / 16; ++ks)
                                mma_ts(tmem + C::kColDV, tmem + C::kColS + b * BQ + (ks >> 1) * 32 + (ks & 1) * 8,
                                       smem_desc_sw128(gb + ks * 2048, C::kQSlab, 1024), idKV,
                                       (it > 0 || ks > 0) ? 1u : 0u);
                        } else {
                            // dK += dS^T Q_i : B = Q_i; A = dS^T from tensor memory beside P (d = 128)
                            // or the dS tile (K-major, 64 q per row)
                            if constexpr (C::kDsInTmem) {
#pragma unroll
                                for (int ks = 0; ks < BQ / 16; ++ks)
                                    mma_ts(tmem + C::kColDK,
                                           tmem + C::kColS + b * BQ + (ks >> 1) * 32 + (ks & 1) * 8 + 16,
                                           smem_desc_sw128(qb + ks * 2048, C::kQSlab, 1024), idKV,
                                           (it > 0 || ks > 0) ? 1u : 0u);
                                mma_commit(bars.kread(b));
                            } else {
#pragma unroll
                                for (int ks = 0; ks < BQ / 16; ++ks)
                                    mma_ss(tmem + C::kColDK, smem_desc_sw128(dsb + ks * 32, 16, 1024),
                                           smem_desc_sw128(qb + ks * 2048, C::kQSlab, 1024), idKV,
                                           (it > 0 || ks > 0) ? 1u : 0u);
                            }
                            mma_commit(bars.dsfree(b));
                        }
                        mma_commit(bars.qempty(s));
                    }
                } else {
                    for (int it = 0; it < n && ok; ++it) {
                        const int g = g0 + it, b = g & 1;
                        if (!(ok = role_wait<D>(bars.pfull(b), (uint32_t)(g >> 1) & 1u, abort_flag, p.dev_status)))
                            break;
                        // one dQ^T buffer: the drain warps must have read dQ^T of block g-1
                        if (g >= 1 &&
                            !(ok = role_wait<D>(bars.dqfree(), (uint32_t)(g - 1) & 1u, abort_flag, p.dev_status)))
                            break;
                        tc_fence_after();
                        const uint32_t dsb = sDs + b * C::kDsTile;
                        // dQ_i^T = K^T dS_i^T : A = K^T (d contiguous), B = dS (q contiguous)
#pragma unroll
                        for (int ks = 0; ks < BKV / 16; ++ks)
                            mma_ss(tmem + C::kColQ, smem_desc_sw128(sK + ks * 2048, C::kDqALbo, 1024),
                                   smem_desc_sw128(dsb + ks * 2048, C::kDsTile, 1024), idQ, ks > 0);
                        mma_commit(bars.dsfree(b));
                        mma_commit(bars.dqfull());
                    }
                }
                // this thread's products of tile T (those reading K, V and dS included)
                if (ok) mma_commit(bars.kvdone());
            }
            if (!ok) {
                // let every MMA this thread issued finish before tensor memory is released
                mma_commit(bars.drain(role));
                mbar_wait(bars.drain(role), 0, abort_flag, p.dev_status);
            }
        }
    } else if (warp < kDqWarp0) {
        // ------------------------------------------------------------ P / dS warps 0-7
        // As in bwd_main: thread = key, warps 0-3 queries 0-31 of a block, warps 4-7 queries 32-63.
        const int h = warp >> 2;
        const int key = (warp & 3) * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const float sl2 = p.scale * kLog2e;
        const uint32_t my_ds_row = (uint32_t)key * 128u;
        uint8_t *ds_gen = sm + C::kDsOff;
        bool ok = true;
        for (int T = 0; T < ntile; ++T) {
            for (int it = 0; it < n && ok; ++it) {
                const int g = T * n + it, s = g % kStages, b = g & 1;
                ok = mbar_wait(bars.sfull(b), (uint32_t)(g >> 1) & 1u, abort_flag, p.dev_status);
                if (ok && g >= 2)
                    ok = mbar_wait(bars.dsfree(b), (uint32_t)((g - 2) >> 1) & 1u, abort_flag, p.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const float *nl2 = ld_f + s * 2 * BQ;  // -LSE log2(e) of the 64 queries, then -D
                const float *ndv = nl2 + BQ;
                uint32_t pk[16], dk[16];
                uint32_t sr[32], pr[32];
                tmem_ld32(lane_base + C::kColS + b * BQ + h * 32, sr);
                tmem_ld32(lane_base + C::kColDP + h * 32, pr);
                tmem_wait_ld();
                reg_fence(sr);
                reg_fence(pr);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.dpfree());
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int q = h * 32 + 2 * t;
                    float4 nl, nd;
                    if ((t & 1) == 0) {
                        nl = *reinterpret_cast<const float4 *>(nl2 + q);
                        nd = *reinterpret_cast<const float4 *>(ndv + q);
                    }
                    const uint64_t l2p = (t & 1) ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y);
                    const uint64_t dvp = (t & 1) ? f2_pack(nd.z, nd.w) : f2_pack(nd.x, nd.y);
                    const uint64_t x2 =
                        f2_fma(f2_pack(__uint_as_float(sr[2 * t]), __uint_as_float(sr[2 * t + 1])), sl2x2, l2p);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    const uint64_t g2 =
                        f2_add(f2_pack(__uint_as_float(pr[2 * t]), __uint_as_float(pr[2 * t + 1])), dvp);
                    float d0, d1;
                    f2_unpack(f2_mul(f2_pack(p0, p1), g2), d0, d1);
                    pk[t] = pack_bf16(p0, p1);
                    dk[t] = pack_bf16(d0, d1);
                }
                tmem_st16(lane_base + C::kColS + b * BQ + h * 32, pk);
                if constexpr (C::kDsInTmem) tmem_st16(lane_base + C::kColS + b * BQ + h * 32 + 16, dk);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = h * 4 + c;
                    const uint32_t off = my_ds_row + (uint32_t)((chunk ^ (key & 7)) * 16);
                    *reinterpret_cast<uint4 *>(ds_gen + b * C::kDsTile + off) =
                        make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.pfull(b));
            }
            // -------------------------------------------------------- dK (warps 0-3), dV (warps 4-7) of tile T
            // The warps meet at the named barriers whatever `ok` says (after a timed-out wait the
            // work is skipped, the barriers kept), so that no warp waits for one that gave up.
            if (ok) {
                ok = mbar_wait(bars.kvdone(), (uint32_t)T & 1u, abort_flag, p.dev_status);
                if (ok && h == 1) ok = mbar_wait(bars.stagefree(), (uint32_t)T & 1u, abort_flag, p.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
            }
            uint8_t *stage = sm + (h == 0 ? C::kDsOff : C::kDqOff);
            const uint32_t acc = lane_base + (h == 0 ? C::kColDK : C::kColDV);
            const float mul = h == 0 ? p.scale : 1.f;
            if (ok) {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t a[32];
                    tmem_ld32(acc + c0, a);
                    tmem_wait_ld();
                    reg_fence(a);
                    uint32_t pa[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        pa[t] = pack_bf16(__uint_as_float(a[2 * t]) * mul, __uint_as_float(a[2 * t + 1]) * mul);
                    uint8_t *slab = stage + (c0 >> 6) * C::kKVSlab + key * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int u = ((c0 & 63) >> 3) + q;  // 16-byte unit within the 128-byte row
                        *reinterpret_cast<uint4 *>(slab + ((u ^ (key & 7)) << 4)) =
                            make_uint4(pa[4 * q], pa[4 * q + 1], pa[4 * q + 2], pa[4 * q + 3]);
                    }
                }
                fence_proxy_async_smem();
            }
            // the accumulators are read: the next tile's first dV and dK (after its first pfull)
            // may overwrite them
            tc_fence_before();
            named_bar_sync(2 + h, 128);
            if ((tid & 127) == 0 && ok) {
                const CUtensorMap *tm = h == 0 ? &tmdK : &tmdV;
                const uint32_t src = smem_addr(stage);
                const int kv0 = tile_kv0(T);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) tma_store_2d(tm, c * 64, kv0, src + c * C::kKVSlab);
                bulk_commit();
                bulk_wait_read_all();
            }
            // both staging tiles have been read: dS and dQ of the next tile may be written there
            named_bar_sync(4, 256);
        }
        if ((tid & 127) == 0) bulk_wait_all();
    } else if (warp < kTmaWarp) {
        // ------------------------------------------------------------ dQ drain warps 8-11
        // As in bwd_main; every drain thread runs the same sequence of named barriers whatever
        // happens (after a failed wait the work is skipped, the barriers kept).
        const int t = tid - kDqWarp0 * 32;  // 0..127 = d index (tensor memory lane); rows >= D are padding
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        float *dq_gen = reinterpret_cast<float *>(sm + C::kDqOff);
        bool alive = true;
        for (int T = 0; T < ntile; ++T) {
            const int head = tile_head(T);
            for (int it = 0; it < n; ++it) {
                const int g = T * n + it;
                bool ok = alive && mbar_wait(bars.dqfull(), (uint32_t)g & 1u, abort_flag, p.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                uint32_t r0[32], r1[32];
                if (ok) {
                    tc_fence_after();
                    tmem_ld32(lane_base + C::kColQ, r0);
                    tmem_ld32(lane_base + C::kColQ + 32, r1);
                    tmem_wait_ld();
                    reg_fence(r0);
                    reg_fence(r1);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.dqfree());
                }
                const size_t q0 = (size_t)head * p.N + (size_t)it * BQ;  // the block's accumulator rows
                if constexpr (D == 64) {
                    // d = 64: straight from registers, each warp adding 32 consecutive floats of one
                    // accumulator row per instruction (measured faster here than the staging tile;
                    // at d = 128 it was 7% slower)
                    if (ok && t < D) {
                        float *dst = dQacc + q0 * D + t;
#pragma unroll
                        for (int q = 0; q < 32; ++q) atomicAdd(dst + (size_t)q * D, __uint_as_float(r0[q]));
#pragma unroll
                        for (int q = 0; q < 32; ++q) atomicAdd(dst + (size_t)(32 + q) * D, __uint_as_float(r1[q]));
                    }
                } else {
                    auto stage = [&](const uint32_t(&r)[32], int hq) {
                        if (t == 0) bulk_wait_read_but_one();
                        named_bar_sync(1, 128);
                        if (ok && t < D) {
                            float *dst = dq_gen + hq * 32 * D;
#pragma unroll
                            for (int q = 0; q < 32; ++q) dst[q * D + t] = __uint_as_float(r[q]);
                            fence_proxy_async_smem();
                        }
                        named_bar_sync(1, 128);
                        if (t == 0 && ok) {
                            bulk_reduce_add_f32(dQacc + (q0 + 32 * hq) * D, sDq + hq * (C::kDqTile / 2),
                                                C::kDqTile / 2);
                            bulk_commit();
                        }
                    };
                    stage(r0, 0);
                    stage(r1, 1);
                }
                alive = alive && ok;
            }
            // the tile's reductions have read the staging tile: the epilogue may stage dV there
            if (t == 0) {
                bulk_wait_read_all();
                if (alive) mbar_arrive(bars.stagefree());
            }
        }
        if (t == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------- 3
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float *__restrict__ acc,
                                                              __nv_bfloat16 *__restrict__ dQ, float scale,
                                                              size_t n8) {
    // four 8-element units per thread and pass, their loads issued before any store
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n8; i0 += 4 * stride) {
        float4 a[4], b[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t i = i0 + u * stride;
            if (i < n8) {
                a[u] = reinterpret_cast<const float4 *>(acc)[2 * i];
                b[u] = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t i = i0 + u * stride;
            if (i < n8) {
                uint4 o;
                o.x = pack_bf16(a[u].x * scale, a[u].y * scale);
                o.y = pack_bf16(a[u].z * scale, a[u].w * scale);
                o.z = pack_bf16(b[u].x * scale, b[u].y * scale);
                o.w = pack_bf16(b[u].z * scale, b[u].w * scale);
                reinterpret_cast<uint4 *>(dQ)[i] = o;
            }
        }
    }
}

// dQ = bf16(s * accumulator) when the accumulator has npad > N rows per head: dQ row
// head * N + q comes from accumulator row head * npad + q.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_rows_kernel(const float *__restrict__ acc,
                                                                   __nv_bfloat16 *__restrict__ dQ, float scale,
                                                                   size_t n8, int N, int npad) {
    constexpr int U = D / 8;  // 8-element units per row
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / U, hh = row / (size_t)N;
        const size_t src = ((hh * (size_t)npad + (row - hh * (size_t)N)) * U + i % U) * 2;
        const float4 a = reinterpret_cast<const float4 *>(acc)[src];
        const float4 b = reinterpret_cast<const float4 *>(acc)[src + 1];
        uint4 o;
        o.x = pack_bf16(a.x * scale, a.y * scale);
        o.y = pack_bf16(a.z * scale, a.w * scale);
        o.z = pack_bf16(b.x * scale, b.y * scale);
        o.w = pack_bf16(b.z * scale, b.w * scale);
        reinterpret_cast<uint4 *>(dQ)[i] = o;
    }
}

// ------------------------------------------------------------------------- 4
// Split tiles: dK and dV rows are bf16 of the fp32 sum of the two query halves (dK is
// already scaled).  One CTA per (split tile, dK or dV).
template <int D>
__global__ void __launch_bounds__(256) bwd_kv_finish_kernel(const float *__restrict__ kvacc,
                                                             __nv_bfloat16 *__restrict__ dK,
                                                             __nv_bfloat16 *__restrict__ dV, int split_from,
                                                             int tiles_per_head, int N) {
    const int s = blockIdx.x >> 1, h = blockIdx.x & 1;
    const int tile = split_from + s;
    const size_t kv0 = (size_t)(tile / tiles_per_head) * N + (size_t)(tile % tiles_per_head) * BKV;
    const float4 *src = reinterpret_cast<const float4 *>(kvacc + ((size_t)s * 2 + h) * BKV * D);
    uint4 *dst = reinterpret_cast<uint4 *>((h == 0 ? dK : dV) + kv0 * D);
    for (int i = threadIdx.x; i < BKV * D / 8; i += blockDim.x) {
        const float4 a = src[2 * i], b = src[2 * i + 1];
        dst[i] = make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(b.x, b.y), pack_bf16(b.z, b.w));
    }
}

template <int D>
cudaError_t launch_d(const Problem &p, const BwdMaps &m, const void *O, const void *dO, const float *LSE,
                     void *dQ, void *dK, void *dV, float *Dv, float *dQacc, float *kvacc, int split,
                     cudaStream_t st) {
    const bool tail = p.N % BKV != 0;
    const int npad = bwd_rows_per_head(p.N);
    const size_t rows = (size_t)p.B * p.H * p.N, prows = (size_t)p.B * p.H * npad;
    const int tiles = (p.N / BKV) * p.B * p.H;
    if (kvacc == nullptr || tail) split = 0;
    {
        ProfScope prof_("bwd_pre", st);
        auto pre = npad != p.N ? bwd_pre_kernel<D, true> : bwd_pre_kernel<D, false>;
        pre<<<(unsigned)((prows + kPreRowsPerBlock<D> - 1) / kPreRowsPerBlock<D>), 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(O), static_cast<const __nv_bfloat16 *>(dO), Dv, dQacc, prows,
            reinterpret_cast<float4 *>(kvacc), bwd_split_bytes(split, D) / sizeof(float4), LSE, Dv + prows, p.N,
            npad);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (tail) {
        auto kt = bwd_main_kernel<D, false, true>;
        e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmemBytes);
        if (e != cudaSuccess) return e;
        {
            ProfScope prof_("bwd_main", st);
            kt<<<dim3((p.N + BKV - 1) / BKV, p.B * p.H), kThreads, BwdCfg<D>::kSmemBytes, st>>>(
                m.q, m.k, m.v, m.dO, m.dk, m.dv, p, Dv + prows, Dv, dQacc, static_cast<__nv_bfloat16 *>(dK),
                static_cast<__nv_bfloat16 *>(dV), INT_MAX, nullptr);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const size_t n8 = rows * D / 8;
        {
            ProfScope prof_("bwd_dq_convert", st);
            const unsigned grid = (unsigned)std::min<size_t>((n8 + 255) / 256, (size_t)device_sm_count() * 16);
            bwd_dq_convert_rows_kernel<D><<<grid, 256, 0, st>>>(
                dQacc, static_cast<__nv_bfloat16 *>(dQ), p.scale, n8, p.N, npad);
        }
        return cudaGetLastError();
    }
    // dense problems: the persistent kernel (every tile has the same query blocks)
    const bool persist = p.mask == nullptr;
    auto kern = bwd_main_kernel<D, false, false>;
    auto kp = bwd_persist_kernel<D>;
    auto kh = bwd_main_kernel<D, true, false>;
    e = persist ? cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmemBytes)
                : cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmemBytes);
    if (e == cudaSuccess && split > 0)
        e = cudaFuncSetAttribute(kh, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    {
        // one timing scope over both launches: together they are the five products of every tile
        ProfScope prof_("bwd_main", st);
        if (persist) {
            const int full = tiles - split;  // tiles of the persistent grid, the rest split in halves
            kp<<<(unsigned)std::min(full, device_sm_count()), kThreads, BwdCfg<D>::kSmemBytes, st>>>(
                m.q, m.k, m.v, m.dO, m.dk, m.dv, p, Dv + rows, Dv, dQacc, full);
        } else {
            kern<<<dim3(p.N / BKV, p.B * p.H), kThreads, BwdCfg<D>::kSmemBytes, st>>>(
                m.q, m.k, m.v, m.dO, m.dk, m.dv, p, Dv + rows, Dv, dQacc, static_cast<__nv_bfloat16 *>(dK),
                static_cast<__nv_bfloat16 *>(dV), tiles - split, kvacc);
        }
        e = cudaGetLastError();
        if (e == cudaSuccess && split > 0) {
            // programmatic dependent launch: the halves may start while the last full tiles run
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(2 * split));
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = BwdCfg<D>::kSmemBytes;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, kh, m.q, m.k, m.v, m.dO, m.dk, m.dv, p, static_cast<const float *>(Dv + rows),
                                   static_cast<const float *>(Dv), dQacc,
                                   static_cast<__nv_bfloat16 *>(dK), static_cast<__nv_bfloat16 *>(dV), tiles - split,
                                   kvacc);
            if (e == cudaSuccess) prof_.add_launch();
        }
    }
    if (e != cudaSuccess) return e;
    if (split > 0) {
        {
            ProfScope prof_("bwd_kv_finish", st);
            bwd_kv_finish_kernel<D><<<(unsigned)(2 * split), 256, 0, st>>>(
                kvacc, static_cast<__nv_bfloat16 *>(dK), static_cast<__nv_bfloat16 *>(dV), tiles - split,
                p.N / BKV, p.N);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t n8 = rows * D / 8;
    {
        ProfScope prof_("bwd_dq_convert", st);
        const unsigned grid = (unsigned)std::min<size_t>((n8 + 255) / 256, (size_t)device_sm_count() * 16);
        bwd_dq_convert_kernel<<<grid, 256, 0, st>>>(
            dQacc, static_cast<__nv_bfloat16 *>(dQ), p.scale, n8);
    }
    return cudaGetLastError();
}

// d = 256: bwd_pre, the two passes of bwd256_sm103.cu, the dQ conversion (no last-wave split).
cudaError_t launch_d256(const Problem &p, const BwdMaps &m, const void *O, const void *dO, const float *LSE,
                        void *dQ, void *dK, void *dV, float *Dv, float *dQacc, cudaStream_t st) {
    constexpr int D = 256;
    const int npad = bwd_rows_per_head(p.N);
    const size_t rows = (size_t)p.B * p.H * p.N, prows = (size_t)p.B * p.H * npad;
    {
        ProfScope prof_("bwd_pre", st);
        auto pre = npad != p.N ? bwd_pre_kernel<D, true> : bwd_pre_kernel<D, false>;
        pre<<<(unsigned)((prows + kPreRowsPerBlock<D> - 1) / kPreRowsPerBlock<D>), 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(O), static_cast<const __nv_bfloat16 *>(dO), Dv, dQacc, prows,
            nullptr, 0, LSE, Dv + prows, p.N, npad);
    }
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_bwd256_main(p, m, Dv + prows, Dv, dQacc, dK, dV, st);
    if (e != cudaSuccess) return e;
    const size_t n8 = rows * D / 8;
    const unsigned grid = (unsigned)std::min<size_t>((n8 + 255) / 256, (size_t)device_sm_count() * 16);
    ProfScope prof_("bwd_dq_convert", st);
    if (npad != p.N)
        bwd_dq_convert_rows_kernel<D><<<grid, 256, 0, st>>>(dQacc, static_cast<__nv_bfloat16 *>(dQ), p.scale, n8,
                                                            p.N, npad);
    else
        bwd_dq_convert_kernel<<<grid, 256, 0, st>>>(dQacc, static_cast<__nv_bfloat16 *>(dQ), p.scale, n8);
    return cudaGetLastError();
}

}  // namespace

int bwd_rows_per_head(int N) { return (N + BQ - 1) / BQ * BQ; }

int bwd_split_tiles(int B, int H, int N) {
    if (N % BKV != 0) return 0;  // partial tiles are never split
    const long long tiles = (long long)B * H * (N / BKV);
    const int sms = device_sm_count();
    const long long r = tiles % sms;
    return (tiles > sms && r > 0 && 2 * r <= sms) ? (int)r : 0;
}

size_t bwd_split_bytes(int split_tiles, int d) { return (size_t)split_tiles * 2 * BKV * d * sizeof(float); }

cudaError_t launch_bwd_bf16(const Problem &p, const BwdMaps &maps, const void *O, const void *dO,
                            const float *LSE, void *dQ, void *dK, void *dV, float *Dv, float *dQacc,
                            float *kvacc, int split_tiles, cudaStream_t st) {
    if (p.B * p.H > 65535) return cudaErrorNotSupported;
    switch (p.d) {
        case 64: return launch_d<64>(p, maps, O, dO, LSE, dQ, dK, dV, Dv, dQacc, kvacc, split_tiles, st);
        case 128: return launch_d<128>(p, maps, O, dO, LSE, dQ, dK, dV, Dv, dQacc, kvacc, split_tiles, st);
        case 256: return launch_d256(p, maps, O, dO, LSE, dQ, dK, dV, Dv, dQacc, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace attn
