// Recompute backward of the fused attention at head dimension d = 256 for sm_103a (bf16 in,
// fp32 accumulation): the same pass and the same chain rule as the d = 64 and d = 128 kernels
// (bwd_sm103.cu), for the d at which "On Fine-Grained I/O Complexity of Attention Backward
// Passes" (gist.science 2410.09397, Theorem 1.1) still puts an SM in the large-cache regime
// M >= d^2 (256 x 256 bf16 is 128 KB).
//
//   P = exp(s Q K^T - LSE),  dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
//   dQ = s dS K,  dK = s dS^T Q.
//
// What changes at d = 256 is what fits on one SM.  A 128-key tile's dK and dV accumulators
// (128 x 256 fp32 each) are 512 tensor-memory columns together, all there is, and its K and V
// (64 KB each) leave no room for a Q/dO ring beside them in 227 KB of shared memory.  So every
// key tile runs two passes, each a CTA of its own, both recomputing S:
//
//   pass B (dK, dQ): K and V resident, the 64-row query blocks that the mask keeps streaming
//     through.  Q arrives in two 128-column halves ("units"; a ring of three unit slots, 48 KB)
//     and dO in one 32 KB slot.  Four tcgen05 products per block:
//       S^T  = K Q_i^T       (128 x 64; issued in two halves, one per unit)
//       dP^T = V dO_i^T      (128 x 64)
//       dK  += dS^T Q_i      (two N = 128 products, one per unit, each releasing its unit)
//       dQ_i^T = K^T dS_i^T  (M = d: two M = 128 products)
//     The thread issuing S^T and dK puts the first half of S^T of block i + 1 before dK of
//     block i and the second half after it: the third unit slot lets the first half load
//     while block i still holds two, and the second can only load once dK of block i has read
//     the slot it takes.  Tensor memory: dK (256 columns), S, dP, dQ^T (2 x 64).  Eight warps
//     turn S and dP into dS (thread = key, each warp 32 queries of a block), one loads, three
//     issue (S^T and dK; dP^T; dQ^T).  dQ^T goes into the fp32 accumulator with atomic adds from
//     registers (a warp adds one 128-byte line of an accumulator row per instruction; no shared
//     memory is left for a staging tile): four drain warps take M half 0 (d 0-127), the eight
//     dS warps M half 1 right after publishing the next block's dS (with the four drain warps
//     alone the pass took 6% longer: their adds, throttled by the memory pipe, held back the
//     buffer's release, and with it dQ^T, dS and the loop).
//   pass A (dV): K resident, Q_i and dO_i in two-stage rings of their own (Q released once S^T
//     has read it, dO with the block's row terms once dV has: a stage shared by both held Q until
//     dV and put the next load's latency between dV and the next S^T, 3.0 ms for this pass on
//     2 x 16 x 8192 x 256); S^T into one of two buffers, P^T written back over it as bf16 pairs
//     by eight warps, dV += P^T dO_i with P^T read from tensor memory.  Tensor memory: dV (256
//     columns), S (2 x 64).
//
// Both passes run as one grid each on the caller's stream, pass B first (its CTAs take about
// two and a half times as long) and pass A as a programmatic dependent launch: neither reads what
// the other writes, so pass A's CTAs take the SMs that pass B's free; pass A's last CTA waits for
// pass B to complete before it ends, so that later work on the stream follows both.  Against the
// one-pass kernel at smaller d the products are 12 N^2 d instead of 10 N^2 d (S^T twice).
//
// Masks, 64-row mask blocks and partial tiles (N % 128 != 0) follow the one-pass kernel: query
// blocks that no kept mask entry covers are skipped, keys of a removed 64-key half get
// P = dS = 0, keys from N on get P = dS = 0 and are not stored, and queries from N on have
// P = 0 from their row terms (the padding rows of bwd_pre).
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "visit_bits.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int D = 256;
constexpr int BKV = 128;  // key rows per CTA
constexpr int BQ = 64;    // query rows per block
constexpr int kThreads = 512;
constexpr int kDqWarp0 = 8;   // pass B: warps 0-7 dS, 8-11 drain dQ^T
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;  // pass B: warps 13, 14, 15 issue; pass A: warp 13
constexpr uint32_t kTmemCols = 512;
constexpr int kKVSlab = BKV * 128;     // 16 KB: 64 columns of a 128-row tile (one TMA box)
constexpr int kKVTile = BKV * D * 2;   // 64 KB
constexpr int kQSlab = BQ * 128;       // 8 KB: 64 columns of a 64-row block
constexpr int kQTile = BQ * D * 2;     // 32 KB
constexpr int kDsTile = BKV * BQ * 2;  // 16 KB: dS^T, 128 rows x 128 B
// visited query blocks as a bit set: up to 32 * kMaxMaskWords 64-row blocks (N <= 65536);
// longer mask columns are read entry by entry
constexpr int kMaxMaskWords = 32;

struct CfgA {
    static constexpr int kStages = 2;
    static constexpr int kKOff = 0;
    static constexpr int kQOff = kKOff + kKVTile;             // Q ring (released by S^T)
    static constexpr int kdOOff = kQOff + kStages * kQTile;   // dO ring (released by dV)
    static constexpr int kLdOff = kdOOff + kStages * kQTile;  // per dO stage: -L2 of 64 rows
    static constexpr int kBarOff = kLdOff + kStages * BQ * 4;
    // kv, qfull[2], qempty[2], dofull[2], doempty[2], sfull[2], pfull[2], kvdone, drain
    static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 1 + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kBitsOff = kMiscOff + 64;
    static constexpr int kSmemBytes = kBitsOff + 4 * kMaxMaskWords + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
    static constexpr uint32_t kColDV = 0, kColS = D;  // dV, then two S buffers of 64 columns
    static_assert(kColS + 2 * BQ <= kTmemCols, "tensor memory budget");
};

struct CfgB {
    static constexpr int kUnits = 3;                   // Q unit slots
    static constexpr int kUnit = 2 * kQSlab;           // 16 KB: 128 columns of a Q block
    static constexpr int kKOff = 0, kVOff = kKVTile;
    static constexpr int kQOff = 2 * kKVTile;          // unit slot u at kQOff + u * kUnit
    static constexpr int kDsOff = kQOff + kUnits * kUnit;
    static constexpr int kdOOff = kDsOff + kDsTile;
    static constexpr int kLdOff = kdOOff + kQTile;     // per unit slot: -L2, -D of 64 rows
    static constexpr int kLdBytes = 2 * BQ * 4;
    static constexpr int kBarOff = kLdOff + kUnits * kLdBytes;
    // kv, qfull[3], qempty[3], dofull, doempty, sfull, sfree, dpfull, dpfree, pfull, dsfree,
    // dqfull, dqfree, kvdone, drain[3]
    static constexpr int kNumBars = 1 + 2 * kUnits + 2 + 4 + 2 + 2 + 1 + 3;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kBitsOff = kMiscOff + 64;
    static constexpr int kSmemBytes = kBitsOff + 4 * kMaxMaskWords + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
    // the epilogue stages the bf16 dK tile (64 KB) over the Q units and the dS tile
    static_assert(kdOOff - kQOff >= kKVTile, "dK staging area");
    static constexpr uint32_t kColDK = 0, kColS = 256, kColDP = 320, kColQ = 384;  // dQ^T: 2 x 64
    static_assert(kColQ + 2 * BQ <= kTmemCols, "tensor memory budget");
};

struct BarsA {
    static_assert(CfgA::kStages == 2 && CfgA::kNumBars == 15, "barrier indices below");
    uint32_t base;
    __device__ uint32_t kv() const { return base; }
    __device__ uint32_t qfull(int s) const { return base + 8u * (1 + s); }
    __device__ uint32_t qempty(int s) const { return base + 8u * (3 + s); }
    __device__ uint32_t dofull(int s) const { return base + 8u * (5 + s); }
    __device__ uint32_t doempty(int s) const { return base + 8u * (7 + s); }
    __device__ uint32_t sfull(int b) const { return base + 8u * (9 + b); }
    __device__ uint32_t pfull(int b) const { return base + 8u * (11 + b); }
    __device__ uint32_t kvdone() const { return base + 8u * 13; }
    __device__ uint32_t drain() const { return base + 8u * 14; }
};

struct BarsB {
    static_assert(CfgB::kUnits == 3 && CfgB::kNumBars == 21, "barrier indices below");
    uint32_t base;
    __device__ uint32_t kv() const { return base; }
    __device__ uint32_t qfull(int u) const { return base + 8u * (1 + u); }
    __device__ uint32_t qempty(int u) const { return base + 8u * (4 + u); }
    __device__ uint32_t dofull() const { return base + 8u * 7; }
    __device__ uint32_t doempty() const { return base + 8u * 8; }
    __device__ uint32_t sfull() const { return base + 8u * 9; }
    __device__ uint32_t sfree() const { return base + 8u * 10; }
    __device__ uint32_t dpfull() const { return base + 8u * 11; }
    __device__ uint32_t dpfree() const { return base + 8u * 12; }
    __device__ uint32_t pfull() const { return base + 8u * 13; }
    __device__ uint32_t dsfree() const { return base + 8u * 14; }
    __device__ uint32_t dqfull() const { return base + 8u * 15; }
    __device__ uint32_t dqfree() const { return base + 8u * 16; }
    __device__ uint32_t kvdone() const { return base + 8u * 17; }
    __device__ uint32_t drain(int r) const { return base + 8u * (18 + r); }
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// The query blocks of one key tile that the block mask keeps (all of them without a mask).
struct QueryBlocks {
    const uint8_t *hm;  // this head's mask, or nullptr
    int mb, mnb, kvt, nq;
    bool tail;
    VisitBits vb;
    bool use_bits;

    // a mask entry covering (the 64 rows of block iq, this tile's 128 keys) is kept
    __device__ bool visited(int iq) const {
        if (hm == nullptr) return true;
        if (mb == 128) return hm[(size_t)(iq >> 1) * mnb + kvt] != 0;
        const uint8_t *r = hm + (size_t)iq * mnb + 2 * kvt;
        if (tail) return (r[0] | (2 * kvt + 1 < mnb ? r[1] : 0)) != 0;  // last column may be absent
        return (r[0] | r[1]) != 0;
    }
    __device__ int count() const {
        if (hm == nullptr) return nq;
        if (use_bits) return vb.count();
        int n = 0;
        for (int iq = 0; iq < nq; ++iq) n += visited(iq) ? 1 : 0;
        return n;
    }
    // the visited block after iq (callers ask only while one remains)
    __device__ int next(int iq) const {
        if (hm == nullptr) return iq + 1;
        if (use_bits) return vb.next(iq);
        do {
            ++iq;
        } while (!visited(iq));
        return iq;
    }
    // 64-row mask blocks: the 64-key half of the tile that key lies in is kept for block iq
    __device__ bool half_kept(int iq, int key) const {
        if (hm == nullptr || mb != 64) return true;
        const int kcol = 2 * kvt + (key >> 6);
        return kcol < mnb && hm[(size_t)iq * mnb + kcol] != 0;
    }
};

// Sets up the CTA's query-block walk: every thread calls it (the bit set is built by all warps;
// the caller's next __syncthreads publishes it).
__device__ __forceinline__ QueryBlocks make_query_blocks(const Problem &p, int head, int kvt, int nq, bool tail,
                                                        uint32_t *words) {
    QueryBlocks v{p.head_mask(head), p.mask_block, p.mask_nb(), kvt, nq, tail, VisitBits{words, (nq + 31) >> 5},
                  false};
    v.use_bits = v.hm != nullptr && v.vb.nwords <= kMaxMaskWords;
    if (v.use_bits) build_visit_bits(words, nq, [&](int iq) { return v.visited(iq); });
    return v;
}

// The bf16 tile of one accumulator (128 rows x 256 fp32 columns of tensor memory, times mul) is
// written out by warps 0-7 (warp w: lanes 32 (w % 4).., columns 128 (w / 4)..): staged in the
// 128-byte-swizzled layout of four 64-column TMA boxes at `stage` and stored with tensor stores,
// or, for the last tile of a head with N % 128 != 0 (whose rows past N belong to the next head),
// row by row from registers.  Both groups of four warps meet at their named barrier whatever
// `ok` says, so that no warp waits there for one that gave up after a timed-out wait.
__device__ __forceinline__ void store_acc_tile(uint32_t acc, float mul, bool ok, bool partial, bool key_ok,
                                               int key, int h, uint8_t *stage, const CUtensorMap *tm, int kv0,
                                               __nv_bfloat16 *out) {
    if (partial) {
        if (!ok) return;
        uint4 *orow = reinterpret_cast<uint4 *>(out + ((size_t)kv0 + key) * D);
#pragma unroll 1
        for (int c0 = h * 128; c0 < h * 128 + 128; c0 += 32) {
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
        return;
    }
    if (ok) {
#pragma unroll 1
        for (int c0 = h * 128; c0 < h * 128 + 128; c0 += 32) {
            uint32_t a[32];
            tmem_ld32(acc + c0, a);
            tmem_wait_ld();
            reg_fence(a);
            uint32_t pa[16];
#pragma unroll
            for (int t = 0; t < 16; ++t)
                pa[t] = pack_bf16(__uint_as_float(a[2 * t]) * mul, __uint_as_float(a[2 * t + 1]) * mul);
            uint8_t *slab = stage + (c0 >> 6) * kKVSlab + key * 128;
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
    if ((threadIdx.x & 127) == 0 && ok) {
        const uint32_t src = smem_addr(stage);
#pragma unroll
        for (int c = 2 * h; c < 2 * h + 2; ++c) tma_store_2d(tm, c * 64, kv0, src + c * kKVSlab);
        bulk_commit();
        bulk_wait_all();
    }
}

// ------------------------------------------------------------------------- pass B: dK, dQ
// Grid (ceil(N / 128), B * H): CTA (x, y) takes key tile x of head y.
template <bool TAIL>
__global__ void __launch_bounds__(kThreads, 1)
bwd256_dkdq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const __grid_constant__ CUtensorMap tmdK, const Problem p, const float *__restrict__ L2,
                   const float *__restrict__ Dv, float *__restrict__ dQacc, __nv_bfloat16 *__restrict__ dK) {
    using C = CfgB;
    // pass A reads nothing this grid writes: let it start on the SMs this grid frees
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const BarsB bars{smem_addr(sm + C::kBarOff)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nq = TAIL ? (p.N + BQ - 1) / BQ : p.N / BQ;
    const int npad = TAIL ? nq * BQ : p.N;  // rows per head of D, L2 and the dQ accumulator
    const int kvt = blockIdx.x, head = blockIdx.y;
    const int kv0 = head * p.N + kvt * BKV;
    const uint32_t sK = smem_addr(sm + C::kKOff), sV = smem_addr(sm + C::kVOff);
    const uint32_t sQ = smem_addr(sm + C::kQOff), sdO = smem_addr(sm + C::kdOOff);
    const uint32_t sDs = smem_addr(sm + C::kDsOff), sLd = smem_addr(sm + C::kLdOff);
    const float *ld_f = reinterpret_cast<const float *>(sm + C::kLdOff);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bars.kv(), 1);
        for (int u = 0; u < C::kUnits; ++u) {
            mbar_init(bars.qfull(u), 1);
            mbar_init(bars.qempty(u), 1);   // the dK product over the unit (issuer 0)
        }
        mbar_init(bars.dofull(), 1);
        mbar_init(bars.doempty(), 1);       // dP^T (issuer 1)
        mbar_init(bars.sfull(), 1);
        mbar_init(bars.sfree(), 8);         // one lane of each dS warp
        mbar_init(bars.dpfull(), 1);
        mbar_init(bars.dpfree(), 8);
        mbar_init(bars.pfull(), 8);
        mbar_init(bars.dsfree(), 2);        // dK (issuer 0) and dQ^T (issuer 2) read dS
        mbar_init(bars.dqfull(), 1);
        mbar_init(bars.dqfree(), 12);       // one lane of each drain warp and of each dS warp
        mbar_init(bars.kvdone(), 1);
        for (int r = 0; r < 3; ++r) mbar_init(bars.drain(r), 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(bars.kv(), 2 * kKVTile);
        for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(sK + c * kKVSlab, &tmK, c * 64, kv0, bars.kv());
            tma_load_2d(sV + c * kKVSlab, &tmV, c * 64, kv0, bars.kv());
        }
    }
    const QueryBlocks qb = make_query_blocks(p, head, kvt, nq, TAIL,
                                             reinterpret_cast<uint32_t *>(sm + C::kBitsOff));
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int n = qb.count();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmdO);
            int iq = -1;
            for (int it = 0; it < n; ++it) {
                iq = qb.next(iq);
                const int q0 = head * p.N + iq * BQ;
                const int ql = TAIL ? head * npad + iq * BQ : q0;  // the block's rows of L2 and D
                // unit 2 it: Q columns 0-127, with the block's row terms
                int u = 2 * it, s = u % C::kUnits;
                if (u >= C::kUnits &&
                    !mbar_wait(bars.qempty(s), ((uint32_t)(u / C::kUnits) & 1u) ^ 1u, abort_flag, p.dev_status))
                    break;
                mbar_arrive_expect_tx(bars.qfull(s), C::kUnit + C::kLdBytes);
                for (int c = 0; c < 2; ++c)
                    tma_load_2d(sQ + s * C::kUnit + c * kQSlab, &tmQ, c * 64, q0, bars.qfull(s));
                bulk_load(sLd + s * C::kLdBytes, L2 + ql, BQ * 4, bars.qfull(s));
                bulk_load(sLd + s * C::kLdBytes + BQ * 4, Dv + ql, BQ * 4, bars.qfull(s));
                // dO_i once dP^T of the block before has read the slot
                if (it >= 1 && !mbar_wait(bars.doempty(), (uint32_t)(it - 1) & 1u, abort_flag, p.dev_status)) break;
                mbar_arrive_expect_tx(bars.dofull(), kQTile);
                for (int c = 0; c < D / 64; ++c) tma_load_2d(sdO + c * kQSlab, &tmdO, c * 64, q0, bars.dofull());
                // unit 2 it + 1: Q columns 128-255
                u = 2 * it + 1;
                s = u % C::kUnits;
                if (u >= C::kUnits &&
                    !mbar_wait(bars.qempty(s), ((uint32_t)(u / C::kUnits) & 1u) ^ 1u, abort_flag, p.dev_status))
                    break;
                mbar_arrive_expect_tx(bars.qfull(s), C::kUnit);
                for (int c = 0; c < 2; ++c)
                    tma_load_2d(sQ + s * C::kUnit + c * kQSlab, &tmQ, 128 + c * 64, q0, bars.qfull(s));
            }
        }
    } else if (warp >= kMmaWarp) {
        // ------------------------------------------------------------ MMA issuers
        const int role = warp - kMmaWarp;  // 0: S^T and dK, 1: dP^T, 2: dQ^T
        if (lane == 0 && n > 0) {
            constexpr uint32_t idSP = idesc_bf16_f32(BKV, BQ, false, false);  // S^T, dP^T
            constexpr uint32_t idK = idesc_bf16_f32(BKV, 128, false, true);   // dK, one unit's columns
            constexpr uint32_t idQ = idesc_bf16_f32(128, BQ, true, true);     // dQ^T, one M half
            bool ok = mbar_wait(bars.kv(), 0, abort_flag, p.dev_status);
            if (role == 0) {
                // S^T_it over unit 2 it + hf (k-steps 8 hf .. 8 hf + 7: the unit's 128 columns of d)
                auto s_half = [&](int it, int hf) -> bool {
                    const int u = 2 * it + hf, s = u % C::kUnits;
                    if (!mbar_wait(bars.qfull(s), (uint32_t)(u / C::kUnits) & 1u, abort_flag, p.dev_status))
                        return false;
                    // one S buffer: the dS warps must have read S^T of the block before
                    if (hf == 0 && it >= 1 &&
                        !mbar_wait(bars.sfree(), (uint32_t)(it - 1) & 1u, abort_flag, p.dev_status))
                        return false;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int ks = 8 * hf + k;
                        const uint32_t ko = (ks >> 2) * kKVSlab + (ks & 3) * 32;
                        const uint32_t qo = s * C::kUnit + (k >> 2) * kQSlab + (k & 3) * 32;
                        mma_ss(tmem + C::kColS, smem_desc_sw128(sK + ko, 16, 1024),
                               smem_desc_sw128(sQ + qo, 16, 1024), idSP, ks > 0);
                    }
                    if (hf == 1) mma_commit(bars.sfull());
                    return true;
                };
                if (ok) ok = s_half(0, 0) && s_half(0, 1);
                for (int it = 0; it < n && ok; ++it) {
                    if (it + 1 < n && !(ok = s_half(it + 1, 0))) break;
                    if (!(ok = mbar_wait(bars.pfull(), (uint32_t)it & 1u, abort_flag, p.dev_status))) break;
                    tc_fence_after();
                    // dK[:, 128 hf ..] += dS^T Q_i[:, 128 hf ..] : A = dS^T (K-major, 64 queries a row),
                    // B = unit 2 it + hf (d contiguous); the commit releases the unit
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int s = (2 * it + hf) % C::kUnits;
#pragma unroll
                        for (int ks = 0; ks < BQ / 16; ++ks)
                            mma_ss(tmem + C::kColDK + hf * 128, smem_desc_sw128(sDs + ks * 32, 16, 1024),
                                   smem_desc_sw128(sQ + s * C::kUnit + ks * 2048, kQSlab, 1024), idK,
                                   (it > 0 || ks > 0) ? 1u : 0u);
                        mma_commit(bars.qempty(s));
                    }
                    mma_commit(bars.dsfree());
                    if (it + 1 < n && !(ok = s_half(it + 1, 1))) break;
                }
                if (ok) mma_commit(bars.kvdone());
            } else if (role == 1) {
                for (int it = 0; it < n && ok; ++it) {
                    if (!(ok = mbar_wait(bars.dofull(), (uint32_t)it & 1u, abort_flag, p.dev_status))) break;
                    // one dP buffer: the dS warps must have read dP^T of the block before
                    if (it >= 1 && !(ok = mbar_wait(bars.dpfree(), (uint32_t)(it - 1) & 1u, abort_flag, p.dev_status)))
                        break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t ko = (ks >> 2) * kKVSlab + (ks & 3) * 32;
                        const uint32_t qo = (ks >> 2) * kQSlab + (ks & 3) * 32;
                        mma_ss(tmem + C::kColDP, smem_desc_sw128(sV + ko, 16, 1024),
                               smem_desc_sw128(sdO + qo, 16, 1024), idSP, ks > 0);
                    }
                    mma_commit(bars.dpfull());
                    mma_commit(bars.doempty());
                }
            } else {
                for (int it = 0; it < n && ok; ++it) {
                    if (!(ok = mbar_wait(bars.pfull(), (uint32_t)it & 1u, abort_flag, p.dev_status))) break;
                    // one dQ^T buffer: the drain warps (M half 0) and the dS warps (M half 1) must
                    // have read dQ^T of the block before
                    if (it >= 1 && !(ok = mbar_wait(bars.dqfree(), (uint32_t)(it - 1) & 1u, abort_flag, p.dev_status)))
                        break;
                    tc_fence_after();
                    // dQ_i^T[128 mh ..] = K^T[128 mh ..] dS_i^T : A = K^T (d contiguous; the half's two
                    // 64-column boxes one leading byte offset apart), B = dS (queries contiguous)
#pragma unroll
                    for (int mh = 0; mh < 2; ++mh) {
#pragma unroll
                        for (int ks = 0; ks < BKV / 16; ++ks)
                            mma_ss(tmem + C::kColQ + mh * BQ,
                                   smem_desc_sw128(sK + mh * 2 * kKVSlab + ks * 2048, kKVSlab, 1024),
                                   smem_desc_sw128(sDs + ks * 2048, kDsTile, 1024), idQ, ks > 0);
                    }
                    mma_commit(bars.dsfree());
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
        // ------------------------------------------------------------ dS warps 0-7
        // Thread = key (tensor memory lane 32 (warp % 4) + lane); warps 0-3 take queries 0-31
        // of each block, warps 4-7 queries 32-63.
        const int h = warp >> 2;
        const int key = (warp & 3) * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const float sl2 = p.scale * kLog2e;
        const bool key_ok = !TAIL || kvt * BKV + key < p.N;
        uint8_t *ds_gen = sm + C::kDsOff;
        int iq = -1, iq_prev = -1;
        bool ok = true;
        // M half 1 of dQ^T of block j (d = 128 + 32 (warp % 4) + lane; queries 32 h ..): read, release,
        // add into the accumulator (the drain warps take M half 0)
        auto drain_half1 = [&](int j, int iqj) -> bool {
            bool w = mbar_wait(bars.dqfull(), (uint32_t)j & 1u, abort_flag, p.dev_status);
            w = __all_sync(0xffffffffu, w);
            if (!w) return false;
            tc_fence_after();
            uint32_t r[32];
            tmem_ld32(lane_base + C::kColQ + BQ + h * 32, r);
            tmem_wait_ld();
            reg_fence(r);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.dqfree());
            float *col = dQacc + (size_t)(TAIL ? head * npad + iqj * BQ : head * p.N + iqj * BQ) * D +
                         (size_t)(h * 32) * D + 128 + key;
#pragma unroll
            for (int q = 0; q < 32; ++q) atomicAdd(col + (size_t)q * D, __uint_as_float(r[q]));
            return true;
        };
        for (int it = 0; it < n; ++it) {
            iq = qb.next(iq);
            const bool row_kept = qb.half_kept(iq, key);  // warp-uniform: 32 keys lie in one half
            ok = mbar_wait(bars.sfull(), (uint32_t)it & 1u, abort_flag, p.dev_status);
            if (ok) ok = mbar_wait(bars.dpfull(), (uint32_t)it & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const float *nl2 = ld_f + ((2 * it) % C::kUnits) * (2 * BQ);  // -L2 of the 64 queries, then -D
            const float *ndv = nl2 + BQ;
            uint32_t sr[32], pr[32], dk[16];
            if (row_kept) {
                tmem_ld32(lane_base + C::kColS + h * 32, sr);
                tmem_ld32(lane_base + C::kColDP + h * 32, pr);
                tmem_wait_ld();
                reg_fence(sr);
                reg_fence(pr);
            }
            // S^T and dP^T are in registers: both buffers may take the next block's products
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bars.sfree());
                mbar_arrive(bars.dpfree());
            }
            if (!row_kept) {
#pragma unroll
                for (int t = 0; t < 16; ++t) dk[t] = 0u;
            } else {
                // two queries per step: x = s log2(e) S - L2, p = 2^x, dS = p (dP - D)
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int q = h * 32 + 2 * t;
                    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[2 * t]), __uint_as_float(sr[2 * t + 1])),
                                               sl2x2, f2_pack(nl2[q], nl2[q + 1]));
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    const uint64_t g2 = f2_add(f2_pack(__uint_as_float(pr[2 * t]), __uint_as_float(pr[2 * t + 1])),
                                               f2_pack(ndv[q], ndv[q + 1]));
                    float d0, d1;
                    f2_unpack(f2_mul(f2_pack(p0, p1), g2), d0, d1);
                    dk[t] = key_ok ? pack_bf16(d0, d1) : 0u;
                }
            }
            // one dS tile: dK and dQ^T of the block before must have read it
            if (it >= 1) {
                ok = mbar_wait(bars.dsfree(), (uint32_t)(it - 1) & 1u, abort_flag, p.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            // dS^T row into shared memory, 128-byte swizzle: 16-byte chunk c at c ^ (row % 8)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int chunk = h * 4 + c;
                *reinterpret_cast<uint4 *>(ds_gen + key * 128 + ((chunk ^ (key & 7)) << 4)) =
                    make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.pfull());
            if (it >= 1 && !drain_half1(it - 1, iq_prev)) { ok = false; break; }
            iq_prev = iq;
        }
        if (ok && n > 0) ok = drain_half1(n - 1, iq_prev);
        // ------------------------------------------------------------ dK epilogue
        // staged over the Q units and the dS tile, once dK and the last dQ^T (which reads dS)
        // are complete
        if (n > 0) {
            if (ok) ok = mbar_wait(bars.kvdone(), 0, abort_flag, p.dev_status);
            if (ok) ok = mbar_wait(bars.dsfree(), (uint32_t)(n - 1) & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            store_acc_tile(lane_base + C::kColDK, p.scale, ok, TAIL && (kvt + 1) * BKV > p.N, key_ok, key, h,
                           sm + C::kQOff, &tmdK, kv0, dK);
        } else if (key_ok) {
            uint4 *orow = reinterpret_cast<uint4 *>(dK + ((size_t)kv0 + key) * D) + h * 16;
            for (int q = 0; q < 16; ++q) orow[q] = make_uint4(0, 0, 0, 0);
        }
    } else if (warp < kTmaWarp) {
        // ------------------------------------------------------------ dQ drain warps 8-11
        // M half 0 of dQ^T (d 0-127; the dS warps take half 1).  Thread t = d index (tensor memory
        // lane); column q = query of the block.  For each query the 32 lanes of a warp add 32
        // consecutive floats of the accumulator row (one 128-byte line; 16-byte adds of four
        // consecutive d after a 4 x 4 lane transpose make the same number of line requests and
        // measured 10% slower on this pass).
        const int t = tid - kDqWarp0 * 32;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        bool alive = true;
        int iq = -1;
        for (int it = 0; it < n; ++it) {
            iq = qb.next(iq);
            bool ok = alive && mbar_wait(bars.dqfull(), (uint32_t)it & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            alive = ok;
            if (!ok) continue;
            tc_fence_after();
            float *row0 = dQacc + (size_t)(TAIL ? head * npad + iq * BQ : head * p.N + iq * BQ) * D + t;
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(lane_base + C::kColQ, r0);
                tmem_ld32(lane_base + C::kColQ + 32, r1);
                tmem_wait_ld();
                reg_fence(r0);
                reg_fence(r1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.dqfree());
                float *col = row0;
#pragma unroll
                for (int q = 0; q < 32; ++q) atomicAdd(col + (size_t)q * D, __uint_as_float(r0[q]));
#pragma unroll
                for (int q = 0; q < 32; ++q) atomicAdd(col + (size_t)(32 + q) * D, __uint_as_float(r1[q]));
            }
        }
    }

    // a tile that visits no query block still received its K (and V) tile: let that copy land first
    if (n == 0 && tid == 0) mbar_wait(bars.kv(), 0, abort_flag, p.dev_status);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------- pass A: dV
template <bool TAIL>
__global__ void __launch_bounds__(kThreads, 1)
bwd256_dv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmdO, const __grid_constant__ CUtensorMap tmdV,
                 const Problem p, const float *__restrict__ L2, __nv_bfloat16 *__restrict__ dV) {
    using C = CfgA;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const BarsA bars{smem_addr(sm + C::kBarOff)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nq = TAIL ? (p.N + BQ - 1) / BQ : p.N / BQ;
    const int npad = TAIL ? nq * BQ : p.N;
    const int kvt = blockIdx.x, head = blockIdx.y;
    const int kv0 = head * p.N + kvt * BKV;
    const uint32_t sK = smem_addr(sm + C::kKOff), sQ = smem_addr(sm + C::kQOff), sdO = smem_addr(sm + C::kdOOff);
    const uint32_t sLd = smem_addr(sm + C::kLdOff);
    const float *ld_f = reinterpret_cast<const float *>(sm + C::kLdOff);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bars.kv(), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bars.qfull(s), 1);
            mbar_init(bars.qempty(s), 1);   // S^T of the stage's block
            mbar_init(bars.dofull(s), 1);
            mbar_init(bars.doempty(s), 1);  // dV of the stage's block
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.sfull(b), 1);
            mbar_init(bars.pfull(b), 8);   // one lane of each P warp
        }
        mbar_init(bars.kvdone(), 1);
        mbar_init(bars.drain(), 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(bars.kv(), kKVTile);
        for (int c = 0; c < D / 64; ++c) tma_load_2d(sK + c * kKVSlab, &tmK, c * 64, kv0, bars.kv());
    }
    const QueryBlocks qb = make_query_blocks(p, head, kvt, nq, TAIL,
                                             reinterpret_cast<uint32_t *>(sm + C::kBitsOff));
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int n = qb.count();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmdO);
            int iq = -1;
            for (int it = 0; it < n; ++it) {
                const int s = it % S;
                const uint32_t ph = ((uint32_t)(it / S) & 1u) ^ 1u;  // the stage's previous use
                iq = qb.next(iq);
                const int q0 = head * p.N + iq * BQ;
                const int ql = TAIL ? head * npad + iq * BQ : q0;
                if (it >= S && !mbar_wait(bars.qempty(s), ph, abort_flag, p.dev_status)) break;
                mbar_arrive_expect_tx(bars.qfull(s), kQTile);
                for (int c = 0; c < D / 64; ++c) tma_load_2d(sQ + s * kQTile + c * kQSlab, &tmQ, c * 64, q0, bars.qfull(s));
                // dO with the row terms: the P warps read those after S^T has released Q
                if (it >= S && !mbar_wait(bars.doempty(s), ph, abort_flag, p.dev_status)) break;
                mbar_arrive_expect_tx(bars.dofull(s), kQTile + BQ * 4);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d(sdO + s * kQTile + c * kQSlab, &tmdO, c * 64, q0, bars.dofull(s));
                bulk_load(sLd + s * BQ * 4, L2 + ql, BQ * 4, bars.dofull(s));
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && n > 0) {
            constexpr uint32_t idS = idesc_bf16_f32(BKV, BQ, false, false);  // S^T
            constexpr uint32_t idV = idesc_bf16_f32(BKV, D, false, true);    // dV
            bool ok = mbar_wait(bars.kv(), 0, abort_flag, p.dev_status);
            // S^T_it into buffer it & 1.  The buffer held P of block it - 2, read by the dV that
            // this thread issued before.
            auto issue_s = [&](int it) -> bool {
                const int s = it % S, b = it & 1;
                if (!mbar_wait(bars.qfull(s), (uint32_t)(it / S) & 1u, abort_flag, p.dev_status)) return false;
                tc_fence_after();
                const uint32_t qb0 = sQ + s * kQTile;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t ko = (ks >> 2) * kKVSlab + (ks & 3) * 32;
                    const uint32_t qo = (ks >> 2) * kQSlab + (ks & 3) * 32;
                    mma_ss(tmem + C::kColS + b * BQ, smem_desc_sw128(sK + ko, 16, 1024),
                           smem_desc_sw128(qb0 + qo, 16, 1024), idS, ks > 0);
                }
                mma_commit(bars.sfull(b));
                mma_commit(bars.qempty(s));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int it = 0; it < n && ok; ++it) {
                const int s = it % S, b = it & 1;
                if (it + 1 < n && !(ok = issue_s(it + 1))) break;
                if (!(ok = mbar_wait(bars.pfull(b), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status))) break;
                if (!(ok = mbar_wait(bars.dofull(s), (uint32_t)(it / S) & 1u, abort_flag, p.dev_status))) break;
                tc_fence_after();
                // dV += P^T dO_i : A = P^T (bf16 pairs; queries 32 h.. at S column 32 h), B = dO_i
                const uint32_t gb = sdO + s * kQTile;
#pragma unroll
                for (int ks = 0; ks < BQ / 16; ++ks)
                    mma_ts(tmem + C::kColDV, tmem + C::kColS + b * BQ + (ks >> 1) * 32 + (ks & 1) * 8,
                           smem_desc_sw128(gb + ks * 2048, kQSlab, 1024), idV, (it > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bars.doempty(s));
            }
            if (ok) {
                mma_commit(bars.kvdone());
            } else {
                mma_commit(bars.drain());
                mbar_wait(bars.drain(), 0, abort_flag, p.dev_status);
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ P warps 0-7
        const int h = warp >> 2;
        const int key = (warp & 3) * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const float sl2 = p.scale * kLog2e;
        const bool key_ok = !TAIL || kvt * BKV + key < p.N;
        int iq = -1;
        bool ok = true;
        for (int it = 0; it < n; ++it) {
            const int s = it % S, b = it & 1;
            iq = qb.next(iq);
            const bool row_kept = key_ok && qb.half_kept(iq, key);
            ok = mbar_wait(bars.sfull(b), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status);
            // the row terms arrive with dO
            if (ok) ok = mbar_wait(bars.dofull(s), (uint32_t)(it / S) & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t pk[16];
            if (__any_sync(0xffffffffu, row_kept)) {
                const float *nl2 = ld_f + s * BQ;
                uint32_t sr[32];
                tmem_ld32(lane_base + C::kColS + b * BQ + h * 32, sr);
                tmem_wait_ld();
                reg_fence(sr);
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int q = h * 32 + 2 * t;
                    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[2 * t]), __uint_as_float(sr[2 * t + 1])),
                                               sl2x2, f2_pack(nl2[q], nl2[q + 1]));
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    pk[t] = row_kept ? pack_bf16(ex2(x0), ex2(x1)) : 0u;
                }
            } else {
#pragma unroll
                for (int t = 0; t < 16; ++t) pk[t] = 0u;
            }
            // P^T as bf16 pairs over the first 16 of this half's own 32 S columns
            tmem_st16(lane_base + C::kColS + b * BQ + h * 32, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.pfull(b));
        }
        if (n > 0) {
            if (ok) ok = mbar_wait(bars.kvdone(), 0, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            // every product that read the rings completed before kvdone: stage dV there
            store_acc_tile(lane_base + C::kColDV, 1.f, ok, TAIL && (kvt + 1) * BKV > p.N, key_ok, key, h,
                           sm + C::kQOff, &tmdV, kv0, dV);
        } else if (key_ok) {
            uint4 *orow = reinterpret_cast<uint4 *>(dV + ((size_t)kv0 + key) * D) + h * 16;
            for (int q = 0; q < 16; ++q) orow[q] = make_uint4(0, 0, 0, 0);
        }
    }

    // a tile that visits no query block still received its K (and V) tile: let that copy land first
    if (n == 0 && tid == 0) mbar_wait(bars.kv(), 0, abort_flag, p.dev_status);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // This grid runs beside pass B as its dependent launch, and later work on the stream (the
    // dQ conversion) reads the accumulator that pass B adds into.  The grid's last CTA (launched
    // last, so it waits only for pass B's tail) ends by waiting for pass B to complete: this grid
    // then completes after pass B.  Its other CTAs leave their SMs at once.
    if (blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <bool TAIL>
cudaError_t launch_passes(const Problem &p, const BwdMaps &m, const float *L2, const float *Dv, float *dQacc,
                          __nv_bfloat16 *dK, __nv_bfloat16 *dV, cudaStream_t st) {
    auto kb = bwd256_dkdq_kernel<TAIL>;
    auto ka = bwd256_dv_kernel<TAIL>;
    cudaError_t e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgB::kSmemBytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgA::kSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((p.N + BKV - 1) / BKV), (unsigned)(p.B * p.H));
    ProfScope prof_("bwd_main", st);
    kb<<<grid, kThreads, CfgB::kSmemBytes, st>>>(m.q, m.k, m.v, m.dO, m.dk, p, L2, Dv, dQacc, dK);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: pass A may start while pass B's last CTAs run
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = CfgA::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, ka, m.q, m.k, m.dO, m.dv, p, L2, dV);
    if (e == cudaSuccess) prof_.add_launch();
    return e;
}

}  // namespace

cudaError_t launch_bwd256_main(const Problem &p, const BwdMaps &maps, const float *L2, const float *Dv,
                               float *dQacc, void *dK, void *dV, cudaStream_t st) {
    auto *k = static_cast<__nv_bfloat16 *>(dK);
    auto *v = static_cast<__nv_bfloat16 *>(dV);
    return p.N % BKV != 0 ? launch_passes<true>(p, maps, L2, Dv, dQacc, k, v, st)
                          : launch_passes<false>(p, maps, L2, Dv, dQacc, k, v, st);
}

}  // namespace attn
