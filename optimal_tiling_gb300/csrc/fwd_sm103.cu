// Fused streaming attention forward for sm_103a (bf16 in, fp32 accumulation).
//
// Method: "The I/O Complexity of Attention" exposition (blog.aeilot.top,
// attention-io-complexity), sections "Softmax without storing the score matrix"
// (the stabilised online update: running max m, sum l, accumulator u, o = u/l)
// and "Large caches: where FlashAttention's I/O comes from" (a query block and
// its output state stay on chip while all of K, V is scanned).  The page's
// schedule is for a generic two-level machine; these kernels are shaped for GB300:
//
//   * a CTA owns 128-row query tiles of one head; K/V are scanned in 128-row
//     blocks through a TMA ring in shared memory (128-byte swizzle);
//   * both products run on tcgen05 with fp32 accumulators in tensor memory:
//     S = Q K^T into a 128-column S buffer, O += P V into a d-column O buffer;
//     P (bf16) is written back over its own S buffer and fed to the second MMA
//     straight from tensor memory;
//   * softmax warps own one query row per thread (TMEM lane = row) and run the
//     softmax, the O rescale and the epilogue; one warp issues TMA, one lane of
//     another allocates tensor memory and issues every MMA;
//   * the running max is kept in the log2 domain (scores scaled by s*log2 e) and
//     O is rescaled only when a row's max grows by more than 8 (a factor 256):
//     the final division uses the same reference max, so the result is the same
//     function and only rounding differs;
//   * key blocks whose mask entries for a query tile are all zero are never
//     loaded or multiplied; with 64-row mask blocks a visited 128-key block can
//     still be removed for one half of the keys or one half of the rows, and
//     the softmax warps drop those 64-column halves (whole 32-column TMEM
//     chunks, the same for every row of a warp) before the max and the exps;
//   * a negative score scale s sets the instruction descriptor's negate-A bit
//     of the S product, so the tensor core returns sign(s) Q K^T and the softmax
//     scales it by |s|.
// Three kernels:
//   fwd_bf16_kernel       one query tile per CTA, S double-buffered so that S of
//                         block j+1 is computed while the softmax of block j runs
//                         (block masks, or N % 256 != 0; d = 64, 128);
//   fwd_bf16_pp_kernel    two query tiles per CTA sharing every K/V block, the
//                         tensor core on one tile while the other's softmax runs
//                         (no mask, N % 256 == 0; d = 64, 128);
//   fwd_bf16_ring_kernel  d = 256: K and V stream through a ring of 32 KB pieces.
// Every mbarrier wait is bounded; an expired wait sets the device status word
// and the CTA unwinds without touching the GPU's state.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "visit_bits.cuh"

namespace attn {
namespace {

using namespace ptx;

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

constexpr int BM = 128;             // query rows per CTA
constexpr int BN = 128;             // keys per streamed block
constexpr int kThreads = 192;       // 4 softmax warps + TMA warp + MMA warp
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol0 = 0, kSCol1 = 128, kOCol = 256;

template <int D>
struct FwdCfg {
    static constexpr int kChunks = D / 64;                     // 64-element (128 B) swizzle atoms per row
    // K/V ring depth: as deep as the shared memory allows (block-sparse masks scatter the
    // key blocks a tile visits, so their loads miss L2 and need the latency covered)
    static constexpr int kStages = D == 64 ? 6 : 3;
    static constexpr int kTileBytes = BM * D * 2;              // Q tile == K tile == V tile bytes
    static constexpr int kChunkBytes = BM * 128;               // one 64-column slab of a tile
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kTileBytes;
    static constexpr int kVOff = kKOff + kStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kStages * kTileBytes;
    // q, kfull[S], kempty[S], vfull[S], vempty[S], sfull[2], pfull[2], drain (PV's completion is
    // read from the release of its V stage)
    static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 1;
    // misc: tensor-memory address (+0), abort flag (+8), per K/V stage the 64-key halves of its
    // block that some row of the tile keeps (+16, 64-row masks)
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kHalvesOff = kMiscOff + 16;
    // visited key blocks as a bit set: masks with up to 32 * kMaxMaskWords blocks per row
    static constexpr int kMaxMaskWords = 256;
    static constexpr int kBitsOff = kMiscOff + 64;
    static constexpr int kSmemBytes = kBitsOff + 4 * kMaxMaskWords + 1024;  // + slack to align the base
    static_assert(kHalvesOff + kStages <= kBitsOff, "misc area");
    static_assert(kChunkBytes == 16384, "slab layout");
    static_assert(kOCol + D <= kTmemCols, "tensor memory budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

struct Bars {
    uint32_t base;
    int stages;
    __device__ uint32_t q() const { return base; }
    __device__ uint32_t kfull(int s) const { return base + 8u * (1 + s); }
    __device__ uint32_t kempty(int s) const { return base + 8u * (1 + stages + s); }
    __device__ uint32_t vfull(int s) const { return base + 8u * (1 + 2 * stages + s); }
    __device__ uint32_t vempty(int s) const { return base + 8u * (1 + 3 * stages + s); }
    __device__ uint32_t sfull(int b) const { return base + 8u * (1 + 4 * stages + b); }
    __device__ uint32_t pfull(int b) const { return base + 8u * (3 + 4 * stages + b); }
    __device__ uint32_t drain() const { return base + 8u * (5 + 4 * stages); }
};

// Key block j (128 keys) is visited by query tile t when any mask entry that
// covers the 128 x 128 square (t, j) is kept: one entry for 128-blocks, four
// for 64-blocks.  hm is this head's [mnb][mnb] mask (nullptr: no mask).
// TAIL (N % 128 != 0): the last tile or key block may cover a single 64-row mask row or column,
// the last one of the mask; the entries past it do not exist and are not read.
template <bool TAIL = false>
__device__ __forceinline__ bool visited(const uint8_t *hm, int mb, int mnb, int t, int j) {
    if (hm == nullptr) return true;
    if (mb == 128) return hm[(size_t)t * mnb + j] != 0;
    const uint8_t *r0 = hm + (size_t)(2 * t) * mnb + 2 * j, *r1 = r0 + mnb;
    if constexpr (TAIL) {
        const bool j1 = 2 * j + 1 < mnb, t1 = 2 * t + 1 < mnb;
        return (r0[0] | (j1 ? r0[1] : 0) | (t1 ? r1[0] : 0) | (t1 && j1 ? r1[1] : 0)) != 0;
    }
    return (r0[0] | r0[1] | r1[0] | r1[1]) != 0;
}

// Instruction descriptors of the S = Q K^T product (128 x 128, both operands K-major), and the
// same with A negated for a negative score scale.
constexpr uint32_t kIdS = idesc_bf16_f32(BM, BN, false, false);
constexpr uint32_t kIdSNeg = kIdS | kIdescNegateA;

// FINE: the mask has 64-row blocks (a visited 128-key block can be removed for a 64-key half
// of a warp's rows, and the softmax then skips that half's scores altogether).
template <int D, bool TAIL, bool FINE>
__global__ void __launch_bounds__(kThreads, 1)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Problem p,
                __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE) {
    using C = FwdCfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Bars bars{smem_addr(sm + C::kBarOff), S};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, head = blockIdx.y;
    const int nb = TAIL ? (p.N + BN - 1) / BN : p.N / BN;  // key blocks (the last one partial under TAIL)
    const uint8_t *hm = p.head_mask(head);
    const int mb = p.mask_block, mnb = p.mask_nb();
    uint32_t *vwords = reinterpret_cast<uint32_t *>(sm + C::kBitsOff);
    // FINE without TAIL: the visit set is over 64-key mask columns (a column is visited when
    // either 64-row half of the tile keeps it), and the visited columns are taken two at a time
    // into one 128-key block: K and V rows of the first in rows 0-63 of the ring stage, of the
    // second in rows 64-127 (K and V maps with 64-row boxes).  A lone last column leaves the upper
    // rows unused: its upper key half counts as removed for every row.
    constexpr bool kPack = FINE && !TAIL;
    const int nunits = kPack ? 2 * nb : nb;  // bit-set units: mask columns or key blocks
    const int nwords = (nunits + 31) >> 5;
    const bool use_bits = hm != nullptr && nwords <= C::kMaxMaskWords;
    const int row0 = head * p.N + tile * BM;  // first row of this tile in the [B*H*N, D] view
    const uint32_t sQ = smem_addr(sm + C::kQOff), sK = smem_addr(sm + C::kKOff), sV = smem_addr(sm + C::kVOff);
    // FINE: per K/V stage, the key halves of its block that some row of the tile keeps (bit 0:
    // keys 0-63), written by the producer before the V load's arrival and read by the issuer after
    // its wait on V, so that PV skips the k-steps of a half no row keeps (their P is zero)
    uint8_t *khalves = sm + C::kHalvesOff;

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bars.q(), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bars.kfull(s), 1);
            mbar_init(bars.kempty(s), 1);
            mbar_init(bars.vfull(s), 1);
            mbar_init(bars.vempty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.sfull(b), 1);
            mbar_init(bars.pfull(b), 4 * 32);
        }
        mbar_init(bars.drain(), 1);
        fence_barrier_init();
        // the Q tile is needed whatever the mask says: start its load before the mask is read
        mbar_arrive_expect_tx(bars.q(), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) tma_load_2d(sQ + c * C::kChunkBytes, &tmQ, c * 64, row0, bars.q());
    }
    // kPack: mask column c of the tile's two mask rows
    auto col_kept = [&](int c) -> bool {
        const uint8_t *r0 = hm + (size_t)(2 * tile) * mnb + c;
        return (r0[0] | r0[mnb]) != 0;
    };
    auto unit_visited = [&](int u) -> bool { return kPack ? col_kept(u) : visited<TAIL>(hm, mb, mnb, tile, u); };
    if (use_bits) build_visit_bits(vwords, nunits, unit_visited);
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const VisitBits vb{vwords, nwords};
    int nu = nunits;  // units (key blocks, or mask columns under kPack) this query tile visits
    if (use_bits) {
        nu = vb.count();
    } else if (hm != nullptr) {  // rows longer than the bit set: read the mask directly
        nu = 0;
        for (int u = 0; u < nunits; ++u) nu += unit_visited(u) ? 1 : 0;
    }
    const int n = kPack ? (nu + 1) / 2 : nu;  // key blocks of the loop
    // the visited unit after u (callers ask only while one remains)
    auto next_block = [&](int u) -> int {
        if (hm == nullptr) return u + 1;
        if (use_bits) return vb.next(u);
        do {
            ++u;
        } while (!unit_visited(u));
        return u;
    };
    // kPack: the two mask columns of block it, c[1] = -1 for a lone last column
    auto block_cols = [&](int it, int &cur, int c[2]) {
        c[0] = cur = next_block(cur);
        c[1] = -1;
        if (2 * it + 1 < nu) c[1] = cur = next_block(cur);
    };

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int j = -1;
            for (int it = 0; it < n; ++it) {
                const int s = it % S;
                const uint32_t ph = (uint32_t)(it / S) & 1u;
                if constexpr (kPack) {
                    int cols[2];
                    block_cols(it, j, cols);
                    const int r0 = head * p.N + cols[0] * 64, r1 = head * p.N + cols[1] * 64;
                    const uint32_t bytes = (cols[1] >= 0 ? 2u : 1u) * (uint32_t)(C::kTileBytes / 2);
                    if (it >= S && !mbar_wait(bars.kempty(s), ph ^ 1u, abort_flag, p.dev_status)) break;
                    mbar_arrive_expect_tx(bars.kfull(s), bytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        const uint32_t dst = sK + s * C::kTileBytes + c * C::kChunkBytes;
                        tma_load_2d(dst, &tmK, c * 64, r0, bars.kfull(s));
                        if (cols[1] >= 0) tma_load_2d(dst + C::kChunkBytes / 2, &tmK, c * 64, r1, bars.kfull(s));
                    }
                    if (it >= S && !mbar_wait(bars.vempty(s), ph ^ 1u, abort_flag, p.dev_status)) break;
                    // every visited column is kept by some row of the tile
                    khalves[s] = cols[1] >= 0 ? 3u : 1u;
                    mbar_arrive_expect_tx(bars.vfull(s), bytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        const uint32_t dst = sV + s * C::kTileBytes + c * C::kChunkBytes;
                        tma_load_2d(dst, &tmV, c * 64, r0, bars.vfull(s));
                        if (cols[1] >= 0) tma_load_2d(dst + C::kChunkBytes / 2, &tmV, c * 64, r1, bars.vfull(s));
                    }
                    continue;
                }
                j = next_block(j);
                const int krow = head * p.N + j * BN;
                if (it >= S && !mbar_wait(bars.kempty(s), ph ^ 1u, abort_flag, p.dev_status)) break;
                mbar_arrive_expect_tx(bars.kfull(s), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_2d(sK + s * C::kTileBytes + c * C::kChunkBytes, &tmK, c * 64, krow, bars.kfull(s));
                if (it >= S && !mbar_wait(bars.vempty(s), ph ^ 1u, abort_flag, p.dev_status)) break;
                if constexpr (FINE) {
                    const uint8_t *r0 = hm + (size_t)(2 * tile) * mnb + 2 * j, *r1 = r0 + mnb;
                    const bool t1 = !TAIL || 2 * tile + 1 < mnb, j1 = !TAIL || 2 * j + 1 < mnb;
                    const bool h0 = (r0[0] | (t1 ? r1[0] : 0)) != 0;
                    const bool h1 = ((j1 ? r0[1] : 0) | (t1 && j1 ? r1[1] : 0)) != 0;
                    khalves[s] = (uint8_t)((h0 ? 1u : 0u) | (h1 ? 2u : 0u));
                }
                mbar_arrive_expect_tx(bars.vfull(s), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_2d(sV + s * C::kTileBytes + c * C::kChunkBytes, &tmV, c * 64, krow, bars.vfull(s));
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n > 0) {
            // a negative scale: S = (-Q) K^T, scaled by |s| in the softmax
            const uint32_t idS = p.scale < 0.f ? kIdSNeg : kIdS;
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
            bool ok = mbar_wait(bars.q(), 0, abort_flag, p.dev_status);
            // S_it = Q K_it^T into S buffer (it & 1)
            auto issue_s = [&](int it) -> bool {
                const int s = it % S;
                if (!mbar_wait(bars.kfull(s), (uint32_t)(it / S) & 1u, abort_flag, p.dev_status)) return false;
                tc_fence_after();
                const uint32_t dcol = tmem + ((it & 1) ? kSCol1 : kSCol0);
                const uint32_t kb = sK + s * C::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
                    mma_ss(dcol, smem_desc_sw128(sQ + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024), idS,
                           ks > 0);
                }
                mma_commit(bars.kempty(s));
                mma_commit(bars.sfull(it & 1));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int it = 0; it < n && ok; ++it) {
                if (it + 1 < n && !(ok = issue_s(it + 1))) break;
                const int s = it % S;
                // V_it was loaded long ago: check it before waiting for P_it, so that only P_it is
                // waited for on the path from the softmax to PV
                if (!(ok = mbar_wait(bars.vfull(s), (uint32_t)(it / S) & 1u, abort_flag, p.dev_status))) break;
                if (!(ok = mbar_wait(bars.pfull(it & 1), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status))) break;
                tc_fence_after();
                const uint32_t pcol = tmem + ((it & 1) ? kSCol1 : kSCol0);
                const uint32_t vb = sV + s * C::kTileBytes;
                const uint32_t kh = FINE ? khalves[s] : 3u;
                if (kh == 3u) {
#pragma unroll
                    for (int ks = 0; ks < BN / 16; ++ks)
                        mma_ts(tmem + kOCol, pcol + ks * 8, smem_desc_sw128(vb + ks * 2048, C::kChunkBytes, 1024),
                               idO, (it > 0 || ks > 0) ? 1u : 0u);
                } else {  // one key half kept by some row: its four k-steps only
                    const int k0 = kh == 1u ? 0 : 4;
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        mma_ts(tmem + kOCol, pcol + (k0 + k4) * 8,
                               smem_desc_sw128(vb + (k0 + k4) * 2048, C::kChunkBytes, 1024), idO,
                               (it > 0 || k4 > 0) ? 1u : 0u);
                }
                // vempty(s) also tells the softmax that PV_it is complete (O may be rescaled, or read
                // after the last block): one commit per block fewer than a barrier of its own
                mma_commit(bars.vempty(s));
            }
            if (!ok) {
                // let every MMA already issued finish before tensor memory is released
                mma_commit(bars.drain());
                mbar_wait(bars.drain(), 0, abort_flag, p.dev_status);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warps 0-3
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float sl2 = fabsf(p.scale) * kLog2e;  // S holds sign(s) Q K^T
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        // 64-row mask blocks: this warp's 32 rows lie in one mask row, so each
        // 64-key half of a visited block is kept or removed for the whole warp.
        constexpr bool fine = FINE;
        // a removed half's scores are not loaded or reduced (FINE and TAIL only)
        constexpr bool kSkipHalves = FINE || TAIL;
        // TAIL: rows 64-127 of the last tile may all lie past N, below the mask's last row
        const bool wrow = !TAIL || 2 * tile + warp / 2 < mnb;
        const uint8_t *wmask = fine && wrow ? hm + (size_t)(2 * tile + warp / 2) * mnb : nullptr;
        int j = -1;  // key block of iteration it (tracked for fine masks and under TAIL)
        for (int it = 0; it < n; ++it) {
            const int b = it & 1;
            bool half_kept[2] = {true, true};
            if constexpr (kPack) {
                int cols[2];
                block_cols(it, j, cols);
                half_kept[0] = wmask[cols[0]] != 0;
                half_kept[1] = cols[1] >= 0 && wmask[cols[1]] != 0;
            } else if (fine) {
                j = next_block(j);
                if (wmask != nullptr) {
                    half_kept[0] = wmask[2 * j] != 0;
                    half_kept[1] = (!TAIL || 2 * j + 1 < mnb) && wmask[2 * j + 1] != 0;
                } else {  // rows past N only (TAIL)
                    half_kept[0] = half_kept[1] = false;
                }
            } else if (TAIL) {
                j = next_block(j);
            }
            // TAIL: keys of the last block from N on do not exist (their rows in the K and V tiles
            // belong to the next head, or read as zeros past the end): their scores are -inf, and a
            // half with no key below N counts as removed
            int lim = BN;
            if constexpr (TAIL) {
                if (j == nb - 1) lim = p.N - j * BN;
                if (lim <= BN / 2) half_kept[1] = false;
            }
            ok = mbar_wait(bars.sfull(b), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t scol = lane_base + (b ? kSCol1 : kSCol0);
            uint32_t r[4][32];
            if (!kSkipHalves || half_kept[0]) {
                tmem_ld32(scol + 0, r[0]);
                tmem_ld32(scol + 32, r[1]);
            }
            if (!kSkipHalves || half_kept[1]) {
                tmem_ld32(scol + 64, r[2]);
                tmem_ld32(scol + 96, r[3]);
            }
            tmem_wait_ld();
            reg_fence(r[0]);
            reg_fence(r[1]);
            reg_fence(r[2]);
            reg_fence(r[3]);
            if constexpr (TAIL) {
                if (lim < BN) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (32 * q + t >= lim) r[q][t] = 0xff800000u;  // -inf
                }
            }
            // row max: four independent chains (one per 32-column chunk), then combined
            float mxq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (kSkipHalves && !half_kept[q >> 1]) {
                    mxq[q] = -INFINITY;
                    continue;
                }
                mxq[q] = fmaxf(__uint_as_float(r[q][0]), __uint_as_float(r[q][1]));
#pragma unroll
                for (int t = 1; t < 16; ++t)
                    mxq[q] = fmax3(mxq[q], __uint_as_float(r[q][2 * t]), __uint_as_float(r[q][2 * t + 1]));
                if (!half_kept[q >> 1]) mxq[q] = -INFINITY;
            }
            const float mx = fmaxf(fmax3(mxq[0], mxq[1], mxq[2]), mxq[3]);
            // a warp with nothing kept so far keeps m_used = -inf
            const float m_new = mx == -INFINITY ? m_used : fmaxf(m_used, mx * sl2);
            float alpha = 1.f;
            if (m_new > m_used + kRescaleThreshold) {
                alpha = ex2(m_used - m_new);
                m_used = m_new;
            }
            // p = 2^(s log2e S - m): pairs on the packed FMA path, exps on MUFU
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
            const uint64_t negm2 = f2_pack(-m_used, -m_used);
            uint64_t sumq[4];  // four independent row-sum chains
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                sumq[q] = f2_pack(0.f, 0.f);
                uint32_t pk[16];
                if (!half_kept[q >> 1]) {
                    // removed half: P = 0, nothing added to the row sum
#pragma unroll
                    for (int t = 0; t < 16; ++t) pk[t] = 0u;
                    tmem_st16(scol + q * 16, pk);
                    continue;
                }
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(r[q][2 * t]), __uint_as_float(r[q][2 * t + 1])),
                                               sl2x2, negm2);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const uint64_t y2 = f2_pack(ex2(x0), ex2(x1));
                    sumq[q] = f2_add(sumq[q], y2);
                    float y0, y1;
                    f2_unpack(y2, y0, y1);
                    pk[t] = pack_bf16(y0, y1);
                }
                tmem_st16(scol + q * 16, pk);
            }
            float rs0, rs1;
            f2_unpack(f2_add(f2_add(sumq[0], sumq[1]), f2_add(sumq[2], sumq[3])), rs0, rs1);
            const float rs = rs0 + rs1;
            l = l * alpha + rs;
            tmem_wait_st();
            if (it > 0) {
                // PV_{it-1} complete: the release of V stage (it-1) % S, use (it-1) / S
                ok = mbar_wait(bars.vempty((it - 1) % S), (uint32_t)((it - 1) / S) & 1u, abort_flag, p.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(lane_base + kOCol + c0, o);
                        tmem_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                        tmem_st32(lane_base + kOCol + c0, o);
                    }
                    tmem_wait_st();
                }
            }
            tc_fence_before();
            mbar_arrive(bars.pfull(b));
        }
        // ------------------------------------------------------------ epilogue
        if (ok && n > 0) {
            ok = mbar_wait(bars.vempty((n - 1) % S), (uint32_t)((n - 1) / S) & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        const size_t grow = (size_t)row0 + tid;
        // rows of this tile below N (TAIL: the last tile of a head is partial)
        const int valid = TAIL ? min(BM, p.N - tile * BM) : BM;
        if (TAIL && n > 0 && valid < BM) {
            // the rows past N belong to the next head: each thread stores its own row, if it
            // exists, instead of one tensor store of the whole tile
            if (ok) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kOCol + c0, o);
                    tmem_wait_ld();
                    reg_fence(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        pk[t] = pack_bf16(__uint_as_float(o[2 * t]) * inv, __uint_as_float(o[2 * t + 1]) * inv);
                    if (tid < valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(O + grow * D + c0);
#pragma unroll
                        for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
                if (tid < valid) LSE[grow] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
            }
        } else if (n > 0) {
            // O leaves through the Q tile (the last MMA that read it completed before PV_{n-1}):
            // rows in the 128-byte-swizzled layout of the 64-column TMA box, then one thread
            // stores the tile.  The four warps meet at the named barrier whatever `ok` says.
            uint8_t *stage = sm + C::kQOff;
            if (ok) {
                // a row whose every visited score was removed (64-row masks) has l = 0:
                // O = 0 and LSE = -inf, with the tensor-memory loads still warp-wide
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kOCol + c0, o);
                    tmem_wait_ld();
                    reg_fence(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        pk[t] = pack_bf16(__uint_as_float(o[2 * t]) * inv, __uint_as_float(o[2 * t + 1]) * inv);
                    uint8_t *slab = stage + (c0 >> 6) * C::kChunkBytes + tid * 128;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int u = ((c0 & 63) >> 3) + v;  // 16-byte unit within the 128-byte row
                        *reinterpret_cast<uint4 *>(slab + ((u ^ (tid & 7)) << 4)) =
                            make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
                LSE[grow] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
                fence_proxy_async_smem();
            }
            named_bar_sync(1, 128);
            if (tid == 0 && ok) {
                const uint32_t src = smem_addr(stage);
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) tma_store_2d(&tmO, c * 64, row0, src + c * C::kChunkBytes);
                bulk_commit();
                bulk_wait_all();
            }
        } else if (tid < valid) {
            // every key block removed: O = 0, LSE = -inf
            uint4 *orow = reinterpret_cast<uint4 *>(O + grow * D);
            for (int v = 0; v < D / 8; ++v) orow[v] = make_uint4(0, 0, 0, 0);
            LSE[grow] = -INFINITY;
        }
    }

    // a tile that visits no key block still received its Q tile: let that copy land first
    if (n == 0 && tid == 0) mbar_wait(bars.q(), 0, abort_flag, p.dev_status);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Two query tiles per CTA ("ping-pong"): 256 query rows, two softmax
// warpgroups (warps 0-3: tile A, warps 4-7: tile B), TMA warp 8, MMA warp 9.
// Tensor memory: S_A, S_B (128 columns each; P overwrites its own S), O_A, O_B
// (d columns each).  MMA order per key block j:
//     PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
// so the tensor core works on one tile while the other tile's softmax runs, and,
// because tcgen05 MMAs of one thread complete in issue order, "S_X(j+1) done"
// also means "PV_X(j) done": the softmax may rescale O_X as soon as it sees
// S_X(j+1).  Used without a block mask (both tiles visit every key block).
constexpr int kPPThreads = 320;
constexpr int kPPTmaWarp = 8;
constexpr int kPPMmaWarp = 9;

template <int D>
struct PPCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kStages = D == 64 ? 4 : 2;
    static constexpr int kTileBytes = BM * D * 2;
    static constexpr int kChunkBytes = BM * 128;
    static constexpr int kQOff = 0;                                // Q_A, Q_B
    static constexpr int kKOff = 2 * kTileBytes;
    static constexpr int kVOff = kKOff + kStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kStages * kTileBytes;
    // q, kfull[S], kempty[S], vfull[S], vempty[S], sfull[2], pfull[2], odone[2], drain
    static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 2 + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 64 + 1024;
    static constexpr uint32_t kOCol0 = 256;
    static __device__ __forceinline__ uint32_t scol(int x) { return x ? 128u : 0u; }
    static_assert(kOCol0 + 2 * D <= kTmemCols, "tensor memory budget");
};

struct PPBars {
    uint32_t base;
    int stages;
    __device__ uint32_t q() const { return base; }
    __device__ uint32_t kfull(int s) const { return base + 8u * (1 + s); }
    __device__ uint32_t kempty(int s) const { return base + 8u * (1 + stages + s); }
    __device__ uint32_t vfull(int s) const { return base + 8u * (1 + 2 * stages + s); }
    __device__ uint32_t vempty(int s) const { return base + 8u * (1 + 3 * stages + s); }
    __device__ uint32_t sfull(int x) const { return base + 8u * (1 + 4 * stages + x); }
    __device__ uint32_t pfull(int x) const { return base + 8u * (3 + 4 * stages + x); }
    __device__ uint32_t odone(int x) const { return base + 8u * (5 + 4 * stages + x); }
    __device__ uint32_t drain() const { return base + 8u * (7 + 4 * stages); }
};

template <int D>
__global__ void __launch_bounds__(kPPThreads, 1)
fwd_bf16_pp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Problem p,
                   __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE) {
    using C = PPCfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const PPBars bars{smem_addr(sm + C::kBarOff), S};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head = blockIdx.y;
    const int n = p.N / BN;                        // key blocks (no mask on this path)
    const int row0 = head * p.N + blockIdx.x * 2 * BM;  // first row of tile A; tile B follows

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bars.q(), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bars.kfull(s), 1);
            mbar_init(bars.kempty(s), 1);
            mbar_init(bars.vfull(s), 1);
            mbar_init(bars.vempty(s), 1);  // unused: a V stage is free when the next K stage is
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bars.sfull(x), 1);
            mbar_init(bars.pfull(x), 128);
            mbar_init(bars.odone(x), 1);
        }
        mbar_init(bars.drain(), 1);
        fence_barrier_init();
    }
    if (warp == kPPMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sQ = smem_addr(sm + C::kQOff), sK = smem_addr(sm + C::kKOff), sV = smem_addr(sm + C::kVOff);

    if (warp == kPPTmaWarp) {
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(bars.q(), 2 * C::kTileBytes);
            for (int x = 0; x < 2; ++x)
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_2d(sQ + x * C::kTileBytes + c * C::kChunkBytes, &tmQ, c * 64, row0 + x * BM, bars.q());
            for (int j = 0; j < n; ++j) {
                const int s = j % S;
                const uint32_t ph = (uint32_t)(j / S) & 1u;
                const int krow = head * p.N + j * BN;
                if (j >= S && !mbar_wait(bars.kempty(s), ph ^ 1u, abort_flag, p.dev_status)) break;
                mbar_arrive_expect_tx(bars.kfull(s), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_2d(sK + s * C::kTileBytes + c * C::kChunkBytes, &tmK, c * 64, krow, bars.kfull(s));
                // V(j - S) was read by PV_A, PV_B(j - S), which complete before S_B(j - S + 1), whose
                // commit releases K(j - S + 1) (kempty completes once per use of a K stage): that
                // release frees V's stage too, one commit per block fewer on the issuing thread
                if (j >= S && !mbar_wait(bars.kempty((j - S + 1) % S), (uint32_t)((j - S + 1) / S) & 1u, abort_flag,
                                         p.dev_status))
                    break;
                mbar_arrive_expect_tx(bars.vfull(s), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_2d(sV + s * C::kTileBytes + c * C::kChunkBytes, &tmV, c * 64, krow, bars.vfull(s));
            }
        }
    } else if (warp == kPPMmaWarp) {
        if (lane == 0) {
            // a negative scale: S = (-Q) K^T, scaled by |s| in the softmax
            const uint32_t idS = p.scale < 0.f ? kIdSNeg : kIdS;
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
            auto mma_s = [&](int x, int j) {
                const uint32_t kb = sK + (j % S) * C::kTileBytes, qb = sQ + x * C::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
                    mma_ss(tmem + C::scol(x), smem_desc_sw128(qb + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024),
                           idS, ks > 0);
                }
                mma_commit(bars.sfull(x));
            };
            auto mma_pv = [&](int x, int j) {
                const uint32_t vb = sV + (j % S) * C::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks)
                    mma_ts(tmem + C::kOCol0 + x * D, tmem + C::scol(x) + ks * 8,
                           smem_desc_sw128(vb + ks * 2048, C::kChunkBytes, 1024), idO, (j > 0 || ks > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(bars.q(), 0, abort_flag, p.dev_status) &&
                      mbar_wait(bars.kfull(0), 0, abort_flag, p.dev_status);
            if (ok) {
                tc_fence_after();
                mma_s(0, 0);
                mma_s(1, 0);
                mma_commit(bars.kempty(0));
            }
            for (int j = 0; j < n && ok; ++j) {
                const int s = j % S;
                const bool more = j + 1 < n;
                const uint32_t ph = (uint32_t)j & 1u;
                // V_j and K_{j+1} were loaded long ago: check them while tile A's softmax still
                // runs, so that only P_A(j) is waited for on the path from softmax to PV
                if (!(ok = mbar_wait(bars.vfull(s), (uint32_t)(j / S) & 1u, abort_flag, p.dev_status))) break;
                if (more && !(ok = mbar_wait(bars.kfull((j + 1) % S), (uint32_t)((j + 1) / S) & 1u, abort_flag,
                                             p.dev_status)))
                    break;
                if (!(ok = mbar_wait(bars.pfull(0), ph, abort_flag, p.dev_status))) break;
                tc_fence_after();
                mma_pv(0, j);
                if (more) mma_s(0, j + 1);
                else mma_commit(bars.odone(0));
                if (!(ok = mbar_wait(bars.pfull(1), ph, abort_flag, p.dev_status))) break;
                tc_fence_after();
                mma_pv(1, j);
                if (more) {
                    mma_s(1, j + 1);
                    mma_commit(bars.kempty((j + 1) % S));
                } else {
                    mma_commit(bars.odone(1));
                }
            }
            if (!ok) {
                mma_commit(bars.drain());
                mbar_wait(bars.drain(), 0, abort_flag, p.dev_status);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax, one tile per warpgroup
        const int x = warp >> 2;  // 0: tile A, 1: tile B
        const int r = tid & 127;  // row within the tile == tensor memory lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t scol = lane_base + C::scol(x);
        const uint32_t ocol = lane_base + C::kOCol0 + x * D;
        const float sl2 = fabsf(p.scale) * kLog2e;  // S holds sign(s) Q K^T
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            ok = mbar_wait(bars.sfull(x), (uint32_t)j & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // S in two 64-column halves, so that only 64 scores are live at a time: the max over
            // both halves, the exps of the high half (still in registers), then the low half
            // loaded again; P of the high half (columns 32..63, which hold S of keys 32..63) is
            // written only after that reload
            uint32_t rr[2][32];
            tmem_ld32(scol + 0, rr[0]);
            tmem_ld32(scol + 32, rr[1]);
            tmem_wait_ld();
            reg_fence(rr[0]);
            reg_fence(rr[1]);
            // row max in four independent chains of 16-column runs (a single chain through the
            // second half made the max a long dependent sequence)
            float mx4[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t *v = &rr[c >> 1][16 * (c & 1)];
                mx4[c] = fmaxf(__uint_as_float(v[0]), __uint_as_float(v[1]));
#pragma unroll
                for (int t = 1; t < 8; ++t) mx4[c] = fmax3(mx4[c], __uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
            }
            tmem_ld32(scol + 64, rr[0]);
            tmem_ld32(scol + 96, rr[1]);
            tmem_wait_ld();
            reg_fence(rr[0]);
            reg_fence(rr[1]);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t *v = &rr[c >> 1][16 * (c & 1)];
#pragma unroll
                for (int t = 0; t < 8; ++t) mx4[c] = fmax3(mx4[c], __uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
            }
            const float mx = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
            const float m_new = fmaxf(m_used, mx * sl2);
            float alpha = 1.f;
            if (m_new > m_used + kRescaleThreshold) {
                alpha = ex2(m_used - m_new);
                m_used = m_new;
            }
            // O_X is complete up to block j-1 (S_X(j) was issued after PV_X(j-1)), and
            // PV_X(j) waits for this warpgroup: rescale it here when a row's max moved.
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(ocol + c0, o);
                    tmem_wait_ld();
                    reg_fence(o);
#pragma unroll
                    for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                    tmem_st32(ocol + c0, o);
                }
            }
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
            const uint64_t negm2 = f2_pack(-m_used, -m_used);
            uint64_t sumq[4];
            uint32_t pkh[2][16];
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                sumq[2 + qq] = f2_pack(0.f, 0.f);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(rr[qq][2 * t]), __uint_as_float(rr[qq][2 * t + 1])),
                                               sl2x2, negm2);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const float y0 = ex2(x0), y1 = ex2(x1);
                    sumq[2 + qq] = f2_add(sumq[2 + qq], f2_pack(y0, y1));
                    pkh[qq][t] = pack_bf16(y0, y1);
                }
            }
            tmem_ld32(scol + 0, rr[0]);
            tmem_ld32(scol + 32, rr[1]);
            tmem_wait_ld();
            reg_fence(rr[0]);
            reg_fence(rr[1]);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                sumq[q] = f2_pack(0.f, 0.f);
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(rr[q][2 * t]), __uint_as_float(rr[q][2 * t + 1])),
                                               sl2x2, negm2);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const float y0 = ex2(x0), y1 = ex2(x1);
                    sumq[q] = f2_add(sumq[q], f2_pack(y0, y1));
                    pk[t] = pack_bf16(y0, y1);
                }
                tmem_st16(scol + q * 16, pk);
            }
            tmem_st16(scol + 32, pkh[0]);
            tmem_st16(scol + 48, pkh[1]);
            float rs0, rs1;
            f2_unpack(f2_add(f2_add(sumq[0], sumq[1]), f2_add(sumq[2], sumq[3])), rs0, rs1);
            l = l * alpha + (rs0 + rs1);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bars.pfull(x));
        }
        if (ok) {
            ok = mbar_wait(bars.odone(x), 0, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        // O leaves through this tile's Q region (the last MMA that read Q_X completed before
        // odone): rows in the 128-byte-swizzled layout of the 64-column TMA box, then one thread
        // stores the tile.  The tile's four warps meet at the named barrier whatever `ok` says.
        uint8_t *stage = sm + C::kQOff + x * C::kTileBytes;
        if (ok) {
            const size_t grow = (size_t)row0 + x * BM + r;
            const float inv = 1.f / l;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(ocol + c0, o);
                tmem_wait_ld();
                reg_fence(o);
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    pk[t] = pack_bf16(__uint_as_float(o[2 * t]) * inv, __uint_as_float(o[2 * t + 1]) * inv);
                uint8_t *slab = stage + (c0 >> 6) * C::kChunkBytes + r * 128;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int u = ((c0 & 63) >> 3) + v;  // 16-byte unit within the 128-byte row
                    *reinterpret_cast<uint4 *>(slab + ((u ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            LSE[grow] = (m_used + __log2f(l)) * kLn2;
            fence_proxy_async_smem();
        }
        named_bar_sync(1 + x, 128);
        if (r == 0 && ok) {
            const uint32_t src = smem_addr(stage);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) tma_store_2d(&tmO, c * 64, row0 + x * BM, src + c * C::kChunkBytes);
            bulk_commit();
            bulk_wait_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kPPMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Two query tiles per CTA under a block mask shared by every head: tile A is query tile t of
// head 2g and tile B the same query tile of head 2g + 1, so both visit the same key blocks and
// alternate on the tensor core exactly as in the two-tile kernel above (MMA order per visited
// block i: PV_A(i), S_A(i+1), PV_B(i), S_B(i+1); one issuing thread).  Their K and V differ, so
// the K and V tiles of both heads stream in, loaded and consumed in that order: K_A(0), K_B(0),
// then V_A(i), K_A(i+1), V_B(i), K_B(i+1) for every visited block, K tiles through a ring of
// their own and V tiles through another.  K piece 2j + x is K of head 2g + x at the j-th visited
// block, V piece 2i + x likewise.  Only the S products commit a release: V piece v is free once
// K piece v + 2 is (PV_x(i) precedes S_x(i+1) in the issuing thread's order), so the issuing
// thread commits four times per visited block instead of six.  Used for 128 x 128 block masks
// shared by all heads (B * H even, d = 64, 128), where pairing two tiles of one head would give
// them different visit lists.
template <int D>
struct PP2Cfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = BM * D * 2;                  // a Q, K or V tile
    static constexpr int kChunkBytes = BM * 128;
    static constexpr int kKSlots = D == 64 ? 6 : 3;               // K ring (tiles of either head)
    static constexpr int kVSlots = D == 64 ? 4 : 2;               // V ring
    static_assert(kKSlots >= kVSlots && kVSlots >= 2, "V releases ride on K releases");
    static constexpr int kQOff = 0;                                // Q_A, Q_B
    static constexpr int kKOff = 2 * kTileBytes;
    static constexpr int kVOff = kKOff + kKSlots * kTileBytes;
    static constexpr int kBarOff = kVOff + kVSlots * kTileBytes;
    // q, kfull[KS], kempty[KS], vfull[VS], sfull[2], pfull[2], odone[2], drain
    static constexpr int kNumBars = 1 + 2 * kKSlots + kVSlots + 2 + 2 + 2 + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    // visited key blocks as a bit set: masks with up to 32 * kMaxMaskWords blocks per row
    static constexpr int kMaxMaskWords = 256;
    static constexpr int kBitsOff = kMiscOff + 64;
    static constexpr int kSmemBytes = kBitsOff + 4 * kMaxMaskWords + 1024;  // + slack to align the base
    static constexpr uint32_t kOCol0 = 256;
    static __device__ __forceinline__ uint32_t scol(int x) { return x ? 128u : 0u; }
    static_assert(kOCol0 + 2 * D <= kTmemCols, "tensor memory budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

template <int KS, int VS>
struct PP2Bars {
    uint32_t base;
    __device__ uint32_t q() const { return base; }
    __device__ uint32_t kfull(int s) const { return base + 8u * (1 + s); }
    __device__ uint32_t kempty(int s) const { return base + 8u * (1 + KS + s); }
    __device__ uint32_t vfull(int s) const { return base + 8u * (1 + 2 * KS + s); }
    __device__ uint32_t sfull(int x) const { return base + 8u * (1 + 2 * KS + VS + x); }
    __device__ uint32_t pfull(int x) const { return base + 8u * (3 + 2 * KS + VS + x); }
    __device__ uint32_t odone(int x) const { return base + 8u * (5 + 2 * KS + VS + x); }
    __device__ uint32_t drain() const { return base + 8u * (7 + 2 * KS + VS); }
};

template <int D>
__global__ void __launch_bounds__(kPPThreads, 1)
fwd_bf16_pp2h_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const Problem p, __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE) {
    using C = PP2Cfg<D>;
    constexpr int KS = C::kKSlots, VS = C::kVSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const PP2Bars<KS, VS> bars{smem_addr(sm + C::kBarOff)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, pair = blockIdx.y;  // heads 2 pair and 2 pair + 1
    const int nb = p.N / BN;
    const uint8_t *hm = p.mask;                      // one 128-block mask for every head
    const int mnb = p.mask_nb();
    uint32_t *vwords = reinterpret_cast<uint32_t *>(sm + C::kBitsOff);
    const int nwords = (nb + 31) >> 5;
    const bool use_bits = nwords <= C::kMaxMaskWords;
    auto kept = [&](int j) { return visited(hm, 128, mnb, tile, j); };
    const uint32_t sQ = smem_addr(sm + C::kQOff), sK = smem_addr(sm + C::kKOff), sV = smem_addr(sm + C::kVOff);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bars.q(), 1);
        for (int s = 0; s < KS; ++s) {
            mbar_init(bars.kfull(s), 1);
            mbar_init(bars.kempty(s), 1);
        }
        for (int s = 0; s < VS; ++s) mbar_init(bars.vfull(s), 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(bars.sfull(x), 1);
            mbar_init(bars.pfull(x), 128);
            mbar_init(bars.odone(x), 1);
        }
        mbar_init(bars.drain(), 1);
        fence_barrier_init();
        // the Q tiles are needed whatever the mask says: start their loads before the mask is read
        mbar_arrive_expect_tx(bars.q(), 2 * C::kTileBytes);
        for (int x = 0; x < 2; ++x)
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_2d(sQ + x * C::kTileBytes + c * C::kChunkBytes, &tmQ, c * 64,
                            (2 * pair + x) * p.N + tile * BM, bars.q());
    }
    if (use_bits) build_visit_bits(vwords, nb, kept);
    if (warp == kPPMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const VisitBits vb{vwords, nwords};
    int n = 0;  // key blocks this query tile visits (in both heads)
    if (use_bits) {
        n = vb.count();
    } else {  // rows longer than the bit set: read the mask directly
        for (int j = 0; j < nb; ++j) n += kept(j) ? 1 : 0;
    }
    // the visited key block after j (callers ask only while one remains)
    auto next_block = [&](int j) -> int {
        if (use_bits) return vb.next(j);
        do {
            ++j;
        } while (!kept(j));
        return j;
    };

    if (warp == kPPTmaWarp) {
        // ------------------------------------------------------------ producer (piece ring)
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int kq = 0, vq = 0;  // next K piece, next V piece
            // K piece kq (K of head 2 pair + x at key block blk) into K slot kq % KS once the S
            // product of K piece kq - KS has completed; V piece vq into V slot vq % VS once V piece
            // vq - VS has been read, which the release of K piece vq - VS + 2 implies (kempty
            // completes once per use of a K slot)
            auto load = [&](int x, bool is_v, int blk) -> bool {
                const int krow = (2 * pair + x) * p.N + blk * BN;
                if (!is_v) {
                    const int slot = kq % KS;
                    if (kq >= KS &&
                        !mbar_wait(bars.kempty(slot), ((uint32_t)(kq / KS) & 1u) ^ 1u, abort_flag, p.dev_status))
                        return false;
                    mbar_arrive_expect_tx(bars.kfull(slot), C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_2d(sK + slot * C::kTileBytes + c * C::kChunkBytes, &tmK, c * 64, krow, bars.kfull(slot));
                    ++kq;
                } else {
                    const int slot = vq % VS;
                    if (vq >= VS) {
                        const int r = vq - VS + 2;
                        if (!mbar_wait(bars.kempty(r % KS), (uint32_t)(r / KS) & 1u, abort_flag, p.dev_status))
                            return false;
                    }
                    mbar_arrive_expect_tx(bars.vfull(slot), C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_2d(sV + slot * C::kTileBytes + c * C::kChunkBytes, &tmV, c * 64, krow, bars.vfull(slot));
                    ++vq;
                }
                return true;
            };
            int jk = next_block(-1), jv = jk;
            bool ok = load(0, false, jk) && load(1, false, jk);
            for (int i = 0; i < n && ok; ++i) {
                const bool more = i + 1 < n;
                if (more) jk = next_block(jk);
                ok = load(0, true, jv) && (!more || load(0, false, jk)) && load(1, true, jv) &&
                     (!more || load(1, false, jk));
                jv = jk;
            }
        }
    } else if (warp == kPPMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n > 0) {
            // a negative scale: S = (-Q) K^T, scaled by |s| in the softmax
            const uint32_t idS = p.scale < 0.f ? kIdSNeg : kIdS;
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
            auto wait_k = [&](int kk) {
                return mbar_wait(bars.kfull(kk % KS), (uint32_t)(kk / KS) & 1u, abort_flag, p.dev_status);
            };
            auto wait_v = [&](int vv) {
                return mbar_wait(bars.vfull(vv % VS), (uint32_t)(vv / VS) & 1u, abort_flag, p.dev_status);
            };
            // S_x from K piece kk; its commit releases K piece kk (and V piece kk - 2, read before it)
            auto mma_s = [&](int x, int kk) {
                const uint32_t kb = sK + (kk % KS) * C::kTileBytes, qb = sQ + x * C::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
                    mma_ss(tmem + C::scol(x), smem_desc_sw128(qb + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024),
                           idS, ks > 0);
                }
                mma_commit(bars.kempty(kk % KS));
                mma_commit(bars.sfull(x));
            };
            // PV_x from V piece vv: no commit of its own (the next S_x's commit covers it)
            auto mma_pv = [&](int x, int vv, bool first) {
                const uint32_t vb = sV + (vv % VS) * C::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks)
                    mma_ts(tmem + C::kOCol0 + x * D, tmem + C::scol(x) + ks * 8,
                           smem_desc_sw128(vb + ks * 2048, C::kChunkBytes, 1024), idO, (!first || ks > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(bars.q(), 0, abort_flag, p.dev_status) && wait_k(0);
            if (ok) {
                tc_fence_after();
                mma_s(0, 0);
                ok = wait_k(1);
            }
            if (ok) {
                tc_fence_after();
                mma_s(1, 1);
            }
            for (int i = 0; i < n && ok; ++i) {
                const bool more = i + 1 < n;
                const uint32_t ph = (uint32_t)i & 1u;
                // V_A(i) and K_A(i+1) were loaded long ago: check them while tile A's softmax still
                // runs, so that only P_A(i) is waited for on the path from softmax to PV
                if (!(ok = wait_v(2 * i))) break;
                if (more && !(ok = wait_k(2 * i + 2))) break;
                if (!(ok = mbar_wait(bars.pfull(0), ph, abort_flag, p.dev_status))) break;
                tc_fence_after();
                mma_pv(0, 2 * i, i == 0);
                if (more) mma_s(0, 2 * i + 2);
                else mma_commit(bars.odone(0));
                if (!(ok = wait_v(2 * i + 1))) break;
                if (more && !(ok = wait_k(2 * i + 3))) break;
                if (!(ok = mbar_wait(bars.pfull(1), ph, abort_flag, p.dev_status))) break;
                tc_fence_after();
                mma_pv(1, 2 * i + 1, i == 0);
                if (more) mma_s(1, 2 * i + 3);
                else mma_commit(bars.odone(1));
            }
            if (!ok) {
                mma_commit(bars.drain());
                mbar_wait(bars.drain(), 0, abort_flag, p.dev_status);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax, one tile per warpgroup
        const int x = warp >> 2;  // 0: tile A (head 2g), 1: tile B (head 2g + 1)
        const int r = tid & 127;  // row within the tile == tensor memory lane
        const int rowx0 = (2 * pair + x) * p.N + tile * BM;  // first row of this warpgroup's tile
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t scol = lane_base + C::scol(x);
        const uint32_t ocol = lane_base + C::kOCol0 + x * D;
        const float sl2 = fabsf(p.scale) * kLog2e;  // S holds sign(s) Q K^T
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            ok = mbar_wait(bars.sfull(x), (uint32_t)j & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // S in two 64-column halves, so that only 64 scores are live at a time: the max over
            // both halves, the exps of the high half (still in registers), then the low half
            // loaded again; P of the high half (columns 32..63, which hold S of keys 32..63) is
            // written only after that reload
            uint32_t rr[2][32];
            tmem_ld32(scol + 0, rr[0]);
            tmem_ld32(scol + 32, rr[1]);
            tmem_wait_ld();
            reg_fence(rr[0]);
            reg_fence(rr[1]);
            // row max in four independent chains of 16-column runs (a single chain through the
            // second half made the max a long dependent sequence)
            float mx4[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t *v = &rr[c >> 1][16 * (c & 1)];
                mx4[c] = fmaxf(__uint_as_float(v[0]), __uint_as_float(v[1]));
#pragma unroll
                for (int t = 1; t < 8; ++t) mx4[c] = fmax3(mx4[c], __uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
            }
            tmem_ld32(scol + 64, rr[0]);
            tmem_ld32(scol + 96, rr[1]);
            tmem_wait_ld();
            reg_fence(rr[0]);
            reg_fence(rr[1]);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t *v = &rr[c >> 1][16 * (c & 1)];
#pragma unroll
                for (int t = 0; t < 8; ++t) mx4[c] = fmax3(mx4[c], __uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
            }
            const float mx = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
            const float m_new = fmaxf(m_used, mx * sl2);
            float alpha = 1.f;
            if (m_new > m_used + kRescaleThreshold) {
                alpha = ex2(m_used - m_new);
                m_used = m_new;
            }
            // O_X is complete up to block j-1 (S_X(j) was issued after PV_X(j-1)), and
            // PV_X(j) waits for this warpgroup: rescale it here when a row's max moved.
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(ocol + c0, o);
                    tmem_wait_ld();
                    reg_fence(o);
#pragma unroll
                    for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                    tmem_st32(ocol + c0, o);
                }
            }
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
            const uint64_t negm2 = f2_pack(-m_used, -m_used);
            uint64_t sumq[4];
            uint32_t pkh[2][16];
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                sumq[2 + qq] = f2_pack(0.f, 0.f);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(rr[qq][2 * t]), __uint_as_float(rr[qq][2 * t + 1])),
                                               sl2x2, negm2);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const float y0 = ex2(x0), y1 = ex2(x1);
                    sumq[2 + qq] = f2_add(sumq[2 + qq], f2_pack(y0, y1));
                    pkh[qq][t] = pack_bf16(y0, y1);
                }
            }
            tmem_ld32(scol + 0, rr[0]);
            tmem_ld32(scol + 32, rr[1]);
            tmem_wait_ld();
            reg_fence(rr[0]);
            reg_fence(rr[1]);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                sumq[q] = f2_pack(0.f, 0.f);
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(rr[q][2 * t]), __uint_as_float(rr[q][2 * t + 1])),
                                               sl2x2, negm2);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const float y0 = ex2(x0), y1 = ex2(x1);
                    sumq[q] = f2_add(sumq[q], f2_pack(y0, y1));
                    pk[t] = pack_bf16(y0, y1);
                }
                tmem_st16(scol + q * 16, pk);
            }
            tmem_st16(scol + 32, pkh[0]);
            tmem_st16(scol + 48, pkh[1]);
            float rs0, rs1;
            f2_unpack(f2_add(f2_add(sumq[0], sumq[1]), f2_add(sumq[2], sumq[3])), rs0, rs1);
            l = l * alpha + (rs0 + rs1);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bars.pfull(x));
        }
        if (n == 0) {
            // every key block removed for this query tile: O = 0, LSE = -inf
            const size_t grow = (size_t)rowx0 + r;
            uint4 *orow = reinterpret_cast<uint4 *>(O + grow * D);
            for (int v = 0; v < D / 8; ++v) orow[v] = make_uint4(0, 0, 0, 0);
            LSE[grow] = -INFINITY;
            ok = false;
        }
        if (ok) {
            ok = mbar_wait(bars.odone(x), 0, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        // O leaves through this tile's Q region (the last MMA that read Q_X completed before
        // odone): rows in the 128-byte-swizzled layout of the 64-column TMA box, then one thread
        // stores the tile.  The tile's four warps meet at the named barrier whatever `ok` says.
        uint8_t *stage = sm + C::kQOff + x * C::kTileBytes;
        if (ok) {
            const size_t grow = (size_t)rowx0 + r;
            const float inv = 1.f / l;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(ocol + c0, o);
                tmem_wait_ld();
                reg_fence(o);
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    pk[t] = pack_bf16(__uint_as_float(o[2 * t]) * inv, __uint_as_float(o[2 * t + 1]) * inv);
                uint8_t *slab = stage + (c0 >> 6) * C::kChunkBytes + r * 128;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int u = ((c0 & 63) >> 3) + v;  // 16-byte unit within the 128-byte row
                    *reinterpret_cast<uint4 *>(slab + ((u ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            LSE[grow] = (m_used + __log2f(l)) * kLn2;
            fence_proxy_async_smem();
        }
        named_bar_sync(1 + x, 128);
        if (r == 0 && ok && n > 0) {
            const uint32_t src = smem_addr(stage);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) tma_store_2d(&tmO, c * 64, rowx0, src + c * C::kChunkBytes);
            bulk_commit();
            bulk_wait_all();
        }
    }

    // a tile pair that visits no key block still received its Q tiles: let those copies land first
    if (n == 0 && tid == 0) mbar_wait(bars.q(), 0, abort_flag, p.dev_status);
    tc_fence_before();
    __syncthreads();
    if (warp == kPPMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// d = 256, one query tile per CTA.  The Q tile takes 64 KB; one K and one V tile
// (64 KB each) fit beside it, but then V of block j+1 can load only after PV of
// block j, and the pass waits for that load every block.  Instead K and V stream
// through a ring of five 32 KB pieces, loaded and consumed in the tensor core's
// order: K of a block as two d-halves (128 keys x 128 columns, the k-steps
// 0..7 and 8..15 of S = Q K^T) and V as two 64-key halves (64 keys x 256
// columns, the k-steps 0..3 and 4..7 of O += P V), so the next block's pieces
// load while the current products run.  Otherwise the single-tile scheme.
template <int D>
struct RingCfg {
    static_assert(D == 256, "the piece ring is laid out for d = 256");
    static constexpr int kChunks = D / 64;                     // 64-column slabs of a row
    static constexpr int kTileBytes = BM * D * 2;              // the Q tile: 64 KB
    static constexpr int kChunkBytes = BM * 128;               // one 64-column slab of a 128-row tile
    static constexpr int kPieces = 5;
    static constexpr int kPieceBytes = 32768;
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kQOff + kTileBytes;
    static constexpr int kBarOff = kRingOff + kPieces * kPieceBytes;
    // q, full[P], empty[P], sfull[2], pfull[2], odone, drain
    static constexpr int kNumBars = 1 + 2 * kPieces + 2 + 2 + 1 + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kMaxMaskWords = 256;
    static constexpr int kBitsOff = kMiscOff + 64;
    static constexpr int kSmemBytes = kBitsOff + 4 * kMaxMaskWords + 1024;  // + slack to align the base
    static_assert(BN * 128 * 2 == kPieceBytes && (BN / 2) * D * 2 == kPieceBytes, "piece sizes");
    static_assert(kOCol + D <= kTmemCols, "tensor memory budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

struct RingBars {
    uint32_t base;
    static constexpr int P = RingCfg<256>::kPieces;
    __device__ uint32_t q() const { return base; }
    __device__ uint32_t full(int s) const { return base + 8u * (1 + s); }
    __device__ uint32_t empty(int s) const { return base + 8u * (1 + P + s); }
    __device__ uint32_t sfull(int b) const { return base + 8u * (1 + 2 * P + b); }
    __device__ uint32_t pfull(int b) const { return base + 8u * (3 + 2 * P + b); }
    __device__ uint32_t odone() const { return base + 8u * (5 + 2 * P); }
    __device__ uint32_t drain() const { return base + 8u * (6 + 2 * P); }
};

template <int D, bool TAIL>
__global__ void __launch_bounds__(kThreads, 1)
fwd_bf16_ring_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Problem p,
                     __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE) {
    using C = RingCfg<D>;
    constexpr int NP = C::kPieces;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const RingBars bars{smem_addr(sm + C::kBarOff)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::kMiscOff + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, head = blockIdx.y;
    const int nb = TAIL ? (p.N + BN - 1) / BN : p.N / BN;  // key blocks (the last one partial under TAIL)
    const uint8_t *hm = p.head_mask(head);
    const int mb = p.mask_block, mnb = p.mask_nb();
    uint32_t *vwords = reinterpret_cast<uint32_t *>(sm + C::kBitsOff);
    const int nwords = (nb + 31) >> 5;
    const bool use_bits = hm != nullptr && nwords <= C::kMaxMaskWords;
    const int row0 = head * p.N + tile * BM;  // first row of this tile in the [B*H*N, D] view
    const uint32_t sQ = smem_addr(sm + C::kQOff), sR = smem_addr(sm + C::kRingOff);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bars.q(), 1);
        for (int s = 0; s < NP; ++s) {
            mbar_init(bars.full(s), 1);
            mbar_init(bars.empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.sfull(b), 1);
            mbar_init(bars.pfull(b), 4 * 32);
        }
        mbar_init(bars.odone(), 1);
        mbar_init(bars.drain(), 1);
        fence_barrier_init();
        // the Q tile is needed whatever the mask says: start its load before the mask is read
        mbar_arrive_expect_tx(bars.q(), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) tma_load_2d(sQ + c * C::kChunkBytes, &tmQ, c * 64, row0, bars.q());
    }
    if (use_bits) build_visit_bits(vwords, nb, [&](int j) { return visited<TAIL>(hm, mb, mnb, tile, j); });
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const VisitBits vb{vwords, nwords};
    int n = nb;  // key blocks this query tile visits
    if (use_bits) {
        n = vb.count();
    } else if (hm != nullptr) {  // rows longer than the bit set: read the mask directly
        n = 0;
        for (int j = 0; j < nb; ++j) n += visited<TAIL>(hm, mb, mnb, tile, j) ? 1 : 0;
    }
    // the visited key block after j (callers ask only while one remains)
    auto next_block = [&](int j) -> int {
        if (hm == nullptr) return j + 1;
        if (use_bits) return vb.next(j);
        do {
            ++j;
        } while (!visited<TAIL>(hm, mb, mnb, tile, j));
        return j;
    };

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer (piece ring)
        // The tensor core's order is S(0), S(1), PV(0), S(2), PV(1), ..., PV(n-1), so pieces are
        // loaded in the order K(0), K(1), V(0), K(2), V(1), ..., K(n-1), V(n-2), V(n-1); piece q
        // goes to slot q % NP once the MMAs of piece q - NP have released it.
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int q = 0;
            auto load = [&](bool is_v, int blk) -> bool {
                const int krow = head * p.N + blk * BN;
                for (int h = 0; h < 2; ++h, ++q) {
                    const int slot = q % NP;
                    if (q >= NP && !mbar_wait(bars.empty(slot), ((uint32_t)(q / NP) & 1u) ^ 1u, abort_flag,
                                              p.dev_status))
                        return false;
                    const uint32_t full = bars.full(slot), dst = sR + slot * C::kPieceBytes;
                    mbar_arrive_expect_tx(full, C::kPieceBytes);
                    if (!is_v) {  // K, columns 128 h .. 128 h + 127: two 128-row boxes
                        for (int c = 0; c < 2; ++c) tma_load_2d(dst + c * C::kChunkBytes, &tmK, (2 * h + c) * 64, krow, full);
                    } else {      // V, keys 64 h .. 64 h + 63: four 64-row boxes (V's map at d = 256)
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_2d(dst + c * (C::kPieceBytes / C::kChunks), &tmV, c * 64, krow + 64 * h, full);
                    }
                }
                return true;
            };
            int jk = next_block(-1), jv = jk;
            bool ok = load(false, jk);
            for (int it = 0; it < n && ok; ++it) {
                if (it + 1 < n) {
                    jk = next_block(jk);
                    if (!(ok = load(false, jk))) break;
                }
                if (!(ok = load(true, jv))) break;
                if (it + 1 < n) jv = next_block(jv);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n > 0) {
            // a negative scale: S = (-Q) K^T, scaled by |s| in the softmax
            const uint32_t idS = p.scale < 0.f ? kIdSNeg : kIdS;
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
            bool ok = mbar_wait(bars.q(), 0, abort_flag, p.dev_status);
            int q = 0;  // next piece of the ring (the producer's order)
            // S_it = Q K_it^T into S buffer (it & 1)
            auto issue_s = [&](int it) -> bool {
                const uint32_t dcol = tmem + ((it & 1) ? kSCol1 : kSCol0);
                for (int h = 0; h < 2; ++h, ++q) {  // d-half h of K_it
                    const int slot = q % NP;
                    if (!mbar_wait(bars.full(slot), (uint32_t)(q / NP) & 1u, abort_flag, p.dev_status)) return false;
                    tc_fence_after();
                    const uint32_t kb = sR + slot * C::kPieceBytes;
#pragma unroll
                    for (int k8 = 0; k8 < 8; ++k8) {
                        const int ks = 8 * h + k8;
                        mma_ss(dcol, smem_desc_sw128(sQ + (ks >> 2) * C::kChunkBytes + (ks & 3) * 32, 16, 1024),
                               smem_desc_sw128(kb + (k8 >> 2) * C::kChunkBytes + (k8 & 3) * 32, 16, 1024), idS, ks > 0);
                    }
                    mma_commit(bars.empty(slot));
                }
                mma_commit(bars.sfull(it & 1));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int it = 0; it < n && ok; ++it) {
                if (it + 1 < n && !(ok = issue_s(it + 1))) break;
                const uint32_t pcol = tmem + ((it & 1) ? kSCol1 : kSCol0);
                // V_it's two 64-key halves are pieces q and q + 1: check both before waiting for P_it,
                // so that only P_it is waited for on the path from the softmax to PV
                const int slot0 = q % NP, slot1 = (q + 1) % NP;
                if (!(ok = mbar_wait(bars.full(slot0), (uint32_t)(q / NP) & 1u, abort_flag, p.dev_status))) break;
                if (!(ok = mbar_wait(bars.full(slot1), (uint32_t)((q + 1) / NP) & 1u, abort_flag, p.dev_status)))
                    break;
                if (!(ok = mbar_wait(bars.pfull(it & 1), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status))) break;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int slot = h ? slot1 : slot0;
                    const uint32_t vb = sR + slot * C::kPieceBytes;  // keys 64 h .. 64 h + 63 of V_it
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        mma_ts(tmem + kOCol, pcol + (4 * h + k4) * 8,
                               smem_desc_sw128(vb + k4 * 2048, C::kPieceBytes / C::kChunks, 1024), idO,
                               (it > 0 || h > 0 || k4 > 0) ? 1u : 0u);
                    mma_commit(bars.empty(slot));
                }
                q += 2;
                mma_commit(bars.odone());
            }
            if (!ok) {
                // let every MMA already issued finish before tensor memory is released
                mma_commit(bars.drain());
                mbar_wait(bars.drain(), 0, abort_flag, p.dev_status);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warps 0-3
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float sl2 = fabsf(p.scale) * kLog2e;  // S holds sign(s) Q K^T
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        // 64-row mask blocks: this warp's 32 rows lie in one mask row, so each
        // 64-key half of a visited block is kept or removed for the whole warp.
        const bool fine = hm != nullptr && mb == 64;
        // TAIL: rows 64-127 of the last tile may all lie past N, below the mask's last row
        const bool wrow = !TAIL || 2 * tile + warp / 2 < mnb;
        const uint8_t *wmask = fine && wrow ? hm + (size_t)(2 * tile + warp / 2) * mnb : nullptr;
        int j = -1;  // key block of iteration it (tracked for fine masks and under TAIL)
        for (int it = 0; it < n; ++it) {
            const int b = it & 1;
            bool half_kept[2] = {true, true};
            if (fine) {
                j = next_block(j);
                if (wmask != nullptr) {
                    half_kept[0] = wmask[2 * j] != 0;
                    half_kept[1] = (!TAIL || 2 * j + 1 < mnb) && wmask[2 * j + 1] != 0;
                } else {  // rows past N only (TAIL)
                    half_kept[0] = half_kept[1] = false;
                }
            } else if (TAIL) {
                j = next_block(j);
            }
            // TAIL: keys of the last block from N on do not exist (their rows in the K and V tiles
            // belong to the next head, or read as zeros past the end): their scores are -inf, and a
            // half with no key below N counts as removed
            int lim = BN;
            if constexpr (TAIL) {
                if (j == nb - 1) lim = p.N - j * BN;
                if (lim <= BN / 2) half_kept[1] = false;
            }
            ok = mbar_wait(bars.sfull(b), (uint32_t)(it >> 1) & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t scol = lane_base + (b ? kSCol1 : kSCol0);
            uint32_t r[4][32];
            tmem_ld32(scol + 0, r[0]);
            tmem_ld32(scol + 32, r[1]);
            tmem_ld32(scol + 64, r[2]);
            tmem_ld32(scol + 96, r[3]);
            tmem_wait_ld();
            reg_fence(r[0]);
            reg_fence(r[1]);
            reg_fence(r[2]);
            reg_fence(r[3]);
            if constexpr (TAIL) {
                if (lim < BN) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (32 * q + t >= lim) r[q][t] = 0xff800000u;  // -inf
                }
            }
            // row max: four independent chains (one per 32-column chunk), then combined
            float mxq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                mxq[q] = fmaxf(__uint_as_float(r[q][0]), __uint_as_float(r[q][1]));
#pragma unroll
                for (int t = 1; t < 16; ++t)
                    mxq[q] = fmax3(mxq[q], __uint_as_float(r[q][2 * t]), __uint_as_float(r[q][2 * t + 1]));
                if (!half_kept[q >> 1]) mxq[q] = -INFINITY;
            }
            const float mx = fmaxf(fmax3(mxq[0], mxq[1], mxq[2]), mxq[3]);
            // a warp with nothing kept so far keeps m_used = -inf
            const float m_new = mx == -INFINITY ? m_used : fmaxf(m_used, mx * sl2);
            float alpha = 1.f;
            if (m_new > m_used + kRescaleThreshold) {
                alpha = ex2(m_used - m_new);
                m_used = m_new;
            }
            // p = 2^(s log2e S - m): pairs on the packed FMA path, exps on MUFU
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
            const uint64_t negm2 = f2_pack(-m_used, -m_used);
            uint64_t sumq[4];  // four independent row-sum chains
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                sumq[q] = f2_pack(0.f, 0.f);
                uint32_t pk[16];
                if (!half_kept[q >> 1]) {
                    // removed half: P = 0, nothing added to the row sum
#pragma unroll
                    for (int t = 0; t < 16; ++t) pk[t] = 0u;
                    tmem_st16(scol + q * 16, pk);
                    continue;
                }
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(r[q][2 * t]), __uint_as_float(r[q][2 * t + 1])),
                                               sl2x2, negm2);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const uint64_t y2 = f2_pack(ex2(x0), ex2(x1));
                    sumq[q] = f2_add(sumq[q], y2);
                    float y0, y1;
                    f2_unpack(y2, y0, y1);
                    pk[t] = pack_bf16(y0, y1);
                }
                tmem_st16(scol + q * 16, pk);
            }
            float rs0, rs1;
            f2_unpack(f2_add(f2_add(sumq[0], sumq[1]), f2_add(sumq[2], sumq[3])), rs0, rs1);
            const float rs = rs0 + rs1;
            l = l * alpha + rs;
            tmem_wait_st();
            if (it > 0) {
                ok = mbar_wait(bars.odone(), (uint32_t)(it - 1) & 1u, abort_flag, p.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(lane_base + kOCol + c0, o);
                        tmem_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                        tmem_st32(lane_base + kOCol + c0, o);
                    }
                    tmem_wait_st();
                }
            }
            tc_fence_before();
            mbar_arrive(bars.pfull(b));
        }
        // ------------------------------------------------------------ epilogue
        if (ok && n > 0) {
            ok = mbar_wait(bars.odone(), (uint32_t)(n - 1) & 1u, abort_flag, p.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        const size_t grow = (size_t)row0 + tid;
        // rows of this tile below N (TAIL: the last tile of a head is partial)
        const int valid = TAIL ? min(BM, p.N - tile * BM) : BM;
        if (TAIL && n > 0 && valid < BM) {
            // the rows past N belong to the next head: each thread stores its own row, if it
            // exists, instead of one tensor store of the whole tile
            if (ok) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kOCol + c0, o);
                    tmem_wait_ld();
                    reg_fence(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        pk[t] = pack_bf16(__uint_as_float(o[2 * t]) * inv, __uint_as_float(o[2 * t + 1]) * inv);
                    if (tid < valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(O + grow * D + c0);
#pragma unroll
                        for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
                if (tid < valid) LSE[grow] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
            }
        } else if (n > 0) {
            // O leaves through the Q tile (the last MMA that read it completed before odone):
            // rows in the 128-byte-swizzled layout of the 64-column TMA box, then one thread
            // stores the tile.  The four warps meet at the named barrier whatever `ok` says.
            uint8_t *stage = sm + C::kQOff;
            if (ok) {
                // a row whose every visited score was removed (64-row masks) has l = 0:
                // O = 0 and LSE = -inf, with the tensor-memory loads still warp-wide
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kOCol + c0, o);
                    tmem_wait_ld();
                    reg_fence(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        pk[t] = pack_bf16(__uint_as_float(o[2 * t]) * inv, __uint_as_float(o[2 * t + 1]) * inv);
                    uint8_t *slab = stage + (c0 >> 6) * C::kChunkBytes + tid * 128;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int u = ((c0 & 63) >> 3) + v;  // 16-byte unit within the 128-byte row
                        *reinterpret_cast<uint4 *>(slab + ((u ^ (tid & 7)) << 4)) =
                            make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
                LSE[grow] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
                fence_proxy_async_smem();
            }
            named_bar_sync(1, 128);
            if (tid == 0 && ok) {
                const uint32_t src = smem_addr(stage);
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) tma_store_2d(&tmO, c * 64, row0, src + c * C::kChunkBytes);
                bulk_commit();
                bulk_wait_all();
            }
        } else if (tid < valid) {
            // every key block removed: O = 0, LSE = -inf
            uint4 *orow = reinterpret_cast<uint4 *>(O + grow * D);
            for (int v = 0; v < D / 8; ++v) orow[v] = make_uint4(0, 0, 0, 0);
            LSE[grow] = -INFINITY;
        }
    }

    // a tile that visits no key block still received its Q tile: let that copy land first
    if (n == 0 && tid == 0) mbar_wait(bars.q(), 0, abort_flag, p.dev_status);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}


template <int D>
cudaError_t launch_pp(const Problem &p, const FwdMaps &m, void *O, float *LSE, cudaStream_t st) {
    auto kern = fwd_bf16_pp_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PPCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.N / (2 * BM), p.B * p.H);
    {
        ProfScope prof_("fwd_bf16", st);
        kern<<<grid, kPPThreads, PPCfg<D>::kSmemBytes, st>>>(m.q, m.k, m.v, m.o, p, static_cast<__nv_bfloat16 *>(O),
                                                              LSE);
    }
    return cudaGetLastError();
}

template <int D, bool TAIL, bool FINE>
cudaError_t launch_d(const Problem &p, const FwdMaps &m, void *O, float *LSE, cudaStream_t st) {
    auto kern = fwd_bf16_kernel<D, TAIL, FINE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + BM - 1) / BM, p.B * p.H);
    {
        ProfScope prof_("fwd_bf16", st);
        kern<<<grid, kThreads, FwdCfg<D>::kSmemBytes, st>>>(m.q, m.k, m.v, m.o, p, static_cast<__nv_bfloat16 *>(O),
                                                            LSE);
    }
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_pp2h(const Problem &p, const FwdMaps &m, void *O, float *LSE, cudaStream_t st) {
    auto kern = fwd_bf16_pp2h_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PP2Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.N / BM, p.B * p.H / 2);
    {
        ProfScope prof_("fwd_bf16", st);
        kern<<<grid, kPPThreads, PP2Cfg<D>::kSmemBytes, st>>>(m.q, m.k, m.v, m.o, p,
                                                               static_cast<__nv_bfloat16 *>(O), LSE);
    }
    return cudaGetLastError();
}

// the single-tile kernel's instantiation: partial last tile, 64-row mask blocks
template <int D>
cudaError_t launch_single(const Problem &p, const FwdMaps &m, void *O, float *LSE, cudaStream_t st, bool tail) {
    const bool fine = p.mask != nullptr && p.mask_block == 64;
    if (tail) return fine ? launch_d<D, true, true>(p, m, O, LSE, st) : launch_d<D, true, false>(p, m, O, LSE, st);
    return fine ? launch_d<D, false, true>(p, m, O, LSE, st) : launch_d<D, false, false>(p, m, O, LSE, st);
}

template <bool TAIL>
cudaError_t launch_ring(const Problem &p, const FwdMaps &m, void *O, float *LSE, cudaStream_t st) {
    auto kern = fwd_bf16_ring_kernel<256, TAIL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RingCfg<256>::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + BM - 1) / BM, p.B * p.H);
    {
        ProfScope prof_("fwd_bf16", st);
        kern<<<grid, kThreads, RingCfg<256>::kSmemBytes, st>>>(m.q, m.k, m.v, m.o, p,
                                                               static_cast<__nv_bfloat16 *>(O), LSE);
    }
    return cudaGetLastError();
}

}  // namespace

bool fwd_kv_half_boxes(const Problem &p) {
    // the single-tile kernel's FINE instantiation without TAIL (launch_single)
    return p.mask != nullptr && p.mask_block == 64 && p.N % BM == 0 && (p.d == 64 || p.d == 128);
}

cudaError_t launch_fwd_bf16(const Problem &p, const FwdMaps &maps, void *O, float *LSE, cudaStream_t st) {
    if (p.B * p.H > 65535) return cudaErrorNotSupported;
    // N % 128 != 0: one query tile per CTA, the last tile and key block partial
    const bool tail = p.N % BM != 0;
    // two query tiles per CTA when both tiles visit every key block
    const bool pp = p.mask == nullptr && p.N % (2 * BM) == 0;
    // or when both are the same query tile of two heads under one 128-block mask for every head
    const bool pp2h =
        !tail && p.mask != nullptr && p.mask_stride == 0 && p.mask_block == 128 && (p.B * p.H) % 2 == 0;
    switch (p.d) {
        case 64:
            return pp     ? launch_pp<64>(p, maps, O, LSE, st)
                   : pp2h ? launch_pp2h<64>(p, maps, O, LSE, st)
                          : launch_single<64>(p, maps, O, LSE, st, tail);
        case 128:
            return pp     ? launch_pp<128>(p, maps, O, LSE, st)
                   : pp2h ? launch_pp2h<128>(p, maps, O, LSE, st)
                          : launch_single<128>(p, maps, O, LSE, st, tail);
        case 256: return tail ? launch_ring<true>(p, maps, O, LSE, st) : launch_ring<false>(p, maps, O, LSE, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace attn
