/*
 * attn.h — C ABI of the GB300 (sm_103a) exact softmax attention library.
 *
 * The operation (all entry points): for every (batch b, head h) independently,
 *
 *     S = s * Q K^T               (N x N scores; s is the caller's score scale)
 *     P = row-softmax(S)          (masked scores count as minus infinity)
 *     O = P V,   LSE_i = ln sum_j exp(S_ij)
 *
 * as defined in "The I/O Complexity of Attention" exposition
 * (blog.aeilot.top, attention-io-complexity), section "Attention as a
 * mathematical problem" (the page omits the 1/sqrt(d) factor; here it is the
 * caller's s).  The fused forward evaluates it with the stabilised online update
 * of the section "Softmax without storing the score matrix" (running max m,
 * sum l and accumulator u kept on chip, O = u / l); the backward is the
 * recompute pass studied by "On Fine-Grained I/O Complexity of Attention
 * Backward Passes" (gist.science 2410.09397); the materialising variant is the
 * small-cache schedule of the first page's section "Small caches: when storing
 * an intermediate matrix helps", which writes the exponentiated score matrix.
 *
 * Conventions common to every call
 *   Layout      Q, K, V, O, dO, dQ, dK, dV: [B][H][N][d], dense, d innermost.
 *               LSE and the backward's D: [B][H][N] fp32.  Element type is the
 *               call's dtype (fp32 or bf16); LSE is always fp32, natural log of
 *               the scaled scores.
 *   Memory      Every pointer is a DEVICE pointer on the current CUDA device,
 *               owned by the caller.  No call allocates device memory; the
 *               library's own device footprint is static (a status word, and
 *               the 64 MiB array of attn_bwd_static_workspace) and is held on
 *               every device the library is loaded on.  Pointers must be
 *               16-byte aligned and must not alias each other.
 *   Block mask  Optional (NULL = keep everything).  A device array of nb x nb
 *               bytes, nb = ceil(N / 128), row-major, shared by all (b, h):
 *               mask[i/128][j/128] == 0 removes score (i, j).  A row with no
 *               kept score gets O = 0, LSE = -inf and passes no gradient.
 *   Stream      `stream` is a cudaStream_t passed as void* (NULL = legacy
 *               default stream).  Every call only enqueues work; nothing waits.
 *   Errors      Arguments are checked before anything is launched; a failed
 *               check returns a status and launches nothing.  A failed launch
 *               returns ATTN_ERR_CUDA.  Kernels never trap: every device-side
 *               wait is bounded, and an expired wait sets a device status word
 *               that attn_device_status() reports as ATTN_ERR_TIMEOUT.
 *   Shapes      fp32: any N >= 1, 1 <= d <= 256 (SIMT kernels).
 *               bf16: fused forward any N >= 1, d in {64, 128, 256}; fused
 *               backward any N >= 1, d in {64, 128, 256}; materialising forward
 *               (N a multiple of 128) d in {64, 128, 256}; materialising
 *               backward (N a multiple of 128) d in {64, 128}.  When 128 does
 *               not divide N, the last 128-row tile of each head is partial:
 *               the kernels read the rows past N (the next head's, or zeros
 *               past the end of the array) and give them no weight, and write
 *               nothing past row N of any head.  All: B * H <= 65535 and
 *               B * H * N <= 2^31 (bf16 backward: B * H * N' <= 2^31, N' = N
 *               rounded up to a multiple of 64).  Anything else returns
 *               ATTN_ERR_UNSUPPORTED.
 *   Scale       Any finite s, of either sign (a non-finite s is
 *               ATTN_ERR_INVALID_ARG).
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, misaligned pointer */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (dtype / d / N combination) */
    ATTN_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed */
    ATTN_ERR_TIMEOUT = 4,      /* a bounded device-side wait expired (reported by attn_device_status) */
    ATTN_ERR_WORKSPACE = 5     /* workspace pointer NULL or smaller than the size query returns */
} attn_status;

typedef enum {
    ATTN_DTYPE_F32 = 0,
    ATTN_DTYPE_BF16 = 1
} attn_dtype;

/*
 * A general block mask, the generalisation of the 128 x 128 block mask that
 * "On Fine-Grained I/O Complexity of Attention Backward Passes" (gist.science
 * 2410.09397, Theorem 4.5, sparse attention stored by non-zero blocks) studies:
 *   blocks       device array; for each (b, h) an nb x nb row-major byte matrix,
 *                nb = ceil(N / block); blocks[i][j] == 0 removes every score
 *                (q, k) with q / block == i and k / block == j.  NULL: no mask.
 *   block        side of a block: 64 or 128 (anything else: ATTN_ERR_INVALID_ARG).
 *   head_stride  bytes between the matrices of consecutive (b, h), index
 *                b * H + h; 0 means one matrix shared by every head; negative
 *                is ATTN_ERR_INVALID_ARG.
 * The struct itself is read on the host during the call; `blocks` is read by
 * the kernels and must stay valid until the call's work on the stream ends.
 */
typedef struct {
    const uint8_t *blocks;
    int block;
    long long head_stride;
} attn_block_mask;

/*
 * attn_fwd — fused streaming forward.
 * In:  Q, K, V [B,H,N,d] (dtype), block_mask (nullable, see above), scale s.
 * Out: O [B,H,N,d] (dtype) = softmax(s Q K^T) V; LSE [B,H,N] fp32.
 * The bf16 path stages Q/K/V tiles with TMA, runs both products on tcgen05
 * into tensor memory (fp32 accumulation) and never writes the score matrix.
 */
ATTN_API attn_status attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                     int B, int H, int N, int d, float scale, attn_dtype dtype,
                     const uint8_t *block_mask, void *stream);

/*
 * attn_fwd_masked — attn_fwd with a general block mask (64- or 128-blocks,
 * shared or per head); `mask` NULL, or mask->blocks NULL, means no mask.  A
 * query row whose every score is removed gets O = 0 and LSE = -inf.  The bf16
 * path visits a 128-key block when any mask entry covering it and the 128-row
 * query tile is kept, and drops the removed 64-key halves inside the softmax.
 */
ATTN_API attn_status attn_fwd_masked(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                     int B, int H, int N, int d, float scale, attn_dtype dtype,
                                     const attn_block_mask *mask, void *stream);

/* Bytes of scratch attn_bwd needs for this shape (0 is a valid answer). */
ATTN_API size_t attn_bwd_workspace_size(int B, int H, int N, int d, attn_dtype dtype);

/*
 * attn_bwd — recompute backward of attn_fwd (chain rule of the definition above):
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_t dO_it O_it,  dS = P o (dP - D),
 *   dQ = s dS K,  dK = s dS^T Q.
 * In:  Q, K, V, O, dO [B,H,N,d] (dtype), LSE [B,H,N] fp32 from attn_fwd on the
 *      same inputs, the same block_mask and scale.
 * Out: dQ, dK, dV [B,H,N,d] (dtype).
 * workspace: device scratch of at least attn_bwd_workspace_size() bytes
 *      (16-byte aligned, contents on entry ignored); it holds D and, for bf16,
 *      LSE log2(e) and the fp32 dQ accumulator (these three with N rounded up
 *      to a multiple of 64 rows per head).  For bf16 without a mask, d < 256
 *      (d = 256 runs two passes per key tile and never splits), when 128
 *      divides N, the current device's SM count does not divide the 128-key
 *      tiles and the last wave of tiles would be at most half full, the size
 *      also covers fp32 dK and dV of
 *      that wave's tiles, which are then split into two query halves each (so
 *      that the wave takes half a tile's time); the size therefore depends on
 *      the current device.  A workspace that holds only those row terms and
 *      the dQ accumulator also works: the last wave is then not split.
 */
ATTN_API attn_status attn_bwd(const void *Q, const void *K, const void *V, const void *O,
                     const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                     int B, int H, int N, int d, float scale, attn_dtype dtype,
                     const uint8_t *block_mask, void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * attn_bwd_masked — attn_bwd with a general block mask (see attn_block_mask);
 * pass the mask the forward that produced O and LSE used.  Rows and columns
 * with no kept score get zero gradients.  workspace as attn_bwd.
 */
ATTN_API attn_status attn_bwd_masked(const void *Q, const void *K, const void *V, const void *O,
                                     const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                                     int B, int H, int N, int d, float scale, attn_dtype dtype,
                                     const attn_block_mask *mask, void *workspace, size_t workspace_bytes,
                                     void *stream);

/*
 * attn_bwd_static_workspace — attn_bwd for callers that cannot allocate device
 * memory (the pages have no counterpart: this is a deployment convenience).
 * Some callers cannot call cudaMalloc: code inside a host framework that owns
 * every device allocation through its own pool, or a latency-critical path that
 * must not allocate after start-up (an allocation can synchronise the device).
 * Same arguments and results as attn_bwd, without the workspace: the scratch
 * comes from a fixed 64 MiB array compiled into the library, held in device
 * memory of every GPU that loads the library until the process exits.
 *   - Shapes whose row-term and dQ scratch exceeds 64 MiB (fp32: B*H*N rows
 *     of 4 bytes; bf16: B*H*N' rows of 8 + 4d bytes, N' = N rounded up to a
 *     multiple of 64; each part rounded up to 256 bytes) return
 *     ATTN_ERR_WORKSPACE and launch nothing (bf16, d = 128: B*H*N up to
 *     about 129,000 rows; fp32: B*H*N up to 16 million rows).  The last-wave
 *     split of attn_bwd is used when its scratch fits as well.
 *   - Arguments are checked as attn_bwd checks them (same statuses) before
 *     the size check and before any CUDA call.
 *   - The first call on a device looks up the array's device address (one
 *     cudaGetSymbolAddress with that device current) and keeps it for the
 *     current CUDA context; a call in a new context (after cudaDeviceReset)
 *     looks it up again.  Make the first call on a device before any stream
 *     capture.  No call allocates.
 *   - Every call on a device shares the array, which keeps the last call's
 *     contents; the kernels rewrite D and zero the dQ accumulator before use.
 *     Calls whose work overlaps on the GPU (e.g. unordered streams) race.
 */
ATTN_API attn_status attn_bwd_static_workspace(const void *Q, const void *K, const void *V, const void *O,
                                               const void *dO, const float *LSE, void *dQ, void *dK,
                                               void *dV, int B, int H, int N, int d, float scale,
                                               attn_dtype dtype, const uint8_t *block_mask, void *stream);

/* Bytes of scratch attn_fwd_materialized needs (the N x N exp-score matrix and row terms). */
ATTN_API size_t attn_fwd_materialized_workspace_size(int B, int H, int N, int d, attn_dtype dtype);

/*
 * attn_fwd_materialized — the small-cache comparison schedule: the exponentiated
 * scores E = exp(s Q K^T - c) are written to HBM (bf16, N x N per head), then
 * O = E V / l and LSE = c + ln l, with l the row sums of E and c_i a per-row
 * upper bound of the scores (s |q_i| max_j |k_j|, so E never overflows).
 * Same inputs and outputs as attn_fwd; bf16 only.  workspace as attn_bwd.
 */
ATTN_API attn_status attn_fwd_materialized(const void *Q, const void *K, const void *V, void *O,
                                  float *LSE, int B, int H, int N, int d, float scale,
                                  attn_dtype dtype, const uint8_t *block_mask,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of scratch attn_bwd_materialized needs (P and dS, N x N bf16 per head, and D). */
ATTN_API size_t attn_bwd_materialized_workspace_size(int B, int H, int N, int d, attn_dtype dtype);

/*
 * attn_bwd_materialized — the small-cache backward schedule of "On Fine-Grained
 * I/O Complexity of Attention Backward Passes" (gist.science 2410.09397,
 * "Algorithm 6": the n x n attention matrices are written to slow memory and
 * read back), as the comparison point for attn_bwd:
 *   D = rowsum(dO o O);  P = exp(s Q K^T - LSE) and dS = P o (dO V^T - D) are
 *   stored in the workspace (bf16, N x N per head);  dV = P^T dO,
 *   dK = s dS^T Q, dQ = s dS K are three GEMMs over them.
 * Same inputs and outputs as attn_bwd; bf16, N % 128 == 0, d in {64, 128}.
 * workspace: at least attn_bwd_materialized_workspace_size() bytes.
 */
ATTN_API attn_status attn_bwd_materialized(const void *Q, const void *K, const void *V, const void *O,
                                           const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                                           int B, int H, int N, int d, float scale, attn_dtype dtype,
                                           const uint8_t *block_mask, void *workspace,
                                           size_t workspace_bytes, void *stream);

/* Bytes of scratch attn_decode needs (partial states per head segment).  The
 * size depends on the current device's SM count: query it with the device that
 * will run attn_decode current. */
ATTN_API size_t attn_decode_workspace_size(int B, int H, int Nq, int Nk, int d, attn_dtype dtype);

/*
 * attn_decode — decode-shaped attention: for every (b, h), Nq queries against
 * Nk keys, O = softmax(s Q K^T) V and LSE, no mask.  "The I/O Complexity of
 * Attention" exposition notes that single-token decoding (query length one)
 * needs a rectangular account rather than the N^2 formula: here every K/V
 * element is read from HBM once and the pass is bandwidth-bound.  The 32-key
 * steps of all heads are cut into one equal range per SM; the partial states
 * (running max, sum, output) of each head segment are merged with the
 * online-softmax rescale rule.
 * Layout: Q, O [B][H][Nq][d]; K, V [B][H][Nk][d]; LSE [B][H][Nq] fp32.
 * bf16 only; 1 <= Nq <= 16, Nk >= 1, d in {64, 128, 256}.
 * workspace: at least attn_decode_workspace_size() bytes, 16-byte aligned.
 */
ATTN_API attn_status attn_decode(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                                 int Nq, int Nk, int d, float scale, attn_dtype dtype, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * attn_device_status — synchronise `stream`, then read and clear the device
 * status word shared by all kernels of this library on the current device.
 * Returns ATTN_ERR_TIMEOUT if a bounded wait expired since the last call,
 * ATTN_ERR_CUDA if the synchronisation failed, ATTN_OK otherwise.
 */
ATTN_API attn_status attn_device_status(void *stream);

/*
 * Launch timing, for measurement tools.  While enabled, every kernel launch of
 * this library is bracketed by a pair of CUDA events recorded on the stream the
 * kernel is launched on (the events are created and owned by the library).
 * attn_profile_query synchronises on the recorded events and returns, for the
 * kernel family `index` (0 <= index < attn_profile_count()), its name, the
 * number of launches and their summed duration in milliseconds.
 * attn_profile_reset drops every record.  Host-side only; off by default.
 */
ATTN_API void attn_profile_enable(int on);
ATTN_API int attn_profile_count(void);
ATTN_API attn_status attn_profile_query(int index, char *name, int name_capacity, int *launches,
                                        double *total_ms);
ATTN_API void attn_profile_reset(void);

/*
 * attn_selftest_timeout — check of the failure path (no counterpart in the
 * pages).  Enqueues a one-CTA kernel that waits, with the library's bounded
 * wait, on an mbarrier nothing completes; after limit_us microseconds (1 to
 * 10,000,000) the wait records a timeout in the device status word and the
 * kernel exits normally.  A following attn_device_status() on the same stream
 * returns ATTN_ERR_TIMEOUT; the CUDA context stays usable.
 */
ATTN_API attn_status attn_selftest_timeout(unsigned int limit_us, void *stream);

/* Static description of a status code (never NULL). */
ATTN_API const char *attn_status_string(attn_status status);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
