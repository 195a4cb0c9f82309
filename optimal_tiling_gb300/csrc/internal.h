// Internal launch interface between the C-ABI host layer (api.cu) and the
// kernel translation units.  Launchers only enqueue work on the given stream
// and return the cudaError_t of the launch; arguments are validated by api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/attn.h"

namespace attn {

// Device status word values (written by kernels, read by attn_device_status).
enum : int {
    kDevOk = 0,
    kDevTimeout = 1,
};

// Opt-in launch timing (attn_profile_* in the C ABI).  A ProfScope placed around
// a kernel launch records a CUDA event pair on the launching stream when
// profiling is enabled, and does nothing otherwise.
class ProfScope {
  public:
    ProfScope(const char *kernel, cudaStream_t st);
    ~ProfScope();
    void add_launch();  // the scope covers one more kernel launch than the first

  private:
    int slot_;
    size_t idx_;
    cudaStream_t st_;
};

// Problem description shared by every launcher.
struct Problem {
    int B, H, N, d;
    float scale;
    const uint8_t *mask;         // device block mask, or nullptr
    int *dev_status;             // device status word
    int mask_block = 128;        // side of a mask block: 64 or 128
    long long mask_stride = 0;   // bytes between the masks of consecutive (b, h); 0 = one mask for all

    // Block mask of head `head` (index b * H + h): row-major [mask_nb()][mask_nb()] bytes.
    __host__ __device__ const uint8_t *head_mask(int head) const {
        return mask ? mask + (size_t)head * (size_t)mask_stride : nullptr;
    }
    __host__ __device__ int mask_nb() const { return (N + mask_block - 1) / mask_block; }
};

// ---- fp32 SIMT path (any N, d <= 256) -------------------------------------
cudaError_t launch_fwd_f32(const Problem &p, const float *Q, const float *K, const float *V,
                           float *O, float *LSE, cudaStream_t st);
cudaError_t launch_bwd_f32(const Problem &p, const float *Q, const float *K, const float *V,
                           const float *O, const float *dO, const float *LSE, float *dQ,
                           float *dK, float *dV, float *D, cudaStream_t st);

// ---- bf16 tcgen05 path ------------------------------------------------------
// Tensor maps are built by the host layer (see tma_desc in api.cu).
struct FwdMaps {
    CUtensorMap q, k, v, o;  // 128-row boxes; at d = 256 V has 64-row boxes (loaded in 64-key halves)
};
// True when the forward kernel for p loads K and V in 64-row boxes (64-row masks, 128 | N,
// d in {64, 128}: the visited 64-key mask columns are packed two to a key block).
bool fwd_kv_half_boxes(const Problem &p);
cudaError_t launch_fwd_bf16(const Problem &p, const FwdMaps &maps, void *O, float *LSE,
                            cudaStream_t st);

struct BwdMaps {
    CUtensorMap q, k, v, dO;
    CUtensorMap dk, dv;  // outputs, 128-row boxes (tensor stores of the dK, dV tiles)
};
// The backward runs one CTA per 128-key tile of one head.  When the SM count does not
// divide the number of tiles and the last wave would be at most half full, the tiles of
// that wave are split into two query halves each (dense problems), so that the wave takes
// half a tile's time; the halves add fp32 partial dK and dV into scratch (kvacc, zeroed by
// the launch) and a small kernel converts them.
// Scratch every backward needs: D (B*H*N fp32) and, for bf16, LSE log2(e) and the fp32 dQ
// accumulator, each rounded up to 256 bytes; the last-wave split's scratch follows it.  The
// bf16 row terms and accumulator hold bwd_rows_per_head(N) rows per head: N rounded up to the
// 64-row query block (the rows past N are padding that the kernels write and read).
size_t bwd_base_bytes(int B, int H, int N, int d, bool bf16);
int bwd_rows_per_head(int N);
int bwd_split_tiles(int B, int H, int N);        // tiles to split, 0 for none (and when 128 does not divide N)
size_t bwd_split_bytes(int split_tiles, int d);  // fp32 dK and dV of the split tiles
cudaError_t launch_bwd_bf16(const Problem &p, const BwdMaps &maps, const void *O,
                            const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                            float *D, float *dQacc, float *kvacc, int split_tiles, cudaStream_t st);

// d = 256: the two passes of the recompute backward (bwd256_sm103.cu) on the row terms and
// accumulator that bwd_pre prepared (L2 = -LSE log2(e), Dv = -D, dQacc zeroed; npad rows per
// head): dK with dQ added into dQacc, then dV.
cudaError_t launch_bwd256_main(const Problem &p, const BwdMaps &maps, const float *L2, const float *Dv,
                               float *dQacc, void *dK, void *dV, cudaStream_t st);

// SM count of the current device (152 when it cannot be asked).
int device_sm_count();

// The calling thread's current CUDA context (cuCtxGetCurrent), or nullptr when none is
// current or the CUDA driver API entry point is unavailable.  Device addresses of the library's
// __device__ variables are cached per context with it.
void *current_context();

// Every check attn_bwd makes on its arguments before any CUDA call, except the workspace's:
// sizes, dtype, null and misaligned pointers, a non-finite scale, supported shapes.
attn_status bwd_args_status(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                            const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int d, float scale,
                            attn_dtype dtype);

struct MatMaps {
    CUtensorMap q, k, e, v;
};
cudaError_t launch_fwd_materialized_bf16(const Problem &p, const MatMaps &maps, const void *Q,
                                         const void *K, void *E, float *rowc, float *rowl,
                                         float *kmax, void *O, float *LSE, cudaStream_t st);

// Materialising backward: Q, K, V, dO with 128-row boxes; P and dS over [B*H*N, N].
struct MatBwdMaps {
    CUtensorMap q, k, v, dO, p, ds;
};
cudaError_t launch_bwd_materialized_bf16(const Problem &p, const MatBwdMaps &maps, const void *O, const void *dO,
                                         const float *LSE, float *Dv, void *dQ, void *dK, void *dV, cudaStream_t st);

// Decode-shaped attention (Nq <= 16 queries against Nk keys): the 32-key steps of all
// heads cut into one equal contiguous range per CTA (one CTA per SM).
struct DecodeShape {
    int B, H, Nq, Nk, d;
    float scale;
    int sph;          // 32-key steps per head
    long long steps;  // steps of all heads
    int ctas;         // CTAs (ranges)
    int max_seg;      // most head segments one range can meet
};
struct DecodeMaps {
    CUtensorMap k, v;  // [B*H*Nk, d] bf16, boxes of 32 rows x 64 columns, 128-byte swizzle
};
DecodeShape decode_shape(int B, int H, int Nq, int Nk, int d, float scale);
size_t decode_workspace_bytes(const DecodeShape &sh);
cudaError_t launch_decode_bf16(const DecodeShape &sh, const DecodeMaps &maps, const void *Q, void *O, float *LSE,
                               float *part, int *dev_status, cudaStream_t st);

// One-CTA kernel whose bounded mbarrier wait expires after limit_ns (self-test).
cudaError_t launch_selftest_wait(int *status, unsigned long long limit_ns, cudaStream_t st);

}  // namespace attn
