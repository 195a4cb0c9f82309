// C-ABI host layer (include/attn.h): argument checks, dispatch by dtype and d,
// TMA descriptor construction, workspace carving and launches on the caller's
// stream.  Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <stdint.h>
#include <string.h>
#include <string>
#include <utility>
#include <vector>

#include "../../include/attn.h"
#include "internal.h"

namespace {

// Device status word shared by every kernel of the library (per device: each
// device that loads the library has its own copy of this variable).
__device__ int g_dev_status;

constexpr int kMaxDevices = 64;
struct StatusAddr {
    void *ctx;   // CUDA context the address was looked up in
    int *ptr;
};
StatusAddr g_status_addr[kMaxDevices];
std::mutex g_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
bool g_ctx_looked_up = false;
std::mutex g_ctx_mu;  // guards the two above only (current_context runs inside g_mu's sections)

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

}  // namespace

namespace attn {

void *current_context() {
    CtxGetCurrentFn fn;
    {
        std::lock_guard<std::mutex> lk(g_ctx_mu);
        if (!g_ctx_looked_up) {
            void *f = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                    cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
            g_ctx_looked_up = true;
        }
        fn = g_ctx_get_current;
    }
    CUcontext c = nullptr;
    if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

}  // namespace attn

namespace {

// Address of the status word on the current device.  It is looked up with the device
// current and kept for the CUDA context it was found in; a call in another context (the
// primary context torn down and created again, e.g. after cudaDeviceReset) looks it up again.
int *device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void *ctx = attn::current_context();
    std::lock_guard<std::mutex> lk(g_mu);
    StatusAddr &a = g_status_addr[dev];
    if (ctx == nullptr || a.ctx != ctx || a.ptr == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dev_status) != cudaSuccess) return nullptr;
        a.ptr = static_cast<int *>(p);
        a.ctx = attn::current_context();  // the lookup makes the device's primary context current
    }
    return a.ptr;
}

EncodeTiledFn encode_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

// 2D bf16 tensor map over a dense [rows][cols] array: boxes of box_rows x 64
// elements (128 bytes), 128-byte swizzle.
bool make_map_bf16(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status check_common(int B, int H, int N, int d, attn_dtype dt) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (dt != ATTN_DTYPE_F32 && dt != ATTN_DTYPE_BF16) return ATTN_ERR_INVALID_ARG;
    // every index fits in 32-bit rows for the tensor maps and in size_t for offsets
    if ((uint64_t)B * H * N > (1ull << 31)) return ATTN_ERR_UNSUPPORTED;
    // the kernels give each (b, h) its own grid row (gridDim.y <= 65535)
    if ((uint64_t)B * H > 65535) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

bool bf16_fwd_shape_ok(int N, int d) { return N >= 1 && (d == 64 || d == 128 || d == 256); }
bool bf16_bwd_shape_ok(int N, int d) { return N >= 1 && (d == 64 || d == 128 || d == 256); }
bool bf16_matfwd_shape_ok(int N, int d) { return N % 128 == 0 && (d == 64 || d == 128 || d == 256); }
bool bf16_matbwd_shape_ok(int N, int d) { return N % 128 == 0 && (d == 64 || d == 128); }

attn_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return ATTN_OK;
    if (e == cudaErrorNotSupported) {
        cudaGetLastError();
        return ATTN_ERR_UNSUPPORTED;
    }
    return ATTN_ERR_CUDA;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }


// ---- launch timing ---------------------------------------------------------
struct ProfFamily {
    std::string name;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev;  // one event pair per scope
    long long launches;                                    // kernels the scopes cover
};
bool g_prof_on = false;
std::vector<ProfFamily> g_prof;
std::mutex g_prof_mu;

}  // namespace

namespace attn {

ProfScope::ProfScope(const char *kernel, cudaStream_t st) : slot_(-1), idx_(0), st_(st) {
    if (!g_prof_on) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    int fam = -1;
    for (size_t i = 0; i < g_prof.size(); ++i)
        if (g_prof[i].name == kernel) fam = (int)i;
    if (fam < 0) {
        g_prof.push_back(ProfFamily{kernel, {}, 0});
        fam = (int)g_prof.size() - 1;
    }
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    if (cudaEventCreate(&b) != cudaSuccess) {
        cudaEventDestroy(a);
        return;
    }
    cudaEventRecord(a, st);
    g_prof[fam].ev.emplace_back(a, b);
    g_prof[fam].launches += 1;
    slot_ = fam;
    idx_ = g_prof[fam].ev.size() - 1;
}

void ProfScope::add_launch() {
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if ((size_t)slot_ < g_prof.size()) g_prof[slot_].launches += 1;
}

ProfScope::~ProfScope() {
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if ((size_t)slot_ < g_prof.size() && idx_ < g_prof[slot_].ev.size())
        cudaEventRecord(g_prof[slot_].ev[idx_].second, st_);
}

size_t bwd_base_bytes(int B, int H, int N, int d, bool bf16) {
    // bf16: rows padded per head to the 64-row query block
    const size_t rows = (size_t)B * H * (bf16 ? bwd_rows_per_head(N) : N);
    // D (and, for bf16, LSE log2(e) after it)
    size_t bytes = ((bf16 ? 2 : 1) * rows * sizeof(float) + 255) / 256 * 256;
    if (bf16) bytes += (rows * (size_t)d * sizeof(float) + 255) / 256 * 256;   // dQ accumulator
    return bytes;
}

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0) {
        cudaGetLastError();
        sms = 152;
    }
    return sms;
}

}  // namespace attn

extern "C" {

void attn_profile_enable(int on) { g_prof_on = on != 0; }

int attn_profile_count(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    return (int)g_prof.size();
}

attn_status attn_profile_query(int index, char *name, int name_capacity, int *launches, double *total_ms) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (index < 0 || index >= (int)g_prof.size()) return ATTN_ERR_INVALID_ARG;
    const ProfFamily &f = g_prof[index];
    if (name && name_capacity > 0) {
        strncpy(name, f.name.c_str(), (size_t)name_capacity - 1);
        name[name_capacity - 1] = 0;
    }
    double tot = 0.0;
    for (const auto &e : f.ev) {
        if (cudaEventSynchronize(e.second) != cudaSuccess) return ATTN_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, e.first, e.second) != cudaSuccess) return ATTN_ERR_CUDA;
        tot += ms;
    }
    if (launches) *launches = (int)f.launches;
    if (total_ms) *total_ms = tot;
    return ATTN_OK;
}

void attn_profile_reset(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto &f : g_prof)
        for (auto &e : f.ev) {
            cudaEventDestroy(e.first);
            cudaEventDestroy(e.second);
        }
    g_prof.clear();
}


const char *attn_status_string(attn_status s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
        case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

}  // extern "C"

namespace {

// Block mask fields: side 64 or 128, head stride >= 0 (0: one mask for every head).
bool mask_ok(int block, long long head_stride) { return (block == 64 || block == 128) && head_stride >= 0; }

attn_status fwd_impl(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N, int d,
                     float scale, attn_dtype dtype, const uint8_t *mask, int mblock, long long mstride,
                     void *stream) {
    attn_status s = check_common(B, H, N, d, dtype);
    if (s != ATTN_OK) return s;
    if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
        return ATTN_ERR_INVALID_ARG;
    if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (dtype == ATTN_DTYPE_F32 && d > 256) return ATTN_ERR_UNSUPPORTED;
    if (dtype == ATTN_DTYPE_BF16 && !bf16_fwd_shape_ok(N, d)) return ATTN_ERR_UNSUPPORTED;
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    attn::Problem p{B, H, N, d, scale, mask, status, mblock, mask ? mstride : 0};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == ATTN_DTYPE_F32) {
        return launch_status(attn::launch_fwd_f32(p, static_cast<const float *>(Q), static_cast<const float *>(K),
                                                  static_cast<const float *>(V), static_cast<float *>(O), LSE, st));
    }
    const uint64_t rows = (uint64_t)B * H * N;
    attn::FwdMaps maps;
    const bool half = attn::fwd_kv_half_boxes(p);  // K and V loaded in 64-key mask columns
    if (!make_map_bf16(&maps.q, Q, d, rows, 128) || !make_map_bf16(&maps.k, K, d, rows, half ? 64 : 128) ||
        !make_map_bf16(&maps.v, V, d, rows, (half || d == 256) ? 64 : 128) || !make_map_bf16(&maps.o, O, d, rows, 128))
        return ATTN_ERR_CUDA;
    return launch_status(attn::launch_fwd_bf16(p, maps, O, LSE, st));
}

}  // namespace

extern "C" {

attn_status attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N,
                     int d, float scale, attn_dtype dtype, const uint8_t *block_mask, void *stream) {
    return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, block_mask, 128, 0, stream);
}

attn_status attn_fwd_masked(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N,
                            int d, float scale, attn_dtype dtype, const attn_block_mask *mask, void *stream) {
    if (mask != nullptr && !mask_ok(mask->block, mask->head_stride)) return ATTN_ERR_INVALID_ARG;
    if (mask == nullptr || mask->blocks == nullptr)
        return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, nullptr, 128, 0, stream);
    return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, dtype, mask->blocks, mask->block, mask->head_stride,
                    stream);
}

size_t attn_bwd_workspace_size(int B, int H, int N, int d, attn_dtype dtype) {
    if (check_common(B, H, N, d, dtype) != ATTN_OK) return 0;
    size_t bytes = attn::bwd_base_bytes(B, H, N, d, dtype == ATTN_DTYPE_BF16);
    if (dtype == ATTN_DTYPE_BF16 && d != 256)  // fp32 partial dK, dV of the last wave's split tiles
        bytes += align_up(attn::bwd_split_bytes(attn::bwd_split_tiles(B, H, N), d), 256);
    return bytes;
}

}  // extern "C"

namespace {

}  // namespace

namespace attn {

attn_status bwd_args_status(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                            const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int d, float scale,
                            attn_dtype dtype) {
    attn_status s = check_common(B, H, N, d, dtype);
    if (s != ATTN_OK) return s;
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return ATTN_ERR_INVALID_ARG;
    const void *ptrs[] = {Q, K, V, O, dO, LSE, dQ, dK, dV};
    for (const void *q : ptrs)
        if (!aligned16(q)) return ATTN_ERR_INVALID_ARG;
    if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (dtype == ATTN_DTYPE_F32 && d > 256) return ATTN_ERR_UNSUPPORTED;
    if (dtype == ATTN_DTYPE_BF16 && !bf16_bwd_shape_ok(N, d)) return ATTN_ERR_UNSUPPORTED;
    // the padded rows of the bf16 row terms and dQ accumulator are indexed in 32 bits too
    if (dtype == ATTN_DTYPE_BF16 && (uint64_t)B * H * bwd_rows_per_head(N) > (1ull << 31))
        return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

}  // namespace attn

namespace {

attn_status bwd_impl(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
                     void *dQ, void *dK, void *dV, int B, int H, int N, int d, float scale, attn_dtype dtype,
                     const uint8_t *mask, int mblock, long long mstride, void *workspace, size_t workspace_bytes,
                     void *stream) {
    attn_status s = attn::bwd_args_status(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype);
    if (s != ATTN_OK) return s;
    const size_t need = attn::bwd_base_bytes(B, H, N, d, dtype == ATTN_DTYPE_BF16);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    attn::Problem p{B, H, N, d, scale, mask, status, mblock, mask ? mstride : 0};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t rows = (size_t)B * H * N;
    float *D = static_cast<float *>(workspace);
    if (dtype == ATTN_DTYPE_F32) {
        return launch_status(attn::launch_bwd_f32(
            p, static_cast<const float *>(Q), static_cast<const float *>(K), static_cast<const float *>(V),
            static_cast<const float *>(O), static_cast<const float *>(dO), LSE, static_cast<float *>(dQ),
            static_cast<float *>(dK), static_cast<float *>(dV), D, st));
    }
    // D, LSE log2(e), then the fp32 dQ accumulator, each with N rounded up to 64 rows per head
    const size_t prows = (size_t)B * H * attn::bwd_rows_per_head(N);
    float *dQacc = reinterpret_cast<float *>(static_cast<char *>(workspace) + align_up(2 * prows * sizeof(float), 256));
    // split the last wave (dense problems) when the workspace also holds the partial dK, dV
    int split = mask == nullptr && d != 256 ? attn::bwd_split_tiles(B, H, N) : 0;  // no split pass at d = 256
    if (split > 0 && workspace_bytes < need + attn::bwd_split_bytes(split, d)) split = 0;
    float *kvacc = split > 0 ? reinterpret_cast<float *>(static_cast<char *>(workspace) + need) : nullptr;
    attn::BwdMaps maps;
    if (!make_map_bf16(&maps.q, Q, d, rows, 64) || !make_map_bf16(&maps.k, K, d, rows, 128) ||
        !make_map_bf16(&maps.v, V, d, rows, 128) || !make_map_bf16(&maps.dO, dO, d, rows, 64) ||
        !make_map_bf16(&maps.dk, dK, d, rows, 128) || !make_map_bf16(&maps.dv, dV, d, rows, 128))
        return ATTN_ERR_CUDA;
    return launch_status(attn::launch_bwd_bf16(p, maps, O, dO, LSE, dQ, dK, dV, D, dQacc, kvacc, split, st));
}

}  // namespace

extern "C" {

attn_status attn_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                     const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int d, float scale,
                     attn_dtype dtype, const uint8_t *block_mask, void *workspace, size_t workspace_bytes,
                     void *stream) {
    return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, block_mask, 128, 0, workspace,
                    workspace_bytes, stream);
}

attn_status attn_bwd_masked(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                            const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int d, float scale,
                            attn_dtype dtype, const attn_block_mask *mask, void *workspace, size_t workspace_bytes,
                            void *stream) {
    if (mask != nullptr && !mask_ok(mask->block, mask->head_stride)) return ATTN_ERR_INVALID_ARG;
    const bool none = mask == nullptr || mask->blocks == nullptr;
    return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, none ? nullptr : mask->blocks,
                    none ? 128 : mask->block, none ? 0 : mask->head_stride, workspace, workspace_bytes, stream);
}

size_t attn_fwd_materialized_workspace_size(int B, int H, int N, int d, attn_dtype dtype) {
    if (check_common(B, H, N, d, dtype) != ATTN_OK || dtype != ATTN_DTYPE_BF16) return 0;
    const size_t heads = (size_t)B * H, rows = heads * N;
    size_t bytes = align_up(heads * (size_t)N * N * 2, 256);   // E, bf16
    bytes += align_up(rows * sizeof(float), 256);               // c (row bound)
    bytes += align_up(rows * sizeof(float), 256);               // l (row sums)
    bytes += align_up(heads * sizeof(float), 256);              // max_j |k_j| per head
    return bytes;
}

attn_status attn_fwd_materialized(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                                  int N, int d, float scale, attn_dtype dtype, const uint8_t *block_mask,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    attn_status s = check_common(B, H, N, d, dtype);
    if (s != ATTN_OK) return s;
    if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
        return ATTN_ERR_INVALID_ARG;
    if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_DTYPE_BF16 || !bf16_matfwd_shape_ok(N, d)) return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_fwd_materialized_workspace_size(B, H, N, d, dtype);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    attn::Problem p{B, H, N, d, scale, block_mask, status};
    const size_t heads = (size_t)B * H, rows = heads * N;
    char *w = static_cast<char *>(workspace);
    void *E = w;
    w += align_up(heads * (size_t)N * N * 2, 256);
    float *rowc = reinterpret_cast<float *>(w);
    w += align_up(rows * sizeof(float), 256);
    float *rowl = reinterpret_cast<float *>(w);
    w += align_up(rows * sizeof(float), 256);
    float *kmax = reinterpret_cast<float *>(w);
    attn::MatMaps maps;
    if (!make_map_bf16(&maps.q, Q, d, rows, 128) || !make_map_bf16(&maps.k, K, d, rows, 128) ||
        !make_map_bf16(&maps.e, E, N, heads * N, 128) || !make_map_bf16(&maps.v, V, d, rows, 128))
        return ATTN_ERR_CUDA;
    return launch_status(attn::launch_fwd_materialized_bf16(p, maps, Q, K, E, rowc, rowl, kmax, O, LSE,
                                                            static_cast<cudaStream_t>(stream)));
}

size_t attn_bwd_materialized_workspace_size(int B, int H, int N, int d, attn_dtype dtype) {
    if (check_common(B, H, N, d, dtype) != ATTN_OK || dtype != ATTN_DTYPE_BF16) return 0;
    const size_t heads = (size_t)B * H, rows = heads * N;
    return 2 * align_up(heads * (size_t)N * N * 2, 256)   // P and dS, bf16
           + align_up(rows * sizeof(float), 256);          // D
}

attn_status attn_bwd_materialized(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                                  const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int d,
                                  float scale, attn_dtype dtype, const uint8_t *block_mask, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    attn_status s = check_common(B, H, N, d, dtype);
    if (s != ATTN_OK) return s;
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return ATTN_ERR_INVALID_ARG;
    const void *ptrs[] = {Q, K, V, O, dO, LSE, dQ, dK, dV};
    for (const void *q : ptrs)
        if (!aligned16(q)) return ATTN_ERR_INVALID_ARG;
    if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_DTYPE_BF16 || !bf16_matbwd_shape_ok(N, d)) return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_bwd_materialized_workspace_size(B, H, N, d, dtype);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    attn::Problem p{B, H, N, d, scale, block_mask, status};
    const size_t heads = (size_t)B * H, rows = heads * N;
    char *w = static_cast<char *>(workspace);
    void *P = w;
    w += align_up(heads * (size_t)N * N * 2, 256);
    void *dS = w;
    w += align_up(heads * (size_t)N * N * 2, 256);
    float *Dv = reinterpret_cast<float *>(w);
    attn::MatBwdMaps maps;
    if (!make_map_bf16(&maps.q, Q, d, rows, 128) || !make_map_bf16(&maps.k, K, d, rows, 128) ||
        !make_map_bf16(&maps.v, V, d, rows, 128) || !make_map_bf16(&maps.dO, dO, d, rows, 128) ||
        !make_map_bf16(&maps.p, P, N, rows, 128) || !make_map_bf16(&maps.ds, dS, N, rows, 128))
        return ATTN_ERR_CUDA;
    return launch_status(attn::launch_bwd_materialized_bf16(p, maps, O, dO, LSE, Dv, dQ, dK, dV,
                                                            static_cast<cudaStream_t>(stream)));
}

namespace {
attn_status check_decode(int B, int H, int Nq, int Nk, int d, attn_dtype dtype) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_DTYPE_F32 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_DTYPE_BF16 || Nq > 16 || !(d == 64 || d == 128 || d == 256)) return ATTN_ERR_UNSUPPORTED;
    if ((uint64_t)B * H > 65535 || (uint64_t)B * H * Nk > (1ull << 31)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}
}  // namespace

size_t attn_decode_workspace_size(int B, int H, int Nq, int Nk, int d, attn_dtype dtype) {
    if (check_decode(B, H, Nq, Nk, d, dtype) != ATTN_OK) return 0;
    return attn::decode_workspace_bytes(attn::decode_shape(B, H, Nq, Nk, d, 1.f));
}

attn_status attn_decode(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int Nq,
                        int Nk, int d, float scale, attn_dtype dtype, void *workspace, size_t workspace_bytes,
                        void *stream) {
    attn_status s = check_decode(B, H, Nq, Nk, d, dtype);
    if (s != ATTN_OK) return s;
    if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
        return ATTN_ERR_INVALID_ARG;
    if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    const attn::DecodeShape sh = attn::decode_shape(B, H, Nq, Nk, d, scale);
    if (workspace == nullptr || workspace_bytes < attn::decode_workspace_bytes(sh) || !aligned16(workspace))
        return ATTN_ERR_WORKSPACE;
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    const uint64_t krows = (uint64_t)B * H * Nk;
    attn::DecodeMaps maps;
    if (!make_map_bf16(&maps.k, K, d, krows, 32) || !make_map_bf16(&maps.v, V, d, krows, 32)) return ATTN_ERR_CUDA;
    return launch_status(attn::launch_decode_bf16(sh, maps, Q, O, LSE, static_cast<float *>(workspace), status,
                                                  static_cast<cudaStream_t>(stream)));
}

attn_status attn_selftest_timeout(unsigned int limit_us, void *stream) {
    if (limit_us == 0 || limit_us > 10000000u) return ATTN_ERR_INVALID_ARG;
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    return launch_status(
        attn::launch_selftest_wait(status, 1000ull * limit_us, static_cast<cudaStream_t>(stream)));
}

attn_status attn_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
        return ATTN_ERR_TIMEOUT;
    }
    return ATTN_OK;
}

}  // extern "C"
