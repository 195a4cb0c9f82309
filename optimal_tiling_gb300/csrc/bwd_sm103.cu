#include "internal.h"
namespace attn {
cudaError_t launch_bwd_bf16(const Problem &, const BwdMaps &, const void *, const void *, const float *, void *,
                            void *, void *, float *, float *, cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace attn
