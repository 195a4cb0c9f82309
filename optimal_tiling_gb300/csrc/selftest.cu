// Self-test of the device-side timeout path shared by every kernel.
//
// A one-CTA kernel initialises an mbarrier that nothing ever arrives on and
// waits for it with the same bounded wait (ptx::mbar_wait) the attention
// kernels use, with a caller-chosen limit.  When the limit passes, the wait
// records a timeout in the library's device status word and returns; the
// kernel then exits normally.  Nothing faults, traps or hangs, and the CUDA
// context stays usable: the host sees ATTN_ERR_TIMEOUT from attn_device_status.
#include "internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

__global__ void selftest_wait_kernel(int *status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ptx::mbar_init(ptx::smem_addr(&bar), 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();
    // phase 0 of this barrier never completes: the wait must give up on its own
    ptx::mbar_wait(ptx::smem_addr(&bar), 0, &abort_flag, status, limit_ns);
    __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(int *status, unsigned long long limit_ns, cudaStream_t st) {
    {
        ProfScope prof_("selftest_wait", st);
        selftest_wait_kernel<<<1, 32, 0, st>>>(status, limit_ns);
    }
    return cudaGetLastError();
}

}  // namespace attn
