// diag.cu -- lora_check_wait_timeout: the library's bounded pipeline wait run
// against an mbarrier that no thread ever completes, so that a caller (or a
// test) can see on a given GPU that a stalled pipeline ends with a status
// word instead of a hang, and that the context stays usable afterwards.
//
// Two warps wait on the same barrier with the tensor-core kernels' own wait
// (tc::mbar_wait_warp): the first to reach the cycle limit sets the CTA's
// abort flag and LORA_ERR_TIMEOUT in *status; the other leaves through the
// abort flag.  Nothing traps, faults or spins without a limit.
#include "internal.h"
#include "tc_common.cuh"

namespace lora {
namespace {

__global__ void __launch_bounds__(64) wait_timeout_kernel(int32_t *status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int32_t abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);  // one arrival completes phase 0; none ever comes
        abort_flag = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    tc::mbar_wait_warp(&bar, 0, &abort_flag, status);
}

}  // namespace
}  // namespace lora

extern "C" LORA_API lora_status_t lora_check_wait_timeout(int32_t *status, lora_stream_t stream)
{
    if (status == nullptr) return LORA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(status) % 4 != 0) return LORA_ERR_ALIGNMENT;
    lora::wait_timeout_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}
