// Self-test of the library's failure path: makes one of the fused kernel's
// bounded waits run out on purpose -- a wait on an mbarrier that nothing
// completes, or on a handoff flag that nothing sets -- and reports what the
// device recorded.  Nothing faults or hangs: the wait gives up after its time
// limit, writes SSD_ERR_DEVICE_TIMEOUT into the status word and returns.
#include <cuda_runtime.h>

#include "ssd_internal.h"
#include "ssd_wait.cuh"

namespace ssd {
namespace {

// words[0]: status word (starts at 0); words[1]: a flag nothing sets.
__global__ void k_selftest_wait(int which, int *words) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    if (which == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
        wait::fwait(&bar, 0, words);      // no arrival ever comes
    } else {
        wait::wait_flag(words + 1, words);
    }
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" SSD_API int ssd_selftest_wait_timeout(int which, int *device_words, void *stream) {
    if ((which != 0 && which != 1) || !device_words || ((uintptr_t)device_words % 4) != 0)
        return SSD_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(device_words, 0, 2 * sizeof(int), st) != cudaSuccess) return SSD_ERR_CUDA;
    k_selftest_wait<<<1, 32, 0, st>>>(which, device_words);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
    int status = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
    if (cudaMemcpy(&status, device_words, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SSD_ERR_CUDA;
    return status;
}
