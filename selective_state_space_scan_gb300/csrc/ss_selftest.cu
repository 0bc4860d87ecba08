// Self-test of the kernels' bounded waits: a wait that nothing will satisfy must give up after
// its limit (~2^31 SM cycles, about a second), record kErrWaitTimeout in the device error word
// and let the kernel finish, so that the context stays usable.  The waits are the library's own
// helpers: the mbarrier wait of the TMA stage ring (device_common.cuh) and the wait for another
// CTA's published state of the balanced schedule (ss_fwd_lane.cuh).  No fault is raised; the
// host reads the outcome with ss_device_error.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "ss_fwd_lane.cuh"

namespace selscan {
namespace {

// kind 0: an mbarrier expecting one arrival that never comes (every thread of a warp waits);
// kind 1: a publication flag that is never set to the awaited epoch.
__global__ void __launch_bounds__(32) ss_wait_selftest_kernel(int kind, const unsigned int* flag, unsigned int* err,
                                                               int* finished) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_word;
    volatile int* abort_flag = &abort_word;
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncwarp();
    if (kind == 0) {
        mbar_wait_bounded(&bar, 0, abort_flag, err);
    } else if (threadIdx.x == 0) {
        wait_published(flag, 1u, err);
    }
    __syncwarp();
    if (threadIdx.x == 0) atomicAdd(finished, 1);
}

}  // namespace
}  // namespace selscan

using namespace selscan;

// Internal test hook (not in the public header): runs one bounded wait that cannot succeed
// (kind 0: mbarrier, 1: publication flag) on the current stream-less default stream, waits for
// the kernel, and returns 1 if it finished (0 if not, -1 on a CUDA error).  The timeout shows
// in the device error word.
extern "C" int ss__wait_timeout_selftest(int kind) {
    if (kind != 0 && kind != 1) return -1;
    unsigned int* err = device_error_word();
    if (!err) return -1;
    void* mem = nullptr;
    if (cudaMalloc(&mem, 256) != cudaSuccess) return -1;
    unsigned int* flag = static_cast<unsigned int*>(mem);            // stays 0: never the awaited epoch
    int* finished = reinterpret_cast<int*>(static_cast<char*>(mem) + 128);
    int done = 0;
    bool ok = cudaMemset(mem, 0, 256) == cudaSuccess;
    if (ok) {
        ss_wait_selftest_kernel<<<1, 32>>>(kind, flag, err, finished);
        ok = cudaGetLastError() == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess &&
             cudaMemcpy(&done, finished, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess;
    }
    cudaFree(mem);
    return ok ? (done == 1 ? 1 : 0) : -1;
}
