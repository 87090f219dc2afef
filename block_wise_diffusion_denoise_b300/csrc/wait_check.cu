// Self-check of the bounded-wait failure path (tt_check_wait_timeout).
//
// Every kernel of the library waits on mbarriers with a poll limit; a wait that
// runs out records TT_ERR_DEVICE_TIMEOUT in the caller's error word and the kernel
// leaves instead of hanging.  This kernel exercises exactly that path: one warp
// initialises a barrier that expects one arrival, never arrives, waits with the
// same bounded wait, and reports.

#include "sm100_ptx.cuh"
#include "tt_common.cuh"
#include "tt_internal.h"

namespace tt {
namespace {

__global__ void wait_check_kernel(uint32_t polls, uint32_t *dev_err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::fence_mbar_init();
    }
    __syncwarp();
    const bool done = sm100::mbar_wait(&bar, 0, polls);   // nothing ever arrives
    if (!done && threadIdx.x == 0) report_error(dev_err, TT_ERR_DEVICE_TIMEOUT);
}

}  // namespace

tt_status launch_wait_check(uint32_t polls, uint32_t *dev_err, cudaStream_t stream) {
    wait_check_kernel<<<1, 32, 0, stream>>>(polls, dev_err);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace tt
