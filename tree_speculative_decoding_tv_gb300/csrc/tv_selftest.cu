// Self-test of the bounded device-side waits.
//
// Every pipelined kernel in this library (the attention, the GDN tree kernel)
// waits on mbarriers with a time limit; when a wait runs out the kernel writes
// TV_ERR_TIMEOUT to the caller's status word, stops, lets its copies land and
// frees its tensor memory, so the context stays usable.  This kernel takes
// that path on purpose and nothing else: it allocates tensor memory, waits on
// an mbarrier that nothing ever arrives at for `limit_ns`, reports the
// timeout, frees the tensor memory and returns.
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr uint32_t kSelftestTmemCols = 32;  // the smallest allocation

__global__ void __launch_bounds__(32, 1) selftest_wait_kernel(uint64_t limit_ns, int32_t *status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    tmem_alloc(smem_u32(&tmem_slot), kSelftestTmemCols);  // the whole warp
    tmem_relinquish();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // Nothing arrives on `bar`, so its phase 0 never completes: the wait ends by its limit.
    mbar_wait_for(b, 0, &abort_flag, status, limit_ns);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem_dealloc(tmem, kSelftestTmemCols);
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, int32_t *status, cudaStream_t stream)
{
    selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace tv
