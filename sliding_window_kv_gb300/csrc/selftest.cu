// selftest.cu -- the bounded-wait path that every kernel of the library shares, run on
// purpose so that failure detection can be tested without a fault.
//
// One warp waits on an mbarrier with mbar_wait, the same bounded wait the attention,
// decode and compaction kernels use for their TMA copies and MMAs. With `complete` set, the
// warp's own arrival completes the phase first and the wait returns at once. Otherwise
// nothing ever arrives: the wait gives up after its limit and the kernel records a time-out
// in the context's error word, as a kernel whose copy never landed would, and returns. No
// copy is in flight and nothing is left pending, so the context stays usable.
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int* err, int complete)
{
    __shared__ __align__(8) uint64_t bar_storage;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (complete && threadIdx.x == 0)
        mbar_arrive(bar);
    const bool ok = mbar_wait(bar, 0);
    if (!ok && threadIdx.x == 0)
        atomicExch(err, kErrTimeout);
}

cudaError_t launch_wait_selftest(int* err, int complete, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(err, complete);
    return cudaGetLastError();
}

}  // namespace vst
