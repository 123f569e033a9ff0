// selftest.cu -- a check of the bounded waits the pipelined kernels use (gdn_pipe.cuh): one CTA
// waits on an mbarrier that either gets its arrival or never does. When nothing arrives, every
// waiting thread gives up after the given number of SM clock cycles, one thread raises
// GDN_DEVERR_TIMEOUT and the kernel returns normally, so the CUDA context stays usable.
#include "gdn_launch.h"
#include "gdn_pipe.cuh"
#include "gdn_tile.cuh"

namespace gdn {

__global__ void wait_selftest_kernel(int32_t *err_flags, long long limit, int arrive)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    const bool ok = mbar_wait(&bar, 0u, &abort_flag, limit);
    if (!ok && (threadIdx.x & 31) == 0) raise_flag(err_flags, GDN_DEVERR_TIMEOUT);
}

}  // namespace gdn

extern "C" int gdn_selftest_bounded_wait(int32_t *err_flags, int64_t limit_cycles, int32_t arrive,
                                         gdn_stream_t stream)
{
    if (!err_flags) return GDN_ERR_NULL;
    if (limit_cycles < 1) return GDN_ERR_ARG;
    gdn::wait_selftest_kernel<<<1, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err_flags, limit_cycles, arrive);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}
