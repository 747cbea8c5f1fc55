// selftest.cu -- exercises the device-side bounded wait on its failure path.
//
// One thread waits on an mbarrier that nothing ever arrives on, through mbar_wait, the
// helper every pipeline wait of the LM-head kernel uses.  The wait must end by its limit
// and raise a bit of the sticky status word, exactly as a stalled pipeline would; the host
// then reads DF2_ERR_TIMEOUT and the context stays usable.
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace df2 {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t *status, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        const bool done = mbar_wait(smem_u32(&bar), 0, &abort_flag, limit_ns);
        if (!done)
            atomicOr(status, kStatusTimeoutSelftest);
    }
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t *status, unsigned long long limit_ns, cudaStream_t stream)
{
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace df2
