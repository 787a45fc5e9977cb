// selftest.cu -- exercises the kernels' bounded mbarrier wait on the device.
//
// One thread initialises an mbarrier that expects one arrival and then waits
// for its first phase with the same bounded wait the attention kernels use.
// Nothing ever arrives, so the wait gives up after the time limit, records
// kStatusWaitTimeout in the per-device status word and the kernel returns: the
// context stays usable and the host reads the code.
#include "device_common.cuh"

namespace apex {
namespace {

__global__ void wait_selftest_kernel(const WaitCtl wc)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbarrier_init();
        mbar_wait(b, 0, wc);  // no arrival: times out
    }
}

}  // namespace

cudaError_t launch_wait_selftest(const WaitCtl &wc, cudaStream_t stream)
{
    wait_selftest_kernel<<<1, 32, 0, stream>>>(wc);
    return cudaGetLastError();
}

}  // namespace apex
