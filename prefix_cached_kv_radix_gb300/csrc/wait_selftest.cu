// Self-test of the bounded wait every kernel of the library uses (rx_device.cuh: mbar_wait).
//
// One CTA waits on an mbarrier that no thread ever arrives at.  The wait gives up after its
// time limit, records RX_DEV_TIMEOUT in the status word and returns, and the kernel ends: the
// path a real kernel takes when a copy or a partner never completes, exercised on purpose
// without faulting or hanging the device (the context stays usable afterwards).
#include <cuda_runtime.h>

#include "radix_attn.h"
#include "rx_common.h"
#include "rx_device.cuh"

namespace rx {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);   // one arrival expected, none will come
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

}  // namespace rx

extern "C" int rx_wait_selftest(int32_t* d_status, uint64_t limit_ns, void* stream) {
    RX_REQUIRE(d_status != nullptr, "rx_wait_selftest: d_status is NULL");
    const uint64_t lim = limit_ns < 1000ull ? 1000ull : (limit_ns > 100000000ull ? 100000000ull : limit_ns);
    rx::wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(d_status, lim);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        rx::set_error("rx_wait_selftest: launch failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}
