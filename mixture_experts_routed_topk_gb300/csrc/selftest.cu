// selftest.cu -- moe_selftest_wait_timeout: runs the kernels' bounded mbarrier wait against a
// barrier that nothing ever arrives on, so the timeout path (status bit, abort flag, clean return)
// can be exercised on a GPU without breaking any real kernel.
#include <cuda_runtime.h>

#include "moe_internal.cuh"
#include "ptx_sm103.cuh"

namespace moe {
namespace {

__global__ void k_selftest_wait(uint32_t* status, unsigned long long timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // expects one arrival that never comes
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, MOE_DEV_TIMEOUT, timeout_ns);
    __syncthreads();
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_selftest_wait_timeout(uint32_t timeout_us, uint32_t* device_status,
                                                  moe_stream_t stream) {
    using namespace moe;
    if (device_status == nullptr || timeout_us == 0 || timeout_us > 2000000u) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(device_status) & 3u) != 0) return MOE_ERR_MISALIGNED;
    DeviceInfo dev;
    moe_status_t st = device_info(&dev);
    if (st != MOE_OK) return st;
    if (!dev.supported) return MOE_ERR_UNSUPPORTED_DEVICE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(device_status, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    k_selftest_wait<<<1, 32, 0, s>>>(device_status, 1000ull * timeout_us);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
