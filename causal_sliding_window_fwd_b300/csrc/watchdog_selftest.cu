// Failure-detection self-test.  One thread waits on an mbarrier that nothing
// will ever complete, through the same bounded wait every pipeline in the
// library uses; when the limit runs out it records NC_ERR_DEVICE_TIMEOUT in
// the device error word and returns, leaving the context usable.
#include <cstdint>
#include <cuda_runtime.h>

#include "nc_attn.h"
#include "nc_kernels.h"
#include "nc_ptx.cuh"

namespace {

__global__ void watchdog_selftest_kernel(long long limit_cycles, int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    nc::mbar_init(&bar, 1);
    nc::fence_barrier_init();
    if (!nc::mbar_wait_limit(&bar, 0, limit_cycles)) nc::set_device_error(err, NC_ERR_DEVICE_TIMEOUT);
}

}  // namespace

extern "C" nc_status nc_debug_watchdog_selftest(unsigned long long limit_cycles, cudaStream_t stream) {
    if (limit_cycles == 0 || limit_cycles > (1ull << 31)) return NC_ERR_INVALID;
    int* err = nc::device_error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>((long long)limit_cycles, err);
    nc::count_launches(1);
    return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}
