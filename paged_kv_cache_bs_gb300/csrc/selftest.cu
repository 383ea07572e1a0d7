// pa_selftest_wait_timeout: proves on a live GPU that the library's bounded waits end with a status
// instead of a hang.  One thread waits on a fresh mbarrier that nothing ever arrives on, with the
// same bounded wait the store, decode and prefill kernels use on their own copies and tensor-core
// work; the wait gives up after `max_cycles`, raises PA_FLAG_TIMEOUT in err_flag and the kernel
// returns, leaving the context usable.
#include <stdio.h>

#include "tc_common.cuh"

namespace pa {
int set_last_error(int code, const char *msg);

namespace {

__global__ void wait_timeout_kernel(long long max_cycles, int32_t *err_flag) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_word;
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);  // one arrival expected, none ever made
        tc::mbar_fence_init();
        abort_word = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait_or_abort(b, 0, max_cycles, &abort_word))
        raise_flag(err_flag, PA_FLAG_TIMEOUT);
}

}  // namespace
}  // namespace pa

extern "C" PA_API int pa_selftest_wait_timeout(int64_t max_cycles, int32_t *err_flag, void *stream) {
    if (max_cycles <= 0 || max_cycles > 4000000000LL || !err_flag)
        return pa::set_last_error(PA_ERR_INVALID_ARG,
                                  "pa_selftest_wait_timeout: max_cycles must be in (0, 4e9] and err_flag non-NULL");
    pa::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(max_cycles, err_flag);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "pa_selftest_wait_timeout launch: %s", cudaGetErrorString(e));
        return pa::set_last_error(PA_ERR_CUDA, msg);
    }
    return pa::set_last_error(PA_OK, "");
}
