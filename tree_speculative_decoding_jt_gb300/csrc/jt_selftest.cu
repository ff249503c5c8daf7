// jt_selftest.cu -- a diagnostic that exercises the device-side timeout path
// of every bounded wait in the library without faulting the GPU.
#include "jt_common.cuh"
#include "jt_internal.h"

namespace jt {

// One CTA waits, with the library's bounded wait, for phase 0 of an
// mbarrier that nothing arrives on.  After the wait limit the helper raises
// DEVERR_TIMEOUT in the error word, sets the abort flag and returns; the
// kernel then exits normally.
__global__ void __launch_bounds__(32) wait_never_kernel(uint32_t* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait_warp(&bar, 0, err, &abort_flag);
}

cudaError_t selftest_wait_timeout_launch(uint32_t* err, cudaStream_t st) {
    return launch_kernel(wait_never_kernel, dim3(1), dim3(32), 0, st, 0, err);
}

}  // namespace jt

using namespace jt;

extern "C" jt_status jt_selftest_wait_timeout(void* ws, size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_selftest_wait_timeout");
    if (!ws || ws_bytes < kWsHeader || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return JT_ERR_WORKSPACE;
    const cudaError_t e = selftest_wait_timeout_launch(static_cast<uint32_t*>(ws), stream);
    if (e == cudaSuccess) return JT_OK;
    return e == cudaErrorInvalidValue ? JT_ERR_INVALID : JT_ERR_CUDA;
}
