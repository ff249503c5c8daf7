// jt_noalloc.cu -- jt_tree_build_noalloc: the draft-tree build with its
// scratch in a fixed, file-scope device array instead of a caller workspace.
//
// Who needs it: a host integration that cannot hand the library a workspace
// at all -- its device memory is owned by another allocator (a serving
// engine's KV-cache pool, a caching allocator it may not call into from the
// thread that drives decoding), or it must not call cudaMalloc/cudaFree in
// the decode loop because those calls synchronise the whole device.  This
// entry point never allocates: the scratch is a static __device__ array
// whose address is looked up once per device.
//
// The kernels are the ones jt_tree_build launches (tree_build_launch); only
// where their scratch lives differs.
#include <mutex>

#include "jt_common.cuh"
#include "jt_internal.h"

namespace jt {

// The scratch: WsHeader (error word and counters, zeroed at every call) then
// the top-W partial and merged tables of the build.
static __device__ __align__(256) char g_noalloc_scratch[JT_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_setup_mu;
char* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call per device); nullptr with *e set when the lookup fails.
char* scratch_for_current_device(cudaError_t* e) {
    int dev = 0;
    *e = cudaGetDevice(&dev);
    if (*e != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *e = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        *e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (*e != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = static_cast<char*>(p);
    }
    return g_scratch_ptr[dev];
}

jt_status status_of(cudaError_t e) {
    if (e == cudaSuccess) return JT_OK;
    if (e == cudaErrorInvalidValue) return JT_ERR_INVALID;
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorNotSupported ||
        e == cudaErrorInvalidDeviceFunction)
        return JT_ERR_UNSUPPORTED;
    return JT_ERR_CUDA;
}

}  // namespace
}  // namespace jt

using namespace jt;

extern "C" jt_status jt_tree_build_noalloc(const float* draft_logits, const int32_t* root_token,
                                           const int32_t* tree_off, int nseq, int N, int W, int64_t V,
                                           int total_nodes, int32_t* parent, int32_t* token,
                                           int32_t* depth, uint32_t* anc, int sync_check,
                                           jt_stream_t stream) {
    JT_RANGE("jt_tree_build_noalloc");
    // the same argument rules as jt_tree_build
    if ((!draft_logits && N > 0) || !root_token || !tree_off || !parent || !token || !depth ||
        !anc || nseq < 1 || nseq > 65535 || N < 0 || N > JT_MAX_N || W < 1 || W > JT_MAX_W ||
        V < W || V > 0x7FFFFFFFll || total_nodes < nseq ||
        static_cast<long long>(nseq) * N > 65535)
        return JT_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(anc) % 16 != 0) return JT_ERR_INVALID;
    // scratch the build needs; beyond the fixed array the call is refused
    // before any device work is enqueued
    const size_t need = kWsHeader + topw_workspace_bytes(static_cast<long long>(nseq) * N, V, W);
    if (need > JT_NOALLOC_SCRATCH_BYTES) return JT_ERR_WORKSPACE;

    cudaError_t e = cudaSuccess;
    char* base = scratch_for_current_device(&e);
    if (!base) return status_of(e);
    // only the header must start at zero: the error word is OR-ed into and
    // the counters are incremented; every table behind it is written before
    // it is read
    e = cudaMemsetAsync(base, 0, sizeof(WsHeader), stream);
    if (e == cudaSuccess)
        e = tree_build_launch(draft_logits, root_token, tree_off, nseq, total_nodes, N, W, V, 0.0, parent, token,
                              depth, anc, base + kWsHeader, reinterpret_cast<uint32_t*>(base), stream);
    if (e != cudaSuccess || !sync_check) return status_of(e);
    // synchronous check: wait for the stream, then read the error word
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return JT_ERR_CUDA;
    uint32_t err = 0;
    e = cudaMemcpy(&err, base, sizeof(err), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return JT_ERR_CUDA;
    if (err & DEVERR_TIMEOUT) return JT_ERR_TIMEOUT;
    if (err & DEVERR_INVALID) return JT_ERR_INVALID;
    return JT_OK;
}
