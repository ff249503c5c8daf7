// tree_attn_f32.cu -- tree-causal paged attention for fp32 inputs on CUDA
// cores (the bf16 tensor-core kernel is in tree_attn.cu; fp32 inputs would
// lose precision in the tensor cores' tf32 mode).
//
// Same semantics as the bf16 path (JetSpec news summary, tree-causal mask;
// "加速AI思考…推测解码新方法" sections 三 and 七): node n attends to prefix
// slots 0..L_b-1 and to the tree slots of its ancestor-or-self set, read
// from the 256-bit sets.  One warp per (node, query head); each lane keeps
// D/32 elements of q and of the running output; per key a warp-shuffle dot
// product and an online-softmax update in fp32.
#include "jt_common.cuh"
#include "jt_internal.h"

namespace jt {

template <int DPL>  // elements per lane = D / 32
__global__ void __launch_bounds__(128)
    tree_attn_f32_kernel(const float* __restrict__ q, const float* __restrict__ kc,
                         const float* __restrict__ vc, const int32_t* __restrict__ block_table,
                         int max_pages, int num_pages, const int32_t* __restrict__ prefix_len,
                         const int32_t* __restrict__ tree_off, const uint32_t* __restrict__ anc,
                         int nseq, int total_nodes, int Hq, int Hkv, float scale,
                         float* __restrict__ out, float* __restrict__ lse, uint32_t* err) {
    constexpr int D = DPL * 32;
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x;
    const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
    if (n >= total_nodes || h >= Hq) return;
    int lo = 0, hi = nseq;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tree_off[mid] <= n) lo = mid; else hi = mid;
    }
    const int b = lo, off = tree_off[b];
    const int B = tree_off[b + 1] - off;
    const int L = prefix_len[b];
    if (B < 1 || B > JT_MAX_TREE || L < 0 || off < 0 || off + B > total_nodes ||
        static_cast<long long>(L) + B > static_cast<long long>(max_pages) * JT_PAGE_SIZE) {
        if (lane == 0) raise_error(err, DEVERR_INVALID);
        return;
    }
    if (n - off >= B) return;  // spare capacity past the last tree
    const int kvh = h / (Hq / Hkv);
    const long long rowid = static_cast<long long>(n) * Hq + h;
    float qv[DPL], acc[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
        qv[k] = q[rowid * D + lane + 32 * k];
        acc[k] = 0.0f;
    }
    float mrun = -INFINITY, lrun = 0.0f;
    bool bad_page = false;
    auto visit = [&](int slot) {
        const long long page = block_table[static_cast<long long>(b) * max_pages + slot / JT_PAGE_SIZE];
        if (page < 0 || page >= num_pages) {  // warp-uniform: every lane reads the same entry
            bad_page = true;
            return;
        }
        const long long base = ((page * JT_PAGE_SIZE + slot % JT_PAGE_SIZE) * Hkv + kvh) * D;
        float d = 0.0f;
#pragma unroll
        for (int k = 0; k < DPL; ++k) d = fmaf(qv[k], kc[base + lane + 32 * k], d);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
        const float s = d * scale;
        const float mnew = fmaxf(mrun, s);
        const float corr = expf(mrun - mnew);
        const float pr = expf(s - mnew);
        lrun = lrun * corr + pr;
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[k] = fmaf(pr, vc[base + lane + 32 * k], acc[k] * corr);
        mrun = mnew;
    };
    for (int slot = 0; slot < L; ++slot) visit(slot);
    const uint32_t* a = anc + static_cast<long long>(n) * 8;
    for (int w = 0; w < 8; ++w) {
        uint32_t bits = a[w];
        while (bits) {
            const int j = 32 * w + __ffs(bits) - 1;
            bits &= bits - 1;
            if (j < B) visit(L + j);
        }
    }
    if (bad_page && lane == 0) raise_error(err, DEVERR_INVALID);
    const float inv = 1.0f / lrun;
#pragma unroll
    for (int k = 0; k < DPL; ++k) out[rowid * D + lane + 32 * k] = acc[k] * inv;
    if (lse && lane == 0) lse[rowid] = mrun + logf(lrun);
}

cudaError_t tree_attn_f32_launch(const float* q, const float* k_cache, const float* v_cache,
                                 const int32_t* block_table, int max_pages, int num_pages,
                                 const int32_t* prefix_len, const int32_t* tree_off,
                                 const uint32_t* anc, int nseq, int total_nodes, int Hq, int Hkv,
                                 int D, float scale, float* out, float* lse, uint32_t* err,
                                 cudaStream_t st) {
    dim3 grid(total_nodes, (Hq + 3) / 4);
#define JT_F32_CASE(DPL_)                                                                      \
    tree_attn_f32_kernel<DPL_><<<grid, 128, 0, st>>>(q, k_cache, v_cache, block_table, max_pages, num_pages, \
                                                     prefix_len, tree_off, anc, nseq, total_nodes, \
                                                     Hq, Hkv, scale, out, lse, err);              \
    return cudaGetLastError();
    switch (D) {
        case 32: JT_F32_CASE(1)
        case 64: JT_F32_CASE(2)
        case 96: JT_F32_CASE(3)
        case 128: JT_F32_CASE(4)
        default: return cudaErrorInvalidValue;
    }
#undef JT_F32_CASE
}

}  // namespace jt
