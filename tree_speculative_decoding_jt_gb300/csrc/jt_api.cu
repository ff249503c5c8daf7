// jt_api.cu -- the extern "C" entry points of libjt (declared in include/jt.h):
// host-side argument checks, workspace carving, kernel launches.
#include <math.h>
#include <string.h>

#include "jt_common.cuh"
#include "jt_internal.h"

namespace jt {

int device_sm_count() {
    static PerDeviceCache cache;
    return cache.get([] {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        return sms;
    });
}

static jt_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return JT_OK;
    if (e == cudaErrorInvalidValue) return JT_ERR_INVALID;
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorNotSupported ||
        e == cudaErrorInvalidDeviceFunction)
        return JT_ERR_UNSUPPORTED;
    return JT_ERR_CUDA;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static jt_status check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (!ws || !aligned(ws, kAlign) || ws_bytes < need) return JT_ERR_WORKSPACE;
    return JT_OK;
}

static size_t build_ws(int nseq, int N, int W, long long V, bool ent = false) {
    return kWsHeader + topw_workspace_bytes(static_cast<long long>(nseq) * N, V, W, ent);
}

}  // namespace jt

using namespace jt;

extern "C" {

int jt_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* jt_status_str(jt_status s) {
    switch (s) {
        case JT_OK: return "JT_OK";
        case JT_ERR_INVALID: return "JT_ERR_INVALID: invalid argument or device array contents";
        case JT_ERR_UNSUPPORTED: return "JT_ERR_UNSUPPORTED: outside this build's limits or GPU";
        case JT_ERR_CUDA: return "JT_ERR_CUDA: a CUDA runtime call failed";
        case JT_ERR_TIMEOUT: return "JT_ERR_TIMEOUT: a bounded device-side wait ran out";
        case JT_ERR_WORKSPACE: return "JT_ERR_WORKSPACE: workspace missing, misaligned or too small";
    }
    return "unknown jt_status";
}

size_t jt_workspace_size(int op, int nseq, int N, int W, int64_t V, int total_nodes, int Hq,
                         int Hkv, int D, int max_pages, int max_tree) {
    switch (op) {
        case JT_OP_TREE_BUILD:
        case JT_OP_TREE_BUILD_MIXED:
            if (nseq < 1 || N < 0 || N > JT_MAX_N || W < 1 || W > JT_MAX_W || V < W) return 0;
            return build_ws(nseq, N, W, V, op == JT_OP_TREE_BUILD_MIXED);
        case JT_OP_TREE_TOPW:
            if (nseq < 0 || W < 1 || W > JT_MAX_W || V < W) return 0;
            return build_ws(nseq, 1, W, V);
        case JT_OP_TREE_ATTN: {
            if (nseq < 1 || total_nodes < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1 ||
                max_pages < 1 || max_tree < 1 || max_tree > JT_MAX_TREE)
                return 0;
            const AttnPlan pl = attn_plan(nseq, Hkv, Hq, D, max_tree, max_pages, JT_DTYPE_BF16);
            return attn_workspace_bytes(pl, total_nodes, Hq, D);
        }
        case JT_OP_VERIFY_ACCEPT:
            if (nseq < 1 || total_nodes < 1) return 0;
            return accept_workspace_bytes(nseq, total_nodes);
        case JT_OP_TREE_POLICY:
            return kWsHeader;
        default:
            return 0;
    }
}

jt_status jt_tree_topw(const float* logits, int64_t rows, int64_t V, int W, int32_t* tok,
                       double* lp, double* lse, void* ws, size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_tree_topw");
    if (!logits || !tok || !lp || !lse || rows < 0 || W < 1 || W > JT_MAX_W || V < W ||
        V > 0x7FFFFFFFll || rows > 65535)
        return JT_ERR_INVALID;
    jt_status s = check_ws(ws, ws_bytes, build_ws(static_cast<int>(rows), 1, W, V));
    if (s != JT_OK) return s;
    if (rows == 0) return JT_OK;
    char* base = static_cast<char*>(ws);
    cudaError_t e = tree_topw_launch(logits, rows, V, W, tok, lp, lse, base + kWsHeader, stream);
    return from_cuda(e);
}

jt_status jt_tree_build_mixed(const float* draft_logits, const int32_t* root_token,
                              const int32_t* tree_off, int nseq, int N, int W, int64_t V,
                              int total_nodes, double alpha, int32_t* parent, int32_t* token,
                              int32_t* depth, uint32_t* anc, void* ws, size_t ws_bytes,
                              jt_stream_t stream) {
    JT_RANGE("jt_tree_build_mixed");
    if ((!draft_logits && N > 0) || !root_token || !tree_off || !parent || !token || !depth ||
        !anc || nseq < 1 || nseq > 65535 || N < 0 || N > JT_MAX_N || W < 1 || W > JT_MAX_W ||
        V < W || V > 0x7FFFFFFFll || total_nodes < nseq ||
        static_cast<long long>(nseq) * N > 65535 || !(alpha >= 0.0 && alpha <= 1.0))
        return JT_ERR_INVALID;
    if (!aligned(anc, 16)) return JT_ERR_INVALID;
    jt_status s = check_ws(ws, ws_bytes, build_ws(nseq, N, W, V, alpha != 0.0));
    if (s != JT_OK) return s;
    char* base = static_cast<char*>(ws);
    cudaError_t e = tree_build_launch(draft_logits, root_token, tree_off, nseq, total_nodes, N, W, V, alpha,
                                      parent, token, depth, anc, base + kWsHeader,
                                      reinterpret_cast<uint32_t*>(base), stream);
    return from_cuda(e);
}

jt_status jt_tree_build(const float* draft_logits, const int32_t* root_token,
                        const int32_t* tree_off, int nseq, int N, int W, int64_t V, int total_nodes,
                        int32_t* parent, int32_t* token, int32_t* depth, uint32_t* anc, void* ws,
                        size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_tree_build");
    return jt_tree_build_mixed(draft_logits, root_token, tree_off, nseq, N, W, V, total_nodes, 0.0, parent,
                               token, depth, anc, ws, ws_bytes, stream);
}

jt_status jt_tree_expand_capped(const int32_t* tok, const double* lp, const int32_t* root_token,
                                const int32_t* tree_off, const int32_t* w_cap, const int32_t* n_cap,
                                int nseq, int N, int W, int total_nodes, int32_t* parent,
                                int32_t* token, int32_t* depth, uint32_t* anc, void* ws,
                                size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_tree_expand_capped");
    if ((N > 0 && (!tok || !lp)) || !root_token || !tree_off || !parent || !token || !depth ||
        !anc || nseq < 1 || nseq > 65535 || N < 0 || N > JT_MAX_N || W < 1 || W > JT_MAX_W ||
        total_nodes < nseq || !aligned(anc, 16))
        return JT_ERR_INVALID;
    jt_status s = check_ws(ws, ws_bytes, kWsHeader);
    if (s != JT_OK) return s;
    char* base = static_cast<char*>(ws);
    cudaError_t e = tree_expand_launch(tok, lp, root_token, tree_off, w_cap, n_cap, nseq, total_nodes, N, W,
                                       parent, token, depth, anc, reinterpret_cast<uint32_t*>(base), stream);
    return from_cuda(e);
}

jt_status jt_tree_expand(const int32_t* tok, const double* lp, const int32_t* root_token,
                         const int32_t* tree_off, int nseq, int N, int W, int total_nodes,
                         int32_t* parent, int32_t* token, int32_t* depth, uint32_t* anc, void* ws,
                         size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_tree_expand");
    return jt_tree_expand_capped(tok, lp, root_token, tree_off, nullptr, nullptr, nseq, N, W, total_nodes,
                                 parent, token, depth, anc, ws, ws_bytes, stream);
}

// Host checks of the policy's parameters (jt_tree_policy's rules); returns
// the per-request budget ceiling, or 0 when a parameter is out of range.
static int policy_params_ok(const jt_policy_params* p, int nseq, int N, int W) {
    if (!p || p->b_min < 1 || p->b_max < p->b_min || p->b_max > JT_MAX_TREE || p->node_cap < 0 ||
        p->w_min < 1 || p->w_min > W || p->n_min < 0 || p->n_min > N || p->n_slack < 0 ||
        p->n_slack > N || !(p->beta > 0.0) || !(p->beta <= 1.0) || p->log_conf != p->log_conf ||
        p->acc_thresh != p->acc_thresh)
        return 0;
    int c = p->b_max;
    if (p->node_cap > 0) {
        const int per = p->node_cap / nseq;
        c = per < p->b_min ? p->b_min : per;
        if (c > p->b_max) c = p->b_max;
    }
    return c;
}

jt_status jt_tree_policy(const double* lp, int nseq, int N, int W, const int32_t* accept_len,
                         const jt_policy_params* params, int32_t* budget_state, double* acc_ema,
                         int32_t* tree_off, int32_t* w_cap, int32_t* n_cap, void* ws,
                         size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_tree_policy");
    if (!lp || !budget_state || !acc_ema || !tree_off || !w_cap || !n_cap || nseq < 1 ||
        nseq > 65535 || N < 1 || N > JT_MAX_N || W < 1 || W > JT_MAX_W ||
        policy_params_ok(params, nseq, N, W) == 0)
        return JT_ERR_INVALID;
    jt_status s = check_ws(ws, ws_bytes, kWsHeader);
    if (s != JT_OK) return s;
    cudaError_t e = tree_policy_launch(lp, nseq, N, W, accept_len, *params, budget_state, acc_ema, tree_off,
                                       w_cap, n_cap, static_cast<uint32_t*>(ws), stream);
    return from_cuda(e);
}

jt_status jt_tree_build_adaptive(const float* draft_logits, const int32_t* root_token, int nseq,
                                 int N, int W, int64_t V, int capacity, const int32_t* accept_len,
                                 const jt_policy_params* params, int32_t* budget_state,
                                 double* acc_ema, int32_t* tree_off, int32_t* w_cap,
                                 int32_t* n_cap, int32_t* parent, int32_t* token, int32_t* depth,
                                 uint32_t* anc, void* ws, size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_tree_build_adaptive");
    if (!draft_logits || !root_token || !budget_state || !acc_ema || !tree_off || !w_cap || !n_cap ||
        !parent || !token || !depth || !anc || nseq < 1 || nseq > 65535 || N < 1 || N > JT_MAX_N ||
        W < 1 || W > JT_MAX_W || V < W || V > 0x7FFFFFFFll || static_cast<long long>(nseq) * N > 65535 ||
        !aligned(anc, 16))
        return JT_ERR_INVALID;
    const int ceil_b = policy_params_ok(params, nseq, N, W);
    if (ceil_b == 0 || static_cast<long long>(capacity) < static_cast<long long>(nseq) * ceil_b)
        return JT_ERR_INVALID;
    jt_status s = check_ws(ws, ws_bytes, build_ws(nseq, N, W, V));
    if (s != JT_OK) return s;
    char* base = static_cast<char*>(ws);
    cudaError_t e = tree_build_adaptive_launch(draft_logits, root_token, nseq, capacity, N, W, V, accept_len,
                                               *params, budget_state, acc_ema, tree_off, w_cap, n_cap, parent,
                                               token, depth, anc, base + kWsHeader,
                                               reinterpret_cast<uint32_t*>(base), stream);
    return from_cuda(e);
}

jt_status jt_tree_attn_paged(const void* q, const void* k_cache, const void* v_cache, int dtype,
                             const int32_t* block_table, int max_pages, int num_pages,
                             const int32_t* prefix_len, const int32_t* tree_off,
                             const uint32_t* anc, int nseq, int total_nodes, int max_tree, int Hq,
                             int Hkv, int D, int page_size, float scale, void* out, float* lse,
                             void* ws, size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_tree_attn_paged");
    if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !tree_off || !anc || !out ||
        nseq < 1 || nseq > 65535 || total_nodes < nseq || max_tree < 1 ||
        max_tree > JT_MAX_TREE || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_pages < 1 ||
        num_pages < 1 || page_size != JT_PAGE_SIZE || !isfinite(scale) ||
        (dtype != JT_DTYPE_BF16 && dtype != JT_DTYPE_F32))
        return JT_ERR_INVALID;
    const int G = Hq / Hkv;
    if (dtype == JT_DTYPE_BF16) {
        if (D != 64 && D != 128) return JT_ERR_UNSUPPORTED;
        if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return JT_ERR_UNSUPPORTED;
        if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
            return JT_ERR_INVALID;
        if (Hkv > 65535) return JT_ERR_UNSUPPORTED;
    } else {
        if (D != 32 && D != 64 && D != 96 && D != 128) return JT_ERR_UNSUPPORTED;
    }
    const AttnPlan pl = attn_plan(nseq, Hkv, Hq, D, max_tree, max_pages, dtype);
    jt_status s = check_ws(ws, ws_bytes, attn_workspace_bytes(pl, total_nodes, Hq, D));
    if (s != JT_OK) return s;
    char* base = static_cast<char*>(ws);
    uint32_t* err = reinterpret_cast<uint32_t*>(base);
    cudaError_t e;
    if (dtype == JT_DTYPE_BF16)
        e = tree_attn_bf16_launch(q, k_cache, v_cache, block_table, max_pages, num_pages,
                                  prefix_len, tree_off, anc, nseq, total_nodes, Hq, Hkv, D, scale,
                                  out, lse, pl, base + kWsHeader, err, stream);
    else
        e = tree_attn_f32_launch(static_cast<const float*>(q), static_cast<const float*>(k_cache),
                                 static_cast<const float*>(v_cache), block_table, max_pages,
                                 num_pages, prefix_len, tree_off, anc, nseq, total_nodes, Hq, Hkv, D, scale,
                                 static_cast<float*>(out), lse, err, stream);
    return from_cuda(e);
}

jt_status jt_verify_accept(const float* target_logits, const int32_t* parent,
                           const int32_t* token, const int32_t* tree_off, int nseq, int N,
                           int64_t V, int total_nodes, int rule, double log_t,
                           int32_t* accept_len, int32_t* path, int32_t* bonus, void* ws,
                           size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_verify_accept");
    if (!target_logits || !parent || !token || !tree_off || !accept_len || !path || !bonus ||
        nseq < 1 || nseq > 8192 || N < 0 || N > JT_MAX_TREE || V < 1 || V > 0x7FFFFFFFll ||
        total_nodes < nseq || (rule != JT_RULE_GREEDY && rule != JT_RULE_MARGIN) ||
        (rule == JT_RULE_MARGIN && !(log_t <= 0.0)))
        return JT_ERR_INVALID;
    jt_status s = check_ws(ws, ws_bytes, accept_workspace_bytes(nseq, total_nodes));
    if (s != JT_OK) return s;
    return from_cuda(verify_accept_launch(target_logits, parent, token, tree_off, nseq, N, V,
                                          total_nodes, rule, log_t, accept_len, path, bonus,
                                          static_cast<char*>(ws), stream));
}

jt_status jt_verify_accept_stochastic(const float* target_logits, const float* draft_logits,
                                      const int32_t* parent, const int32_t* token,
                                      const int32_t* tree_off, int nseq, int N, int64_t V,
                                      int total_nodes, const double* u_accept, const double* u_bonus,
                                      int32_t* accept_len, int32_t* path, int32_t* bonus, void* ws,
                                      size_t ws_bytes, jt_stream_t stream) {
    JT_RANGE("jt_verify_accept_stochastic");
    if (!target_logits || (!draft_logits && N > 0) || !parent || !token || !tree_off || !u_accept ||
        !u_bonus || !accept_len || !path || !bonus || nseq < 1 || nseq > 8192 || N < 0 ||
        N > JT_MAX_TREE || V < 1 || V > 0x7FFFFFFFll || total_nodes < nseq)
        return JT_ERR_INVALID;
    if (V > JT_STOCHASTIC_MAX_V) return JT_ERR_UNSUPPORTED;
    jt_status s = check_ws(ws, ws_bytes, accept_workspace_bytes(nseq, total_nodes));
    if (s != JT_OK) return s;
    return from_cuda(verify_stochastic_launch(target_logits, draft_logits, parent, token, tree_off, nseq, N, V,
                                              total_nodes, u_accept, u_bonus, accept_len, path, bonus,
                                              static_cast<char*>(ws), stream));
}

jt_status jt_check(void* ws, jt_stream_t stream) {
    JT_RANGE("jt_check");
    if (!ws) return JT_ERR_WORKSPACE;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return JT_ERR_CUDA;
    uint32_t err = 0;
    e = cudaMemcpy(&err, ws, sizeof(err), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return JT_ERR_CUDA;
    if (err) {
        const uint32_t zero = 0;
        if (cudaMemcpy(ws, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return JT_ERR_CUDA;
    }
    if (err & DEVERR_TIMEOUT) return JT_ERR_TIMEOUT;
    if (err & DEVERR_INVALID) return JT_ERR_INVALID;
    return JT_OK;
}

}  // extern "C"
