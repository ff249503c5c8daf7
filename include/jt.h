/*
 * jt.h -- C ABI of libjt, the GB300 (sm_103a) hot path of JetSpec-style tree
 * speculative decoding: draft-tree build, tree-causal paged attention and
 * tree acceptance.
 *
 * Conventions shared by every entry point
 *  - Array arguments are DEVICE pointers owned by the caller, unless a
 *    comment says "host".  The library allocates no memory and keeps no
 *    state besides a per-device cache of device properties (and the fixed
 *    scratch array behind jt_tree_build_noalloc).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Outputs are valid once the stream reaches the call.
 *    Some kernels are launched as programmatic dependents of the kernel
 *    before them on the stream (they may become resident early); each one
 *    waits for that kernel to finish before it reads or writes global
 *    memory, so ordinary stream order holds whatever ran before.
 *  - Arguments checkable on the host (null pointers, sizes, limits, the
 *    workspace size) are checked before anything is enqueued; on failure the
 *    call returns JT_ERR_INVALID / JT_ERR_UNSUPPORTED / JT_ERR_WORKSPACE and
 *    writes nothing.
 *  - Contents of device arrays (tree offsets, prefix lengths, tree
 *    structure) are checked on the device; an offending sequence is skipped
 *    (its outputs are left untouched) and a flag is raised in the first
 *    word of the workspace.  jt_check() synchronises the stream and turns
 *    that flag into a status.  Device-side waits are bounded in time; a wait
 *    that runs out raises JT_ERR_TIMEOUT the same way.
 *  - Every call needs a caller-allocated device workspace of at least
 *    jt_workspace_size(...) bytes, 256-byte aligned, whose first 256 bytes
 *    (the header holding the error word) are ZERO before its first use
 *    (e.g. one cudaMemset after allocating it).  Calls never clear the
 *    header themselves: a raised flag stays set until jt_check() reads and
 *    clears it.  Calls that share one workspace must not overlap on the
 *    device.
 *
 * Tree layout shared by the three steps
 *  - nseq sequences; sequence b owns global node indices
 *    tree_off[b] .. tree_off[b+1]-1 (tree_off: int32 [nseq+1], tree_off[0]=0),
 *    so its budget is B_b = tree_off[b+1] - tree_off[b], 1 <= B_b <= 256.
 *  - Within a sequence, nodes are numbered 0..B_b-1 in the order the
 *    best-first expansion pops them; node 0 is the root (the last verified
 *    token); parent[] holds LOCAL indices (root: -1) and parent < child.
 *  - anc: uint32 [total_nodes, 8], a 256-bit ancestor-or-self set per node:
 *    bit j of word w is set when local node 32*w + j is the node itself or
 *    one of its ancestors.
 *  - total_nodes (host) is the capacity of the node-indexed arrays and must
 *    be >= tree_off[nseq]; it may be larger (tree offsets written on the
 *    device by jt_tree_policy, whose total the host does not know).  Rows at
 *    or beyond tree_off[nseq] are neither read nor written.
 *
 * Sources (prose pages; no code is printed there):
 *  [JS-news] JetSpec news summary (mlqm.cn/news/158889): tree-causal
 *      attention mask; building the candidate tree from one forward's
 *      per-depth logits, top-W per depth, cumulative draft log-prob, greedy
 *      fill to the budget B, depth at most N; longest consistent prefix.
 *  [JS-art] "加速AI思考：UC San Diego等机构研究出让大模型“一心多用”的推测解码新方法":
 *      section 三 (mask, one-forward verification), section 五 (best-first
 *      expansion with a priority queue), section 七 (paged tree attention
 *      without a dense mask).
 *  [AS] "AdaptiveSpec：免训练推测解码方案提速56%的技术解析", section
 *      "逐步Margin规则": accept when p(draft)/p(top1) >= t; section
 *      "逐步树策略：动态调整草稿树规模": per-step tree size from the draft's
 *      top-1 confidence and the rolling acceptance history.
 *  [SD] speculative-decoding overview, chooseai.io/news/6515, section
 *      "推测解码是什么：草稿模型先猜，目标模型验收" (rejection-sampling acceptance).
 */
#ifndef JT_H
#define JT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so that users need no CUDA
 * header to include this file. */
typedef struct CUstream_st* jt_stream_t;

typedef enum {
    JT_OK = 0,
    JT_ERR_INVALID = -1,      /* bad argument, or bad device-side array contents */
    JT_ERR_UNSUPPORTED = -2,  /* valid but outside this build's limits (dtype, D, G, GPU) */
    JT_ERR_CUDA = -3,         /* a CUDA runtime call failed */
    JT_ERR_TIMEOUT = -4,      /* a bounded device-side wait ran out */
    JT_ERR_WORKSPACE = -5     /* workspace missing, misaligned or too small */
} jt_status;

typedef enum { JT_DTYPE_F32 = 0, JT_DTYPE_BF16 = 1 } jt_dtype;
typedef enum { JT_RULE_GREEDY = 0, JT_RULE_MARGIN = 1 } jt_rule;
typedef enum { JT_OP_TREE_BUILD = 0, JT_OP_TREE_ATTN = 1, JT_OP_VERIFY_ACCEPT = 2,
               JT_OP_TREE_TOPW = 3, JT_OP_TREE_BUILD_MIXED = 4, JT_OP_TREE_POLICY = 5 } jt_op;

/* Limits of this build. */
#define JT_MAX_TREE 256   /* B_b (bitset width) */
#define JT_MAX_W 8        /* draft width W */
#define JT_MAX_N 64       /* draft depth N */
#define JT_PAGE_SIZE 16   /* KV page size in tokens */

/*
 * Workspace bytes needed by one call of `op` with these sizes (arguments an
 * op does not use are ignored; pass 0).  Depends on the current device's SM
 * count for JT_OP_TREE_ATTN.  Returns 0 for invalid sizes.
 *   TREE_BUILD:    nseq, N, W, V
 *   TREE_BUILD_MIXED: nseq, N, W, V
 *   TREE_POLICY:   (256 bytes: the header only; jt_tree_expand and
 *                  jt_tree_expand_capped need the same)
 *   TREE_TOPW:     nseq*N rows given as nseq (N=1), W, V
 *   TREE_ATTN:     nseq, total_nodes, Hq, Hkv, D, max_pages, max_tree
 *   VERIFY_ACCEPT: nseq, total_nodes
 */
size_t jt_workspace_size(int op, int nseq, int N, int W, int64_t V, int total_nodes,
                         int Hq, int Hkv, int D, int max_pages, int max_tree);

/*
 * jt_tree_build -- draft-tree construction ([JS-news] tree construction;
 * [JS-art] section 五).
 *   draft_logits: fp32 [nseq, N, V]; row (b, d) is the draft distribution
 *                 for depth d+1 of sequence b (shared by every node of that
 *                 depth).
 *   root_token:   int32 [nseq], token of each root.
 *   tree_off:     int32 [nseq+1], budgets B_b as described above; the full
 *                 W-ary tree of depth N must hold at least B_b nodes.
 *   total_nodes:  capacity >= tree_off[nseq] (host value; sizes the outputs).
 * Step 1 takes, per row, the top-W tokens (logit descending, token id
 * ascending) and lse = log sum exp(z).  Step 2 runs best-first expansion:
 * a queue of candidate nodes keyed by (cumulative log-prob descending, depth
 * ascending, token ascending, parent index ascending); the best candidate is
 * popped and becomes the next node; its W children (depth < N) are pushed;
 * stop at B_b nodes.  Log-probs and scores are fp64.
 * Outputs (global node index): parent (local), token, depth (int32
 * [total_nodes]) and anc (uint32 [total_nodes, 8]).
 */
jt_status jt_tree_build(const float* draft_logits, const int32_t* root_token,
                        const int32_t* tree_off, int nseq, int N, int W, int64_t V,
                        int total_nodes, int32_t* parent, int32_t* token, int32_t* depth,
                        uint32_t* anc, void* ws, size_t ws_bytes, jt_stream_t stream);

/*
 * jt_tree_build_mixed -- jt_tree_build with entropy-mixed step scores
 * ([JS-art] section 五: besides the cumulative probability, the authors
 * score candidates by the information entropy at each position and by a
 * weighted mix of the two).  Reading: the step from depth d to d+1 through
 * token x adds
 *     (1 - alpha) * lp_d(x) - alpha * H_d,
 * H_d = lse_d - sum_v softmax(z_d)_v * z_d,v the natural-log entropy of
 * draft row d (masked entries, z = -inf, add 0), evaluated in fp64 as
 * ((1 - alpha) * lp) - (alpha * H); a candidate of probability 0 (lp =
 * -inf) keeps -inf under every weight.
 *   alpha: in [0, 1]; 0 gives exactly jt_tree_build's trees (the same
 *          kernels run); 1 is the pure entropy score, under which every
 *          node of a depth ties and the queue's tie-breaks (depth, then
 *          token, then parent) decide.  Outside [0, 1]: JT_ERR_INVALID.
 * Every step still adds a value <= 0; the expansion (queue key and
 * tie-breaks), outputs, limits and error behaviour are those of
 * jt_tree_build.  The entropy sum is accumulated in float-float (about
 * 1e-12 relative), so trees equal the fp64 definition's except where two
 * different candidate scores lie closer than that.
 * Workspace: jt_workspace_size(JT_OP_TREE_BUILD_MIXED, nseq, N, W, V).
 */
jt_status jt_tree_build_mixed(const float* draft_logits, const int32_t* root_token,
                              const int32_t* tree_off, int nseq, int N, int W, int64_t V,
                              int total_nodes, double alpha, int32_t* parent, int32_t* token,
                              int32_t* depth, uint32_t* anc, void* ws, size_t ws_bytes,
                              jt_stream_t stream);

/*
 * jt_tree_build_noalloc -- jt_tree_build with no caller workspace and no
 * allocation.  The pages have no counterpart: this entry point exists for
 * host integrations that cannot give the library device memory (memory owned
 * by another allocator, or a decode loop that must not call cudaMalloc, which
 * synchronises the device).
 *   Arguments, outputs and results are those of jt_tree_build; the scratch
 *   is a fixed device array of JT_NOALLOC_SCRATCH_BYTES inside the library.
 *   It must hold 256 bytes of header plus the build's tables, i.e.
 *   jt_workspace_size(JT_OP_TREE_BUILD, nseq, N, W, V) bytes (about 4096
 *   draft rows nseq*N at V = 151936, W = 4); a larger need returns
 *   JT_ERR_WORKSPACE before anything is enqueued.
 *   sync_check: 0 = asynchronous, like jt_tree_build (device-side errors are
 *   then not reported); nonzero = synchronise `stream` after the launch and
 *   return the device-side status (JT_ERR_INVALID / JT_ERR_TIMEOUT).
 *   The first call on a device looks up the array's address
 *   (cudaGetSymbolAddress); make it before any stream capture.
 *   There is ONE scratch array per device: calls whose executions overlap on
 *   the device (different streams, or different host threads without
 *   ordering) race on it and give wrong trees.  Serialise them.
 */
#define JT_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)
jt_status jt_tree_build_noalloc(const float* draft_logits, const int32_t* root_token,
                                const int32_t* tree_off, int nseq, int N, int W, int64_t V,
                                int total_nodes, int32_t* parent, int32_t* token, int32_t* depth,
                                uint32_t* anc, int sync_check, jt_stream_t stream);

/*
 * jt_tree_topw -- step 1 of jt_tree_build alone, on `rows` rows of V fp32
 * logits: tok int32 [rows, W], lp fp64 [rows, W] (= z[tok] - lse), lse fp64
 * [rows].  Same kernels as jt_tree_build.
 */
jt_status jt_tree_topw(const float* logits, int64_t rows, int64_t V, int W, int32_t* tok,
                       double* lp, double* lse, void* ws, size_t ws_bytes, jt_stream_t stream);

/*
 * jt_tree_expand -- step 2 of jt_tree_build alone, from given per-depth
 * tables tok int32 [nseq, N, W] and lp fp64 [nseq, N, W] (row d = candidates
 * of depth d+1, best first).  Same outputs as jt_tree_build.  Needs a
 * workspace of at least 256 bytes (only its error word is used).
 */
jt_status jt_tree_expand(const int32_t* tok, const double* lp, const int32_t* root_token,
                         const int32_t* tree_off, int nseq, int N, int W, int total_nodes,
                         int32_t* parent, int32_t* token, int32_t* depth, uint32_t* anc,
                         void* ws, size_t ws_bytes, jt_stream_t stream);

/*
 * jt_tree_expand_capped -- jt_tree_expand with per-sequence caps on the
 * tree's width and depth ([AS] per-step tree policy: each request's tree
 * gets its own depth, width and node count).
 *   w_cap: int32 [nseq] or NULL; sequence b uses only the first w_cap[b]
 *          candidates of every row (1 <= w_cap[b] <= W).
 *   n_cap: int32 [nseq] or NULL; nodes of depth n_cap[b] get no children
 *          (0 <= n_cap[b] <= N).
 * The tree is then the best-first expansion of the capped full tree; B_b
 * must fit it.  A cap out of range or a budget beyond the capped tree
 * skips the sequence and raises JT_ERR_INVALID (device-side).  With both
 * caps NULL this is jt_tree_expand.  Workspace: 256 bytes.
 */
jt_status jt_tree_expand_capped(const int32_t* tok, const double* lp, const int32_t* root_token,
                                const int32_t* tree_off, const int32_t* w_cap, const int32_t* n_cap,
                                int nseq, int N, int W, int total_nodes, int32_t* parent,
                                int32_t* token, int32_t* depth, uint32_t* anc, void* ws,
                                size_t ws_bytes, jt_stream_t stream);

/*
 * Parameters of the adaptive tree policy (host struct, read at the call).
 */
typedef struct {
    int32_t b_min;     /* budget floor, 1 <= b_min */
    int32_t b_max;     /* budget ceiling, b_min <= b_max <= JT_MAX_TREE */
    int32_t node_cap;  /* node budget of the whole batch, 0 = none; the
                          per-request ceiling is then
                          min(b_max, max(b_min, node_cap / nseq)) */
    int32_t w_min;     /* width when the draft is not confident, 1..W */
    int32_t n_min;     /* depth floor, 0..N */
    int32_t n_slack;   /* depth beyond the rolling accepted length, 0..N */
    double beta;       /* weight of the newest accepted length in the
                          rolling average, 0 < beta <= 1 */
    double log_conf;   /* confidence threshold on the log of the draft's
                          top-1 probability at depth 1 (not NaN) */
    double acc_thresh; /* threshold on the rolling accepted length, in
                          tokens (not NaN) */
} jt_policy_params;

/*
 * jt_tree_policy -- per-request tree size for the next step ([AS] section
 * "逐步树策略：动态调整草稿树规模": the draft's top-1 confidence and the
 * rolling acceptance history set depth, width and node count; the tree
 * grows when both are high and shrinks in the opposite case; [JS-art]
 * section 七: large budgets stop paying as the batch grows).  The pages
 * give no formula; this is the rule, per request b:
 *   ema   <- (1 - beta) * ema + beta * accept_len[b]   (if accept_len[b] >= 0)
 *   conf  =  lp[b, 0, 0] >= log_conf;  hot = ema >= acc_thresh
 *   B     <- clamp(B, b_min, ceil); then min(2B, ceil) if conf and hot,
 *            max(B / 2, b_min) if neither, else unchanged
 *   n_cap =  clamp(floor(ema) + n_slack, n_min, N);  w_cap = conf ? W : w_min
 *   budget = min(B, nodes of the full w_cap-ary tree of depth n_cap)
 *   tree_off = exclusive prefix sum of the budgets (tree_off[0] = 0)
 * fp64 operations are rounded one at a time (no fused multiply-add).
 *   lp:           fp64 [nseq, N, W], the per-depth table of jt_tree_topw.
 *   accept_len:   int32 [nseq] or NULL: accepted length of each request's
 *                 previous step (jt_verify_accept*), -1 = none observed.
 *   budget_state: int32 [nseq], in/out: the controller's B (not clipped to
 *                 the tree); initialise to the first budget wanted.
 *   acc_ema:      fp64 [nseq], in/out: the rolling accepted length (>= 0,
 *                 finite); initialise to a prior, e.g. acc_thresh.
 *   tree_off:     int32 [nseq+1] out; w_cap, n_cap: int32 [nseq] out, for
 *                 jt_tree_expand_capped.  tree_off[nseq] <= nseq * ceil.
 * A request whose accept_len is outside [-1, N] or whose acc_ema is
 * negative or not finite gets a root-only tree (budget 1, n_cap 0), keeps
 * its state and raises JT_ERR_INVALID (device-side).  One CTA; N >= 1.
 * Workspace: jt_workspace_size(JT_OP_TREE_POLICY, ...) = 256 bytes.
 */
jt_status jt_tree_policy(const double* lp, int nseq, int N, int W, const int32_t* accept_len,
                         const jt_policy_params* params, int32_t* budget_state, double* acc_ema,
                         int32_t* tree_off, int32_t* w_cap, int32_t* n_cap, void* ws,
                         size_t ws_bytes, jt_stream_t stream);

/*
 * jt_tree_build_adaptive -- jt_tree_topw, jt_tree_policy and
 * jt_tree_expand_capped in one call, with no host round trip: the budgets
 * stay on the device.
 *   capacity: host, >= nseq * ceil (ceil as in jt_tree_policy); sizes
 *             parent/token/depth [capacity] and anc [capacity, 8] like
 *             total_nodes elsewhere.  Pass it as total_nodes, and the
 *             policy's ceiling as max_tree, to jt_tree_attn_paged.
 * Other arguments as in jt_tree_build and jt_tree_policy (root_token
 * [nseq]; tree_off, w_cap, n_cap are outputs).  Workspace:
 * jt_workspace_size(JT_OP_TREE_BUILD, nseq, N, W, V).
 */
jt_status jt_tree_build_adaptive(const float* draft_logits, const int32_t* root_token, int nseq,
                                 int N, int W, int64_t V, int capacity, const int32_t* accept_len,
                                 const jt_policy_params* params, int32_t* budget_state,
                                 double* acc_ema, int32_t* tree_off, int32_t* w_cap,
                                 int32_t* n_cap, int32_t* parent, int32_t* token, int32_t* depth,
                                 uint32_t* anc, void* ws, size_t ws_bytes, jt_stream_t stream);

/*
 * jt_tree_attn_paged -- tree-causal attention over a paged KV cache
 * ([JS-news] tree-causal attention mask; [JS-art] sections 三 and 七).
 *   q:        [total_nodes, Hq, D] (dtype), the tree nodes' queries.
 *   k_cache, v_cache: [num_pages, page_size, Hkv, D] (dtype).
 *   dtype:    JT_DTYPE_BF16 (tensor-core path: D in {64,128},
 *             Hq/Hkv in {1,2,4,8,16}) or JT_DTYPE_F32 (D in {32,64,96,128}).
 *   block_table: int32 [nseq, max_pages]; logical page p of sequence b is
 *             physical page block_table[b*max_pages + p].  Entries past the
 *             pages a sequence uses are never read.
 *   prefix_len: int32 [nseq], L_b cached tokens in logical slots 0..L_b-1.
 *             Tree node i of sequence b has its K/V (written by the caller)
 *             in logical slot L_b + i; L_b + B_b <= max_pages*page_size.
 *   anc:      the ancestor-or-self sets of the tree (see above).
 *   max_tree: max_b B_b (host value; an upper bound used for sizing).
 *   page_size: must be JT_PAGE_SIZE.  scale: softmax scale (e.g. 1/sqrt(D)).
 * The bf16 path runs one work slot per SM (one CTA); the key tiles of all
 * (sequence, KV head, query-tile pair) units are split into equal ranges,
 * one per slot, planned on the device from prefix_len and tree_off.  A unit
 * cut by a range boundary is merged from fp32 partials in the workspace by
 * the slot that finishes its piece last.  For D = 128, when every
 * (sequence, KV head) has one query-tile pair at max_tree (max_tree <=
 * 2 * 128 / (Hq/Hkv) nodes), a slot is a cluster of two CTAs on two SMs
 * sharing each MMA (tcgen05 cta_group::2; one slot per resident pair).
 * The environment variable JT_ATTN_KERNEL = "pair" or "single" overrides
 * that choice (read at every call and by jt_workspace_size); both kernels
 * agree within the bf16 tolerance.  Workspace:
 * jt_workspace_size(JT_OP_TREE_ATTN, nseq, 0, 0, 0, total_nodes, Hq, Hkv,
 * D, max_pages, max_tree) = 256 + 16 * slots + O(nseq) + 2 * slots * 256 *
 * (D + 2) * 4 bytes (about 40 MB at D = 128 on 152 SMs), sized for the
 * current device and kernel choice and serving that device only.  Its
 * first 256 + 16 * SMs bytes (rounded up to 256; the header and the merge
 * counts) must be zero before its first use, like every header; they stay
 * valid from call to call (counts carry the number of the call that wrote
 * them, whatever the grid of the calls before), so they never need
 * clearing again.
 * Node n of sequence b, query head h (KV head h / (Hq/Hkv)) attends to
 * slots 0..L_b-1 and to slot L_b + j for every j in anc(n): never to a
 * sibling or a descendant.  No dense mask is formed.
 *   out:      [total_nodes, Hq, D] (bf16 for the bf16 path, fp32 for fp32):
 *             softmax(scale * q.K^T) V, fp32 accumulation, one rounding.
 *   lse:      fp32 [total_nodes, Hq] or NULL: natural-log sum of
 *             exp(scale * q.k) over the visible keys.
 */
jt_status jt_tree_attn_paged(const void* q, const void* k_cache, const void* v_cache, int dtype,
                             const int32_t* block_table, int max_pages, int num_pages,
                             const int32_t* prefix_len, const int32_t* tree_off,
                             const uint32_t* anc, int nseq, int total_nodes, int max_tree,
                             int Hq, int Hkv, int D, int page_size, float scale, void* out,
                             float* lse, void* ws, size_t ws_bytes, jt_stream_t stream);

/*
 * jt_verify_accept -- tree acceptance ([JS-art] section 三; [AS] margin rule).
 *   target_logits: fp32 [total_nodes, V]; row u = the target's logits
 *             after node u (it verifies u's children and gives u's bonus).
 *   parent, token: the tree (local parent indices, topological order).
 *   N:        maximum depth (width of `path` is N+1).
 *   rule:     JT_RULE_GREEDY: child c of an accepted node u is accepted
 *             when token[c] == argmax(row u) (lowest id on ties; first such
 *             child in node order).
 *             JT_RULE_MARGIN: child c of u passes when
 *             (double)row_u[token c] - (double)max(row u) >= log_t, i.e.
 *             p(draft)/p(top1) >= t; a node is reached when every edge of
 *             its root path passes; the result is the deepest reached node
 *             (lowest index on ties).
 *   log_t:    log(t) in fp64, t in (0, 1] (margin rule only).
 * Outputs per sequence: accept_len int32 [nseq] (accepted draft tokens =
 * depth of the final node), path int32 [nseq, N+1] (local node at each depth
 * of the accepted path, root first, -1 after the end), bonus int32 [nseq]
 * (argmax of the final node's row).  Only rows on reached nodes are read.
 */
jt_status jt_verify_accept(const float* target_logits, const int32_t* parent,
                           const int32_t* token, const int32_t* tree_off, int nseq, int N,
                           int64_t V, int total_nodes, int rule, double log_t,
                           int32_t* accept_len, int32_t* path, int32_t* bonus, void* ws,
                           size_t ws_bytes, jt_stream_t stream);

/*
 * jt_verify_accept_stochastic -- temperature-1 tree acceptance by rejection
 * sampling ([SD] acceptance paragraph; [AS] section "严格的token匹配验证机制":
 * accept a drafted token x with probability min(1, p(x)/q(x)); after a
 * rejection draw from norm(max(0, p - q))).
 *   target_logits: fp32 [total_nodes, V]; row u is the target after node u.
 *   draft_logits:  fp32 [nseq, N, V]; row (b, d) is the draft distribution
 *                  of depth d+1 (the rows the tree was built from).
 *   u_accept, u_bonus: fp64 [total_nodes], the caller's uniforms in [0, 1):
 *                  u_accept[c] decides the test of node c, u_bonus[u] the
 *                  bonus draw when the walk stops at node u.
 * From the root: the current node's children are tried in node order
 * against a running residual r (first r = p = softmax of the node's target
 * row; q = softmax of the draft row of the children's depth, both at
 * temperature 1): child c with token t is accepted when
 * u_accept[c] < min(1, r(t)/q(t)); after a rejection r <- norm(max(0, r - q)).
 * An accepted child becomes the current node.  When no child is accepted
 * (or there is none) the bonus is the smallest token x with
 * r(0) + ... + r(x) > u_bonus[u] * sum(r).  Outputs as jt_verify_accept.
 * Softmax and sums are fp32: a decision whose uniform lies within ~1e-5 of
 * its threshold can differ from an fp64 evaluation.
 * V <= JT_STOCHASTIC_MAX_V (the vocabulary is held in shared memory across
 * one thread-block cluster per sequence), else JT_ERR_UNSUPPORTED.
 * Workspace: jt_workspace_size(JT_OP_VERIFY_ACCEPT, nseq, ...).
 */
#define JT_STOCHASTIC_MAX_V 409600
jt_status jt_verify_accept_stochastic(const float* target_logits, const float* draft_logits,
                                      const int32_t* parent, const int32_t* token,
                                      const int32_t* tree_off, int nseq, int N, int64_t V,
                                      int total_nodes, const double* u_accept, const double* u_bonus,
                                      int32_t* accept_len, int32_t* path, int32_t* bonus, void* ws,
                                      size_t ws_bytes, jt_stream_t stream);

/*
 * jt_check -- synchronise `stream`, read the device-side error flag of a
 * workspace used by an earlier call, clear it, and return the matching
 * status (JT_OK, JT_ERR_INVALID, JT_ERR_TIMEOUT or JT_ERR_CUDA).
 */
jt_status jt_check(void* ws, jt_stream_t stream);

/*
 * jt_selftest_wait_timeout -- diagnostic of the device-side failure path
 * (no counterpart in the pages).  Launches one 32-thread CTA that waits,
 * with the same bounded wait every kernel of the library uses, for an
 * mbarrier phase that nothing completes.  After the library's wait limit
 * (2 s) the wait gives up, raises the timeout flag in the workspace's error
 * word and the kernel exits normally: the next jt_check(ws, stream) returns
 * JT_ERR_TIMEOUT and the CUDA context stays usable.  No fault, trap or
 * unbounded wait is involved.
 *   ws: a workspace of at least 256 bytes (only its error word is used).
 */
jt_status jt_selftest_wait_timeout(void* ws, size_t ws_bytes, jt_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* jt_status_str(jt_status status);

/* Library ABI version (major*10000 + minor*100 + patch). */
int jt_version(void);

#ifdef __cplusplus
}
#endif
#endif /* JT_H */
