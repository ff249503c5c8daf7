/*
 * jt_oracle.c -- plain, slow, obviously-correct CPU oracle for the tree
 * speculative decoding hot path (tree build, tree-causal paged attention,
 * tree acceptance).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library: every step is written out here in fp64 with plain loops.
 *
 * Sources (the method is described in prose only; no code is printed there):
 *  [JS-news]  JetSpec news summary, mlqm.cn/news/158889, paragraph on
 *             building the candidate tree (top W per depth, greedy fill
 *             to the budget) and on the tree-causal attention mask.
 *  [JS-art]   "加速AI思考：UC San Diego等机构研究出让大模型“一心多用”的推测解码新方法",
 *             section 三 (tree-causal mask, parallel verification) and
 *             section 五 (tree construction: priority queue, cumulative
 *             log-prob, W, B).
 *  [AS]       "AdaptiveSpec：免训练推测解码方案提速56%的技术解析",
 *             section "逐步Margin规则" (accept if p(draft)/p(top1) >= t,
 *             worked example 0.30/0.35 ~ 0.86 >= 0.8).
 *
 * Readings taken where the pages leave a step open (each is listed in the
 * design notes of the repository):
 *  - draft logits are per depth: row d of a sequence scores every node at
 *    depth d+1, so all nodes of one depth share the same W candidates;
 *  - the budget B counts tree nodes including the root, and a node counts
 *    when it is popped from the priority queue (its pushed children are only
 *    candidates);
 *  - queue order key: score descending, then depth ascending, then token id
 *    ascending, then parent index ascending; top-W order: logit descending,
 *    token id ascending; argmax ties: lowest token id;
 *  - node numbering is pop order (topological: parent index < child index);
 *  - row u of the target logits is the target's next-token distribution after
 *    node u: it verifies u's children and supplies the bonus token at u;
 *  - the margin rule is applied per edge at the parent's row, in log space:
 *    z[tok] - max(z) >= log(t), with log(t) supplied by the caller.
 *
 * Precision: every arithmetic step is fp64.  fp32 and bf16 inputs are
 * converted exactly.  exp/log are the C library's double routines.
 *
 * Parity pins (tests/test_oracle_*.py): brute-force path enumeration, W=1
 * chain == causal attention (library SDPA), per-node brute-force attention,
 * sibling/descendant perturbation invariance, page permutation invariance,
 * constant-key closed form, the AdaptiveSpec worked example, brute-force
 * acceptance on tiny trees, t=1 margin == greedy.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define JTO_OK 0
#define JTO_ERR_INVALID (-1)
#define JTO_MAX_TREE 256

/* ------------------------------------------------------------------------ */
/* small helpers                                                             */
/* ------------------------------------------------------------------------ */

/* bf16 -> double, exact: a bf16 is the top 16 bits of an IEEE binary32. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element of a q/k/v array given as fp32 (dtype 0) or bf16 (dtype 1). */
static double load_elem(const void* base, int dtype, int64_t idx)
{
    if (dtype == 0) return (double)((const float*)base)[idx];
    return bf16_to_double(((const uint16_t*)base)[idx]);
}

/* Index of the largest entry of a row; ties go to the lowest index. */
static int64_t row_argmax(const float* z, int64_t V)
{
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
        if (z[v] > z[best]) best = v;
    return best;
}

/* Number of nodes of a full W-ary tree of depth N, including the root,
 * saturated at cap. */
static int64_t full_tree_nodes(int N, int W, int64_t cap)
{
    int64_t total = 1, level = 1;
    for (int d = 1; d <= N; ++d) {
        level *= W;
        total += level;
        if (total >= cap || level >= cap) return cap;
    }
    return total;
}

/* ------------------------------------------------------------------------ */
/* Tree build, step 1: top-W per depth and log-softmax normaliser.           */
/* [JS-news]: one forward gives the logits of every depth; each depth keeps  */
/* its top-W candidates.  The branch score uses log-probabilities, so each   */
/* row also needs lse = log sum_v exp(z_v).                                  */
/* ------------------------------------------------------------------------ */

/*
 * z: [rows, V] fp32.  Outputs per row r: tok[r*W + k] (k-th best id by
 * logit descending, id ascending), lp[r*W + k] = z[tok] - lse[r],
 * lse[r] = m + log(sum_v exp(z_v - m)) with m the row maximum; the sum runs
 * over v = 0..V-1 in order.
 */
int jto_topw_lse(const float* z, int64_t rows, int64_t V, int W,
                 int32_t* tok, double* lp, double* lse)
{
    if (!z || !tok || !lp || !lse || rows < 0 || V < 1 || W < 1 || W > V)
        return JTO_ERR_INVALID;
    char* taken = (char*)calloc((size_t)V, 1);
    if (!taken) return JTO_ERR_INVALID;
    for (int64_t r = 0; r < rows; ++r) {
        const float* row = z + r * V;
        double m = (double)row[row_argmax(row, V)];
        double S = 0.0;
        for (int64_t v = 0; v < V; ++v) S += exp((double)row[v] - m);
        double L = m + log(S);
        lse[r] = L;
        memset(taken, 0, (size_t)V);
        /* W selection passes: each pass takes the best id not yet taken. */
        for (int k = 0; k < W; ++k) {
            int64_t best = -1;
            for (int64_t v = 0; v < V; ++v) {
                if (taken[v]) continue;
                if (best < 0 || row[v] > row[best]) best = v;
            }
            taken[best] = 1;
            tok[r * W + k] = (int32_t)best;
            lp[r * W + k] = (double)row[best] - L;
        }
    }
    free(taken);
    return JTO_OK;
}

/* ------------------------------------------------------------------------ */
/* Tree build, step 2: best-first expansion.                                 */
/* [JS-art] section 五: a priority queue holds candidate nodes, the priority */
/* is the cumulative log-probability of the node's path; repeatedly pop the  */
/* best node, give it (up to) W children, push them, until the tree holds B  */
/* nodes.  Depth never exceeds N ([JS-news]).                                */
/* ------------------------------------------------------------------------ */

typedef struct {
    double score;   /* cumulative draft log-prob of the path root..node     */
    int depth;      /* 1..N                                                 */
    int token;      /* draft token of the node                              */
    int parent;     /* local index of the parent (already in the tree)      */
    int alive;      /* still in the queue                                   */
} jto_cand;

/* 1 if candidate a comes out of the queue before candidate b. */
static int cand_before(const jto_cand* a, const jto_cand* b)
{
    if (a->score != b->score) return a->score > b->score;
    if (a->depth != b->depth) return a->depth < b->depth;
    if (a->token != b->token) return a->token < b->token;
    return a->parent < b->parent;
}

/*
 * Expansion from given per-depth tables (tok/lp: [nseq, N, W]; row d holds
 * the candidates of depth d+1, best first).  Writes, for every sequence b
 * and local node i < B_b = tree_off[b+1]-tree_off[b], at global index
 * tree_off[b]+i: parent (local, -1 for the root), token, depth, the path
 * score, and the 256-bit ancestor-or-self set anc[.., 8] (bit j of word w
 * marks local node 32w+j).  gap[b] (optional) receives the smallest score
 * difference between the popped candidate and the best remaining one over
 * all pops of sequence b (+inf if never two candidates): a decision closer
 * than rounding noise is reported, not hidden.
 *
 * Optional per-sequence caps (either pointer may be NULL = no cap): w_cap[b]
 * in [1, W] keeps only the first w_cap[b] candidates of every row, n_cap[b]
 * in [0, N] stops the tree at depth n_cap[b] (nodes of that depth get no
 * children).  The budget must fit the capped full tree.
 */
static int expand_impl(const int32_t* tok, const double* lp, const int32_t* root_token,
                       const int32_t* tree_off, const int32_t* w_cap, const int32_t* n_cap,
                       int nseq, int N, int W, int32_t* parent, int32_t* token, int32_t* depth,
                       uint32_t* anc, double* score, double* gap)
{
    if (!tok || !lp || !root_token || !tree_off || nseq < 0 || N < 0 || W < 1)
        return JTO_ERR_INVALID;
    for (int b = 0; b < nseq; ++b) {
        int B = tree_off[b + 1] - tree_off[b];
        int Wb = w_cap ? w_cap[b] : W;
        int Nb = n_cap ? n_cap[b] : N;
        if (Wb < 1 || Wb > W || Nb < 0 || Nb > N) return JTO_ERR_INVALID;
        if (B < 1 || B > JTO_MAX_TREE || B > full_tree_nodes(Nb, Wb, JTO_MAX_TREE + 1))
            return JTO_ERR_INVALID;
    }
    /* every popped node pushes at most W candidates */
    jto_cand* q = (jto_cand*)malloc(sizeof(jto_cand) * (size_t)(JTO_MAX_TREE * W + 1));
    if (!q) return JTO_ERR_INVALID;

    for (int b = 0; b < nseq; ++b) {
        const int off = tree_off[b];
        const int B = tree_off[b + 1] - off;
        const int Wb = w_cap ? w_cap[b] : W;
        const int Nb = n_cap ? n_cap[b] : N;
        const int32_t* tk = tok + (int64_t)b * N * W;
        const double* lq = lp + (int64_t)b * N * W;
        double sc[JTO_MAX_TREE];
        int dp[JTO_MAX_TREE];
        int nq = 0;
        double min_gap = INFINITY;

        /* node 0: the root (the last verified token), score 0 */
        parent[off] = -1;
        token[off] = root_token[b];
        depth[off] = 0;
        sc[0] = 0.0;
        dp[0] = 0;
        int count = 1;
        /* push the root's children */
        if (Nb >= 1)
            for (int k = 0; k < Wb; ++k) {
                jto_cand c = { sc[0] + lq[k], 1, tk[k], 0, 1 };
                q[nq++] = c;
            }
        while (count < B) {
            /* pop: linear scan for the best live candidate */
            int best = -1;
            for (int i = 0; i < nq; ++i)
                if (q[i].alive && (best < 0 || cand_before(&q[i], &q[best]))) best = i;
            if (best < 0) break; /* cannot happen: B <= full tree size */
            /* runner-up, for the decision-gap report */
            int second = -1;
            for (int i = 0; i < nq; ++i)
                if (q[i].alive && i != best && (second < 0 || cand_before(&q[i], &q[second])))
                    second = i;
            if (second >= 0) {
                double g = q[best].score - q[second].score;
                if (g < min_gap) min_gap = g;
            }
            jto_cand c = q[best];
            q[best].alive = 0;
            const int n = count++;
            parent[off + n] = c.parent;
            token[off + n] = c.token;
            depth[off + n] = c.depth;
            sc[n] = c.score;
            dp[n] = c.depth;
            /* push its children (row c.depth scores depth c.depth+1) */
            if (c.depth < Nb)
                for (int k = 0; k < Wb; ++k) {
                    jto_cand ch = { sc[n] + lq[(int64_t)c.depth * W + k], c.depth + 1,
                                    tk[(int64_t)c.depth * W + k], n, 1 };
                    q[nq++] = ch;
                }
        }
        (void)dp;
        /* ancestor-or-self sets, by walking parent pointers */
        for (int n = 0; n < B; ++n) {
            uint32_t* a = anc ? anc + (int64_t)(off + n) * 8 : NULL;
            if (a) {
                for (int w = 0; w < 8; ++w) a[w] = 0u;
                for (int u = n; u >= 0; u = parent[off + u]) a[u >> 5] |= 1u << (u & 31);
            }
            if (score) score[off + n] = sc[n];
        }
        if (gap) gap[b] = min_gap;
    }
    free(q);
    return JTO_OK;
}

int jto_tree_expand(const int32_t* tok, const double* lp, const int32_t* root_token,
                    const int32_t* tree_off, int nseq, int N, int W,
                    int32_t* parent, int32_t* token, int32_t* depth, uint32_t* anc,
                    double* score, double* gap)
{
    return expand_impl(tok, lp, root_token, tree_off, NULL, NULL, nseq, N, W, parent, token, depth,
                       anc, score, gap);
}

int jto_tree_expand_capped(const int32_t* tok, const double* lp, const int32_t* root_token,
                           const int32_t* tree_off, const int32_t* w_cap, const int32_t* n_cap,
                           int nseq, int N, int W, int32_t* parent, int32_t* token, int32_t* depth,
                           uint32_t* anc, double* score, double* gap)
{
    return expand_impl(tok, lp, root_token, tree_off, w_cap, n_cap, nseq, N, W, parent, token, depth,
                       anc, score, gap);
}

/* Full tree build: top-W/lse on every (sequence, depth) row, then expansion.
 * draft_logits: [nseq, N, V] fp32.  tok_out/lp_out ([nseq,N,W]) and
 * lse_out ([nseq,N]) are optional copies of the step-1 tables. */
int jto_tree_build(const float* draft_logits, const int32_t* root_token, const int32_t* tree_off,
                   int nseq, int N, int W, int64_t V,
                   int32_t* parent, int32_t* token, int32_t* depth, uint32_t* anc,
                   double* score, double* gap,
                   int32_t* tok_out, double* lp_out, double* lse_out)
{
    if (!draft_logits || nseq < 0 || N < 0 || W < 1 || V < W) return JTO_ERR_INVALID;
    int64_t rows = (int64_t)nseq * N;
    int32_t* tk = tok_out ? tok_out : (int32_t*)malloc(sizeof(int32_t) * (size_t)(rows * W + 1));
    double* l = lp_out ? lp_out : (double*)malloc(sizeof(double) * (size_t)(rows * W + 1));
    double* s = lse_out ? lse_out : (double*)malloc(sizeof(double) * (size_t)(rows + 1));
    int rc = (tk && l && s) ? JTO_OK : JTO_ERR_INVALID;
    if (rc == JTO_OK) rc = jto_topw_lse(draft_logits, rows, V, W, tk, l, s);
    if (rc == JTO_OK)
        rc = jto_tree_expand(tk, l, root_token, tree_off, nseq, N, W, parent, token, depth, anc,
                             score, gap);
    if (!tok_out) free(tk);
    if (!lp_out) free(l);
    if (!lse_out) free(s);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Tree-causal paged attention.                                              */
/* [JS-news] / [JS-art] section 三: every tree node sees the original prefix */
/* and its own ancestors on its branch (itself included), never siblings or  */
/* descendants.  [JS-art] section 七: the K/V live in a paged cache; the     */
/* mask is never expanded into a dense matrix.  Here the visible key list of */
/* a node is built explicitly by walking parent pointers.                    */
/* ------------------------------------------------------------------------ */

/*
 * q: [total, Hq, D]; k_cache, v_cache: [pages, page_size, Hkv, D]; dtype 0 =
 * fp32, 1 = bf16 (all three alike).  block_table: [nseq, max_pages]: logical
 * page p of sequence b lives in physical page block_table[b*max_pages+p].
 * Sequence b has prefix_len[b] = L_b cached tokens in logical slots
 * 0..L_b-1, and tree node i (local) in slot L_b + i.  Query head h reads KV
 * head h / (Hq/Hkv).
 *
 * rows: optional list of global node indices to evaluate (n_rows entries);
 * NULL means all nodes 0..total-1 (n_rows = total).  out: [n_rows, Hq, D],
 * lse: [n_rows, Hq] (natural log of sum exp(scale * q.k) over visible keys).
 */
int jto_tree_attn(const void* q, const void* k_cache, const void* v_cache, int dtype,
                  const int32_t* block_table, int max_pages, const int32_t* prefix_len,
                  const int32_t* tree_off, const int32_t* parent, int nseq, int Hq, int Hkv,
                  int D, int page_size, double scale, const int32_t* rows, int64_t n_rows,
                  double* out, double* lse)
{
    if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !tree_off || !parent ||
        !out || nseq < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1 || page_size < 1 ||
        (dtype != 0 && dtype != 1))
        return JTO_ERR_INVALID;
    const int G = Hq / Hkv;
    const int64_t total = tree_off[nseq];
    if (!rows) n_rows = total;
    int64_t max_keys = 0;
    for (int b = 0; b < nseq; ++b) {
        int64_t n = (int64_t)prefix_len[b] + (tree_off[b + 1] - tree_off[b]);
        if ((n + page_size - 1) / page_size > max_pages) return JTO_ERR_INVALID;
        if (n > max_keys) max_keys = n;
    }
    int64_t* slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)(max_keys + 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_keys + 1));
    int32_t path[JTO_MAX_TREE];
    if (!slot || !s) { free(slot); free(s); return JTO_ERR_INVALID; }

    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t n = rows ? rows[r] : r;
        if (n < 0 || n >= total) { free(slot); free(s); return JTO_ERR_INVALID; }
        int b = 0;
        while (!(tree_off[b] <= n && n < tree_off[b + 1])) ++b;
        const int64_t L = prefix_len[b];
        const int i = (int)(n - tree_off[b]);

        /* visible keys: prefix slots 0..L-1, then the root..i ancestor path */
        int64_t nk = 0;
        for (int64_t t = 0; t < L; ++t) slot[nk++] = t;
        int plen = 0;
        for (int u = i; u >= 0; u = parent[tree_off[b] + u]) path[plen++] = u;
        for (int p = plen - 1; p >= 0; --p) slot[nk++] = L + path[p];

        for (int h = 0; h < Hq; ++h) {
            const int kvh = h / G;
            const int64_t qbase = (n * Hq + h) * (int64_t)D;
            double m = -INFINITY;
            for (int64_t j = 0; j < nk; ++j) {
                const int64_t page = block_table[(int64_t)b * max_pages + slot[j] / page_size];
                const int64_t kbase = ((page * page_size + slot[j] % page_size) * Hkv + kvh) * (int64_t)D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += load_elem(q, dtype, qbase + d) * load_elem(k_cache, dtype, kbase + d);
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < nk; ++j) {
                s[j] = exp(s[j] - m); /* unnormalised probability */
                l += s[j];
            }
            double* o = out + (r * Hq + h) * (int64_t)D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t j = 0; j < nk; ++j) {
                const int64_t page = block_table[(int64_t)b * max_pages + slot[j] / page_size];
                const int64_t vbase = ((page * page_size + slot[j] % page_size) * Hkv + kvh) * (int64_t)D;
                for (int d = 0; d < D; ++d) o[d] += s[j] * load_elem(v_cache, dtype, vbase + d);
            }
            for (int d = 0; d < D; ++d) o[d] /= l;
            if (lse) lse[r * Hq + h] = m + log(l);
        }
    }
    free(slot);
    free(s);
    return JTO_OK;
}

/* ------------------------------------------------------------------------ */
/* Acceptance.                                                               */
/* [JS-art] section 三 / [JS-news]: the target verifies the whole tree in    */
/* one forward; along each path take the longest accepted prefix; adopt the  */
/* longest.  Greedy (temperature 0) rule: a drafted token is accepted when   */
/* it equals the target's argmax.  [AS] "逐步Margin规则": accept the drafted */
/* token when p_target(draft) / p_target(top1) >= t.                         */
/* ------------------------------------------------------------------------ */

/*
 * target_logits: [total, V] fp32, row u = target logits after node u.
 * parent/token: per node, local indices (root = -1).  rule 0 = greedy,
 * 1 = margin with threshold log_t = log(t).  Outputs per sequence b:
 * accept_len[b] = number of accepted draft tokens (depth of the final node),
 * path[b*(N+1) + k] = local node at depth k of the accepted path (root at 0),
 * -1 after its end; bonus[b] = argmax of the final node's row.
 * Depth is recomputed here by walking parent pointers.
 */
int jto_verify_accept(const float* target_logits, const int32_t* parent, const int32_t* token,
                      const int32_t* tree_off, int nseq, int N, int64_t V, int rule, double log_t,
                      int32_t* accept_len, int32_t* path, int32_t* bonus)
{
    if (!target_logits || !parent || !token || !tree_off || !accept_len || !path || !bonus ||
        nseq < 0 || N < 0 || V < 1 || (rule != 0 && rule != 1))
        return JTO_ERR_INVALID;
    for (int b = 0; b < nseq; ++b) {
        const int off = tree_off[b];
        const int B = tree_off[b + 1] - off;
        if (B < 1 || B > JTO_MAX_TREE) return JTO_ERR_INVALID;
        int dep[JTO_MAX_TREE];
        if (parent[off] != -1) return JTO_ERR_INVALID;
        for (int n = 1; n < B; ++n)
            if (parent[off + n] < 0 || parent[off + n] >= n) return JTO_ERR_INVALID;
        for (int n = 0; n < B; ++n) {
            int d = 0;
            for (int u = n; parent[off + u] >= 0; u = parent[off + u]) ++d;
            dep[n] = d;
            if (d > N) return JTO_ERR_INVALID;
        }
        int final_node = 0;
        if (rule == 0) {
            int u = 0;
            for (;;) {
                const int64_t a = row_argmax(target_logits + (int64_t)(off + u) * V, V);
                int next = -1;
                for (int c = 0; c < B; ++c)
                    if (parent[off + c] == u && token[off + c] == a) { next = c; break; }
                if (next < 0) break;
                u = next;
            }
            final_node = u;
        } else {
            /* ok[c]: the edge parent(c) -> c passes the margin test at the
             * parent's row; reach[c]: every edge root..c passes. */
            int reach[JTO_MAX_TREE];
            reach[0] = 1;
            for (int c = 1; c < B; ++c) {
                const int p = parent[off + c];
                const float* zp = target_logits + (int64_t)(off + p) * V;
                const double zmax = (double)zp[row_argmax(zp, V)];
                const int ok = ((double)zp[token[off + c]] - zmax) >= log_t;
                reach[c] = ok && reach[p]; /* p < c: already decided */
            }
            for (int c = 1; c < B; ++c)
                if (reach[c] && dep[c] > dep[final_node]) final_node = c;
        }
        accept_len[b] = dep[final_node];
        for (int k = 0; k <= N; ++k) path[(int64_t)b * (N + 1) + k] = -1;
        for (int u = final_node; u >= 0; u = parent[off + u])
            path[(int64_t)b * (N + 1) + dep[u]] = u;
        bonus[b] = (int32_t)row_argmax(target_logits + (int64_t)(off + final_node) * V, V);
    }
    return JTO_OK;
}

/* ------------------------------------------------------------------------ */
/* Stochastic (temperature 1) tree acceptance.                               */
/* [SD-overview] chooseai.io/news/6515, section "推测解码是什么：草稿模型先猜，  */
/* 目标模型验收", and [AS] section "严格的token匹配验证机制": a drafted token x is   */
/* accepted with probability min(1, p(x)/q(x)), p the target and q the draft */
/* distribution; after a rejection the next token is drawn from             */
/* norm(max(0, p - q)).                                                      */
/* Tree reading (the pages describe one chain): at the current node u the   */
/* children are tried in node order against a running residual r (r = p_u  */
/* at first); child c with token t is accepted when u_accept[c] <            */
/* min(1, r(t)/q(t)); after a rejection r <- norm(max(0, r - q)).  An        */
/* accepted child becomes the current node.  When every child is rejected,  */
/* or u has none, the bonus token is drawn from r by inverse CDF with        */
/* u_bonus[u]: the smallest x with r(0) + ... + r(x) > u_bonus[u] * sum(r).  */
/* p_u = softmax(target row u), q = softmax(draft row of the children's     */
/* depth), both at temperature 1.                                            */
/* ------------------------------------------------------------------------ */

/* softmax of a float row in fp64 (max-subtracted) */
static void softmax_row(const float* z, int64_t V, double* p)
{
    double m = -INFINITY;
    for (int64_t i = 0; i < V; ++i)
        if ((double)z[i] > m) m = (double)z[i];
    double s = 0.0;
    for (int64_t i = 0; i < V; ++i) {
        p[i] = exp((double)z[i] - m);
        s += p[i];
    }
    for (int64_t i = 0; i < V; ++i) p[i] /= s;
}

/*
 * draft_logits: [nseq, N, V] fp32 (row d = draft distribution of depth d+1).
 * u_accept, u_bonus: [total] uniforms in [0, 1) (u_accept of a root and
 * u_bonus of a node the walk never stops at are unused).
 * Outputs as jto_verify_accept.  Optional outputs (NULL to skip), so that a
 * caller can tell rounding-sensitive cases apart: min_margin[b] = the
 * smallest |u_accept - min(1, ratio)| over the acceptance tests taken for
 * sequence b (infinity when there were none); final_r[b*V + x] = the
 * normalised residual the bonus was drawn from; final_u[b] = the uniform of
 * that draw.
 */
int jto_verify_accept_stochastic(const float* target_logits, const float* draft_logits,
                                 const int32_t* parent, const int32_t* token,
                                 const int32_t* tree_off, int nseq, int N, int64_t V,
                                 const double* u_accept, const double* u_bonus,
                                 int32_t* accept_len, int32_t* path, int32_t* bonus,
                                 double* min_margin, double* final_r, double* final_u)
{
    if (!target_logits || (!draft_logits && N > 0) || !parent || !token || !tree_off ||
        !u_accept || !u_bonus || !accept_len || !path || !bonus || nseq < 0 || N < 0 || V < 1)
        return JTO_ERR_INVALID;
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    if (!r || !q) {
        free(r);
        free(q);
        return JTO_ERR_INVALID;
    }
    int status = JTO_OK;
    for (int b = 0; b < nseq && status == JTO_OK; ++b) {
        const int off = tree_off[b];
        const int B = tree_off[b + 1] - off;
        if (B < 1 || B > JTO_MAX_TREE || parent[off] != -1) { status = JTO_ERR_INVALID; break; }
        for (int n = 1; n < B; ++n)
            if (parent[off + n] < 0 || parent[off + n] >= n || token[off + n] < 0 ||
                token[off + n] >= V)
                status = JTO_ERR_INVALID;
        if (status != JTO_OK) break;
        double margin = INFINITY;
        int u = 0, d = 0;
        int32_t* pb = path + (int64_t)b * (N + 1);
        for (int k = 0; k <= N; ++k) pb[k] = -1;
        pb[0] = 0;
        for (;;) {
            softmax_row(target_logits + (int64_t)(off + u) * V, V, r);
            int next = -1;
            if (d < N) {
                int have_child = 0;
                for (int c = u + 1; c < B; ++c)
                    if (parent[off + c] == u) { have_child = 1; break; }
                if (have_child)
                    softmax_row(draft_logits + ((int64_t)b * N + d) * V, V, q);
                for (int c = u + 1; c < B && next < 0; ++c) {
                    if (parent[off + c] != u) continue;
                    const int t = token[off + c];
                    const double ratio = (q[t] > 0.0) ? r[t] / q[t] : INFINITY;
                    const double a = ratio < 1.0 ? ratio : 1.0;
                    const double ua = u_accept[off + c];
                    if (fabs(ua - a) < margin) margin = fabs(ua - a);
                    if (ua < a) {
                        next = c;
                    } else {
                        double z = 0.0;
                        for (int64_t x = 0; x < V; ++x) {
                            r[x] = r[x] - q[x] > 0.0 ? r[x] - q[x] : 0.0;
                            z += r[x];
                        }
                        for (int64_t x = 0; x < V; ++x) r[x] /= z;
                    }
                }
            }
            if (next < 0) break;
            u = next;
            ++d;
            pb[d] = u;
        }
        /* bonus: inverse CDF of r with u_bonus[u] */
        double total = 0.0;
        for (int64_t x = 0; x < V; ++x) total += r[x];
        const double target = u_bonus[off + u] * total;
        double cum = 0.0;
        int64_t pick = -1;
        for (int64_t x = 0; x < V; ++x) {
            if (r[x] <= 0.0) continue;
            cum += r[x];
            if (cum > target) {
                pick = x;
                break;
            }
        }
        if (pick < 0) { /* rounding left target at the very top: the last bin */
            for (int64_t x = V - 1; x >= 0; --x)
                if (r[x] > 0.0) { pick = x; break; }
        }
        accept_len[b] = d;
        bonus[b] = (int32_t)pick;
        if (min_margin) min_margin[b] = margin;
        if (final_r)
            for (int64_t x = 0; x < V; ++x) final_r[(int64_t)b * V + x] = r[x] / total;
        if (final_u) final_u[b] = u_bonus[off + u];
    }
    free(r);
    free(q);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Tree build with entropy-mixed scoring.                                    */
/* [JS-art] section 五 also reports scoring variants: the information        */
/* entropy at each position, and a weighted mix of the cumulative            */
/* probability and the entropy.  Reading: each step from depth d to d+1 adds */
/* (1 - alpha) * lp_d(token) - alpha * H_d, with H_d the entropy (natural    */
/* log) of draft row d and alpha in [0, 1]; alpha = 0 is the plain build    */
/* and alpha = 1 the pure entropy score.  A candidate of probability 0       */
/* (lp = -inf) keeps the score -inf under every weight.  Every step still    */
/* adds a value <= 0; the best-first queue (with its tie-breaks) is the      */
/* plain build's, fed the mixed table.                                       */
/* ------------------------------------------------------------------------ */
int jto_tree_build_mixed(const float* draft_logits, const int32_t* root_token, const int32_t* tree_off,
                         int nseq, int N, int W, int64_t V, double alpha,
                         int32_t* parent, int32_t* token, int32_t* depth, uint32_t* anc,
                         double* score, double* gap, double* entropy_out)
{
    if (!draft_logits || nseq < 0 || N < 0 || W < 1 || V < W || !(alpha >= 0.0) || !(alpha <= 1.0))
        return JTO_ERR_INVALID;
    int64_t rows = (int64_t)nseq * N;
    int32_t* tk = (int32_t*)malloc(sizeof(int32_t) * (size_t)(rows * W + 1));
    double* l = (double*)malloc(sizeof(double) * (size_t)(rows * W + 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(rows + 1));
    int rc = (tk && l && s) ? JTO_OK : JTO_ERR_INVALID;
    if (rc == JTO_OK) rc = jto_topw_lse(draft_logits, rows, V, W, tk, l, s);
    if (rc == JTO_OK) {
        for (int64_t r = 0; r < rows; ++r) {
            /* H = -sum p log p = lse - sum p z, p = exp(z - lse), sum in order;
               a masked entry (z = -inf, p = 0) adds nothing (0 log 0 = 0) */
            const float* row = draft_logits + r * V;
            double pz = 0.0;
            for (int64_t v = 0; v < V; ++v)
                if (row[v] != -INFINITY) pz += exp((double)row[v] - s[r]) * (double)row[v];
            const double H = s[r] - pz;
            if (entropy_out) entropy_out[r] = H;
            for (int k = 0; k < W; ++k) {
                if (l[r * W + k] == -INFINITY) continue; /* probability 0 stays -inf */
                const double a = (1.0 - alpha) * l[r * W + k];
                const double b = alpha * H;
                l[r * W + k] = a - b;
            }
        }
        rc = jto_tree_expand(tk, l, root_token, tree_off, nseq, N, W, parent, token, depth, anc,
                             score, gap);
    }
    free(tk);
    free(l);
    free(s);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Adaptive per-request tree policy.                                         */
/* [AS] section "逐步树策略：动态调整草稿树规模": two signals, the draft's      */
/* top-1 confidence and the rolling acceptance history, set the depth, width */
/* and node count of every request's tree; the tree grows when recent        */
/* acceptance is high and the draft confident, and shrinks in the opposite   */
/* case.  [JS-art] section 七: large budgets stop paying as the batch grows, */
/* and budgets that follow the load are named as future work.               */
/* Reading (the pages give no formula), per request b and step:              */
/*   ema   <- (1 - beta) * ema + beta * accept_len[b]   (when observed, >= 0) */
/*   conf  =  lp[b, 0, 0] >= log_conf    (log top-1 draft prob., depth 1)    */
/*   hot   =  ema >= acc_thresh                                              */
/*   ceil  =  b_max, or min(b_max, max(b_min, node_cap / nseq)) if node_cap  */
/*   B     <- clamp(B, b_min, ceil); then 2B (<= ceil) if conf and hot,      */
/*            B/2 (>= b_min) if neither, unchanged otherwise                 */
/*   n_cap =  clamp(floor(ema) + n_slack, n_min, N), 0 <= n_slack <= N       */
/*   w_cap =  conf ? W : w_min                                               */
/*   emitted budget = min(B, nodes of the full w_cap-ary tree of depth n_cap) */
/*   tree_off = exclusive prefix sum of the emitted budgets                  */
/* Depth, width and node count each move with the signals (none shrinks    */
/* when a signal rises), so the emitted budget is monotone in both.          */
/* budget_state keeps the controller's B (not the emitted one).             */
/* ------------------------------------------------------------------------ */
int jto_tree_policy(const double* lp, int nseq, int N, int W, const int32_t* accept_len,
                    int b_min, int b_max, int node_cap, int w_min, int n_min, int n_slack,
                    double beta, double log_conf, double acc_thresh,
                    int32_t* budget_state, double* acc_ema,
                    int32_t* tree_off, int32_t* w_cap, int32_t* n_cap)
{
    if (!lp || !budget_state || !acc_ema || !tree_off || !w_cap || !n_cap || nseq < 1 || N < 1 ||
        W < 1 || b_min < 1 || b_max < b_min || b_max > JTO_MAX_TREE || node_cap < 0 || w_min < 1 ||
        w_min > W || n_min < 0 || n_min > N || n_slack < 0 || n_slack > N || !(beta > 0.0) ||
        !(beta <= 1.0) ||
        log_conf != log_conf || !(acc_thresh == acc_thresh))
        return JTO_ERR_INVALID;
    for (int b = 0; b < nseq; ++b) {
        const int acc = accept_len ? accept_len[b] : -1;
        if (acc < -1 || acc > N || !(acc_ema[b] >= 0.0) || acc_ema[b] == INFINITY)
            return JTO_ERR_INVALID;
    }
    int ceil_b = b_max;
    if (node_cap > 0) {
        int per = node_cap / nseq;
        if (per < b_min) per = b_min;
        if (per < ceil_b) ceil_b = per;
    }
    tree_off[0] = 0;
    for (int b = 0; b < nseq; ++b) {
        double ema = acc_ema[b];
        const int acc = accept_len ? accept_len[b] : -1;
        if (acc >= 0) {
            const double x = (1.0 - beta) * ema;
            const double y = beta * (double)acc;
            ema = x + y;
        }
        const int conf = lp[(int64_t)b * N * W] >= log_conf;
        const int hot = ema >= acc_thresh;
        int B = budget_state[b];
        if (B < b_min) B = b_min;
        if (B > ceil_b) B = ceil_b;
        if (conf && hot) {
            B = 2 * B;
            if (B > ceil_b) B = ceil_b;
        } else if (!conf && !hot) {
            B = B / 2;
            if (B < b_min) B = b_min;
        }
        int nc;
        if (floor(ema) >= (double)N) {
            nc = N;
        } else {
            nc = (int)floor(ema) + n_slack;
            if (nc > N) nc = N;
        }
        if (nc < n_min) nc = n_min;
        const int wc = conf ? W : w_min;
        int64_t full = full_tree_nodes(nc, wc, JTO_MAX_TREE + 1);
        const int emit = (int64_t)B < full ? B : (int)full;
        budget_state[b] = B;
        acc_ema[b] = ema;
        w_cap[b] = wc;
        n_cap[b] = nc;
        tree_off[b + 1] = tree_off[b] + emit;
    }
    return JTO_OK;
}
