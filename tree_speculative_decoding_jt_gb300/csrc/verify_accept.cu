// verify_accept.cu -- tree acceptance on CUDA cores.
//
// Follows "加速AI思考…推测解码新方法" section 三 and the JetSpec news summary
// (after one verification forward over the whole tree, keep the longest
// prefix the target agrees with, along the best path) and AdaptiveSpec's
// "逐步Margin规则" (accept a drafted token when p(draft)/p(top1) >= t).
//
// One thread-block cluster per sequence walks its tree level by level.  At
// level d the frontier is the set of reached nodes of depth d (one node under
// the greedy rule).  Phase 1: every warp of the cluster streams 2048-entry
// chunks of the frontier rows (coalesced 16-byte loads) and folds a packed
// 64-bit key (order-preserving value, inverted id) into its CTA's slot for
// the row with a shared-memory atomicMax; the word holds the row maximum and
// its lowest-id argmax.  Phase 2: rank 0 combines the ranks' words through
// distributed shared memory, tests every child of the frontier against the
// row keys (one thread per child) and compacts the accepted ones, in node
// order, into the next frontier.  Hardware cluster
// barriers separate the phases.  Only rows of reached nodes are read:
// (accepted length + 1) rows per sequence under the greedy rule.
#include <cooperative_groups.h>

#include "jt_common.cuh"
#include "jt_internal.h"

namespace cg = cooperative_groups;

namespace jt {

constexpr int kAccThreads = 256;
constexpr int kAccChunk = 2048;  // entries per warp work item (one load round per level)

size_t accept_workspace_bytes(int /*nseq*/, int /*total_nodes*/) { return kWsHeader; }

__device__ __forceinline__ unsigned long long pack_argmax_key(float v, long long id) {
    return (static_cast<unsigned long long>(float_order_key(v)) << 32) |
           static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}

template <bool VEC>
__global__ void __launch_bounds__(kAccThreads)
    accept_cluster_kernel(const float* __restrict__ z, const int32_t* __restrict__ parent,
                          const int32_t* __restrict__ token, const int32_t* __restrict__ tree_off,
                          int total_nodes, int N, long long V, int rule, double log_t,
                          int32_t* __restrict__ accept_len, int32_t* __restrict__ path,
                          int32_t* __restrict__ bonus, uint32_t* err) {
    __shared__ unsigned long long s_part[JT_MAX_TREE];    // this CTA's key per frontier slot
    __shared__ unsigned long long s_rowkey[JT_MAX_TREE];  // rank 0: combined key per slot
    __shared__ int s_front[2][JT_MAX_TREE];               // frontier lists (node ids, ascending)
    __shared__ int s_slot[JT_MAX_TREE];                   // rank 0: node -> frontier slot
    __shared__ int s_par[JT_MAX_TREE], s_tok[JT_MAX_TREE];
    __shared__ int s_wcnt[kAccThreads / 32];
    __shared__ int s_n[2];
    __shared__ int s_done, s_final;
    __shared__ unsigned long long s_finalkey;

    cg::cluster_group cl = cg::this_cluster();
    const unsigned rank = cl.block_rank(), csize = cl.num_blocks();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / csize;
    const int off = tree_off[b];
    const int B = tree_off[b + 1] - off;
    if (B < 1 || B > JT_MAX_TREE || off < 0 || off + B > total_nodes) {
        if (rank == 0 && tid == 0) raise_error(err, DEVERR_INVALID);
        return;  // the whole cluster leaves before any cluster barrier
    }
    // rank 0 fetches the tree now; the loads land while phase 1 streams rows
    int my_par = -1, my_tok = 0;
    if (rank == 0 && tid < B) {
        my_par = parent[off + tid];
        my_tok = token[off + tid];
    }
    if (tid == 0) {
        s_front[0][0] = 0;
        s_n[0] = 1;
        s_done = 0;
        s_final = 0;
    }
    for (int i = tid; i < JT_MAX_TREE; i += kAccThreads) {
        s_part[i] = 0ull;
        s_rowkey[i] = 0ull;
    }
    cl.sync();
    int* fr0 = cl.map_shared_rank(&s_front[0][0], 0);
    int* n0 = cl.map_shared_rank(s_n, 0);
    int* done0 = cl.map_shared_rank(&s_done, 0);

    const long long C = (V + kAccChunk - 1) / kAccChunk;
    const int gw = static_cast<int>(rank) * (kAccThreads / 32) + warp;
    const int nw = static_cast<int>(csize) * (kAccThreads / 32);
    bool finished = false;
    for (int lvl = 0; lvl <= N; ++lvl) {
        const int cur = lvl & 1, nxt = cur ^ 1;
        const int n = s_n[cur];
        // ---- phase 1: row keys of the frontier
        for (long long it = gw; it < n * C; it += nw) {
            const int i = static_cast<int>(it / C);
            const long long c = it - static_cast<long long>(i) * C;
            const float* zr = z + static_cast<long long>(off + s_front[cur][i]) * V;
            const long long begin = c * kAccChunk, end = min(V, begin + kAccChunk);
            unsigned long long best = 0ull;
            if (VEC) {
                float4 f[kAccChunk / 128];
#pragma unroll
                for (int q = 0; q < kAccChunk / 128; ++q) {
                    const long long e = begin + 4ll * (lane + 32 * q);
                    f[q] = (e < end) ? __ldg(reinterpret_cast<const float4*>(zr + e))
                                     : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                }
#pragma unroll
                for (int q = 0; q < kAccChunk / 128; ++q) {
                    const long long e = begin + 4ll * (lane + 32 * q);
                    if (e < end) {
                        JT_DCHECK(f[q].x == f[q].x && f[q].y == f[q].y && f[q].z == f[q].z && f[q].w == f[q].w,
                                  err);
                        best = max(best, pack_argmax_key(f[q].x, e));
                        best = max(best, pack_argmax_key(f[q].y, e + 1));
                        best = max(best, pack_argmax_key(f[q].z, e + 2));
                        best = max(best, pack_argmax_key(f[q].w, e + 3));
                    }
                }
            } else {
                for (long long e = begin + lane; e < end; e += 32) {
                    const float v = __ldg(zr + e);
                    JT_DCHECK(v == v, err);  // a NaN logit has no place in the argmax order
                    best = max(best, pack_argmax_key(v, e));
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
            if (lane == 0) atomicMax(&s_part[i], best);
        }
        if (lvl == 0 && rank == 0) {
            s_par[tid] = my_par;
            s_tok[tid] = my_tok;
            JT_DCHECK(tid != 0 || my_par == -1, err);  // node 0 is the root
        }
        cl.sync();
        // ---- phase 2 (rank 0): combine the ranks' keys, test the children
        if (rank == 0) {
            for (int q = tid; q < n * static_cast<int>(csize); q += kAccThreads) {
                const int i = q / static_cast<int>(csize);
                const unsigned r = static_cast<unsigned>(q) % csize;
                atomicMax(&s_rowkey[i], cl.map_shared_rank(s_part, r)[i]);
            }
            s_slot[tid] = -1;
            __syncthreads();
            if (tid < n) s_slot[s_front[cur][tid]] = tid;
            __syncthreads();
            const int c = tid;  // one thread per child
            bool acc = false;
            if (c >= 1 && c < B) {
                const int p = s_par[c];
                const int tk = s_tok[c];
                if (p < 0 || p >= c || tk < 0 || tk >= V) {
                    raise_error(err, DEVERR_INVALID);
                } else if (s_slot[p] >= 0) {
                    const unsigned long long key = s_rowkey[s_slot[p]];
                    if (rule == JT_RULE_GREEDY) {
                        acc = static_cast<uint32_t>(tk) == 0xFFFFFFFFu - static_cast<uint32_t>(key);
                    } else {
                        const float zmax = float_from_order_key(static_cast<uint32_t>(key >> 32));
                        const float zt = z[static_cast<long long>(off + p) * V + tk];
                        acc = (static_cast<double>(zt) - static_cast<double>(zmax)) >= log_t;
                    }
                }
            }
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, acc);
            if (lane == 0) s_wcnt[warp] = __popc(bal);
            __syncthreads();
            int wbase = 0, cnt = 0;
#pragma unroll
            for (int w = 0; w < kAccThreads / 32; ++w) {
                wbase += (w < warp) ? s_wcnt[w] : 0;
                cnt += s_wcnt[w];
            }
            if (acc) s_front[nxt][wbase + __popc(bal & ((1u << lane) - 1u))] = c;
            if (rule == JT_RULE_GREEDY && cnt > 1) cnt = 1;  // first accepted child in node order
            if (tid == 0) {
                if (cnt == 0) {  // frontier lists are ascending: slot 0 is the lowest node
                    s_final = s_front[cur][0];
                    s_finalkey = s_rowkey[0];
                    s_done = 1;
                }
                s_n[nxt] = cnt;
            }
            __syncthreads();
            for (int i = tid; i < n; i += kAccThreads) s_rowkey[i] = 0ull;  // next level's slots
        }
        cl.sync();
        for (int i = tid; i < JT_MAX_TREE; i += kAccThreads) s_part[i] = 0ull;  // next level's slots
        if (*done0) {
            finished = true;
            break;
        }
        const int nn = n0[nxt];
        if (rank != 0)
            for (int i = tid; i < nn; i += kAccThreads) s_front[nxt][i] = fr0[nxt * JT_MAX_TREE + i];
        if (tid == 0) s_n[nxt] = nn;
        __syncthreads();
    }

    // epilogue: path, accepted length, bonus token
    if (rank == 0 && warp == 0) {
        if (!finished) {  // tree deeper than N
            if (lane == 0) raise_error(err, DEVERR_INVALID);
        } else {
            const int f = s_final;
            int d = 0;  // the chain root..f was validated edge by edge when it was accepted
            for (int u = f; d <= N && s_par[u] >= 0; u = s_par[u]) ++d;
            int32_t* pb = path + static_cast<long long>(b) * (N + 1);
            for (int k = lane; k <= N; k += 32) pb[k] = -1;
            __syncwarp();
            if (lane == 0 && d <= N) {
                int k = d;
                for (int u = f; u >= 0 && k >= 0; u = s_par[u]) pb[k--] = u;
                accept_len[b] = d;
                bonus[b] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(s_finalkey));
            } else if (lane == 0) {
                raise_error(err, DEVERR_INVALID);
            }
        }
    }
    cl.sync();  // rank 0's shared memory stays alive until every rank is done with it
}

// Largest cluster size (16, 8, 4, 2, 1) the current device can schedule for
// this kernel (asked once per device).
template <bool VEC>
static int accept_cluster_size_uncached() {
    cudaFuncSetAttribute(accept_cluster_kernel<VEC>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    for (int cs = 16; cs >= 1; cs >>= 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3(kAccThreads);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = cs;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, accept_cluster_kernel<VEC>, &cfg) == cudaSuccess &&
            nclusters > 0)
            return cs;
        cudaGetLastError();
    }
    return 1;
}

template <bool VEC>
static int accept_cluster_size() {
    static PerDeviceCache cache;
    return cache.get(accept_cluster_size_uncached<VEC>);
}

template <bool VEC>
static cudaError_t launch_accept(const float* z, const int32_t* parent, const int32_t* token,
                                 const int32_t* tree_off, int nseq, int N, long long V,
                                 int total_nodes, int rule, double log_t, int32_t* accept_len,
                                 int32_t* path, int32_t* bonus, uint32_t* err, cudaStream_t st) {
    const int cs = accept_cluster_size<VEC>();
    return launch_kernel(accept_cluster_kernel<VEC>, dim3(static_cast<unsigned>(nseq) * cs), dim3(kAccThreads),
                      0, st, static_cast<unsigned>(cs), z, parent, token, tree_off, total_nodes, N, V, rule,
                      log_t, accept_len, path, bonus, err);
}

cudaError_t verify_accept_launch(const float* z, const int32_t* parent, const int32_t* token,
                                 const int32_t* tree_off, int nseq, int N, long long V,
                                 int total_nodes, int rule, double log_t, int32_t* accept_len,
                                 int32_t* path, int32_t* bonus, char* ws, cudaStream_t st) {
    uint32_t* err = reinterpret_cast<uint32_t*>(ws);
    const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
    if (vec)
        return launch_accept<true>(z, parent, token, tree_off, nseq, N, V, total_nodes, rule, log_t,
                                   accept_len, path, bonus, err, st);
    return launch_accept<false>(z, parent, token, tree_off, nseq, N, V, total_nodes, rule, log_t,
                                accept_len, path, bonus, err, st);
}

}  // namespace jt
