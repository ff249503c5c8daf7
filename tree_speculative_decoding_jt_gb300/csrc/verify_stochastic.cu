// verify_stochastic.cu -- temperature-1 tree acceptance by rejection
// sampling against a running residual.
//
// Rule (speculative-decoding overview, chooseai.io/news/6515, section
// "推测解码是什么：草稿模型先猜，目标模型验收"; AdaptiveSpec, section
// "严格的token匹配验证机制"): a drafted token x is accepted with probability
// min(1, p(x)/q(x)); after a rejection the next token comes from
// norm(max(0, p - q)).  On the tree: at the current node the children are
// tried in node order against the residual r (r = p at first); after each
// rejection r <- norm(max(0, r - q)); an accepted child becomes the current
// node; when no child is accepted (or there is none) the bonus token is the
// inverse-CDF draw from r.  p = softmax of the node's target row, q = softmax
// of the draft row of the children's depth, both at temperature 1.  The
// caller supplies the uniforms (one per node for its acceptance test, one per
// node for a bonus draw there).
//
// One thread-block cluster per sequence; the vocabulary is split into one
// contiguous chunk per CTA, held in shared memory as r and q (fp32).  Every
// CTA takes every decision itself from values exchanged through distributed
// shared memory (per-CTA (max, sum) pairs, per-CTA residual sums and the two
// entries r(t), q(t) of a tested token), combined in the same order on every
// CTA, so all CTAs agree without a broadcast.  Hardware cluster barriers
// separate the exchanges; all CTAs execute exactly the same barrier
// sequence (their control flow depends only on exchanged, identical values).
#include <cooperative_groups.h>

#include "jt_common.cuh"
#include "jt_internal.h"

namespace cg = cooperative_groups;

namespace jt {

constexpr int kStThreads = 256;
constexpr int kStWarps = kStThreads / 32;

struct StSlot {   // one exchange: per-CTA values read by every CTA
    float m_p, s_p, m_q, s_q;  // max and sum of exp(x - max) of the target / draft chunk
    float rsum;                // sum of the current residual over the chunk
};

struct StShared {
    StSlot slot[2];            // double-buffered by exchange parity
    float red_m[kStWarps], red_s[kStWarps], red_m2[kStWarps], red_s2[kStWarps];  // block reductions
    float scan[kStThreads];
    int par[JT_MAX_TREE], tok[JT_MAX_TREE];
};

// Block-wide max of two values; results valid in every thread.
__device__ __forceinline__ void block_max2(float& a, float& b, StShared& sh) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
        b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, o));
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sh.red_m[warp] = a;
        sh.red_m2[warp] = b;
    }
    __syncthreads();
    a = b = -INFINITY;
    for (int w = 0; w < kStWarps; ++w) {
        a = fmaxf(a, sh.red_m[w]);
        b = fmaxf(b, sh.red_m2[w]);
    }
    __syncthreads();
}

// Block-wide sum of two values (fixed order); results valid in every thread.
__device__ __forceinline__ void block_sum2(float& a, float& b, StShared& sh) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        b += __shfl_xor_sync(0xFFFFFFFFu, b, o);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sh.red_s[warp] = a;
        sh.red_s2[warp] = b;
    }
    __syncthreads();
    a = b = 0.0f;
    for (int w = 0; w < kStWarps; ++w) {
        a += sh.red_s[w];
        b += sh.red_s2[w];
    }
    __syncthreads();
}

__device__ __forceinline__ float block_sum(float v, StShared& sh) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sh.red_s[warp] = v;
    __syncthreads();
    float t = 0.0f;
    for (int w = 0; w < kStWarps; ++w) t += sh.red_s[w];
    __syncthreads();
    return t;
}

__global__ void __launch_bounds__(kStThreads)
    accept_stochastic_kernel(const float* __restrict__ z, const float* __restrict__ zd,
                             const int32_t* __restrict__ parent, const int32_t* __restrict__ token,
                             const int32_t* __restrict__ tree_off, int total_nodes, int N, long long V,
                             int chunk, const double* __restrict__ u_accept,
                             const double* __restrict__ u_bonus, int32_t* __restrict__ accept_len,
                             int32_t* __restrict__ path, int32_t* __restrict__ bonus, uint32_t* err) {
    extern __shared__ __align__(16) unsigned char st_dyn[];
    float* r = reinterpret_cast<float*>(st_dyn);  // [chunk] residual, r / Z is the distribution
    float* q = r + chunk;                         // [chunk] exp(draft - max), q / Sq is the distribution
    __shared__ StShared sh;

    cg::cluster_group cl = cg::this_cluster();
    const unsigned rank = cl.block_rank(), cs = cl.num_blocks();
    const int tid = threadIdx.x;
    const int b = blockIdx.x / cs;
    const int off = tree_off[b];
    const int B = tree_off[b + 1] - off;
    bool bad = B < 1 || B > JT_MAX_TREE || off < 0 || off + B > total_nodes;
    if (!bad) {
        for (int i = tid; i < B; i += kStThreads) {
            const int pa = parent[off + i], tk = token[off + i];
            sh.par[i] = pa;
            sh.tok[i] = tk;
            if ((i == 0 && pa != -1) || (i > 0 && (pa < 0 || pa >= i || tk < 0 || tk >= V))) bad = true;
        }
    }
    if (__syncthreads_or(bad)) {  // identical on every CTA of the cluster: all leave together
        if (rank == 0 && tid == 0) raise_error(err, DEVERR_INVALID);
        return;
    }
    const long long x0 = static_cast<long long>(rank) * chunk;
    const int n_loc = static_cast<int>(max(0ll, min(static_cast<long long>(chunk), V - x0)));

    int u = 0, d = 0, ex = 0;  // current node, its depth, exchange parity
    int32_t* pb = path + static_cast<long long>(b) * (N + 1);
    if (rank == 0)
        for (int k = tid; k <= N; k += kStThreads) pb[k] = (k == 0) ? 0 : -1;
    for (;;) {
        int first_child = -1;
        if (d < N)
            for (int c = u + 1; c < B; ++c)
                if (sh.par[c] == u) {
                    first_child = c;
                    break;
                }
        const bool has_children = first_child >= 0;
        // ---- target row of u and draft row of depth d: max pass, then one
        // exp per entry; r holds exp(z - max) (r / Z is p), q holds
        // exp(zd - max) (q / Sq is the draft distribution)
        const float* zr = z + static_cast<long long>(off + u) * V + x0;
        const float* dr = zd + (static_cast<long long>(b) * N + d) * V + x0;
        float mp = -INFINITY, mq = -INFINITY;
        for (int i = tid; i < n_loc; i += kStThreads) {
            const float zv = zr[i];
            r[i] = zv;
            mp = fmaxf(mp, zv);
            JT_DCHECK(zv == zv, err);  // a NaN logit leaves the softmax undefined
            if (has_children) {
                const float dv = dr[i];
                q[i] = dv;
                mq = fmaxf(mq, dv);
                JT_DCHECK(dv == dv, err);
            }
        }
        block_max2(mp, mq, sh);
        if (tid == 0) sh.slot[ex].m_p = mp, sh.slot[ex].m_q = mq;
        cl.sync();
        float Mp = -INFINITY, Mq = -INFINITY;
        for (unsigned k = 0; k < cs; ++k) {
            const StSlot* o = cl.map_shared_rank(&sh.slot[ex], k);
            Mp = fmaxf(Mp, o->m_p);
            Mq = fmaxf(Mq, o->m_q);
        }
        ex ^= 1;
        float sp = 0.0f, sq = 0.0f;
        for (int i = tid; i < n_loc; i += kStThreads) {
            const float e = __expf(r[i] - Mp);
            r[i] = e;
            sp += e;
            if (has_children) {
                const float eq = __expf(q[i] - Mq);
                q[i] = eq;
                sq += eq;
            }
        }
        block_sum2(sp, sq, sh);
        if (tid == 0) sh.slot[ex].s_p = sp, sh.slot[ex].s_q = sq;
        cl.sync();  // r and q of every chunk are final for the tests below
        float Sp = 0.0f, Sq = 0.0f;
        for (unsigned k = 0; k < cs; ++k) {  // same order on every CTA
            const StSlot* o = cl.map_shared_rank(&sh.slot[ex], k);
            Sp += o->s_p;
            Sq += o->s_q;
        }
        ex ^= 1;
        const float inv_q = has_children ? 1.0f / Sq : 0.0f;
        // ---- children in node order
        float Z = Sp;  // r / Z is the current residual distribution
        int next = -1;
        for (int c = first_child; has_children && c < B && next < 0; ++c) {
            if (sh.par[c] != u) continue;
            const int t = sh.tok[c];
            const unsigned owner = static_cast<unsigned>(t / chunk);
            const int lt = t - static_cast<int>(owner) * chunk;
            const float rt = cl.map_shared_rank(r, owner)[lt] / Z;
            const float qt = cl.map_shared_rank(q, owner)[lt] * inv_q;
            const float ratio = (qt > 0.0f) ? rt / qt : INFINITY;
            const double a = ratio < 1.0f ? static_cast<double>(ratio) : 1.0;
            if (u_accept[off + c] < a) {
                next = c;
                break;
            }
            // rejected: r <- max(0, r/Z - q); new Z = sum r over the cluster
            cl.sync();  // every CTA has read r(t) before any chunk changes
            const float invZ = 1.0f / Z;
            float ls = 0.0f;
            for (int i = tid; i < n_loc; i += kStThreads) {
                const float v = fmaxf(r[i] * invZ - q[i] * inv_q, 0.0f);
                r[i] = v;
                ls += v;
            }
            ls = block_sum(ls, sh);
            if (tid == 0) sh.slot[ex].rsum = ls;
            cl.sync();
            float zs = 0.0f;
            for (unsigned k = 0; k < cs; ++k) zs += cl.map_shared_rank(&sh.slot[ex], k)->rsum;
            ex ^= 1;
            Z = zs;
        }
        if (next >= 0) {
            cl.sync();  // the next level rewrites r and q
            u = next;
            ++d;
            if (rank == 0 && tid == 0) pb[d] = u;
            continue;
        }
        // ---- bonus: inverse CDF of r over the vocabulary order
        // per-thread contiguous ranges of the chunk, block scan, CTA prefix
        const int per = (n_loc + kStThreads - 1) / kStThreads;
        const int i0 = tid * per, i1 = min(n_loc, i0 + per);
        float ts = 0.0f;
        for (int i = i0; i < i1; ++i) ts += r[i];
        sh.scan[tid] = ts;
        const float cta_sum = block_sum(ts, sh);
        if (tid == 0) sh.slot[ex].rsum = cta_sum;
        cl.sync();
        float before = 0.0f, total = 0.0f;
        for (unsigned k = 0; k < cs; ++k) {
            const float v = cl.map_shared_rank(&sh.slot[ex], k)->rsum;
            if (k < rank) before += v;
            total += v;
        }
        const float target = static_cast<float>(u_bonus[off + u] * static_cast<double>(total));
        // this CTA owns the draw when before <= target < before + cta_sum; the
        // last CTA with mass also takes a target past the total (rounding)
        if (tid == 0) {
            float acc = before;
            int pick = -1;
            for (int tt = 0; tt < kStThreads && pick < 0; ++tt) {
                const float nx = acc + sh.scan[tt];
                if (nx > target && sh.scan[tt] > 0.0f) {
                    for (int i = tt * per; i < min(n_loc, tt * per + per); ++i) {
                        if (r[i] <= 0.0f) continue;
                        acc += r[i];
                        if (acc > target) {
                            pick = i;
                            break;
                        }
                    }
                    if (pick < 0) acc = nx;
                } else {
                    acc = nx;
                }
            }
            bool take = pick >= 0 && target >= before;
            if (!take && target >= before + cta_sum && cta_sum > 0.0f) {
                // past every bin of this CTA: the draw belongs here only when
                // no later CTA has mass
                bool later = false;
                for (unsigned k = rank + 1; k < cs; ++k)
                    if (cl.map_shared_rank(&sh.slot[ex], k)->rsum > 0.0f) later = true;
                if (!later) {
                    for (int i = n_loc - 1; i >= 0; --i)
                        if (r[i] > 0.0f) {
                            pick = i;
                            break;
                        }
                    take = pick >= 0;
                }
            }
            if (take) {
                bonus[b] = static_cast<int32_t>(x0 + pick);
                accept_len[b] = d;
            }
        }
        break;
    }
    cl.sync();  // shared memory stays alive until every CTA has read it
}

// Largest cluster size (16, 8, 4, 2, 1) that fits with `smem` bytes of
// dynamic shared memory per CTA.
static int stochastic_cluster_size(long long V) {
    cudaFuncSetAttribute(accept_stochastic_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    for (int cs = 16; cs >= 1; cs >>= 1) {
        const long long chunk = (V + cs - 1) / cs;
        const size_t smem = static_cast<size_t>(chunk) * 2 * sizeof(float);
        if (smem > 200 * 1024) continue;
        if (cudaFuncSetAttribute(accept_stochastic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3(kStThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = cs;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, accept_stochastic_kernel, &cfg) == cudaSuccess && n > 0)
            return cs;
        cudaGetLastError();
    }
    return 0;
}

cudaError_t verify_stochastic_launch(const float* z, const float* zd, const int32_t* parent,
                                     const int32_t* token, const int32_t* tree_off, int nseq, int N,
                                     long long V, int total_nodes, const double* u_accept,
                                     const double* u_bonus, int32_t* accept_len, int32_t* path,
                                     int32_t* bonus, char* ws, cudaStream_t st) {
    uint32_t* err = reinterpret_cast<uint32_t*>(ws);
    static PerDeviceCache cache;  // per device and vocabulary size
    const int cs = cache.get([V] { return stochastic_cluster_size(V); }, V);
    if (cs == 0) return cudaErrorNotSupported;
    const long long chunk = (V + cs - 1) / cs;
    const size_t smem = static_cast<size_t>(chunk) * 2 * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(accept_stochastic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_kernel(accept_stochastic_kernel, dim3(static_cast<unsigned>(nseq) * cs), dim3(kStThreads), smem,
                         st, static_cast<unsigned>(cs), z, zd, parent, token, tree_off, total_nodes, N, V,
                         static_cast<int>(chunk), u_accept, u_bonus, accept_len, path, bonus, err);
}

}  // namespace jt
