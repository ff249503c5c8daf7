// verify_accept.cu -- tree acceptance on CUDA cores.
//
// Follows "加速AI思考…推测解码新方法" section 三 and the JetSpec news summary
// (after one verification forward over the whole tree, keep the longest
// prefix the target agrees with, along the best path) and AdaptiveSpec's
// "逐步Margin规则" (accept a drafted token when p(draft)/p(top1) >= t).
//
// One cooperative kernel walks all sequences level by level.  At level d
// the frontier of a sequence is the set of reached nodes of depth d (one
// node under the greedy rule).  Phase 1: every CTA streams 4096-entry chunks
// of the frontier rows (vectorised coalesced loads) and folds a packed
// (order-preserving value, inverted id) 64-bit key into the row's slot with
// atomicMax, which yields max and lowest-id argmax in one word.  Phase 2:
// one warp per sequence tests the frontier's children against those keys and
// forms the next frontier.  Only rows of reached nodes are read, so a step
// costs (accepted length + 1) rows under the greedy rule instead of B rows.
// Grid-wide barriers are bounded in time (error flag, then exit).
#include "jt_common.cuh"
#include "jt_internal.h"

namespace jt {

constexpr int kAccThreads = 256;
constexpr int kAccChunk = 4096;
constexpr int kAccMaxSeq = 8192;

struct AcceptWs {
    WsHeader* hdr;
    unsigned long long* keys;  // [total_nodes]
    int* frontier;             // [nseq][2][JT_MAX_TREE]
    int* fcount;               // [nseq][2]
    int* final_node;           // [nseq]
    int* state;                // [nseq]: 0 walking, 1 done, 2 invalid
};

size_t accept_workspace_bytes(int nseq, int total_nodes) {
    size_t b = kWsHeader;
    b += align_up(sizeof(unsigned long long) * static_cast<size_t>(total_nodes));
    b += align_up(sizeof(int) * static_cast<size_t>(nseq) * 2 * JT_MAX_TREE);
    b += align_up(sizeof(int) * static_cast<size_t>(nseq) * 2);
    b += align_up(sizeof(int) * static_cast<size_t>(nseq));
    b += align_up(sizeof(int) * static_cast<size_t>(nseq));
    return b;
}

static AcceptWs carve_accept(char* ws, int nseq, int total_nodes) {
    AcceptWs w;
    w.hdr = reinterpret_cast<WsHeader*>(ws);
    char* p = ws + kWsHeader;
    w.keys = reinterpret_cast<unsigned long long*>(p);
    p += align_up(sizeof(unsigned long long) * static_cast<size_t>(total_nodes));
    w.frontier = reinterpret_cast<int*>(p);
    p += align_up(sizeof(int) * static_cast<size_t>(nseq) * 2 * JT_MAX_TREE);
    w.fcount = reinterpret_cast<int*>(p);
    p += align_up(sizeof(int) * static_cast<size_t>(nseq) * 2);
    w.final_node = reinterpret_cast<int*>(p);
    p += align_up(sizeof(int) * static_cast<size_t>(nseq));
    w.state = reinterpret_cast<int*>(p);
    return w;
}

// Grid-wide barrier over co-resident CTAs (cooperative launch).  Returns
// false, with DEVERR_TIMEOUT raised, if the others do not arrive in time.
__device__ __forceinline__ bool grid_barrier(WsHeader* hdr, unsigned nblocks) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        volatile unsigned* gen = &hdr->bar_gen;
        const unsigned g = *gen;
        __threadfence();
        const unsigned arrived = atomicAdd(&hdr->bar_count, 1u);
        if (arrived == nblocks - 1) {
            atomicExch(&hdr->bar_count, 0u);
            __threadfence();
            atomicAdd(&hdr->bar_gen, 1u);
        } else {
            const unsigned long long t0 = globaltimer_ns();
            while (*gen == g) {
                __nanosleep(64);
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    raise_error(&hdr->err, DEVERR_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ unsigned long long pack_argmax_key(float v, long long id) {
    return (static_cast<unsigned long long>(float_order_key(v)) << 32) |
           static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}

template <bool VEC>
__global__ void __launch_bounds__(kAccThreads)
    accept_kernel(const float* __restrict__ z, const int32_t* __restrict__ parent,
                  const int32_t* __restrict__ token, const int32_t* __restrict__ tree_off,
                  int nseq, int total_nodes, int N, long long V, int rule, double log_t,
                  int32_t* __restrict__ accept_len, int32_t* __restrict__ path,
                  int32_t* __restrict__ bonus, AcceptWs w) {
    extern __shared__ int s_prefix[];  // [nseq + 1]
    __shared__ unsigned long long s_red[kAccThreads / 32];
    __shared__ uint32_t s_mask[kAccThreads / 32][8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned nblocks = gridDim.x;
    const int gwarp = blockIdx.x * (kAccThreads / 32) + warp;
    const int nwarps = gridDim.x * (kAccThreads / 32);
    const long long C = (V + kAccChunk - 1) / kAccChunk;

    // prologue: root of every sequence is the level-0 frontier
    for (int b = blockIdx.x * kAccThreads + tid; b < nseq; b += gridDim.x * kAccThreads) {
        const int B = tree_off[b + 1] - tree_off[b];
        const bool ok = (B >= 1 && B <= JT_MAX_TREE && tree_off[b] >= 0 &&
                         tree_off[b + 1] <= total_nodes);
        if (!ok) raise_error(&w.hdr->err, DEVERR_INVALID);
        w.state[b] = ok ? 0 : 2;
        w.frontier[(b * 2 + 0) * JT_MAX_TREE] = 0;
        w.fcount[b * 2 + 0] = ok ? 1 : 0;
        w.fcount[b * 2 + 1] = 0;
        w.final_node[b] = 0;
        if (ok) w.keys[tree_off[b]] = 0ull;
    }
    if (!grid_barrier(w.hdr, nblocks)) return;

    for (int lvl = 0; lvl <= N; ++lvl) {
        const int cur = lvl & 1, nxt = cur ^ 1;

        // ---- phase 1: packed max/argmax keys of the frontier rows
        if (warp == 0) {
            // exclusive prefix of frontier sizes over the sequences still
            // walking (finished or invalid ones contribute nothing)
            const int per = (nseq + 31) / 32;
            const int lo = lane * per, hi = min(nseq, lo + per);
            int sum = 0;
            for (int b = lo; b < hi; ++b)
                sum += (w.state[b] == 0) ? min(w.fcount[b * 2 + cur], JT_MAX_TREE) : 0;
            int incl = sum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
                if (lane >= off) incl += t;
            }
            int run = incl - sum;
            for (int b = lo; b < hi; ++b) {
                s_prefix[b] = run;
                run += (w.state[b] == 0) ? min(w.fcount[b * 2 + cur], JT_MAX_TREE) : 0;
            }
            if (lane == 31) s_prefix[nseq] = incl;
        }
        __syncthreads();
        const long long total_rows = s_prefix[nseq];
        for (long long it = blockIdx.x; it < total_rows * C; it += gridDim.x) {
            const long long r = it / C;
            const long long c = it - r * C;
            int lo = 0, hi = nseq;  // last b with s_prefix[b] <= r
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_prefix[mid] <= r) lo = mid; else hi = mid;
            }
            const int b = lo;
            const int u = w.frontier[(b * 2 + cur) * JT_MAX_TREE + (r - s_prefix[b])];
            const long long grow = tree_off[b] + u;
            const float* zr = z + grow * V;
            const long long begin = c * kAccChunk, end = min(V, begin + kAccChunk);
            unsigned long long best = 0ull;
            if (VEC) {
#pragma unroll
                for (int i = 0; i < kAccChunk / (4 * kAccThreads); ++i) {
                    const long long e = begin + 4ll * (tid + kAccThreads * i);
                    if (e < end) {
                        const float4 f = __ldg(reinterpret_cast<const float4*>(zr + e));
                        best = max(best, pack_argmax_key(f.x, e));
                        best = max(best, pack_argmax_key(f.y, e + 1));
                        best = max(best, pack_argmax_key(f.z, e + 2));
                        best = max(best, pack_argmax_key(f.w, e + 3));
                    }
                }
            } else {
                for (long long e = begin + tid; e < end; e += kAccThreads)
                    best = max(best, pack_argmax_key(__ldg(zr + e), e));
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, off));
            if (lane == 0) s_red[warp] = best;
            __syncthreads();
            if (tid == 0) {
                for (int i = 1; i < kAccThreads / 32; ++i) best = max(best, s_red[i]);
                atomicMax(&w.keys[grow], best);
            }
            __syncthreads();
        }
        if (!grid_barrier(w.hdr, nblocks)) return;
        // The counter of the next level was last read before the barrier
        // just passed and is next incremented after the following one.
        if (blockIdx.x == 0 && tid == 0) w.hdr->active[nxt] = 0u;

        // ---- phase 2: one warp per sequence tests the frontier's children
        for (int b = gwarp; b < nseq; b += nwarps) {
            if (w.state[b] != 0) continue;
            const int off = tree_off[b];
            const int B = tree_off[b + 1] - off;
            const int ncur = w.fcount[b * 2 + cur];
            const int* fl = w.frontier + (b * 2 + cur) * JT_MAX_TREE;
            if (lane < 8) s_mask[warp][lane] = 0u;
            __syncwarp();
            int fmin = JT_MAX_TREE;
            for (int i = lane; i < ncur; i += 32) {
                const int u = fl[i];
                atomicOr(&s_mask[warp][u >> 5], 1u << (u & 31));
                fmin = min(fmin, u);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) fmin = min(fmin, __shfl_xor_sync(0xFFFFFFFFu, fmin, o));
            __syncwarp();
            int* nl = w.frontier + (b * 2 + nxt) * JT_MAX_TREE;
            int cnt = 0;
            for (int c0 = 1; c0 < B; c0 += 32) {
                const int c = c0 + lane;
                bool acc = false;
                if (c < B) {
                    const int p = parent[off + c];
                    const int tk = token[off + c];
                    if (p < 0 || p >= c || tk < 0 || tk >= V) {
                        raise_error(&w.hdr->err, DEVERR_INVALID);
                    } else if ((s_mask[warp][p >> 5] >> (p & 31)) & 1u) {
                        const unsigned long long key = w.keys[off + p];
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
                if (acc) {
                    const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
                    nl[pos] = c;
                    w.keys[off + c] = 0ull;
                }
                cnt += __popc(bal);
            }
            if (rule == JT_RULE_GREEDY && cnt > 1) cnt = 1;  // first accepted child in node order
            if (lane == 0) {
                if (cnt == 0) {
                    w.final_node[b] = fmin;
                    w.state[b] = 1;
                    w.fcount[b * 2 + nxt] = 0;
                } else {
                    w.fcount[b * 2 + nxt] = cnt;
                    atomicAdd(&w.hdr->active[cur], 1u);
                }
            }
        }
        if (!grid_barrier(w.hdr, nblocks)) return;
        if (*reinterpret_cast<volatile unsigned*>(&w.hdr->active[cur]) == 0u) break;
    }

    // epilogue: path, accepted length, bonus token
    for (int b = gwarp; b < nseq; b += nwarps) {
        const int st = w.state[b];
        if (st == 2) continue;
        if (st != 1) {  // deeper than N
            if (lane == 0) raise_error(&w.hdr->err, DEVERR_INVALID);
            continue;
        }
        const int off = tree_off[b];
        const int f = w.final_node[b];
        int d = 0;  // the chain root..f was validated edge by edge when it was accepted
        for (int u = f; d <= N && parent[off + u] >= 0; u = parent[off + u]) ++d;
        if (d > N) {
            if (lane == 0) raise_error(&w.hdr->err, DEVERR_INVALID);
            continue;
        }
        int32_t* pb = path + static_cast<long long>(b) * (N + 1);
        for (int k = lane; k <= N; k += 32) pb[k] = -1;
        __syncwarp();
        if (lane == 0) {
            int k = d;
            for (int u = f; u >= 0 && k >= 0; u = parent[off + u]) pb[k--] = u;
            accept_len[b] = d;
            bonus[b] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(w.keys[off + f]));
        }
    }
}

cudaError_t verify_accept_launch(const float* z, const int32_t* parent, const int32_t* token,
                                 const int32_t* tree_off, int nseq, int N, long long V,
                                 int total_nodes, int rule, double log_t, int32_t* accept_len,
                                 int32_t* path, int32_t* bonus, char* ws, cudaStream_t st) {
    if (nseq > kAccMaxSeq) return cudaErrorInvalidValue;
    AcceptWs w = carve_accept(ws, nseq, total_nodes);
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(WsHeader), st);
    if (e != cudaSuccess) return e;
    const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
    const void* fn = vec ? reinterpret_cast<const void*>(&accept_kernel<true>)
                         : reinterpret_cast<const void*>(&accept_kernel<false>);
    const size_t smem = sizeof(int) * static_cast<size_t>(nseq + 1);
    int dev = 0, occ = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kAccThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    // one CTA per 4096-entry chunk of one row per sequence (the greedy
    // frontier), at least 16, at most what is co-resident: fewer CTAs make
    // the grid barriers cheaper
    const long long chunks = static_cast<long long>(nseq) * ((V + kAccChunk - 1) / kAccChunk);
    const long long cap = static_cast<long long>(device_sm_count()) * (occ < 2 ? occ : 2);
    const int grid = static_cast<int>(chunks < 16 ? (cap < 16 ? cap : 16) : (chunks < cap ? chunks : cap));
    void* args[] = {(void*)&z,      (void*)&parent, (void*)&token, (void*)&tree_off,
                    (void*)&nseq,   (void*)&total_nodes, (void*)&N, (void*)&V, (void*)&rule,
                    (void*)&log_t,  (void*)&accept_len, (void*)&path, (void*)&bonus,
                    (void*)&w};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kAccThreads), args, smem, st);
}

}  // namespace jt
