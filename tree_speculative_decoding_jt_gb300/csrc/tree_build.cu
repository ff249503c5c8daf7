// tree_build.cu -- draft-tree construction on CUDA cores.
//
// Follows the JetSpec news summary (tree construction: one forward gives the
// logits of every depth, keep the top-W per depth, score branches by the
// cumulative draft log-probability and fill greedily up to the budget B,
// depth at most N) and "加速AI思考…推测解码新方法" section 五 (best-first
// expansion with a priority queue: pop the best node, give it up to W
// children, push them, stop at B nodes).
//
// Kernels
//   topw_partial_kernel  one CTA per (row, chunk of 256 x 16 or 32 entries):
//                        vectorised coalesced loads, per-thread top-W in
//                        registers, warp-shuffle merge; chunk max and the
//                        chunk's sum of exp(z - max) from the table-driven
//                        fp32 exp with float-float accumulation (and, for the
//                        entropy-mixed build, the sum of exp(z - max) * z).
//   topw_merge_kernel    one warp per row: merges the chunk partials into
//                        top-W ids, log-probs (or mixed step scores) and lse.
//   expand_kernel        one CTA per sequence: builds the B-1 best nodes of
//                        the (optionally width/depth-capped) full tree level
//                        by level with rank-by-binary-search merges, then
//                        derives the 256-bit ancestor sets.
//   tree_policy_kernel   one CTA: the adaptive per-request budget, width and
//                        depth caps and the tree offsets (AdaptiveSpec's
//                        per-step tree policy).
#include <float.h>

#include <algorithm>

#include "ffexp.cuh"
#include "jt_common.cuh"
#include "jt_internal.h"

namespace jt {

constexpr int kTopwThreads = 256;
constexpr int kTopwPerThread = 32;     // entries per thread with many rows
constexpr int kTopwPerThreadMin = 16;  // with few rows: more, shorter CTAs
constexpr int kExpandThreads = 1024;  // ranking uses all; set-sized steps use the first 256
constexpr unsigned kFull = 0xFFFFFFFFu;

struct ExpTable {
    float hi[64];
    float lo[64];
};

// (value desc, id asc); id -1 marks an empty entry and loses every tie.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && static_cast<unsigned>(ia) < static_cast<unsigned>(ib));
}

template <int W>
struct TopList {
    float v[W];
    int id[W];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int k = 0; k < W; ++k) {
            v[k] = -INFINITY;
            id[k] = -1;
        }
    }
    __device__ __forceinline__ void push(float x, int i) {
        if (!better(x, i, v[W - 1], id[W - 1])) return;
        bool placed = false;
#pragma unroll
        for (int k = W - 1; k >= 1; --k) {
            if (!placed) {
                if (better(x, i, v[k - 1], id[k - 1])) {
                    v[k] = v[k - 1];
                    id[k] = id[k - 1];
                } else {
                    v[k] = x;
                    id[k] = i;
                    placed = true;
                }
            }
        }
        if (!placed) {
            v[0] = x;
            id[0] = i;
        }
    }
    __device__ __forceinline__ void pop_front() {
#pragma unroll
        for (int k = 0; k < W - 1; ++k) {
            v[k] = v[k + 1];
            id[k] = id[k + 1];
        }
        v[W - 1] = -INFINITY;
        id[W - 1] = -1;
    }
};

// Merge the 32 lanes' sorted lists into the warp's top-W (result in every
// lane): W rounds of a shuffle arg-max over the lanes' heads.
template <int W>
__device__ __forceinline__ void warp_merge(TopList<W>& L, float (&rv)[W], int (&rid)[W]) {
#pragma unroll
    for (int r = 0; r < W; ++r) {
        float bv = L.v[0];
        int bi = L.id[0];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, off);
            const int oi = __shfl_xor_sync(kFull, bi, off);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        rv[r] = bv;
        rid[r] = bi;
        if (bi != -1 && L.id[0] == bi) L.pop_front();
    }
}

__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    return x;
}
__device__ __forceinline__ ffloat warp_sum_ff(ffloat x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        ffloat o;
        o.hi = __shfl_xor_sync(kFull, x.hi, off);
        o.lo = __shfl_xor_sync(kFull, x.lo, off);
        x = ff_add(x, o);
    }
    return x;
}
__device__ __forceinline__ float warp_max_f(float x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, off));
    return x;
}

// ---------------------------------------------------------------------------
// Step 1a: per-chunk top-W, max and sum of exp(z - max).
// grid = (splits, rows); chunk = kTopwThreads*kTopwPerThread entries; every
// thread holds kTopwPerThread entries in registers (ids increase with the
// slot index, out-of-range slots form a suffix).
//   top-W: each lane tracks the arg-max of its own entries (strict '>' over
//   ascending slots keeps the lowest id among equal values); W warp rounds
//   take the best lane head (value desc, id asc) and let the winning lane
//   rescan its remaining entries; warp 0 then merges the warps' lists the
//   same way.  Exact under ties, and the per-entry cost is a few compares.
//   sum: per warp, exp(z - warp max) summed in float-float from the
//   table-driven exp; warp 0 rescales the warp sums to the chunk maximum.
// ---------------------------------------------------------------------------
// Packed fp32 pairs: one instruction computes two independent lanes of
// data on sm_100 and later, each lane rounded exactly like the scalar
// operation (round to nearest, no fusion beyond what is written).
struct F2 {
    float x, y;
};
__device__ __forceinline__ F2 f2(float a, float b) { return F2{a, b}; }
__device__ __forceinline__ F2 f2(float a) { return F2{a, a}; }
#define JT_F2_OP(NAME, INSTR)                                                                                     \
    __device__ __forceinline__ F2 NAME(F2 a, F2 b) {                                                              \
        F2 d;                                                                                                     \
        asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t" INSTR             \
            " d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"                                                           \
            : "=f"(d.x), "=f"(d.y)                                                                                \
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                                            \
        return d;                                                                                                 \
    }
JT_F2_OP(add2, "add.rn.f32x2")
JT_F2_OP(sub2, "sub.rn.f32x2")
JT_F2_OP(mul2, "mul.rn.f32x2")
#undef JT_F2_OP
__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
    F2 d;
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// Error-free sum of two pairs (two_sum on each lane).
__device__ __forceinline__ void two_sum2(F2 a, F2 b, F2& s, F2& e) {
    s = add2(a, b);
    const F2 bb = sub2(s, a);
    e = add2(sub2(a, sub2(s, bb)), sub2(b, bb));
}

// ffexp_in_range (ffexp.cuh: Tang's table-driven exp with error-free
// transforms) on two entries at once: the same operations, each lane
// rounded as there, with the negated reduction constants folded into the
// multiplications (exact).
__device__ __forceinline__ void ffexp_pair(F2 xh, F2 xl, const float* tab_hi, const float* tab_lo, F2& yh,
                                           F2& yl) {
    const F2 tk = fma2(xh, f2(kExpInvL), f2(kRoundMagic));
    const F2 kf = sub2(tk, f2(kRoundMagic));
    const int k0 = static_cast<int>(__float_as_uint(tk.x)) - 0x4B400000;
    const int k1 = static_cast<int>(__float_as_uint(tk.y)) - 0x4B400000;
    const F2 r1 = fma2(kf, f2(-kExpC1), xh);  // exact
    const F2 rh = fma2(kf, f2(-kExpC2), r1);  // exact
    const F2 rl = fma2(kf, f2(-kExpC3), xl);
    const F2 rc = add2(rh, rl);
    F2 p = fma2(rc, f2(1.0f / 120.0f), f2(1.0f / 24.0f));
    p = fma2(rc, p, f2(1.0f / 6.0f));
    p = fma2(rc, p, f2(0.5f));
    p = mul2(mul2(rc, rc), p);
    const F2 q = add2(rl, p);
    const F2 th = f2(tab_hi[k0 & 63], tab_hi[k1 & 63]), tl = f2(tab_lo[k0 & 63], tab_lo[k1 & 63]);
    const F2 prod = mul2(th, rh);
    const F2 perr = fma2(th, rh, sub2(f2(0.0f), prod));
    const F2 small = fma2(th, q, add2(fma2(tl, rh, tl), perr));
    const F2 sm = add2(th, prod);  // |th| > |prod|: Fast2Sum
    const F2 e = add2(sub2(th, sm), prod);
    const F2 sc = f2(jt_pow2i(k0 >> 6), jt_pow2i(k1 >> 6));
    yh = mul2(sm, sc);
    yl = mul2(add2(e, small), sc);
}

template <bool VEC>
__device__ __forceinline__ long long topw_slot_id(long long begin, int tid, int s) {
    return VEC ? begin + 4ll * (tid + kTopwThreads * (s >> 2)) + (s & 3)
               : begin + tid + static_cast<long long>(kTopwThreads) * s;
}

// Best two remaining in-range slots of this lane (value desc, slot asc);
// `avail` has a bit per slot still eligible (in range and not taken).  The
// eligible slots are scanned once; a lane only rescans after both of its
// heads were taken (rare: two of the warp's top-W in one lane).
template <int PER>
__device__ __forceinline__ void lane_best2(const float (&x)[PER], uint32_t avail, float& v1,
                                           int& s1, float& v2, int& s2) {
    v1 = v2 = -INFINITY;
    s1 = s2 = -1;
#pragma unroll
    for (int s = 0; s < PER; ++s) {
        if ((avail >> s) & 1u) {
            const float xs = x[s];
            if (s1 < 0 || xs > v1) {
                v2 = v1;
                s2 = s1;
                v1 = xs;
                s1 = s;
            } else if (s2 < 0 || xs > v2) {
                v2 = xs;
                s2 = s;
            }
        }
    }
}

// One round of the warp arg-max over (value, id) heads (id -1 = empty).
__device__ __forceinline__ void warp_best(float& v, int& id) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(kFull, v, off);
        const int oi = __shfl_xor_sync(kFull, id, off);
        if (better(ov, oi, v, id)) {
            v = ov;
            id = oi;
        }
    }
}

// ENT: also sum exp(z - max) * z (float-float) for the row entropy
// H = lse - sum p z of the entropy-mixed build.
template <int W, bool VEC, int PER, bool ENT>
__global__ void __launch_bounds__(kTopwThreads)
    topw_partial_kernel(const float* __restrict__ z, long long V, int splits, ExpTable tab,
                        float* __restrict__ part_v, int* __restrict__ part_id,
                        float* __restrict__ part_m, float2* __restrict__ part_s,
                        float2* __restrict__ part_t) {
    constexpr int CH = kTopwThreads * PER;
    constexpr int NW = kTopwThreads / 32;
    __shared__ float s_thi[64], s_tlo[64];
    __shared__ float s_wv[NW][W];
    __shared__ int s_wi[NW][W];
    __shared__ float s_wmax[NW];
    __shared__ float2 s_wsum[NW];
    __shared__ float2 s_wt[NW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long row = blockIdx.y;
    const int sp = blockIdx.x;
    if (tid < 64) {
        s_thi[tid] = tab.hi[tid];
        s_tlo[tid] = tab.lo[tid];
    }
    const float* zr = z + row * V;
    const long long begin = static_cast<long long>(sp) * CH;
    const long long end = min(V, begin + CH);

    float x[PER];
    if (VEC) {
#pragma unroll
        for (int i = 0; i < PER / 4; ++i) {
            const long long e = begin + 4ll * (tid + kTopwThreads * i);
            float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (e < end) f = __ldg(reinterpret_cast<const float4*>(zr + e));
            x[4 * i + 0] = f.x;
            x[4 * i + 1] = f.y;
            x[4 * i + 2] = f.z;
            x[4 * i + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const long long e = begin + tid + static_cast<long long>(kTopwThreads) * i;
            x[i] = (e < end) ? __ldg(zr + e) : -INFINITY;
        }
    }
    // in-range slots form a prefix of the lane's slots
    int nvalid = 0;
    if (VEC) {
        const long long g = (end - begin - 4ll * tid + 4ll * kTopwThreads - 1) / (4ll * kTopwThreads);
        nvalid = 4 * static_cast<int>(max(0ll, min(static_cast<long long>(PER / 4), g)));
    } else {
        const long long g = (end - begin - tid + kTopwThreads - 1) / kTopwThreads;
        nvalid = static_cast<int>(max(0ll, min(static_cast<long long>(PER), g)));
    }
    uint32_t avail = (nvalid >= 32) ? 0xFFFFFFFFu : ((1u << nvalid) - 1u);
    float bv, bv2;
    int bs, bs2;
    lane_best2(x, avail, bv, bs, bv2, bs2);

    // warp maximum, then this lane's share of sum exp(z - max) (float-float)
    const float mw = warp_max_f(bv);
    __syncthreads();  // exp table ready
    float acc_hi = 0.0f, acc_lo = 0.0f, tac_hi = 0.0f, tac_lo = 0.0f;
    if (mw != -INFINITY) {
        // entries more than 87 below the maximum (and -inf padding) are
        // lifted to max - 87 (~87 after rounding): they then add ~1e-38 each
        // instead of 0, far below the sum's rounding (the sum is >= 1)
        const float floor_v = mw - 87.0f;
        if (!ENT) {
            // two entries per step on packed fp32 pairs, two running sums
            // (even and odd slots) joined in float-float at the end
            F2 ah = f2(0.0f), al = f2(0.0f);
#pragma unroll
            for (int i = 0; i < PER; i += 2) {
                const F2 xc = f2(fmaxf(x[i], floor_v), fmaxf(x[i + 1], floor_v));
                F2 dh, dl;
                two_sum2(xc, f2(-mw), dh, dl);
                F2 yh, yl;
                ffexp_pair(f2(fmaxf(dh.x, -87.0f), fmaxf(dh.y, -87.0f)), dl, s_thi, s_tlo, yh, yl);
                F2 sum, err;
                two_sum2(ah, yh, sum, err);
                ah = sum;
                al = add2(al, add2(err, yl));
            }
            const ffloat sa = ff_add(ff_norm(ah.x, al.x), ff_norm(ah.y, al.y));
            acc_hi = sa.hi;
            acc_lo = sa.lo;
        }
#pragma unroll
        for (int i = 0; ENT && i < PER; ++i) {
            const float xc = fmaxf(x[i], floor_v);
            float dh, dl;
            two_sum(xc, -mw, dh, dl);
            const ffloat y = ffexp_in_range(fmaxf(dh, -87.0f), dl, s_thi, s_tlo);
            float sum, err;
            two_sum(acc_hi, y.hi, sum, err);
            acc_hi = sum;
            acc_lo = jt_add(acc_lo, jt_add(err, y.lo));
            if (ENT) {  // y * xc as a float pair, summed the same way
                const float ph = jt_mul(y.hi, xc);
                const float pl = jt_fmaf(y.lo, xc, jt_fmaf(y.hi, xc, -ph));
                two_sum(tac_hi, ph, sum, err);
                tac_hi = sum;
                tac_lo = jt_add(tac_lo, jt_add(err, pl));
            }
        }
    }
#ifdef JT_CHECKS
    {   // a NaN logit poisons the sum (the clamps above would hide it), so the
        // row's lse is NaN and the expansion's check reports it
        bool bad = false;
#pragma unroll
        for (int i = 0; i < PER; ++i) bad |= (x[i] != x[i]);
        if (bad) acc_hi = __int_as_float(0x7FC00000);
    }
#endif
    pdl_trigger();  // the row merge may be scheduled; it waits for this grid's writes
    const ffloat Sw = warp_sum_ff(ff_norm(acc_hi, acc_lo));
    ffloat Tw;
    Tw.hi = Tw.lo = 0.0f;
    if (ENT) Tw = warp_sum_ff(ff_norm(tac_hi, tac_lo));

    // warp top-W: W extraction rounds over the lanes' heads
#pragma unroll
    for (int r = 0; r < W; ++r) {
        float v = bv;
        int id = (bs >= 0) ? static_cast<int>(topw_slot_id<VEC>(begin, tid, bs)) : -1;
        const int mine = id;
        warp_best(v, id);
        if (lane == 0) {
            s_wv[warp][r] = v;
            s_wi[warp][r] = id;
        }
        if (id != -1 && id == mine) {  // this lane's head was taken
            avail &= ~(1u << bs);
            if (bs2 >= 0) {
                bv = bv2;
                bs = bs2;
                bs2 = -1;  // the next head after this one needs a rescan
            } else {
                float v3;
                int s3;
                lane_best2(x, avail, bv, bs, v3, s3);
                bv2 = v3;
                bs2 = s3;
            }
        }
    }
    if (lane == 0) {
        s_wmax[warp] = mw;
        s_wsum[warp] = make_float2(Sw.hi, Sw.lo);
        if (ENT) s_wt[warp] = make_float2(Tw.hi, Tw.lo);
    }
    __syncthreads();
    if (warp == 0) {
        // chunk max and sum: rescale each warp's sum to the chunk maximum
        float m = (lane < NW) ? s_wmax[lane] : -INFINITY;
        m = warp_max_f(m);
        ffloat S, T;
        S.hi = S.lo = T.hi = T.lo = 0.0f;
        if (lane < NW && m != -INFINITY) {
            const float mj = s_wmax[lane];
            if (mj != -INFINITY) {
                float dh, dl;
                two_sum(mj, -m, dh, dl);
                const ffloat f = ffexp(dh, dl, s_thi, s_tlo);
                ffloat Sj;
                Sj.hi = s_wsum[lane].x;
                Sj.lo = s_wsum[lane].y;
                S = ff_mul(Sj, f);
                if (ENT) {
                    ffloat Tj;
                    Tj.hi = s_wt[lane].x;
                    Tj.lo = s_wt[lane].y;
                    T = ff_mul(Tj, f);
                }
            }
        }
        S = warp_sum_ff(S);
        if (ENT) T = warp_sum_ff(T);
        // chunk top-W from the warps' sorted lists (NW*W <= 64 entries; each
        // lane holds up to two, best first)
        constexpr int PL = (NW * W + 31) / 32;
        float hv[PL];
        int hi[PL];
#pragma unroll
        for (int q = 0; q < PL; ++q) {
            const int c = lane + 32 * q;
            hv[q] = (c < NW * W) ? s_wv[c / W][c % W] : -INFINITY;
            hi[q] = (c < NW * W) ? s_wi[c / W][c % W] : -1;
        }
        if (PL == 2 && better(hv[PL - 1], hi[PL - 1], hv[0], hi[0])) {
            const float tv = hv[0];
            const int ti = hi[0];
            hv[0] = hv[PL - 1];
            hi[0] = hi[PL - 1];
            hv[PL - 1] = tv;
            hi[PL - 1] = ti;
        }
        const long long p = row * splits + sp;
#pragma unroll
        for (int r = 0; r < W; ++r) {
            float v = hv[0];
            int id = hi[0];
            const int mine = id;
            warp_best(v, id);
            if (lane == 0) {
                part_v[p * W + r] = v;
                part_id[p * W + r] = id;
            }
            if (id != -1 && id == mine) {  // pop this lane's head
#pragma unroll
                for (int q = 0; q + 1 < PL; ++q) {
                    hv[q] = hv[q + 1];
                    hi[q] = hi[q + 1];
                }
                hv[PL - 1] = -INFINITY;
                hi[PL - 1] = -1;
            }
        }
        if (lane == 0) {
            part_m[p] = m;
            part_s[p] = make_float2(S.hi, S.lo);
            if (ENT) part_t[p] = make_float2(T.hi, T.lo);
        }
    }
}

// Merge the partials of one row (whole warp): top-W ids/values and lse.
// lse = M + log(sum_j S_j exp(m_j - M)) in float-float: the chunk sums are
// rescaled with the table-driven exp, and log is one fp32 logf refined by a
// Newton step (y = y0 + e - e^2/2 with 1 + e = S exp(-y0)), accurate to
// ~1e-11; only the final assembly and lp = z - lse are fp64.
// ENT: also merge the sum exp(z - max) * z partials and return the row
// entropy H = lse - sum p z.
template <int W, bool ENT, int R = 4>
__device__ __forceinline__ void merge_row(const float* __restrict__ part_v,
                                          const int* __restrict__ part_id,
                                          const float* __restrict__ part_m,
                                          const float2* __restrict__ part_s,
                                          const float2* __restrict__ part_t, int splits,
                                          long long row, int lane, const float* tab_hi,
                                          const float* tab_lo, int (&tok)[W], double (&lp)[W],
                                          double& lse, double& H) {
    const long long base = row * splits;
    // the row's first 32 * R chunk loads are issued up front (one memory
    // round trip): lane handles chunks s = lane + 32 r, r < R; any further
    // chunks (R = 4 covers 512k vocabulary entries) are read in a loop
    constexpr int kMergeR = R;
    float pm[kMergeR];
    float2 ps[kMergeR], pt[kMergeR];
    float pv[kMergeR][W];
    int pi[kMergeR][W];
#pragma unroll
    for (int r = 0; r < kMergeR; ++r) {
        const int s = lane + 32 * r;
        const bool in = s < splits;
        pm[r] = in ? part_m[base + s] : -INFINITY;
        ps[r] = in ? part_s[base + s] : make_float2(0.0f, 0.0f);
        pt[r] = (ENT && in) ? part_t[base + s] : make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < W; ++k) {
            pv[r][k] = in ? part_v[(base + s) * W + k] : -INFINITY;
            pi[r][k] = in ? part_id[(base + s) * W + k] : -1;
        }
    }
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMergeR; ++r) M = fmaxf(M, pm[r]);
    for (int s = lane + 32 * kMergeR; s < splits; s += 32) M = fmaxf(M, part_m[base + s]);
    M = warp_max_f(M);
    ffloat S, T;
    S.hi = S.lo = T.hi = T.lo = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
        for (int r = 0; r < kMergeR; ++r) {
            if (pm[r] != -INFINITY) {
                float dh, dl;
                two_sum(pm[r], -M, dh, dl);
                const ffloat f = ffexp(dh, dl, tab_hi, tab_lo);
                ffloat Sj;
                Sj.hi = ps[r].x;
                Sj.lo = ps[r].y;
                S = ff_add(S, ff_mul(Sj, f));
                if (ENT) {
                    ffloat Tj;
                    Tj.hi = pt[r].x;
                    Tj.lo = pt[r].y;
                    T = ff_add(T, ff_mul(Tj, f));
                }
            }
        }
        for (int s = lane + 32 * kMergeR; s < splits; s += 32) {
            const float ms = part_m[base + s];
            if (ms != -INFINITY) {
                float dh, dl;
                two_sum(ms, -M, dh, dl);
                const ffloat f = ffexp(dh, dl, tab_hi, tab_lo);
                const float2 q = part_s[base + s];
                ffloat Sj;
                Sj.hi = q.x;
                Sj.lo = q.y;
                S = ff_add(S, ff_mul(Sj, f));
                if (ENT) {
                    const float2 qt = part_t[base + s];
                    ffloat Tj;
                    Tj.hi = qt.x;
                    Tj.lo = qt.y;
                    T = ff_add(T, ff_mul(Tj, f));
                }
            }
        }
    }
    S = warp_sum_ff(S);
    if (ENT) T = warp_sum_ff(T);
    if (M == -INFINITY) {
        lse = -INFINITY;
    } else {
        const float y0 = logf(S.hi);
        const ffloat t = ff_mul(S, ffexp(-y0, 0.0f, tab_hi, tab_lo));
        float e = jt_add(jt_add(t.hi, -1.0f), t.lo);
        e = jt_add(e, -0.5f * e * e);
        lse = static_cast<double>(M) + (static_cast<double>(y0) + static_cast<double>(e));
    }

    H = 0.0;
    if (ENT && M != -INFINITY)
        H = lse - (static_cast<double>(T.hi) + static_cast<double>(T.lo)) /
                      (static_cast<double>(S.hi) + static_cast<double>(S.lo));

    TopList<W> L;
    L.init();
#pragma unroll
    for (int r = 0; r < kMergeR; ++r)
#pragma unroll
        for (int k = 0; k < W; ++k) L.push(pv[r][k], pi[r][k]);
    for (int s = lane + 32 * kMergeR; s < splits; s += 32)
#pragma unroll
        for (int k = 0; k < W; ++k) L.push(part_v[(base + s) * W + k], part_id[(base + s) * W + k]);
    float rv[W];
    int rid[W];
    warp_merge<W>(L, rv, rid);
#pragma unroll
    for (int k = 0; k < W; ++k) {
        tok[k] = rid[k];
        lp[k] = static_cast<double>(rv[k]) - lse;
    }
}

// Entropy-mixed step scores of one merged row: ((1 - alpha) * lp) - (alpha *
// H), each operation rounded on its own (no fused multiply-add), as the fp64
// definition evaluates it; probability 0 stays at -inf.  The expansion needs
// each row in queue-key order (score desc, token asc): equal scores (every
// candidate at alpha = 1, rare rounding collisions below it) go by token.
template <int W>
__device__ __forceinline__ void mixed_scores(int (&tok)[W], double (&lp)[W], double H, double alpha) {
#pragma unroll
    for (int k = 0; k < W; ++k)
        if (lp[k] != -INFINITY) lp[k] = __dsub_rn(__dmul_rn(1.0 - alpha, lp[k]), __dmul_rn(alpha, H));
#pragma unroll
    for (int i = 0; i + 1 < W; ++i)
#pragma unroll
        for (int j = 0; j + 1 < W - i; ++j)
            if (lp[j + 1] > lp[j] || (lp[j + 1] == lp[j] && tok[j + 1] < tok[j])) {
                const double tl = lp[j];
                lp[j] = lp[j + 1];
                lp[j + 1] = tl;
                const int tt = tok[j];
                tok[j] = tok[j + 1];
                tok[j + 1] = tt;
            }
}

// ---------------------------------------------------------------------------
// Step 1b: merge the partials, one warp per row (the adaptive build and
// jt_tree_topw; the plain and mixed builds merge inside the expansion).
// ---------------------------------------------------------------------------
template <int W, bool ENT>
__global__ void __launch_bounds__(256)
    topw_merge_kernel(const float* __restrict__ part_v, const int* __restrict__ part_id,
                      const float* __restrict__ part_m, const float2* __restrict__ part_s,
                      const float2* __restrict__ part_t, int splits, long long rows, ExpTable tab,
                      double alpha, int32_t* __restrict__ tok_out, double* __restrict__ lp_out,
                      double* __restrict__ lse_out) {
    __shared__ float s_thi[64], s_tlo[64];
    if (threadIdx.x < 64) {
        s_thi[threadIdx.x] = tab.hi[threadIdx.x];
        s_tlo[threadIdx.x] = tab.lo[threadIdx.x];
    }
    __syncthreads();
    pdl_wait();     // the partials are complete and visible
    pdl_trigger();  // the expansion may be scheduled (it waits for this grid)
    const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    int tok[W];
    double lp[W], lse, H;
    merge_row<W, ENT>(part_v, part_id, part_m, part_s, part_t, splits, row, lane, s_thi, s_tlo, tok, lp,
                      lse, H);
    if (lane == 0) {
        if (ENT) mixed_scores<W>(tok, lp, H, alpha);
#pragma unroll
        for (int k = 0; k < W; ++k) {
            tok_out[row * W + k] = tok[k];
            lp_out[row * W + k] = lp[k];
        }
        lse_out[row] = lse;
    }
}

// ---------------------------------------------------------------------------
// Step 2: best-first expansion, one CTA per sequence.
//
// The nodes best-first pops, in pop order, are exactly the B-1 best non-root
// nodes of the full depth-N tree (or of the tree cut at depth n_cap and
// width w_cap) under the queue key, in key order: a child never beats its
// parent (step scores -- log-probs, or the entropy-mixed scores -- are <= 0,
// and depth breaks exact ties in the parent's favour) and a later sibling
// never beats an earlier one (each table row is in queue-key order).  So
// instead of B-1 dependent pops the CTA builds that set level by level.  S
// holds the best candidates seen so far, sorted by key and cut to B-1.  At
// level d every depth-d entry of S generates its children (depth d+1) that
// beat S's current (B-1)-th entry (any other child has B-1 better nodes, and
// so has every descendant).  Those children form W runs, one per child rank
// k, each already sorted (the parents are sorted and the k-th log-prob is
// shared).  Every candidate's new position is its index in its own sorted
// run plus, per other run, a binary search for the number of better entries;
// no sort is needed.  After the last level S is the pop sequence.  Scores are
// the same fp64 root-to-node sums as the reference definition, so the integer
// outputs are identical.
// ---------------------------------------------------------------------------
constexpr int kExpCap = JT_MAX_TREE + JT_MAX_TREE * JT_MAX_W;  // set + all new children

// Tie key (larger = earlier): depth asc, token asc, parent position asc.
// The parent field only ever decides between children of the same depth
// created at the same level, whose parent positions refer to the same
// (sorted) set.
__device__ __forceinline__ unsigned long long make_k2(int depth, int token, int parent_pos) {
    return (static_cast<unsigned long long>(255 - depth) << 56) |
           (static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(token)) << 24) |
           static_cast<unsigned long long>(0xFFFFFF - (parent_pos + 1));
}
__device__ __forceinline__ int k2_depth(unsigned long long k2) { return 255 - static_cast<int>(k2 >> 56); }
__device__ __forceinline__ int k2_token(unsigned long long k2) {
    return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>((k2 >> 24) & 0xFFFFFFFFull));
}

__device__ __forceinline__ double double_from_order_key(unsigned long long k) {
    const unsigned long long u = (k & 0x8000000000000000ull) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k;
    return __longlong_as_double(static_cast<long long>(u));
}

__device__ __forceinline__ bool key_better(unsigned long long a1, unsigned long long a2,
                                           unsigned long long b1, unsigned long long b2) {
    return a1 > b1 || (a1 == b1 && a2 > b2);
}

// Number of entries of a[0, len) (sorted best first) better than (x1, x2):
// a binary search on the score key alone, then, only when the score is tied,
// one on the tie key inside the equal-score range.
__device__ __forceinline__ int count_better(const unsigned long long* a1, const unsigned long long* a2,
                                            int len, unsigned long long x1, unsigned long long x2) {
    int lo = 0, hi = len;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a1[mid] > x1) lo = mid + 1;
        else hi = mid;
    }
    if (lo < len && a1[lo] == x1) {
        hi = len;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (a1[mid] == x1 && a2[mid] > x2) lo = mid + 1;
            else hi = mid;
        }
    }
    return lo;
}

__host__ __device__ inline int full_tree_nodes(int N, int W, int cap) {
    long long total = 1, level = 1;
    for (int d = 1; d <= N; ++d) {
        level *= W;
        total += level;
        if (total >= cap || level >= cap) return cap;
    }
    return static_cast<int>(total);
}

// Barrier among the first kSetWarps warps only (named barrier 1): the
// set-sized steps run on them while the other warps wait at the next full
// barrier without spending issue slots.
constexpr int kSetWarps = JT_MAX_TREE / 32;
__device__ __forceinline__ void set_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kSetWarps * 32) : "memory");
}

// Inclusive prefix sum of v over threads 0..255; called by warps 0..7 only.
// s_warp[kSetWarps - 1] ends as the total.
__device__ __forceinline__ int set_incl_scan(int v, int* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) s_warp[warp] = v;
    set_sync();
    if (warp == 0) {
        int w = (lane < kSetWarps) ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < kSetWarps; o <<= 1) {
            const int t = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += t;
        }
        if (lane < kSetWarps) s_warp[lane] = w;
    }
    set_sync();
    if (warp > 0) v += s_warp[warp - 1];
    return v;
}

// w_cap / n_cap (optional, per sequence): only the first w_cap[b] candidates
// of every row are children, and nodes of depth n_cap[b] get none.
// The top-W partials of a build whose rows the expansion merges itself.
struct MergeIn {
    const float* v;
    const int* id;
    const float* m;
    const float2* s;
    const float2* t;
    int splits;
    double alpha;
    ExpTable tab;
};

template <int W, int MODE>  // MODE 0: tok_in / lp_in given; 1: merge the partials; 2: merge, mixed scores
__global__ void __launch_bounds__(kExpandThreads, 1)
    expand_kernel(const int32_t* __restrict__ tok_in, const double* __restrict__ lp_in, const MergeIn mi,
                  const int32_t* __restrict__ root_token, const int32_t* __restrict__ tree_off,
                  const int32_t* __restrict__ w_cap, const int32_t* __restrict__ n_cap,
                  int total_nodes, int N, int32_t* __restrict__ parent, int32_t* __restrict__ token,
                  int32_t* __restrict__ depth, uint32_t* __restrict__ anc, uint32_t* err) {
    extern __shared__ __align__(16) unsigned char dsm[];
    // two buffers c = 0, 1 of (score key, tie key, parent position), each
    // kExpCap entries: score keys at kb + 2c*kExpCap, tie keys right after
    unsigned long long* const kb = reinterpret_cast<unsigned long long*>(dsm);  // [kExpCap] x 4
    short* const pb = reinterpret_cast<short*>(kb + 4 * kExpCap);               // [kExpCap] x 2
    short* const rank_of = pb + 2 * kExpCap;                                   // [kExpCap]
    auto kb1 = [&](int c) { return kb + 2 * c * kExpCap; };
    auto kb2 = [&](int c) { return kb + (2 * c + 1) * kExpCap; };
    auto pbuf = [&](int c) { return pb + c * kExpCap; };
    __shared__ int s_tok[JT_MAX_N * W];
    __shared__ double s_lp[JT_MAX_N * W];
    __shared__ short s_front[JT_MAX_TREE];
    __shared__ int s_warp[kExpandThreads / 32];
    __shared__ int s_cnt[kSetWarps][W];
    __shared__ int s_L[W];

    __shared__ float s_thi[MODE ? 64 : 1], s_tlo[MODE ? 64 : 1];
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    if (MODE && tid < 64) {
        s_thi[tid] = mi.tab.hi[tid];
        s_tlo[tid] = mi.tab.lo[tid];
    }
    pdl_wait();     // the tables (or partials) are complete and visible
    pdl_trigger();  // the next kernel may be scheduled (it waits for this grid)
    if (MODE) {
        // the N top-W rows of this sequence from the partials, one warp each
        __syncthreads();  // exp table ready
        for (int d = tid >> 5; d < N; d += kExpandThreads / 32) {
            int tk[W];
            double lp[W], lse, H;
            merge_row<W, MODE == 2, 1>(mi.v, mi.id, mi.m, mi.s, mi.t, mi.splits, static_cast<long long>(b) * N + d,
                                       tid & 31, s_thi, s_tlo, tk, lp, lse, H);
            if ((tid & 31) == 0) {
                if (MODE == 2) mixed_scores<W>(tk, lp, H, mi.alpha);
#pragma unroll
                for (int k = 0; k < W; ++k) {
                    s_tok[d * W + k] = tk[k];
                    s_lp[d * W + k] = lp[k];
                    JT_DCHECK(lp[k] == lp[k] && tk[k] >= 0, err);  // a NaN draft logit makes the row NaN
                }
            }
        }
    } else {
        // The table loads do not depend on the offsets: issue both together.
        for (int i = tid; i < N * W; i += kExpandThreads) {
            s_tok[i] = tok_in[static_cast<long long>(b) * N * W + i];
            s_lp[i] = lp_in[static_cast<long long>(b) * N * W + i];
            // a NaN draft logit makes its row's lse (so every lp) NaN
            JT_DCHECK(s_lp[i] == s_lp[i] && s_tok[i] >= 0, err);
        }
    }
    const int off = tree_off[b];
    const int B = tree_off[b + 1] - off;
    const int Wb = w_cap ? w_cap[b] : W;
    const int Nb = n_cap ? n_cap[b] : N;
    // Uniform over the block: every thread returns or none does.
    if (Wb < 1 || Wb > W || Nb < 0 || Nb > N || B < 1 || B > JT_MAX_TREE ||
        B > full_tree_nodes(Nb, Wb, JT_MAX_TREE + 1) || off < 0 || off + B > total_nodes) {
        if (tid == 0) raise_error(err, DEVERR_INVALID);
        return;
    }
    __syncthreads();

    const int K = B - 1;  // non-root nodes
    const int lane = tid & 31, warp = tid >> 5;
    int m = 0;            // size of the sorted set S (buffer cb)
    int cb = 0;
    for (int d = 0; d < Nb && K > 0; ++d) {
        unsigned long long* k1 = kb1(cb);
        unsigned long long* k2 = kb2(cb);
        short* par = pbuf(cb);
        if (warp < kSetWarps) {
            // frontier: the root at d == 0, else S's depth-d entries (ascending positions)
            int nf;
            if (d == 0) {
                if (tid == 0) s_front[0] = -1;
                nf = 1;
            } else {
                const int is_f = (tid < m && k2_depth(k2[tid]) == d) ? 1 : 0;  // m <= 255
                const int incl = set_incl_scan(is_f, s_warp);
                if (is_f) s_front[incl - 1] = static_cast<short>(tid);
                nf = s_warp[kSetWarps - 1];
            }
            set_sync();
            // children of frontier entry e better than S's (B-1)-th entry
            const bool full = (m >= K);
            const unsigned long long t1 = full ? k1[K - 1] : 0ull, t2 = full ? k2[K - 1] : 0ull;
            const int e = tid;
            int pos = -2, c = 0;
            unsigned long long ck[W];
            if (e < nf) {
                pos = s_front[e];
                const double su = (pos < 0) ? 0.0 : double_from_order_key(k1[pos]);
#pragma unroll
                for (int k = 0; k < W; ++k) {
                    ck[k] = double_order_key(__dadd_rn(su, s_lp[d * W + k]));
                    if (c == k && k < Wb &&
                        (!full || key_better(ck[k], make_k2(d + 1, s_tok[d * W + k], pos), t1, t2)))
                        ++c;
                }
            }
            // run k = children of rank k of entries 0..L_k-1 (L_k
            // non-increasing in k), counted with per-warp ballots
#pragma unroll
            for (int k = 0; k < W; ++k) {
                const unsigned bal = __ballot_sync(kFull, e < nf && c > k);
                if (lane == 0) s_cnt[warp][k] = __popc(bal);
            }
            set_sync();
            if (warp == 0 && lane < W) {
                int l = 0;
#pragma unroll
                for (int w = 0; w < kSetWarps; ++w) l += s_cnt[w][lane];
                s_L[lane] = l;
            }
            set_sync();
            int Rk = 0;  // start of run k
#pragma unroll
            for (int k = 0; k < W; ++k) {
                if (k < c) {
                    const int x = m + Rk + e;
                    k1[x] = ck[k];
                    k2[x] = make_k2(d + 1, s_tok[d * W + k], pos);
                    par[x] = static_cast<short>(pos);
                }
                Rk += s_L[k];
            }
        }
        __syncthreads();
        int L[W], R[W];
        int total = 0;
#pragma unroll
        for (int k = 0; k < W; ++k) {
            L[k] = s_L[k];
            R[k] = total;
            total += L[k];
        }
        if (total == 0) break;
        // rank of every candidate in S + runs; a candidate stops searching as
        // soon as its partial rank reaches B-1 (it is dropped)
        const int M = m + total;
        for (int x = tid; x < M; x += kExpandThreads) {
            const unsigned long long x1 = k1[x], x2 = k2[x];
            int rank, own = -1;
            if (x < m) {
                rank = x;
            } else {
                const int y = x - m;
                int rbase = 0;
#pragma unroll
                for (int k = 0; k < W; ++k)
                    if (y >= R[k] && y < R[k] + L[k]) {
                        own = k;
                        rbase = R[k];
                    }
                rank = y - rbase;
                if (rank < K) rank += count_better(k1, k2, m, x1, x2);
            }
#pragma unroll
            for (int k = 0; k < W; ++k)
                if (rank < K && k != own && L[k] > 0)
                    rank += count_better(k1 + m + R[k], k2 + m + R[k], L[k], x1, x2);
            rank_of[x] = static_cast<short>(rank < K ? rank : -2);
        }
        __syncthreads();
        unsigned long long* n1 = kb1(cb ^ 1);
        unsigned long long* n2 = kb2(cb ^ 1);
        short* npar = pbuf(cb ^ 1);
        for (int x = tid; x < M; x += kExpandThreads) {
            const int r = rank_of[x];
            if (r >= 0) {
                const int pp = par[x];
                n1[r] = k1[x];
                n2[r] = k2[x];
                npar[r] = static_cast<short>(pp < 0 ? pp : rank_of[pp]);
            }
        }
        __syncthreads();
        cb ^= 1;
        m = min(K, M);
    }
    if (m != K) {  // cannot happen when B fits the full tree
        if (tid == 0) raise_error(err, DEVERR_INVALID);
        return;
    }

    // outputs: node 0 = root, node p+1 = S[p]; ancestor-or-self sets
    const unsigned long long* k2f = kb2(cb);
    const short* parf = pbuf(cb);
    for (int n = tid; n < B; n += kExpandThreads) {
        int pn, tn, dn;
        if (n == 0) {
            pn = -1;
            tn = root_token[b];
            dn = 0;
            JT_DCHECK(tn >= 0, err);
        } else {
            pn = parf[n - 1] + 1;
            tn = k2_token(k2f[n - 1]);
            dn = k2_depth(k2f[n - 1]);
        }
        uint32_t a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        int u = n;
        for (int steps = 0; u >= 0 && steps <= JT_MAX_N; ++steps) {
#pragma unroll
            for (int w = 0; w < 8; ++w)
                if (w == (u >> 5)) a[w] |= 1u << (u & 31);
            u = (u == 0) ? -1 : parf[u - 1] + 1;
        }
        const long long g = off + n;
        parent[g] = pn;
        token[g] = tn;
        depth[g] = dn;
        uint4* ap = reinterpret_cast<uint4*>(anc + g * 8);
        ap[0] = make_uint4(a[0], a[1], a[2], a[3]);
        ap[1] = make_uint4(a[4], a[5], a[6], a[7]);
    }
}

constexpr size_t kExpandSmem = sizeof(unsigned long long) * 4 * kExpCap + sizeof(short) * 3 * kExpCap;

// ---------------------------------------------------------------------------
// Adaptive per-request tree policy (AdaptiveSpec, per-step tree policy: the
// draft's top-1 confidence and the rolling acceptance history set the depth,
// width and node count of each request's tree; it grows when both are high
// and shrinks in the opposite case).  Per request b:
//   ema  <- (1 - beta) * ema + beta * accept_len[b]      (when observed)
//   conf =  lp[b, 0, 0] >= log_conf,  hot = ema >= acc_thresh
//   B    <- clamp(B, b_min, ceil); 2B (<= ceil) if conf && hot, B/2 (>= b_min)
//           if neither, else unchanged
//   n_cap = clamp(floor(ema) + n_slack, n_min, N),  w_cap = conf ? W : w_min
//   budget = min(B, full w_cap-ary tree of depth n_cap)
// and tree_off = exclusive prefix sum of the budgets.  One CTA walks the
// requests 1024 at a time with a block scan and a running carry.  fp64
// operations are rounded one by one (no fused multiply-add), like the
// definition, so every decision is reproducible bit for bit.
// ---------------------------------------------------------------------------
constexpr int kPolicyThreads = 1024;

__global__ void __launch_bounds__(kPolicyThreads)
    tree_policy_kernel(const double* __restrict__ lp, int nseq, int N, int W,
                       const int32_t* __restrict__ accept_len, jt_policy_params prm, int ceil_b,
                       int32_t* __restrict__ budget_state, double* __restrict__ acc_ema,
                       int32_t* __restrict__ tree_off, int32_t* __restrict__ w_cap,
                       int32_t* __restrict__ n_cap, uint32_t* err) {
    __shared__ int s_warp[kPolicyThreads / 32];
    __shared__ int s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_carry = 0;
        tree_off[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < nseq; base += kPolicyThreads) {
        const int b = base + tid;
        int emit = 0;
        if (b < nseq) {
            double ema = acc_ema[b];
            const int acc = accept_len ? accept_len[b] : -1;
            if (acc < -1 || acc > N || !(ema >= 0.0) || ema == INFINITY) {
                // invalid state: root-only tree, state left as it was
                raise_error(err, DEVERR_INVALID);
                emit = 1;
                w_cap[b] = W;
                n_cap[b] = 0;
            } else {
                if (acc >= 0)
                    ema = __dadd_rn(__dmul_rn(1.0 - prm.beta, ema), __dmul_rn(prm.beta, static_cast<double>(acc)));
                const bool conf = lp[static_cast<long long>(b) * N * W] >= prm.log_conf;
                const bool hot = ema >= prm.acc_thresh;
                int B = min(max(budget_state[b], prm.b_min), ceil_b);
                if (conf && hot) B = min(2 * B, ceil_b);
                else if (!conf && !hot) B = max(B / 2, prm.b_min);
                const double fl = floor(ema);
                int nc = (fl >= static_cast<double>(N)) ? N : min(static_cast<int>(fl) + prm.n_slack, N);
                nc = max(nc, prm.n_min);
                const int wc = conf ? W : prm.w_min;
                emit = min(B, full_tree_nodes(nc, wc, JT_MAX_TREE + 1));
                budget_state[b] = B;
                acc_ema[b] = ema;
                w_cap[b] = wc;
                n_cap[b] = nc;
            }
        }
        // inclusive block scan of emit
        int v = emit;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31) s_warp[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int w = s_warp[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(kFull, w, o);
                if (lane >= o) w += t;
            }
            s_warp[lane] = w;
        }
        __syncthreads();
        const int incl = v + (warp > 0 ? s_warp[warp - 1] : 0);
        if (b < nseq) tree_off[b + 1] = s_carry + incl;
        __syncthreads();
        if (tid == 0) s_carry += s_warp[kPolicyThreads / 32 - 1];
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
static const ExpTable& exp_table() {
    static const ExpTable tab = [] {
        ExpTable t;
        ffexp_table(t.hi, t.lo);
        return t;
    }();
    return tab;
}

// One-time attribute set-up per device; the first call on a device should
// come before any stream capture.
template <int W, int MODE = 0>
static cudaError_t set_expand_smem() {
    static PerDeviceCache done;
    return static_cast<cudaError_t>(done.get([] {
        return static_cast<int>(cudaFuncSetAttribute(expand_kernel<W, MODE>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     static_cast<int>(kExpandSmem)));
    }));
}

static MergeIn no_merge() {
    MergeIn mi = {};
    return mi;
}

static int topw_splits(long long V, int per) {
    const long long CH = static_cast<long long>(kTopwThreads) * per;
    return static_cast<int>((V + CH - 1) / CH);
}

// Entries per thread: 32, or 16 when 32 would give fewer than four CTAs per
// SM (few rows: shorter per-thread chains, more CTAs).
static int topw_per_thread(long long rows, long long V) {
    const long long ctas = rows * topw_splits(V, kTopwPerThread);
    return (ctas < 4ll * device_sm_count()) ? kTopwPerThreadMin : kTopwPerThread;
}

size_t topw_workspace_bytes(long long rows, long long V, int W, bool ent) {
    const long long p = rows * topw_splits(V, topw_per_thread(rows, V));
    size_t bytes = 0;
    bytes += align_up(rows * W * sizeof(int32_t));  // merged tables (tree build)
    bytes += align_up(rows * W * sizeof(double));
    bytes += align_up(rows * sizeof(double));
    bytes += align_up(p * W * sizeof(float));
    bytes += align_up(p * W * sizeof(int));
    bytes += align_up(p * sizeof(float));
    bytes += align_up(p * sizeof(float2));
    if (ent) bytes += align_up(p * sizeof(float2));  // entropy partials
    return bytes;
}

struct TopwParts {
    int32_t* tok;
    double* lp;
    double* lse;
    float* v;
    int* id;
    float* m;
    float2* s;
    float2* t;  // entropy partials (mixed build only)
    int splits;
};

static TopwParts carve_topw(char* base, long long rows, long long V, int W, int per) {
    TopwParts t;
    t.splits = topw_splits(V, per);
    const long long p = rows * t.splits;
    t.tok = reinterpret_cast<int32_t*>(base);
    base += align_up(rows * W * sizeof(int32_t));
    t.lp = reinterpret_cast<double*>(base);
    base += align_up(rows * W * sizeof(double));
    t.lse = reinterpret_cast<double*>(base);
    base += align_up(rows * sizeof(double));
    t.v = reinterpret_cast<float*>(base);
    base += align_up(p * W * sizeof(float));
    t.id = reinterpret_cast<int*>(base);
    base += align_up(p * W * sizeof(int));
    t.m = reinterpret_cast<float*>(base);
    base += align_up(p * sizeof(float));
    t.s = reinterpret_cast<float2*>(base);
    base += align_up(p * sizeof(float2));
    t.t = reinterpret_cast<float2*>(base);
    return t;
}

template <int W, bool ENT>
static cudaError_t launch_topw_partial(const float* z, long long rows, long long V, int per, TopwParts& t,
                                       cudaStream_t st) {
    const ExpTable& tab = exp_table();
    const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
    dim3 grid(t.splits, static_cast<unsigned>(rows));
#define JT_TOPW_LAUNCH(VEC_, PER_)                                                                       \
    return launch_kernel(topw_partial_kernel<W, VEC_, PER_, ENT>, grid, dim3(kTopwThreads), 0, st, 0, z, \
                         V, t.splits, tab, t.v, t.id, t.m, t.s, t.t)
    if (per == kTopwPerThreadMin) {
        if (vec) JT_TOPW_LAUNCH(true, kTopwPerThreadMin);
        JT_TOPW_LAUNCH(false, kTopwPerThreadMin);
    }
    if (vec) JT_TOPW_LAUNCH(true, kTopwPerThread);
    JT_TOPW_LAUNCH(false, kTopwPerThread);
#undef JT_TOPW_LAUNCH
}

template <int W>
static cudaError_t run_topw(const float* z, long long rows, long long V, int32_t* tok, double* lp,
                            double* lse, char* ws_parts, cudaStream_t st) {
    const int per = topw_per_thread(rows, V);
    TopwParts t = carve_topw(ws_parts, rows, V, W, per);
    cudaError_t e = launch_topw_partial<W, false>(z, rows, V, per, t, st);
    if (e != cudaSuccess) return e;
    const long long warps_per_block = 8;
    const unsigned blocks = static_cast<unsigned>((rows + warps_per_block - 1) / warps_per_block);
    return launch_kernel_pdl(topw_merge_kernel<W, false>, dim3(blocks), dim3(256), 0, st, t.v, t.id, t.m, t.s,
                             t.t, t.splits, rows, exp_table(), 0.0, tok, lp, lse);
}

// alpha > 0: entropy-mixed step scores (1 - alpha) * lp - alpha * H(row);
// alpha == 0 runs the plain build's kernels.
template <int W>
static cudaError_t run_build(const float* z, const int32_t* root_token, const int32_t* tree_off,
                             int nseq, int total_nodes, int N, long long V, double alpha, int32_t* parent,
                             int32_t* token, int32_t* depth, uint32_t* anc, char* ws_parts,
                             uint32_t* err, cudaStream_t st) {
    const long long rows = static_cast<long long>(nseq) * N;
    const int per = topw_per_thread(rows, V);
    TopwParts t = carve_topw(ws_parts, rows, V, W, per);
    const bool ent = alpha != 0.0;
    if (rows > 0) {
        cudaError_t e = ent ? launch_topw_partial<W, true>(z, rows, V, per, t, st)
                            : launch_topw_partial<W, false>(z, rows, V, per, t, st);
        if (e != cudaSuccess) return e;
    }
    // the expansion merges each sequence's rows from the partials itself
    // (one launch fewer on the critical path)
    MergeIn mi;
    mi.v = t.v;
    mi.id = t.id;
    mi.m = t.m;
    mi.s = t.s;
    mi.t = t.t;
    mi.splits = t.splits;
    mi.alpha = alpha;
    mi.tab = exp_table();
    const int32_t* none = nullptr;
    if (ent) {
        cudaError_t ea = set_expand_smem<W, 2>();
        if (ea != cudaSuccess) return ea;
        return launch_kernel_pdl(expand_kernel<W, 2>, dim3(nseq), dim3(kExpandThreads), kExpandSmem, st, none,
                                 static_cast<const double*>(nullptr), mi, root_token, tree_off, none, none,
                                 total_nodes, N, parent, token, depth, anc, err);
    }
    cudaError_t ea = set_expand_smem<W, 1>();
    if (ea != cudaSuccess) return ea;
    return launch_kernel_pdl(expand_kernel<W, 1>, dim3(nseq), dim3(kExpandThreads), kExpandSmem, st, none,
                             static_cast<const double*>(nullptr), mi, root_token, tree_off, none, none, total_nodes,
                             N, parent, token, depth, anc, err);
}

static int policy_ceiling(const jt_policy_params& prm, int nseq) {
    int c = prm.b_max;
    if (prm.node_cap > 0) c = std::min(c, std::max(prm.b_min, prm.node_cap / nseq));
    return c;
}

cudaError_t tree_policy_launch(const double* lp, int nseq, int N, int W, const int32_t* accept_len,
                               const jt_policy_params& prm, int32_t* budget_state, double* acc_ema,
                               int32_t* tree_off, int32_t* w_cap, int32_t* n_cap, uint32_t* err,
                               cudaStream_t st) {
    return launch_kernel(tree_policy_kernel, dim3(1), dim3(kPolicyThreads), 0, st, 0, lp, nseq, N, W, accept_len,
                         prm, policy_ceiling(prm, nseq), budget_state, acc_ema, tree_off, w_cap, n_cap, err);
}

// top-W tables -> policy (budgets, caps, tree_off) -> capped expansion
template <int W>
static cudaError_t run_build_adaptive(const float* z, const int32_t* root_token, int nseq, int capacity, int N,
                                      long long V, const int32_t* accept_len, const jt_policy_params& prm,
                                      int32_t* budget_state, double* acc_ema, int32_t* tree_off,
                                      int32_t* w_cap, int32_t* n_cap, int32_t* parent, int32_t* token,
                                      int32_t* depth, uint32_t* anc, char* ws_parts, uint32_t* err,
                                      cudaStream_t st) {
    const long long rows = static_cast<long long>(nseq) * N;
    const int per = topw_per_thread(rows, V);
    TopwParts t = carve_topw(ws_parts, rows, V, W, per);
    cudaError_t e = launch_topw_partial<W, false>(z, rows, V, per, t, st);
    if (e != cudaSuccess) return e;
    const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
    e = launch_kernel_pdl(topw_merge_kernel<W, false>, dim3(blocks), dim3(256), 0, st, t.v, t.id, t.m, t.s,
                          t.t, t.splits, rows, exp_table(), 0.0, t.tok, t.lp, t.lse);
    if (e != cudaSuccess) return e;
    e = tree_policy_launch(t.lp, nseq, N, W, accept_len, prm, budget_state, acc_ema, tree_off, w_cap, n_cap,
                           err, st);
    if (e != cudaSuccess) return e;
    e = set_expand_smem<W>();
    if (e != cudaSuccess) return e;
    return launch_kernel(expand_kernel<W, 0>, dim3(nseq), dim3(kExpandThreads), kExpandSmem, st, 0, t.tok, t.lp,
                         no_merge(), root_token, static_cast<const int32_t*>(tree_off), static_cast<const int32_t*>(w_cap),
                         static_cast<const int32_t*>(n_cap), capacity, N, parent, token, depth, anc, err);
}

template <int W>
static cudaError_t run_expand(const int32_t* tok, const double* lp, const int32_t* root_token,
                              const int32_t* tree_off, const int32_t* w_cap, const int32_t* n_cap, int nseq,
                              int total_nodes, int N, int32_t* parent, int32_t* token, int32_t* depth,
                              uint32_t* anc, uint32_t* err, cudaStream_t st) {
    cudaError_t ea = set_expand_smem<W>();
    if (ea != cudaSuccess) return ea;
    return launch_kernel_pdl(expand_kernel<W, 0>, dim3(nseq), dim3(kExpandThreads), kExpandSmem, st, tok, lp,
                             no_merge(), root_token, tree_off, w_cap, n_cap, total_nodes, N, parent, token, depth,
                             anc, err);
}

#define JT_DISPATCH_W(W, CALL)           \
    switch (W) {                          \
        case 1: { constexpr int kW = 1; return CALL; } \
        case 2: { constexpr int kW = 2; return CALL; } \
        case 3: { constexpr int kW = 3; return CALL; } \
        case 4: { constexpr int kW = 4; return CALL; } \
        case 5: { constexpr int kW = 5; return CALL; } \
        case 6: { constexpr int kW = 6; return CALL; } \
        case 7: { constexpr int kW = 7; return CALL; } \
        case 8: { constexpr int kW = 8; return CALL; } \
        default: return cudaErrorInvalidValue; \
    }

cudaError_t tree_topw_launch(const float* z, long long rows, long long V, int W, int32_t* tok,
                             double* lp, double* lse, char* ws_parts, cudaStream_t st) {
    JT_DISPATCH_W(W, run_topw<kW>(z, rows, V, tok, lp, lse, ws_parts, st));
}

cudaError_t tree_build_launch(const float* z, const int32_t* root_token, const int32_t* tree_off,
                              int nseq, int total_nodes, int N, int W, long long V, double alpha,
                              int32_t* parent, int32_t* token, int32_t* depth, uint32_t* anc, char* ws_parts,
                              uint32_t* err, cudaStream_t st) {
    JT_DISPATCH_W(W, run_build<kW>(z, root_token, tree_off, nseq, total_nodes, N, V, alpha, parent, token, depth,
                                   anc, ws_parts, err, st));
}

cudaError_t tree_expand_launch(const int32_t* tok, const double* lp, const int32_t* root_token,
                               const int32_t* tree_off, const int32_t* w_cap, const int32_t* n_cap, int nseq,
                               int total_nodes, int N, int W, int32_t* parent, int32_t* token, int32_t* depth,
                               uint32_t* anc, uint32_t* err, cudaStream_t st) {
    JT_DISPATCH_W(W, run_expand<kW>(tok, lp, root_token, tree_off, w_cap, n_cap, nseq, total_nodes, N, parent,
                                    token, depth, anc, err, st));
}

cudaError_t tree_build_adaptive_launch(const float* z, const int32_t* root_token, int nseq, int capacity, int N,
                                       int W, long long V, const int32_t* accept_len, const jt_policy_params& prm,
                                       int32_t* budget_state, double* acc_ema, int32_t* tree_off, int32_t* w_cap,
                                       int32_t* n_cap, int32_t* parent, int32_t* token, int32_t* depth,
                                       uint32_t* anc, char* ws_parts, uint32_t* err, cudaStream_t st) {
    JT_DISPATCH_W(W, run_build_adaptive<kW>(z, root_token, nseq, capacity, N, V, accept_len, prm, budget_state,
                                            acc_ema, tree_off, w_cap, n_cap, parent, token, depth, anc, ws_parts,
                                            err, st));
}

}  // namespace jt
