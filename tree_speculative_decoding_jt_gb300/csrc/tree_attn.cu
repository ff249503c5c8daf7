// tree_attn.cu -- tree-causal attention over a paged bf16 KV cache on the
// sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Semantics (JetSpec news summary, tree-causal attention mask; "加速AI思考…
// 推测解码新方法" sections 三 and 七): tree node n of sequence b attends to
// every prefix slot 0..L_b-1 and to the tree slot L_b+j of each node j in
// its ancestor-or-self set, never to a sibling or a descendant; the mask is
// read from 256-bit ancestor sets, never expanded into a dense matrix.  The
// pages' own kernel (SM90, CuTe DSL, shared-memory mask staging) is prior
// art; this is a Blackwell design.
//
// Work unit (one CTA): sequence b, KV head g, two 128-row query tiles A and
// B (each = 128/G tree nodes x the G query heads of that KV head: GQA heads
// share K/V because they are stacked in the MMA's M dimension), and a
// contiguous range of 128-key tiles of the logical key sequence (prefix +
// tree tail).  Both query tiles consume every K/V tile, halving the paged TMA
// traffic per FLOP.  Keys past the last node of tile B are never loaded
// (ancestors have smaller indices).  Several key ranges of one unit (KV
// split) are merged by tree_attn_combine_kernel.
//
// Warp roles (320 threads):
//   warps 0-3 / 4-7  softmax + epilogue of query tile A / B, one query row
//                    per thread (TMEM lane);
//   warp 8           TMA producer: both Q tiles once, then per KV tile one
//                    16-row box per 16-token page for K and for V (128-byte
//                    swizzle); page ids are held in registers, loaded two
//                    groups of four tiles ahead; zero-fills V rows past the
//                    last needed slot of the final tile;
//   warp 9           TMEM allocator and single-thread MMA issuer.
// TMEM (512 columns): per query tile X, S_X (128 fp32 columns) and O_X (D
// fp32 columns).  Per KV tile j: S_X = Q_X K^T (SS MMA, K-major operands,
// M=128, N=128, K=D); softmax X reads S_X and writes P_X (bf16, packed in
// pairs) over the first 64 columns of S_X; O_X += P_X V (TS MMA: A = P_X
// from TMEM, B = V MN-major, N=D).  Issue order per KV tile: PV_A(j),
// QK_A(j+1), PV_B(j), QK_B(j+1): the tensor core runs tile A's MMAs while
// softmax B works and the other way round.  MMAs from one thread execute in
// issue order, so QK_X(j+1) overwrites S_X only after PV_X(j) has read P_X,
// and the completion of QK_X(j+1) tells softmax X that O_X holds PV_X(j).
// Online softmax in the log2 domain, two passes over S in TMEM (row max,
// then exp and P), lazy rescaling of O (only when the running max grows by
// more than 2^8).  All waits are bounded in time.
#include "jt_common.cuh"
#include "jt_internal.h"

namespace jt {

constexpr int kAttnThreads = 320;
constexpr int kStages = 2;   // K ring and V ring depth
constexpr int kTileN = 128;  // keys per KV tile
constexpr int kTileM = 128;  // query rows per query tile
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxSplits = 32;

struct AttnParams {
    const int32_t* block_table;
    const int32_t* prefix_len;
    const int32_t* tree_off;
    const uint32_t* anc;
    __nv_bfloat16* out;
    float* lse;
    float* part_o;   // [total*Hq*splits, D] when splits > 1
    float2* part_ml; // [total*Hq*splits]: running max (log2 units), sum
    uint32_t* err;
    int max_pages, num_pages, nseq, total_nodes, Hq, G, npt, splits;
    float scale_log2;
};

template <int D>
struct SmemLayout {
    static constexpr int kChunks = D / 64;            // 64-element (128-byte) column blocks
    static constexpr int kChunkBytes = kTileM * 128;  // 128 rows x 128 bytes
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kQ = 0;                      // Q_A, Q_B
    static constexpr int kK = kQ + 2 * kTileBytes;
    static constexpr int kV = kK + kStages * kTileBytes;
    static constexpr int kBar = kV + kStages * kTileBytes;
    static constexpr int kBytes = kBar + 256;
    static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};

struct Bars {
    uint64_t q_full;
    uint64_t k_full[kStages];
    uint64_t v_full[kStages];
    uint64_t k_empty[kStages];
    uint64_t v_empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_final[2];
    uint64_t v_last;
    uint64_t mma_final;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Visibility of 32 consecutive keys starting at tree-relative position rel0
// (bit c <-> rel0 + c): negative positions are prefix slots (visible),
// positions in [0, 256) read the ancestor-or-self set a[], the rest are not
// visible.
__device__ __forceinline__ uint32_t visible_bits(const uint32_t (&a)[8], int rel0) {
    if (rel0 >= JT_MAX_TREE) return 0u;
    if (rel0 + 32 <= 0) return 0xFFFFFFFFu;
    const int w0 = rel0 >> 5;  // floor division
    const int sh = rel0 & 31;
    uint32_t lo = 0u, hi = 0u;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        if (w == w0) lo = a[w];
        if (w == w0 + 1) hi = a[w];
    }
    if (w0 < 0) lo = 0xFFFFFFFFu;
    return sh ? ((lo >> sh) | (hi << (32 - sh))) : lo;
}

// The 128 fp32 scores of this thread's S row, held in registers as four
// 32-column chunks (one TMEM round trip per tile).
struct SRow {
    uint32_t c[4][32];
};

__device__ __forceinline__ void load_srow(uint32_t tS, SRow& s) {
    tmem_ld32(tS, s.c[0]);
    tmem_ld32(tS + 32, s.c[1]);
    tmem_ld32(tS + 64, s.c[2]);
    tmem_ld32(tS + 96, s.c[3]);
    tmem_wait_ld();
}

// Columns whose key (tree-relative position rel0 + c) is not visible -> -inf.
__device__ __forceinline__ void mask_srow(SRow& s, const uint32_t (&a)[8], int rel0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t vis = visible_bits(a, rel0 + 32 * q);
#pragma unroll
        for (int c = 0; c < 32; ++c)
            if (!((vis >> c) & 1u)) s.c[q][c] = __float_as_uint(-INFINITY);
    }
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed fp32 pair arithmetic (one instruction per two lanes of data on
// sm_100 and later): (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1), and the sum.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ float max_srow(const SRow& s) {
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            m0 = fmax3(m0, __uint_as_float(s.c[q][c]), __uint_as_float(s.c[q][c + 1]));
            m1 = fmax3(m1, __uint_as_float(s.c[q][c + 2]), __uint_as_float(s.c[q][c + 3]));
        }
    return fmaxf(m0, m1);
}

// P = exp2(s * sl2 - m), packed to bf16 pairs into the first 64 columns of
// the S region (the scores are already in registers); returns the row sum.
// Per pair of scores: one packed FMA, two ex2, one packed add, one convert.
__device__ __forceinline__ float exp_store_srow(const SRow& s, uint32_t tS, float sl2, float m) {
    float a0 = 0.0f, a1 = 0.0f, b0 = 0.0f, b1 = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        uint32_t pk[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int c2 = (q & 1) * 8 + c;
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(s.c[q >> 1][2 * c2]), __uint_as_float(s.c[q >> 1][2 * c2 + 1]), sl2, sl2,
                  -m, -m);
            const float e0 = ex2_approx(x0);
            const float e1 = ex2_approx(x1);
            if (c & 1)
                fadd2(b0, b1, b0, b1, e0, e1);
            else
                fadd2(a0, a1, a0, a1, e0, e1);
            pk[c] = pack_bf16x2(e0, e1);
        }
        tmem_st8(tS + 8 * q, pk);
    }
    return (a0 + a1) + (b0 + b1);
}

// Tile range [t0, t0 + count) of split sp for a unit whose needed keys end
// at valid_end; returns the count.
__device__ __forceinline__ int split_range(int valid_end, int splits, int sp, int& t0) {
    const int T = (valid_end + kTileN - 1) / kTileN;
    const int tps = (T + splits - 1) / splits;
    t0 = sp * tps;
    const int t1 = min(T, t0 + tps);
    return max(0, t1 - t0);
}

// Keys needed by the unit of query-tile pair mp: through the last node of
// its second tile.
__device__ __forceinline__ int unit_valid_end(int L, int B, int mp, int npt) {
    return L + min(B, (2 * mp + 2) * npt);
}

// Operand descriptors are built once (dq: Q tile, dk / dv: K / V stage) and
// stepped by adding the byte offset / 16 to the start-address field (the
// field cannot carry: shared memory addresses stay below 256 KB).  The whole
// MMA warp calls these; one elected lane issues, with as few instructions per
// MMA as possible because the softmax warps compete for the same issue slots.

// S (+)= Q K^T: 8 (D = 128) or 4 (D = 64) MMAs of K = 16.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tS, uint64_t dq, uint64_t dk) {
    using SL = SmemLayout<D>;
    constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kTileN, false);
    if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = ((kk >> 2) * SL::kChunkBytes + (kk & 3) * 32) >> 4;
            mma_ss(tS, dq + ko, dk + ko, idesc, kk > 0 ? 1u : 0u);
        }
    }
    __syncwarp();
}

// O (+)= P V with P (bf16 pairs) in the first 64 columns of S: 8 MMAs of K = 16.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tS, uint64_t dv, bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16_f32(kTileM, D, true);
    if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
            mma_ts(tS + 128, tS + kk * 8, dv + kk * ((16 * 128) >> 4), idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
    __syncwarp();
}

// tcgen05.commit from the elected lane (the lane that issued the MMAs).
__device__ __forceinline__ void commit_warp(uint64_t* bar) {
    if (elect_one()) mma_commit(bar);
    __syncwarp();
}

// Page ids of 4 consecutive tiles (group g4): lane l holds page l%8 of tile
// 4*g4 + l/8 of the unit.
__device__ __forceinline__ int bt_group(const AttnParams& p, int b, int t0, int nt, int valid_end,
                                        int g4, int lane) {
    const int tile = 4 * g4 + (lane >> 3);
    const int slot = (t0 + tile) * kTileN + (lane & 7) * JT_PAGE_SIZE;
    return (tile < nt && slot < valid_end)
               ? p.block_table[static_cast<long long>(b) * p.max_pages + slot / JT_PAGE_SIZE]
               : 0;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
    using SL = SmemLayout<D>;
    constexpr int kTileBytes = SL::kTileBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + SL::kBar);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, g = blockIdx.y;
    const int mp = blockIdx.x / p.splits, sp = blockIdx.x % p.splits;
    // Set-up that reads no global memory (barriers, TMEM, tensor-map
    // prefetch) runs before the wait for the previous kernel, overlapping
    // its tail when this grid is launched as its programmatic dependent.
    if (tid == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bars->s_full[x], 1);
            mbar_init(&bars->p_full[x], 128);
            mbar_init(&bars->o_final[x], 1);
        }
        mbar_init(&bars->v_last, 1);
        mbar_init(&bars->mma_final, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 9) tmem_alloc(&bars->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    volatile int* abort = &bars->abort;

    pdl_wait();  // no global memory is read before the previous kernel's writes are visible
    const int off = p.tree_off[b];
    const int B = p.tree_off[b + 1] - off;
    const int L = p.prefix_len[b];
    const int m0 = 2 * mp;                    // query tile A; tile B = m0 + 1
    bool run = m0 * p.npt < B;                // else the pair lies past this sequence's tree
    if (run && (B > JT_MAX_TREE || L < 0 || off < 0 || off + B > p.total_nodes ||
                static_cast<long long>(L) + B > static_cast<long long>(p.max_pages) * JT_PAGE_SIZE)) {
        if (tid == 0) raise_error(p.err, DEVERR_INVALID);
        run = false;
    }
    const bool hasB = (m0 + 1) * p.npt < B;
    const int n_end = min(B, (m0 + 2) * p.npt);
    const int valid_end = L + n_end;
    int t0 = 0;
    const int nt = run ? split_range(valid_end, p.splits, sp, t0) : 0;
    if (nt == 0) {  // nothing to do (or an empty split, which the combine skips too)
        if (warp == 9) tmem_dealloc(tmem, 512);  // no tcgen05 operation was issued
        return;
    }

    uint8_t* sQ = smem + SL::kQ;
    uint8_t* sK = smem + SL::kK;
    uint8_t* sV = smem + SL::kV;

    if (warp == 8) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars->q_full, (hasB ? 2 : 1) * kTileBytes);
            for (int x = 0; x < (hasB ? 2 : 1); ++x)
                for (int c = 0; c < SL::kChunks; ++c)
                    tma_load_3d(sQ + x * kTileBytes + c * SL::kChunkBytes, &tm_q, &bars->q_full,
                                c * 64, g * p.G, off + (m0 + x) * p.npt);
        }
        // page ids held in registers, loaded two groups of four tiles ahead
        int bt_cur = bt_group(p, b, t0, nt, valid_end, 0, lane);
        int bt_nxt = bt_group(p, b, t0, nt, valid_end, 1, lane);
        int bt_nn = bt_group(p, b, t0, nt, valid_end, 2, lane);
        int issued = 0;
        for (int j = 0; j < nt; ++j) {
            const int st = j % kStages;
            const uint32_t empty_parity = ((j / kStages) & 1) ^ 1;
            if (j > 0 && (j & 3) == 0) {
                bt_cur = bt_nxt;
                bt_nxt = bt_nn;
                bt_nn = bt_group(p, b, t0, nt, valid_end, (j >> 2) + 2, lane);
            }
            const int slot0 = (t0 + j) * kTileN;
            const int nvalid = min(kTileN, valid_end - slot0);
            const int npg = (nvalid + JT_PAGE_SIZE - 1) / JT_PAGE_SIZE;
            const int pid = __shfl_sync(0xFFFFFFFFu, bt_cur, ((j & 3) << 3) + (lane & 7));
            JT_DCHECK(lane >= npg || (pid >= 0 && pid < p.num_pages), p.err);  // block-table entry in the pool
            const uint32_t bytes = npg * SL::kChunks * (JT_PAGE_SIZE * 128);
            // K of tile j: its slot is free once QK^T of tile j-kStages is done
            if (j >= kStages && !mbar_wait_warp(&bars->k_empty[st], empty_parity, p.err, abort)) break;
            if (lane == 0) mbar_arrive_expect_tx(&bars->k_full[st], bytes);
            __syncwarp();
            if (lane < npg)
                for (int c = 0; c < SL::kChunks; ++c)
                    tma_load_4d(sK + st * kTileBytes + c * SL::kChunkBytes + lane * (JT_PAGE_SIZE * 128),
                                &tm_k, &bars->k_full[st], c * 64, g, 0, pid);
            // V of tile j: free once PV of tile j-kStages is done
            if (j >= kStages && !mbar_wait_warp(&bars->v_empty[st], empty_parity, p.err, abort)) break;
            if (lane == 0) mbar_arrive_expect_tx(&bars->v_full[st], bytes);
            __syncwarp();
            if (lane < npg)
                for (int c = 0; c < SL::kChunks; ++c)
                    tma_load_4d(sV + st * kTileBytes + c * SL::kChunkBytes + lane * (JT_PAGE_SIZE * 128),
                                &tm_v, &bars->v_full[st], c * 64, g, 0, pid);
            issued = j + 1;
            if (j == nt - 1) {
                // final tile: once its V has landed, zero rows past the last
                // needed slot (stale or foreign data; P is 0 there but
                // 0 * NaN would not be), then release it to the MMA warp
                if (!mbar_wait_warp(&bars->v_full[st], (j / kStages) & 1, p.err, abort)) break;
                uint8_t* vt = sV + st * kTileBytes;
                const int n16 = (kTileN - nvalid) * 8;  // 16-byte pieces per column block
                for (int c = 0; c < SL::kChunks; ++c)
                    for (int idx = lane; idx < n16; idx += 32)
                        reinterpret_cast<uint4*>(vt + c * SL::kChunkBytes + (nvalid + (idx >> 3)) * 128)[idx & 7] =
                            make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->v_last);
            }
        }
        // on abort: let copies already in flight land before the CTA exits
        if (*abort) {
            for (int j = max(0, issued - kStages); j < issued; ++j) {
                mbar_wait(&bars->k_full[j % kStages], (j / kStages) & 1, p.err, nullptr);
                mbar_wait(&bars->v_full[j % kStages], (j / kStages) & 1, p.err, nullptr);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA
        // the whole warp runs this loop (uniform control flow, operands in
        // uniform registers); one elected lane issues every tcgen05 op
        using SLm = SmemLayout<D>;
        const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), SLm::kChunkBytes, 1024);
        constexpr uint32_t kTileStep = SLm::kTileBytes >> 4;  // one tile / stage in 16-byte units
        const int nx = hasB ? 2 : 1;
        bool ok = mbar_wait_warp(&bars->q_full, 0, p.err, abort) &&
                  mbar_wait_warp(&bars->k_full[0], 0, p.err, abort);
        if (ok) {
            tc_fence_after();
            for (int x = 0; x < nx; ++x) {
                issue_qk<D>(tmem + 256 * x, dq0 + x * kTileStep, dk0);
                commit_warp(&bars->s_full[x]);
            }
            commit_warp(&bars->k_empty[0]);
        }
        for (int j = 0; ok && j < nt; ++j) {
            const int st = j % kStages;
            const bool more = j + 1 < nt;
            for (int x = 0; ok && x < nx; ++x) {
                ok = mbar_wait_warp(&bars->p_full[x], j & 1, p.err, abort);
                if (ok && x == 0)
                    ok = (j == nt - 1) ? mbar_wait_warp(&bars->v_last, 0, p.err, abort)
                                       : mbar_wait_warp(&bars->v_full[st], (j / kStages) & 1, p.err, abort);
                if (!ok) break;
                tc_fence_after();
                issue_pv<D>(tmem + 256 * x, dv0 + st * kTileStep, j > 0);
                if (x == nx - 1) commit_warp(&bars->v_empty[st]);
                if (!more) {
                    commit_warp(&bars->o_final[x]);
                } else {
                    if (x == 0) ok = mbar_wait_warp(&bars->k_full[(j + 1) % kStages],
                                                    ((j + 1) / kStages) & 1, p.err, abort);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk<D>(tmem + 256 * x, dq0 + x * kTileStep, dk0 + ((j + 1) % kStages) * kTileStep);
                    commit_warp(&bars->s_full[x]);
                    if (x == nx - 1) commit_warp(&bars->k_empty[(j + 1) % kStages]);
                }
            }
        }
        // every MMA issued above completes before TMEM is released
        commit_warp(&bars->mma_final);
        mbar_wait_warp(&bars->mma_final, 0, p.err, nullptr);
    } else if (warp < 4 || hasB) {
        // ---------------------------------------------- softmax of tile X
        const int x = warp >> 2;
        const int r = tid & 127;  // query row = TMEM lane
        const int node = (m0 + x) * p.npt + r / p.G;
        const int head = g * p.G + r % p.G;
        const bool valid_row = node < n_end;
        uint32_t a[8];
#pragma unroll
        for (int w = 0; w < 8; ++w)
            a[w] = valid_row ? p.anc[static_cast<long long>(off + node) * 8 + w] : 0u;
#ifdef JT_CHECKS
        if (valid_row) {  // a node's set holds the node itself and only nodes before it
            bool ok_set = true;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const int lo = 32 * w;
                const uint32_t allowed = node >= lo + 31 ? 0xFFFFFFFFu : (node < lo ? 0u : (2u << (node - lo)) - 1u);
                if (a[w] & ~allowed) ok_set = false;
                if (node >= lo && node < lo + 32 && !((a[w] >> (node - lo)) & 1u)) ok_set = false;
            }
            JT_DCHECK(ok_set, p.err);
        }
#endif
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + 256 * x + lane_off, tO = tS + 128;
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.0f;
        bool ok = true;
        for (int j = 0; j < nt && ok; ++j) {
            if (!mbar_wait_warp(&bars->s_full[x], j & 1, p.err, abort)) { ok = false; break; }
            tc_fence_after();
            const int slot0 = (t0 + j) * kTileN;
            const bool tail = slot0 + kTileN > L;
            SRow sr;
            load_srow(tS, sr);
            if (tail) mask_srow(sr, a, slot0 - L);  // tiles inside the prefix need no mask
            const float mx = max_srow(sr);
            const float mx_s = mx * sl2;
            bool resc = false;
            float factor = 1.0f;
            if (mx_s > m_run + kRescaleLog2 || m_run == -INFINITY) {
                const float m_new = fmaxf(m_run, mx_s);
                if (m_run != -INFINITY) {
                    factor = ex2_approx(m_run - m_new);
                    resc = j > 0;
                } else {
                    factor = 0.0f;
                }
                l_run *= factor;
                m_run = m_new;
            }
            // P = exp2(s*scale*log2e - m), written over S (bf16 pairs)
            const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
            l_run += exp_store_srow(sr, tS, sl2, m_use);
            if (__any_sync(0xFFFFFFFFu, resc)) {
                // O_X from the earlier tiles, rescaled before PV_X(j) adds to it
                // (S_X(j) done implies PV_X(j-1) done: O_X is current)
#pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t v[32];
                    tmem_ld32(tO + q * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        v[c] = __float_as_uint(__uint_as_float(v[c]) * (resc ? factor : 1.0f));
                    tmem_st32(tO + q * 32, v);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_full[x]);
        }
        // epilogue (the split combine may be scheduled; it waits for this grid)
        pdl_trigger();
        if (ok && mbar_wait_warp(&bars->o_final[x], 0, p.err, abort)) {
            tc_fence_after();
            const long long rowid = static_cast<long long>(off + node) * p.Hq + head;
            const float inv = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
            // Every QK_X MMA completed before o_final[X], so the Q_X tile is
            // free: each warp stages its 32 rows there, one 128-byte piece
            // of each row at a time (16-byte slots XOR-swizzled by row, so
            // both the row-wise writes and the line-wise reads are free of
            // bank conflicts), and 8 lanes then store each row's piece as
            // one full 128-byte line.
            uint8_t* stage = sQ + x * kTileBytes + (warp & 3) * 4096;
            const int sub = lane & 7;  // 16-byte slot of the piece
            const bool piece_f32 = p.splits > 1;
            constexpr int kPiecesF32 = D / 32, kPiecesBf16 = D / 64;
            const int pieces = piece_f32 ? kPiecesF32 : kPiecesBf16;
#pragma unroll 1
            for (int h = 0; h < pieces; ++h) {
                uint4 slot[8];
                if (piece_f32) {
                    uint32_t v[32];
                    tmem_ld32(tO + h * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 8; ++c) slot[c] = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                } else {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tO + h * 64, v0);
                    tmem_ld32(tO + h * 64 + 32, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        slot[c] = make_uint4(
                            pack_bf16x2(__uint_as_float(v0[8 * c + 0]) * inv, __uint_as_float(v0[8 * c + 1]) * inv),
                            pack_bf16x2(__uint_as_float(v0[8 * c + 2]) * inv, __uint_as_float(v0[8 * c + 3]) * inv),
                            pack_bf16x2(__uint_as_float(v0[8 * c + 4]) * inv, __uint_as_float(v0[8 * c + 5]) * inv),
                            pack_bf16x2(__uint_as_float(v0[8 * c + 6]) * inv, __uint_as_float(v0[8 * c + 7]) * inv));
                        slot[4 + c] = make_uint4(
                            pack_bf16x2(__uint_as_float(v1[8 * c + 0]) * inv, __uint_as_float(v1[8 * c + 1]) * inv),
                            pack_bf16x2(__uint_as_float(v1[8 * c + 2]) * inv, __uint_as_float(v1[8 * c + 3]) * inv),
                            pack_bf16x2(__uint_as_float(v1[8 * c + 4]) * inv, __uint_as_float(v1[8 * c + 5]) * inv),
                            pack_bf16x2(__uint_as_float(v1[8 * c + 6]) * inv, __uint_as_float(v1[8 * c + 7]) * inv));
                    }
                }
                uint4* my_row = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c) my_row[c ^ (lane & 7)] = slot[c];
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = 4 * i + (lane >> 3);  // staged row this lane copies
                    const long long rid = __shfl_sync(0xFFFFFFFFu, rowid, rr);
                    const bool rvalid = __shfl_sync(0xFFFFFFFFu, valid_row, rr);
                    const uint4 val = reinterpret_cast<const uint4*>(stage + rr * 128)[sub ^ (rr & 7)];
                    if (rvalid) {
                        if (piece_f32)
                            reinterpret_cast<uint4*>(p.part_o + (rid * p.splits + sp) * D + h * 32)[sub] = val;
                        else
                            reinterpret_cast<uint4*>(p.out + rid * D + h * 64)[sub] = val;
                    }
                }
                __syncwarp();  // the next piece overwrites the stage
            }
            if (valid_row) {
                if (p.splits == 1) {
                    if (p.lse) p.lse[rowid] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
                } else {
                    p.part_ml[rowid * p.splits + sp] = make_float2(m_run, l_run);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Merge the KV-split partials of every (node, head) row.  One warp per row.
template <int D>
__global__ void __launch_bounds__(128)
    tree_attn_combine_kernel(const AttnParams p, int total_nodes) {
    pdl_wait();  // the partials are complete and visible
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x;
    const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
    if (n >= total_nodes || h >= p.Hq) return;
    int lo = 0, hi = p.nseq;  // sequence of node n
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.tree_off[mid] <= n) lo = mid; else hi = mid;
    }
    const int b = lo, off = p.tree_off[b];
    const int B = p.tree_off[b + 1] - off;
    const int L = p.prefix_len[b];
    if (B < 1 || B > JT_MAX_TREE || L < 0 || off < 0 || off + B > p.total_nodes ||
        static_cast<long long>(L) + B > static_cast<long long>(p.max_pages) * JT_PAGE_SIZE)
        return;  // reported by the main kernel
    const int node = n - off;
    if (node >= B) return;  // spare capacity past the last tree
    const int valid_end = unit_valid_end(L, B, (node / p.npt) >> 1, p.npt);
    const long long rowid = static_cast<long long>(n) * p.Hq + h;
    float M = -INFINITY;
    int ns = 0;
    for (int s = 0; s < p.splits; ++s) {
        int t0;
        if (split_range(valid_end, p.splits, s, t0) == 0) break;
        M = fmaxf(M, p.part_ml[rowid * p.splits + s].x);
        ns = s + 1;
    }
    float acc[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) acc[k] = 0.0f;
    float lsum = 0.0f;
    for (int s = 0; s < ns; ++s) {
        const float2 ml = p.part_ml[rowid * p.splits + s];
        const float wgt = (ml.x == -INFINITY) ? 0.0f : exp2f(ml.x - M);
        lsum += wgt * ml.y;
        const float* po = p.part_o + (rowid * p.splits + s) * D;
#pragma unroll
        for (int k = 0; k < D / 32; ++k) acc[k] += wgt * po[lane + 32 * k];
    }
    const float inv = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) p.out[rowid * D + lane + 32 * k] = __float2bfloat16_rn(acc[k] * inv);
    if (lane == 0 && p.lse) p.lse[rowid] = (M + log2f(lsum)) * 0.6931471805599453f;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                      const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                      const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                      CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled_t get_encode_fn() {
    static PFN_encodeTiled_t fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiled_t>(ptr);
    }
    return fn;
}

AttnPlan attn_plan(int nseq, int Hkv, int Hq, int max_tree, int max_pages, int dtype) {
    AttnPlan pl;
    const int G = Hq / Hkv;
    pl.rows_per_tile_nodes = kTileM / G;
    pl.mtiles = (max_tree + pl.rows_per_tile_nodes - 1) / pl.rows_per_tile_nodes;
    pl.splits = 1;
    if (dtype == JT_DTYPE_BF16) {
        const long long units = static_cast<long long>(nseq) * Hkv * ((pl.mtiles + 1) / 2);
        const int sms = device_sm_count();
        const int tmax = (max_pages * JT_PAGE_SIZE + kTileN - 1) / kTileN;
        if (units > 0 && units < sms) {
            int s = static_cast<int>(sms / units);
            s = min(s, max(1, tmax / 2));
            pl.splits = max(1, min(s, kMaxSplits));
        }
    }
    return pl;
}

size_t attn_workspace_bytes(const AttnPlan& p, int total_nodes, int Hq, int D) {
    size_t b = kWsHeader;
    if (p.splits > 1) {
        const size_t rows = static_cast<size_t>(total_nodes) * Hq * p.splits;
        b += align_up(rows * D * sizeof(float));
        b += align_up(rows * sizeof(float2));
    }
    return b;
}

template <int D>
static cudaError_t launch_bf16(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int max_pages, int num_pages,
                               const int32_t* prefix_len, const int32_t* tree_off,
                               const uint32_t* anc, int nseq, int total_nodes, int Hq, int Hkv,
                               float scale, void* out, float* lse, const AttnPlan& plan,
                               char* ws_parts, uint32_t* err, cudaStream_t st) {
    PFN_encodeTiled_t enc = get_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int G = Hq / Hkv;
    CUtensorMap tq, tk, tv;
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                                    static_cast<cuuint64_t>(total_nodes)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                       static_cast<cuuint64_t>(Hq) * D * 2};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G),
                                   static_cast<cuuint32_t>(plan.rows_per_tile_nodes)};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                                    JT_PAGE_SIZE, static_cast<cuuint64_t>(num_pages)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                       static_cast<cuuint64_t>(Hkv) * D * 2,
                                       static_cast<cuuint64_t>(JT_PAGE_SIZE) * Hkv * D * 2};
        const cuuint32_t box[4] = {64, 1, JT_PAGE_SIZE, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(k_cache), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        if (enc(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(v_cache), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    AttnParams prm;
    prm.block_table = block_table;
    prm.prefix_len = prefix_len;
    prm.tree_off = tree_off;
    prm.anc = anc;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.lse = lse;
    prm.part_o = nullptr;
    prm.part_ml = nullptr;
    if (plan.splits > 1) {
        const size_t rows = static_cast<size_t>(total_nodes) * Hq * plan.splits;
        prm.part_o = reinterpret_cast<float*>(ws_parts);
        prm.part_ml = reinterpret_cast<float2*>(ws_parts + align_up(rows * D * sizeof(float)));
    }
    prm.err = err;
    prm.max_pages = max_pages;
    prm.num_pages = num_pages;
    prm.nseq = nseq;
    prm.total_nodes = total_nodes;
    prm.Hq = Hq;
    prm.G = G;
    prm.npt = plan.rows_per_tile_nodes;
    prm.splits = plan.splits;
    prm.scale_log2 = scale * 1.4426950408889634f;

    using SL = SmemLayout<D>;
    static PerDeviceCache attr;  // the shared-memory opt-in is per device
    const cudaError_t ea = static_cast<cudaError_t>(attr.get([] {
        return static_cast<int>(cudaFuncSetAttribute(tree_attn_tc_kernel<D>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, SL::kAlloc));
    }));
    if (ea != cudaSuccess) return ea;
    dim3 grid(((plan.mtiles + 1) / 2) * plan.splits, Hkv, nseq);
    cudaError_t e = launch_kernel_pdl(tree_attn_tc_kernel<D>, grid, dim3(kAttnThreads), SL::kAlloc, st, tq, tk,
                                      tv, prm);
    if (e != cudaSuccess || plan.splits == 1) return e;
    dim3 cgrid(total_nodes, (Hq + 3) / 4);
    return launch_kernel_pdl(tree_attn_combine_kernel<D>, cgrid, dim3(128), 0, st, prm, total_nodes);
}

cudaError_t tree_attn_bf16_launch(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, int max_pages, int num_pages,
                                  const int32_t* prefix_len, const int32_t* tree_off,
                                  const uint32_t* anc, int nseq, int total_nodes, int Hq, int Hkv,
                                  int D, float scale, void* out, float* lse, const AttnPlan& plan,
                                  char* ws_parts, uint32_t* err, cudaStream_t st) {
    if (D == 128)
        return launch_bf16<128>(q, k_cache, v_cache, block_table, max_pages, num_pages, prefix_len,
                                tree_off, anc, nseq, total_nodes, Hq, Hkv, scale, out, lse, plan,
                                ws_parts, err, st);
    if (D == 64)
        return launch_bf16<64>(q, k_cache, v_cache, block_table, max_pages, num_pages, prefix_len,
                               tree_off, anc, nseq, total_nodes, Hq, Hkv, scale, out, lse, plan,
                               ws_parts, err, st);
    return cudaErrorInvalidValue;
}

}  // namespace jt
