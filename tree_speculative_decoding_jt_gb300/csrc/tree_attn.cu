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
// Work.  A unit is (sequence b, KV head g, query-tile pair mp): two 128-row
// query tiles A = 2mp and B = 2mp+1 (each = 128/G tree nodes x the G query
// heads of KV head g, which share K/V because they are stacked in the MMA's
// M dimension; B is absent when the tree ends inside A) against the 128-key
// tiles 0..T_u-1 of the sequence's logical keys (prefix + tree through the
// last node of tile B; ancestors have smaller indices, so no later key is
// ever visible).  Units are laid end to end in (b, g, mp) order and the
// T_total key tiles of all units are cut into one equal range of
// P = ceil(T_total / slots) tiles per work slot -- one CTA per SM in the
// single-SM kernel below, one CTA pair per two SMs in the CTA-pair kernel
// further down (head dim 128; the host picks it when every (sequence, KV
// head) has one query-tile pair): every SM gets the same tile count
// whatever the prefix lengths, so there is no tail wave and no straggler.
// A slot walks the pieces of units in its range; a unit cut
// by a range boundary leaves fp32 partials (O, running max, sum) from each
// CTA that holds a piece of it, and the CTA that finishes its piece last
// merges them (an atomic count per cut unit, tagged with the call's number
// so that counts left by earlier calls never need clearing; no CTA ever
// waits for another).  Only the first and the last piece of a CTA can be
// cut, so two partial slots per CTA suffice.  Each CTA derives the whole
// plan from prefix_len and tree_off on the device, so sequence lengths never
// visit the host.  With few units (a batch of one: every unit would be cut
// into many pieces whose merge lands on one CTA's critical path) the launch
// runs in split mode instead: one CTA per (unit, key split), the splits'
// partials merged by tree_attn_combine_kernel, one warp per query row.
//
// Single-SM kernel, warp roles (320 threads):
//   warps 0-3 / 4-7  softmax + epilogue of query tile A / B, one query row
//                    per thread (TMEM lane);
//   warp 8           planner, then TMA producer: per piece the Q tiles, then
//                    per KV tile one 16-row box per 16-token page for K and
//                    for V (128-byte swizzle); page ids are held in
//                    registers, loaded two groups of four tiles ahead; zero-
//                    fills V rows past the last needed slot of a unit's
//                    final tile;
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
// Across pieces the barrier phases run on (global tile and piece counters);
// the next piece's first PV_X overwrites O_X only after softmax X has read
// it out, because softmax X reads O_X before it releases that PV.
// Online softmax in the log2 domain, two passes over S in TMEM (row max,
// then exp and P), lazy rescaling of O (only when the running max grows by
// more than 2^8).  All waits are bounded in time.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "jt_common.cuh"
#include "jt_internal.h"

namespace jt {

constexpr int kAttnThreads = 320;
constexpr int kStages = 2;   // K ring and V ring depth
constexpr int kTileN = 128;  // keys per KV tile
constexpr int kTileM = 128;  // query rows per query tile
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxMergeIn = 4;  // other pieces whose (m, l) a merging row loads in one batch

struct AttnParams {
    const int32_t* block_table;
    const int32_t* prefix_len;
    const int32_t* tree_off;
    const uint32_t* anc;
    __nv_bfloat16* out;
    float* lse;
    float* part_o;    // [2 * grid][2][128][D]: partial O of the pieces of cut units
    float2* part_ml;  // [2 * grid][2][128]: their running max (log2 units) and sum
    int* plan;        // [2 + nseq + 1]: T_total, P, then each sequence's first global tile
    unsigned long long* tickets;    // CTA arrivals over all calls (workspace header)
    unsigned long long* merge_cnt;  // [grid][2]: (call number << 32) | pieces done, per cut unit and query tile
    uint32_t* err;
    int max_pages, num_pages, nseq, total_nodes, Hq, Hkv, G, npt;
    int splits, npairs;  // split mode (splits > 0): CTA c = unit c / splits, key split c % splits
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
    static constexpr int kStage = kV + kStages * kTileBytes;  // epilogue staging, 4 KB per softmax warp
    static constexpr int kBar = kStage + 8 * 4096;
    static constexpr int kBytes = kBar + 512;
    static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};

struct Bars {
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t k_full[kStages];
    uint64_t v_full[kStages];
    uint64_t k_empty[kStages];
    uint64_t v_empty[kStages];
    uint64_t v_last[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_final[2];
    uint64_t mma_final;
    uint32_t tmem_base;
    int abort;
    // the CTA's start position, published by the planner
    int w_b, w_g, w_mp, w_t, w_quota, w_P;
    uint32_t call_id;  // this call's number (+1) on this workspace
    int merge_flag[2];  // per query tile: this CTA finished the last piece of a cut unit
    uint64_t msync[2];  // per query tile: its four softmax warps meet (merge of a cut unit)
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// ---------------------------------------------------------------------------
// The work plan (shared by the main kernel's roles and the combine)
// ---------------------------------------------------------------------------
struct SeqInfo {
    int L, B, off;
    int np;  // query-tile pairs (0: no tree, or contents out of range)
};

__device__ __forceinline__ SeqInfo load_seq(const AttnParams& p, int b) {
    SeqInfo s;
    s.off = p.tree_off[b];
    s.B = p.tree_off[b + 1] - s.off;
    s.L = p.prefix_len[b];
    const bool ok = s.B >= 0 && s.B <= JT_MAX_TREE && s.L >= 0 && s.off >= 0 && s.off + s.B <= p.total_nodes &&
                    static_cast<long long>(s.L) + s.B <= static_cast<long long>(p.max_pages) * JT_PAGE_SIZE;
    s.np = ok ? ((s.B + p.npt - 1) / p.npt + 1) / 2 : (s.B == 0 ? 0 : -1);
    return s;
}

// Keys needed by pair mp: through the last node of its second tile.
__device__ __forceinline__ int unit_end(const SeqInfo& s, int mp, int npt) {
    return s.L + min(s.B, (2 * mp + 2) * npt);
}
__device__ __forceinline__ int unit_tiles(const SeqInfo& s, int mp, int npt) {
    return (unit_end(s, mp, npt) + kTileN - 1) / kTileN;
}
// Key tiles of all pairs of one KV head.
__device__ __forceinline__ int head_tiles(const SeqInfo& s, int npt) {
    int t = 0;
    for (int mp = 0; mp < s.np; ++mp) t += unit_tiles(s, mp, npt);
    return t;
}

// One piece: key tiles [t0, t0 + nt) of unit (b, g, mp), which has T tiles.
// slot: the partial slot the piece writes, or -1 when it is the whole unit.
struct Piece {
    SeqInfo s;
    int b, g, mp, t0, nt, T, slot;
    int gpos;  // global tile index of the piece's first tile
};

// Walks the pieces of one work slot's tile range in order.  Every role runs
// its own copy over the same start position, so all roles see the same
// pieces.  A work slot is one CTA of the single-SM kernel, or one CTA pair.
struct Walker {
    SeqInfo s;
    int b, g, mp, t, remaining, piece, gpos, work;

    template <typename BarsT>
    __device__ __forceinline__ void init(const AttnParams& p, const BarsT* bars, int work_slot) {
        b = bars->w_b;
        g = bars->w_g;
        mp = bars->w_mp;
        t = bars->w_t;
        remaining = bars->w_quota;
        work = work_slot;
        gpos = work * bars->w_P;
        piece = 0;
        if (remaining > 0) s = load_seq(p, b);
    }

    __device__ __forceinline__ bool next(const AttnParams& p, Piece& pc) {
        if (remaining <= 0) return false;
        const int T = unit_tiles(s, mp, p.npt);
        const int nt = min(T - t, remaining);
        pc.s = s;
        pc.b = b;
        pc.g = g;
        pc.mp = mp;
        pc.t0 = t;
        pc.nt = nt;
        pc.T = T;
        pc.slot = (t == 0 && nt == T) ? -1 : 2 * work + (piece == 0 ? 0 : 1);
        pc.gpos = gpos;
        gpos += nt;
        remaining -= nt;
        t += nt;
        ++piece;
        if (t == T && remaining > 0) {  // on to the next unit in (b, g, mp) order
            t = 0;
            if (++mp >= s.np) {
                mp = 0;
                if (++g >= p.Hkv) {
                    g = 0;
                    do {
                        ++b;
                        s = load_seq(p, b);
                    } while (s.np <= 0 && b + 1 < p.nseq);
                }
            }
        }
        return true;
    }
};

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// The planner (one warp): the total tile count, the range of work slot
// `work` (of nwork) and the unit and tile that range starts at.  With rec
// set (one CTA of work slot 0) it also records the plan (T_total, P and each
// sequence's first global tile) and reports sequences whose offsets or
// lengths are out of range.
template <typename BarsT>
__device__ void plan_cta(const AttnParams& p, BarsT* bars, int lane, int work, int nwork, bool rec) {
    const int H = p.Hkv;
    long long total = 0;
    for (int base = 0; base < p.nseq; base += 32) {
        const int b = base + lane;
        int t = 0;
        if (b < p.nseq) {
            const SeqInfo s = load_seq(p, b);
            if (s.np < 0) {
                if (rec) raise_error(p.err, DEVERR_INVALID);
            } else {
                t = H * head_tiles(s, p.npt);
            }
        }
        total += warp_sum(t);
    }
    if (total > 0x7FFFFFFFll) {  // beyond the int tile arithmetic: refuse the launch's work
        if (rec && lane == 0) raise_error(p.err, DEVERR_INVALID);
        total = 0;
    }
    const int T_total = static_cast<int>(total);
    const int P = T_total > 0 ? (T_total + nwork - 1) / nwork : 0;
    const long long start = static_cast<long long>(work) * P;
    int quota = (start < T_total) ? static_cast<int>(min(static_cast<long long>(P), T_total - start)) : 0;
    if (rec && lane == 0) {
        p.plan[0] = T_total;
        p.plan[1] = P;
    }
    // second pass: the sequence holding tile `start` (and, on CTA 0, every
    // sequence's first global tile)
    int found_b = -1, found_rel = 0;
    int acc = 0;
    for (int base = 0; base < p.nseq && (rec || found_b < 0); base += 32) {
        const int b = base + lane;
        int t = 0;
        if (b < p.nseq) {
            const SeqInfo s = load_seq(p, b);
            if (s.np > 0) t = H * head_tiles(s, p.npt);
        }
        int incl = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += u;
        }
        const int excl = acc + incl - t;
        if (rec && b < p.nseq) p.plan[2 + b] = excl;
        const bool here = t > 0 && start >= excl && start < excl + t;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, here);
        if (m && found_b < 0) {
            const int src = __ffs(m) - 1;
            found_b = base + src;
            found_rel = static_cast<int>(start) - __shfl_sync(0xFFFFFFFFu, excl, src);
        }
        acc += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (rec && lane == 0) p.plan[2 + p.nseq] = acc;
    if (found_b < 0) quota = 0;
    if (lane == 0) {
        int g = 0, mp = 0, t = 0;
        if (quota > 0) {
            const SeqInfo s = load_seq(p, found_b);
            const int ht = head_tiles(s, p.npt);
            g = found_rel / ht;
            int r = found_rel - g * ht;
            while (mp < s.np - 1 && r >= unit_tiles(s, mp, p.npt)) {
                r -= unit_tiles(s, mp, p.npt);
                ++mp;
            }
            t = r;
        }
        bars->w_b = found_b;
        bars->w_g = g;
        bars->w_mp = mp;
        bars->w_t = t;
        bars->w_quota = quota;
        bars->w_P = P;
    }
}

// Split mode: work slot c holds unit u = c / splits of the dense (b, g, mp)
// layout (npairs pairs per KV head), key split c % splits of ceil(T /
// splits) tiles.  Slots whose pair lies past the sequence's tree, or whose
// split is empty, get no tiles.  rec: report bad sequence contents.
__device__ __forceinline__ int split_tiles(int T, int splits) { return (T + splits - 1) / splits; }

template <typename BarsT>
__device__ void plan_cta_split(const AttnParams& p, BarsT* bars, int lane, int c, bool rec) {
    const int u = c / p.splits, sp = c % p.splits;
    const int b = u / (p.Hkv * p.npairs);
    const int rem = u % (p.Hkv * p.npairs);
    int quota = 0, t0 = 0;
    if (b < p.nseq) {
        const SeqInfo s = load_seq(p, b);
        if (s.np < 0 && rec && lane == 0) raise_error(p.err, DEVERR_INVALID);
        // the recording CTA also reports the other sequences' bad contents
        if (rec)
            for (int bb = lane; bb < p.nseq; bb += 32)
                if (bb != b && load_seq(p, bb).np < 0) raise_error(p.err, DEVERR_INVALID);
        const int mp = rem % p.npairs;
        if (mp < s.np) {
            const int T = unit_tiles(s, mp, p.npt);
            const int tps = split_tiles(T, p.splits);
            t0 = sp * tps;
            quota = max(0, min(T, t0 + tps) - t0);
        }
    }
    if (lane == 0) {
        bars->w_b = b;
        bars->w_g = rem / p.npairs;
        bars->w_mp = rem % p.npairs;
        bars->w_t = t0;
        bars->w_quota = quota;
        bars->w_P = 0;
    }
}

// The CTAs holding the pieces of the unit that starts at global tile U and
// has T tiles (range length P): c0 .. c0 + n - 1; slot of piece k.
struct CutUnit {
    int c0, n, slot0;
    __device__ __forceinline__ CutUnit(int U, int T, int P) {
        c0 = U / P;
        n = (U + T - 1) / P - c0 + 1;
        slot0 = 2 * c0 + (U == c0 * P ? 0 : 1);
    }
    __device__ __forceinline__ int slot(int k) const { return k == 0 ? slot0 : 2 * (c0 + k); }
};

// Stage this warp's 32 rows' 128-byte pieces (slot[8] = this thread's row)
// through shared memory (16-byte slots XOR-swizzled by row: conflict-free
// both ways) and store each row's piece as one full line: dst(rr) gives the
// destination of staged row rr (nullptr: skip).
template <typename Dst>
__device__ __forceinline__ void stage_store(uint8_t* stage, int lane, const uint4 (&slot)[8], Dst dst) {
    uint4* my_row = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c) my_row[c ^ (lane & 7)] = slot[c];
    __syncwarp();
    const int sub = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + (lane >> 3);  // staged row this lane copies
        const uint4 val = reinterpret_cast<const uint4*>(stage + rr * 128)[sub ^ (rr & 7)];
        uint4* d = dst(rr);
        if (d) d[sub] = val;
    }
    __syncwarp();  // the next piece overwrites the stage
}

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

// The same maximum over eight independent chains (a shorter dependency
// chain, for kernels with registers to spare).
__device__ __forceinline__ float max_srow8(const SRow& s) {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = fmaxf(__uint_as_float(s.c[i >> 1][(i & 1) * 16]), __uint_as_float(s.c[i >> 1][(i & 1) * 16 + 1]));
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int c = 2; c < 16; c += 2)
            m[i] = fmax3(m[i], __uint_as_float(s.c[i >> 1][(i & 1) * 16 + c]),
                         __uint_as_float(s.c[i >> 1][(i & 1) * 16 + c + 1]));
    return fmaxf(fmax3(m[0], m[1], m[2]), fmax3(fmax3(m[3], m[4], m[5]), m[6], m[7]));
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

// Page ids of 4 consecutive tiles (group g4) of a piece: lane l holds page
// l%8 of tile 4*g4 + l/8 of the piece.
__device__ __forceinline__ int bt_group(const AttnParams& p, const Piece& pc, int valid_end, int g4, int lane) {
    const int tile = 4 * g4 + (lane >> 3);
    const int slot = (pc.t0 + tile) * kTileN + (lane & 7) * JT_PAGE_SIZE;
    return (tile < pc.nt && slot < valid_end)
               ? p.block_table[static_cast<long long>(pc.b) * p.max_pages + slot / JT_PAGE_SIZE]
               : 0;
}

// Call numbers for the merge counts.  Every CTA of a call draws from the
// workspace's ticket counter: the recording CTA (the first of work slot 0)
// draws kTicketQuantum - (CTAs - 1) tickets and every other CTA one, so a
// call draws exactly kTicketQuantum tickets whatever its grid, and all its
// CTAs compute the same number, ticket / kTicketQuantum + 1.
constexpr unsigned long long kTicketQuantum = 1ull << 24;

__device__ __forceinline__ uint32_t draw_call_id(unsigned long long* tickets, bool first, unsigned ctas) {
    const unsigned long long t = atomicAdd(tickets, first ? kTicketQuantum - (ctas - 1u) : 1ull);
    return static_cast<uint32_t>(t / kTicketQuantum) + 1u;
}

// Output of one piece for this thread's query row (tile X, row r): the
// normalised bf16 row and its lse when the piece is a whole unit, else the
// fp32 partial row; when this work slot completes a cut unit, the merge of
// all its pieces.  O_X is read from TMEM at tO (complete: the caller has
// waited for the piece's last PV).  The four softmax warps of tile X call
// this together; sync4(i) is their i-th meeting of this merge (bounded:
// false when it gives up, the error already raised).
template <int D, typename BarsT, typename Sync4>
__device__ __forceinline__ void piece_output(const AttnParams& p, const Piece& pc, BarsT* bars, int work, int x,
                                             int r, int lane, int node, int head, bool valid_row, uint32_t tO,
                                             uint8_t* stage, float m_run, float l_run, Sync4&& sync4) {
    const long long rowid = static_cast<long long>(pc.s.off + node) * p.Hq + head;
    const bool partial = pc.slot >= 0;
    const long long prow = (static_cast<long long>(pc.slot) * 2 + x) * kTileM + r;  // partial row
    const float inv = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
    // Each warp stages its 32 output rows in its own 4 KB of shared
    // memory, one 128-byte piece of each row at a time, and stores
    // full lines (stage_store).
    if (partial) {
#pragma unroll 1
        for (int h = 0; h < D / 32; ++h) {
            uint32_t v[32];
            tmem_ld32(tO + h * 32, v);
            tmem_wait_ld();
            uint4 slot[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) slot[c] = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            stage_store(stage, lane, slot, [&](int rr) {
                const long long pr = __shfl_sync(0xFFFFFFFFu, prow, rr);
                return reinterpret_cast<uint4*>(p.part_o + pr * D + h * 32);
            });
        }
        p.part_ml[prow] = make_float2(m_run, l_run);
    } else {
#pragma unroll 1
        for (int h = 0; h < D / 64; ++h) {
            uint32_t v0[32], v1[32];
            tmem_ld32(tO + h * 64, v0);
            tmem_ld32(tO + h * 64 + 32, v1);
            tmem_wait_ld();
            uint4 slot[8];
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
            stage_store(stage, lane, slot, [&](int rr) {
                const long long rid = __shfl_sync(0xFFFFFFFFu, rowid, rr);
                const bool rvalid = __shfl_sync(0xFFFFFFFFu, valid_row, rr);
                return rvalid ? reinterpret_cast<uint4*>(p.out + rid * D + h * 64) : nullptr;
            });
        }
        if (valid_row && p.lse) p.lse[rowid] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
    }
    if (partial && p.splits == 0) {
        // count this piece done; the CTA that completes the unit
        // merges every piece's partial rows (its own included).  Each
        // query tile's four warps do this on their own (sync4, count and
        // flag per tile), so neither tile's warps ever wait for the
        // other's.
        const CutUnit cu(pc.gpos - pc.t0, pc.T, bars->w_P);
        __threadfence();  // this thread's partial rows are visible GPU-wide
        if (!sync4(0)) return;
        if (r == 0) {
            const uint32_t cid = bars->call_id;
            unsigned long long* ctr = p.merge_cnt + 2 * cu.c0 + x;
            unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr), assumed, nv;
            do {  // a count from an earlier call restarts at this call's first piece
                assumed = old;
                nv = ((assumed >> 32) == cid) ? assumed + 1ull
                                              : ((static_cast<unsigned long long>(cid) << 32) | 1ull);
                old = atomicCAS(ctr, assumed, nv);
            } while (old != assumed);
            bars->merge_flag[x] = static_cast<int>(nv & 0xFFFFFFFFull) == cu.n;
            __threadfence();  // the other pieces' rows are read after this count
        }
        if (!sync4(1)) return;
        if (bars->merge_flag[x]) {  // uniform over the tile's warps
            // merge this row over the unit's pieces: M = max m_k,
            // O = sum 2^(m_k - M) O_k / sum 2^(m_k - M) l_k.  This
            // CTA's own piece is still in TMEM (O_X) and registers
            // (m_run, l_run); the other pieces come from L2, each
            // half row (64 columns) one batch of 16 loads in flight.
            const int own = work - cu.c0;
            float mk[kMaxMergeIn], lk[kMaxMergeIn];
            float M = m_run;
#pragma unroll
            for (int i = 0; i < kMaxMergeIn; ++i) {  // every other piece's (m, l) in one round trip
                const int k = i < own ? i : i + 1;
                mk[i] = -INFINITY;
                lk[i] = 0.0f;
                if (k < cu.n) {
                    const float2 ml = __ldcg(&p.part_ml[(static_cast<long long>(cu.slot(k)) * 2 + x) * kTileM + r]);
                    mk[i] = ml.x;
                    lk[i] = ml.y;
                }
            }
            for (int k0 = kMaxMergeIn; k0 + 1 < cu.n; ++k0) {  // beyond the unrolled pieces (rare)
                const int k = k0 < own ? k0 : k0 + 1;
                M = fmaxf(M, __ldcg(&p.part_ml[(static_cast<long long>(cu.slot(k)) * 2 + x) * kTileM + r]).x);
            }
#pragma unroll
            for (int i = 0; i < kMaxMergeIn; ++i) M = fmaxf(M, mk[i]);
            // weights and sums in piece order, whichever CTA merges,
            // so that every call rounds the same way
            const float w_own = (m_run == -INFINITY) ? 0.0f : exp2f(m_run - M);
#pragma unroll
            for (int i = 0; i < kMaxMergeIn; ++i) mk[i] = (mk[i] == -INFINITY) ? 0.0f : exp2f(mk[i] - M);
            auto weight_of = [&](int k) {  // piece k's weight (k != own)
                const int i = k < own ? k : k - 1;
                float w = mk[0];
#pragma unroll
                for (int j = 1; j < kMaxMergeIn; ++j)
                    if (j == i) w = mk[j];
                if (i >= kMaxMergeIn) {
                    const float ms = __ldcg(&p.part_ml[(static_cast<long long>(cu.slot(k)) * 2 + x) * kTileM + r]).x;
                    w = (ms == -INFINITY) ? 0.0f : exp2f(ms - M);
                }
                return w;
            };
            auto sum_of = [&](int k) {  // piece k's row sum (k != own)
                const int i = k < own ? k : k - 1;
                float l = lk[0];
#pragma unroll
                for (int j = 1; j < kMaxMergeIn; ++j)
                    if (j == i) l = lk[j];
                if (i >= kMaxMergeIn) l = __ldcg(&p.part_ml[(static_cast<long long>(cu.slot(k)) * 2 + x) * kTileM + r]).y;
                return l;
            };
            float lsum = 0.0f;
            for (int k = 0; k < cu.n; ++k) lsum += (k == own) ? w_own * l_run : weight_of(k) * sum_of(k);
            const float minv = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;
#pragma unroll 1
            for (int h = 0; h < D / 64; ++h) {
                uint32_t packed[32];  // the 64 output columns of this staged piece, bf16 pairs
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int col = h * 64 + half * 32;
                    float acc[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) acc[c] = 0.0f;
#pragma unroll 1
                    for (int k = 0; k < cu.n; ++k) {
                        if (k == own) {  // this CTA's piece, from TMEM (k is the same for the whole warp)
                            uint32_t v[32];
                            tmem_ld32(tO + col, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 32; ++c) acc[c] += w_own * __uint_as_float(v[c]);
                        } else {
                            const long long pr = (static_cast<long long>(cu.slot(k)) * 2 + x) * kTileM + r;
                            const float wgt = weight_of(k);
                            const float4* po = reinterpret_cast<const float4*>(p.part_o + pr * D + col);
                            float4 q[8];
#pragma unroll
                            for (int c = 0; c < 8; ++c) q[c] = __ldcg(po + c);
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                acc[4 * c + 0] += wgt * q[c].x;
                                acc[4 * c + 1] += wgt * q[c].y;
                                acc[4 * c + 2] += wgt * q[c].z;
                                acc[4 * c + 3] += wgt * q[c].w;
                            }
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        packed[half * 16 + c] = pack_bf16x2(acc[2 * c] * minv, acc[2 * c + 1] * minv);
                }
                uint4 slot[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    slot[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
                stage_store(stage, lane, slot, [&](int rr) {
                    const long long rid = __shfl_sync(0xFFFFFFFFu, rowid, rr);
                    const bool rvalid = __shfl_sync(0xFFFFFFFFu, valid_row, rr);
                    return rvalid ? reinterpret_cast<uint4*>(p.out + rid * D + h * 64) : nullptr;
                });
            }
            if (valid_row && p.lse) p.lse[rowid] = (M + log2f(lsum)) * 0.6931471805599453f;
        }
    }
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
    const int work = blockIdx.x;  // one work slot per CTA
    // Set-up that reads no global memory (barriers, TMEM, tensor-map
    // prefetch) runs before the wait for the previous kernel, overlapping
    // its tail when this grid is launched as its programmatic dependent.
    if (tid == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_empty[s], 1);
            mbar_init(&bars->v_last[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bars->s_full[x], 1);
            mbar_init(&bars->p_full[x], 128);
            mbar_init(&bars->o_final[x], 1);
            mbar_init(&bars->msync[x], 4);
        }
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
    pdl_wait();  // no global memory is read before the previous kernel's writes are visible
    if (warp == 8) {
        if (p.splits > 0)
            plan_cta_split(p, bars, lane, blockIdx.x, blockIdx.x == 0);
        else
            plan_cta(p, bars, lane, blockIdx.x, gridDim.x, blockIdx.x == 0);
    }
    if (tid == 0)  // every CTA of a call draws its tickets before anything can fail
        bars->call_id = draw_call_id(p.tickets, blockIdx.x == 0, gridDim.x);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    volatile int* abort = &bars->abort;
    if (bars->w_quota <= 0) {  // no tiles for this CTA
        if (warp == 9) tmem_dealloc(tmem, 512);  // no tcgen05 operation was issued
        return;
    }

    uint8_t* sQ = smem + SL::kQ;
    uint8_t* sK = smem + SL::kK;
    uint8_t* sV = smem + SL::kV;
    const int npt = p.npt;

    if (warp == 8) {
        // ------------------------------------------------------------ TMA
        Walker w;
        w.init(p, bars, work);
        Piece pc;
        int jj = 0, npc = 0, q_pending = 0;
        int k_iss = 0, v_iss = 0;  // K / V tiles whose copies have been issued
        int vl[kStages] = {0, 0};
        while (!*abort && w.next(p, pc)) {
            const bool hasB = (2 * pc.mp + 1) * npt < pc.s.B;
            const int valid_end = unit_end(pc.s, pc.mp, npt);
            // Q of this piece: the Q tiles are free once every QK of the
            // previous piece has completed
            if (npc > 0 && !mbar_wait_warp(&bars->q_empty, (npc - 1) & 1, p.err, abort)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->q_full, (hasB ? 2 : 1) * kTileBytes);
                for (int x = 0; x < (hasB ? 2 : 1); ++x)
                    for (int c = 0; c < SL::kChunks; ++c)
                        tma_load_3d(sQ + x * kTileBytes + c * SL::kChunkBytes, &tm_q, &bars->q_full, c * 64,
                                    pc.g * p.G, pc.s.off + (2 * pc.mp + x) * npt);
            }
            q_pending = npc + 1;
            // page ids held in registers, loaded two groups of four tiles ahead
            int bt_cur = bt_group(p, pc, valid_end, 0, lane);
            int bt_nxt = bt_group(p, pc, valid_end, 1, lane);
            int bt_nn = bt_group(p, pc, valid_end, 2, lane);
            bool ok = true;
            for (int j = 0; j < pc.nt; ++j, ++jj) {
                const int st = jj % kStages;
                const uint32_t empty_parity = ((jj / kStages) & 1) ^ 1;
                if (j > 0 && (j & 3) == 0) {
                    bt_cur = bt_nxt;
                    bt_nxt = bt_nn;
                    bt_nn = bt_group(p, pc, valid_end, (j >> 2) + 2, lane);
                }
                const int slot0 = (pc.t0 + j) * kTileN;
                const int nvalid = min(kTileN, valid_end - slot0);
                const int npg = (nvalid + JT_PAGE_SIZE - 1) / JT_PAGE_SIZE;
                const int pid = __shfl_sync(0xFFFFFFFFu, bt_cur, ((j & 3) << 3) + (lane & 7));
                JT_DCHECK(lane >= npg || (pid >= 0 && pid < p.num_pages), p.err);  // block-table entry in the pool
                const uint32_t bytes = npg * SL::kChunks * (JT_PAGE_SIZE * 128);
                // K of tile jj: its slot is free once QK^T of tile jj-kStages is done
                if (jj >= kStages && !mbar_wait_warp(&bars->k_empty[st], empty_parity, p.err, abort)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&bars->k_full[st], bytes);
                __syncwarp();
                if (lane < npg)
                    for (int c = 0; c < SL::kChunks; ++c)
                        tma_load_4d(sK + st * kTileBytes + c * SL::kChunkBytes + lane * (JT_PAGE_SIZE * 128),
                                    &tm_k, &bars->k_full[st], c * 64, pc.g, 0, pid);
                k_iss = jj + 1;
                // V of tile jj: free once PV of tile jj-kStages is done
                if (jj >= kStages && !mbar_wait_warp(&bars->v_empty[st], empty_parity, p.err, abort)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&bars->v_full[st], bytes);
                __syncwarp();
                if (lane < npg)
                    for (int c = 0; c < SL::kChunks; ++c)
                        tma_load_4d(sV + st * kTileBytes + c * SL::kChunkBytes + lane * (JT_PAGE_SIZE * 128),
                                    &tm_v, &bars->v_full[st], c * 64, pc.g, 0, pid);
                v_iss = jj + 1;
                if (pc.t0 + j == pc.T - 1) {
                    // the unit's final tile: once its V has landed, zero the
                    // rows past the last needed slot (stale or foreign data;
                    // P is 0 there but 0 * NaN would not be), then release
                    // it to the MMA warp
                    if (!mbar_wait_warp(&bars->v_full[st], (jj / kStages) & 1, p.err, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* vt = sV + st * kTileBytes;
                    const int n16 = (kTileN - nvalid) * 8;  // 16-byte pieces per column block
                    for (int c = 0; c < SL::kChunks; ++c)
                        for (int idx = lane; idx < n16; idx += 32)
                            reinterpret_cast<uint4*>(vt + c * SL::kChunkBytes + (nvalid + (idx >> 3)) * 128)[idx & 7] =
                                make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->v_last[st]);
                    ++vl[st];
                }
            }
            if (!ok) break;
            ++npc;
        }
        // on abort: let copies already in flight land before the CTA exits
        if (*abort) {
            for (int j = max(0, k_iss - kStages); j < k_iss; ++j)
                mbar_wait(&bars->k_full[j % kStages], (j / kStages) & 1, p.err, nullptr);
            for (int j = max(0, v_iss - kStages); j < v_iss; ++j)
                mbar_wait(&bars->v_full[j % kStages], (j / kStages) & 1, p.err, nullptr);
            if (q_pending > 0) mbar_wait(&bars->q_full, (q_pending - 1) & 1, p.err, nullptr);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA
        // the whole warp runs this loop (uniform control flow, operands in
        // uniform registers); one elected lane issues every tcgen05 op
        const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), SL::kChunkBytes, 1024);
        constexpr uint32_t kTileStep = SL::kTileBytes >> 4;  // one tile / stage in 16-byte units
        Walker w;
        w.init(p, bars, work);
        Piece pc;
        int jj = 0, npc = 0;
        int cnt[2] = {0, 0};  // tiles handed to each query tile's softmax so far
        int vl[kStages] = {0, 0};
        bool ok = true;
        while (ok && w.next(p, pc)) {
            const int nx = ((2 * pc.mp + 1) * npt < pc.s.B) ? 2 : 1;
            ok = mbar_wait_warp(&bars->q_full, npc & 1, p.err, abort) &&
                 mbar_wait_warp(&bars->k_full[jj % kStages], (jj / kStages) & 1, p.err, abort);
            if (!ok) break;
            tc_fence_after();
            for (int x = 0; x < nx; ++x) {
                issue_qk<D>(tmem + 256 * x, dq0 + x * kTileStep, dk0 + (jj % kStages) * kTileStep);
                commit_warp(&bars->s_full[x]);
            }
            commit_warp(&bars->k_empty[jj % kStages]);
            if (pc.nt == 1) commit_warp(&bars->q_empty);  // the piece's last QK is issued
            for (int j = 0; ok && j < pc.nt; ++j, ++jj) {
                const int st = jj % kStages;
                const bool more = j + 1 < pc.nt;
                const bool unit_final = pc.t0 + j == pc.T - 1;
                for (int x = 0; ok && x < nx; ++x) {
                    ok = mbar_wait_warp(&bars->p_full[x], cnt[x] & 1, p.err, abort);
                    if (ok && x == 0)
                        ok = unit_final ? mbar_wait_warp(&bars->v_last[st], vl[st] & 1, p.err, abort)
                                        : mbar_wait_warp(&bars->v_full[st], (jj / kStages) & 1, p.err, abort);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv<D>(tmem + 256 * x, dv0 + st * kTileStep, j > 0);
                    if (x == nx - 1) commit_warp(&bars->v_empty[st]);
                    if (!more) {
                        commit_warp(&bars->o_final[x]);
                    } else {
                        const int st1 = (jj + 1) % kStages;
                        if (x == 0) ok = mbar_wait_warp(&bars->k_full[st1], ((jj + 1) / kStages) & 1, p.err, abort);
                        if (!ok) break;
                        tc_fence_after();
                        issue_qk<D>(tmem + 256 * x, dq0 + x * kTileStep, dk0 + st1 * kTileStep);
                        commit_warp(&bars->s_full[x]);
                        if (x == nx - 1) commit_warp(&bars->k_empty[st1]);
                    }
                    ++cnt[x];
                }
                if (unit_final) ++vl[st];
                if (ok && j == pc.nt - 2) commit_warp(&bars->q_empty);  // the piece's last QK is issued
            }
            ++npc;
        }
        // every MMA issued above completes before TMEM is released
        commit_warp(&bars->mma_final);
        mbar_wait_warp(&bars->mma_final, 0, p.err, nullptr);
    } else {
        // ---------------------------------------------- softmax of tile X
        const int x = warp >> 2;
        const int r = tid & 127;  // query row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + 256 * x + lane_off, tO = tS + 128;
        const float sl2 = p.scale_log2;
        uint8_t* stage = smem + SL::kStage + warp * 4096;
        Walker w;
        w.init(p, bars, work);
        Piece pc;
        int cnt = 0, nfin = 0;
        // the tile's four softmax warps meet (bounded; one phase of msync
        // per meeting, and no warp can be a meeting ahead of another).  A
        // merge meets exactly twice, so meeting i of it completes a phase
        // of parity i.
        auto sync4 = [&](int i) -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->msync[x]);
            return mbar_wait_warp(&bars->msync[x], static_cast<uint32_t>(i), p.err, abort);
        };
        bool ok = true;
        while (ok && w.next(p, pc)) {
            if (x == 1 && (2 * pc.mp + 1) * npt >= pc.s.B) continue;  // tile B absent from this unit
            const int L = pc.s.L;
            const int n_end = min(pc.s.B, (2 * pc.mp + 2) * npt);
            const int node = (2 * pc.mp + x) * npt + r / p.G;
            const int head = pc.g * p.G + r % p.G;
            const bool valid_row = node < n_end;
            uint32_t a[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                a[k] = valid_row ? p.anc[static_cast<long long>(pc.s.off + node) * 8 + k] : 0u;
#ifdef JT_CHECKS
            if (valid_row) {  // a node's set holds the node itself and only nodes before it
                bool ok_set = true;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int lo = 32 * k;
                    const uint32_t allowed =
                        node >= lo + 31 ? 0xFFFFFFFFu : (node < lo ? 0u : (2u << (node - lo)) - 1u);
                    if (a[k] & ~allowed) ok_set = false;
                    if (node >= lo && node < lo + 32 && !((a[k] >> (node - lo)) & 1u)) ok_set = false;
                }
                JT_DCHECK(ok_set, p.err);
            }
#endif
            float m_run = -INFINITY, l_run = 0.0f;
            for (int j = 0; j < pc.nt; ++j, ++cnt) {
                if (!mbar_wait_warp(&bars->s_full[x], cnt & 1, p.err, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int slot0 = (pc.t0 + j) * kTileN;
                SRow sr;
                load_srow(tS, sr);
                if (slot0 + kTileN > L) mask_srow(sr, a, slot0 - L);  // tiles inside the prefix need no mask
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
            if (!ok) break;
            // epilogue of the piece (after the CTA's last piece the combine may
            // be scheduled; it waits for this grid)
            if (w.remaining <= 0) pdl_trigger();
            if (!mbar_wait_warp(&bars->o_final[x], nfin & 1, p.err, abort)) {
                ok = false;
                break;
            }
            ++nfin;
            tc_fence_after();
            piece_output<D>(p, pc, bars, work, x, r, lane, node, head, valid_row, tO, stage, m_run, l_run, sync4);
            // O_X has been read (tcgen05.wait::ld above) before this thread
            // arrives on p_full[X] for the next piece's first tile, which is
            // what lets the MMA warp overwrite O_X
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ===========================================================================
// CTA-pair kernel (D = 128)
//
// The two CTAs of a cluster (a pair, on two SMs) run one work slot: CTA
// rank X takes query tile X of each unit, and one tcgen05.mma.cta_group::2
// of M = 256 covers both tiles, issued by CTA 0 (the leader).  Each CTA
// holds its half of every K tile (keys 64X..64X+63, all 128 dims) and of
// every V tile (all 128 keys, dims 64X..64X+63); the MMA reads B's halves
// from both CTAs, so a unit's K/V cross HBM and shared memory once while
// each SM's tensor core does the MMAs of its own 128 rows.  Against the
// single-SM kernel this halves each SM's K/V operand reads per MMA (a
// quarter of its shared-memory reads) and leaves room in TMEM for three S
// buffers: per CTA S0, S1, S2 (128 columns each) and O (128).  MMAs from
// one thread run in issue order, and QK(t) may overwrite S(t mod 3) only
// after PV(t-3) has read P(t-3) from it.  Softmax releases P(t) without
// waiting for PV(t-1) (O is rescaled only when a row's maximum grows by
// more than 2^32, and only then does the softmax wait for that PV), so the
// tensor core scores tiles up to three ahead of the softmax and never
// waits for it in between.
//
// Warp roles (224 threads per CTA):
//   warps 0-3  softmax + epilogue of this CTA's query tile, one row per
//              thread (TMEM lane);
//   warp 4     planner, then TMA producer of this CTA's Q tile and K halves
//              (the leader's barriers count both CTAs' bytes);
//   warp 5     TMEM allocation; in the leader, the single-thread MMA issuer;
//   warp 6     TMA producer of this CTA's V halves.
// Issue order per piece: QK(0), QK(1), QK(2), then per tile j: PV(j),
// QK(j+3) (later, when its K lands late).  Per tile the eight softmax
// warps of the pair arrive on the leader's p_full[j mod 3]; S(t) needs
// PV(t-3) issued, so neither CTA's softmax runs more than two tiles ahead
// of the other's.  PV(t) commits a phase of o_done[t mod 3]: when a warp
// waits for PV(t-1) (a rescale at tile t) or for the piece's last PV,
// PV(t-4) (resp. the one three before the last) has completed, S(t)
// having, and the next PV on that barrier is not issued (it needs this
// warp's P), so that barrier is within one phase of the wait.
// ===========================================================================
constexpr int kPairThreads = 224;
constexpr int kPairKStages = 6;  // K ring depth (half tiles): a K slot frees at QK, early
constexpr int kPairVStages = 4;  // V ring depth (half tiles): a V slot frees at PV
// Lazy rescaling threshold of the pair kernel (log2 units): O is rescaled
// only when a row's running maximum grows by more than this.  Until then P
// = exp2(s - m) stays below 2^32 and O and the row sum below ~2^60 times
// their values: far inside fp32 and bf16 range, with no loss of relative
// precision.
constexpr float kPairRescaleLog2 = 32.0f;

struct PairSmem {
    static constexpr int kQChunk = kTileM * 128;  // 128 query rows x 64 dims
    static constexpr int kQBytes = 2 * kQChunk;
    static constexpr int kKChunk = 64 * 128;      // 64 keys x 64 dims
    static constexpr int kKHalf = 2 * kKChunk;    // this CTA's 64 keys x 128 dims
    static constexpr int kVHalf = kTileN * 128;   // 128 keys x this CTA's 64 dims
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kQBytes;
    static constexpr int kV = kK + kPairKStages * kKHalf;
    static constexpr int kStage = kV + kPairVStages * kVHalf;  // epilogue staging, 4 KB per softmax warp
    static constexpr int kBar = kStage + 4 * 4096;
    static constexpr int kBytes = kBar + 512;
    static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};

struct PairBars {
    uint64_t q_full;                // leader: both CTAs' Q tiles have landed
    uint64_t q_empty;               // every QK of the piece has completed
    uint64_t k_full[kPairKStages];   // leader: both halves of the stage's K tile have landed
    uint64_t k_empty[kPairKStages];  // QK of the stage's tile has completed
    uint64_t v_full[kPairVStages];   // leader: both halves of the stage's V tile have landed
    uint64_t v_empty[kPairVStages];  // PV of the stage's tile has completed
    uint64_t v_own[kPairVStages];    // this CTA's half of a unit-final V tile has landed
    uint64_t v_last[kPairVStages];   // leader: both halves of a unit-final V tile are zero-filled
    uint64_t s_full[3];             // S buffer X holds QK of its latest tile
    uint64_t p_full[3];             // leader: P of the tile in S buffer X, from the pair's 8 softmax warps
    uint64_t o_done[3];             // one phase per PV of a tile t with t mod 3 == X
    uint64_t mma_final;             // every MMA of the pair has completed
    uint32_t tmem_base;
    int abort;
    int w_b, w_g, w_mp, w_t, w_quota, w_P;
    uint32_t call_id;
    int merge_flag[2];
    uint64_t msync[2];  // this CTA's four softmax warps meet (merge of a cut unit)
};
static_assert(sizeof(PairBars) <= 512, "barrier block");

__device__ __forceinline__ void commit_pair_warp(uint64_t* bar) {
    if (elect_one()) mma_commit_pair(bar);
    __syncwarp();
}

// S (+)= Q K^T over the pair: 8 MMAs of M = 256, N = 128, K = 16.
__device__ __forceinline__ void issue_qk_pair(uint32_t tS, uint64_t dq, uint64_t dk) {
    constexpr uint32_t idesc = idesc_bf16_f32(2 * kTileM, kTileN, false);
    if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t qo = ((kk >> 2) * PairSmem::kQChunk + (kk & 3) * 32) >> 4;
            const uint32_t ko = ((kk >> 2) * PairSmem::kKChunk + (kk & 3) * 32) >> 4;
            mma_ss_pair(tS, dq + qo, dk + ko, idesc, kk > 0 ? 1u : 0u);
        }
    }
    __syncwarp();
}

// O (+)= P V over the pair, P (bf16 pairs) in the first 64 columns of an S
// buffer: 8 MMAs of M = 256, N = 128, K = 16.
__device__ __forceinline__ void issue_pv_pair(uint32_t tO, uint32_t tP, uint64_t dv, bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16_f32(2 * kTileM, 128, true);
    if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
            mma_ts_pair(tO, tP + kk * 8, dv + kk * ((16 * 128) >> 4), idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
    __syncwarp();
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    tree_attn_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
    constexpr int D = 128;
    using SL = PairSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    PairBars* bars = reinterpret_cast<PairBars*>(smem + SL::kBar);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();  // 0: the leader, which issues the pair's MMAs
    const int work = static_cast<int>(blockIdx.x >> 1), nwork = static_cast<int>(gridDim.x >> 1);
    if (tid == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int s = 0; s < kPairKStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < kPairVStages; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
            mbar_init(&bars->v_own[s], 1);
            mbar_init(&bars->v_last[s], 2);
        }
        for (int x = 0; x < 3; ++x) {
            mbar_init(&bars->s_full[x], 1);
            mbar_init(&bars->p_full[x], 8);
            mbar_init(&bars->o_done[x], 1);
        }
        for (int x = 0; x < 2; ++x) mbar_init(&bars->msync[x], 4);
        mbar_init(&bars->mma_final, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 5) tmem_alloc_pair(&bars->tmem_base, 512);
    cluster_sync();  // both CTAs' barriers exist before any copy, commit or arrive crosses the pair
    pdl_wait();
    if (warp == 4) {
        const bool rec = work == 0 && rank == 0;
        if (p.splits > 0)
            plan_cta_split(p, bars, lane, work, rec);
        else
            plan_cta(p, bars, lane, work, nwork, rec);
    }
    if (tid == 0) bars->call_id = draw_call_id(p.tickets, work == 0 && rank == 0, gridDim.x);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    volatile int* abort = &bars->abort;
    const bool has_work = bars->w_quota > 0;  // the same in both CTAs: one plan per work slot

    uint8_t* sQ = smem + SL::kQ;
    uint8_t* sK = smem + SL::kK;
    uint8_t* sV = smem + SL::kV;
    const int npt = p.npt;

    if (!has_work) {
        // nothing issued: both CTAs go straight to the teardown
    } else if (warp == 4 || warp == 6) {
        // ------------------------------------------------------------ TMA
        // warp 4: Q and K, warp 6: V.  Each walks the pieces on its own, so
        // K copies run ahead of V's (a K slot frees at QK, a V slot at PV).
        const bool kw = warp == 4;
        const int nst = kw ? kPairKStages : kPairVStages;
        Walker w;
        w.init(p, bars, work);
        Piece pc;
        int jj = 0, npc = 0, q_pending = 0;
        int iss = 0;  // tiles whose copies this warp has issued
        int vo[kPairVStages] = {0, 0, 0, 0};
        const uint32_t lead_q = cluster_map(&bars->q_full, 0);
        bool ok = true;
        while (ok && !*abort && w.next(p, pc)) {
            const int valid_end = unit_end(pc.s, pc.mp, npt);
            if (kw) {
                // Q of this piece (this CTA's tile; the peer's tile may lie
                // past the tree: its rows are then never written out)
                if (npc > 0 && !mbar_wait_warp(&bars->q_empty, (npc - 1) & 1, p.err, abort)) break;
                if (lane == 0) {
                    if (rank == 0) mbar_arrive_expect_tx(&bars->q_full, 2 * SL::kQBytes);
                    for (int c = 0; c < 2; ++c)
                        tma_load_3d_pair(sQ + c * SL::kQChunk, &tm_q, lead_q, c * 64, pc.g * p.G,
                                         pc.s.off + (2 * pc.mp + static_cast<int>(rank)) * npt);
                }
                q_pending = npc + 1;
            }
            int bt_cur = bt_group(p, pc, valid_end, 0, lane);
            int bt_nxt = bt_group(p, pc, valid_end, 1, lane);
            int bt_nn = bt_group(p, pc, valid_end, 2, lane);
            for (int j = 0; j < pc.nt; ++j, ++jj) {
                const int st = jj % nst;
                const uint32_t empty_parity = ((jj / nst) & 1) ^ 1;
                if (j > 0 && (j & 3) == 0) {
                    bt_cur = bt_nxt;
                    bt_nxt = bt_nn;
                    bt_nn = bt_group(p, pc, valid_end, (j >> 2) + 2, lane);
                }
                const int slot0 = (pc.t0 + j) * kTileN;
                const int nvalid = min(kTileN, valid_end - slot0);
                const int npg = (nvalid + JT_PAGE_SIZE - 1) / JT_PAGE_SIZE;
                const int pid = __shfl_sync(0xFFFFFFFFu, bt_cur, ((j & 3) << 3) + (lane & 7));
                JT_DCHECK(lane >= npg || (pid >= 0 && pid < p.num_pages), p.err);  // block-table entry in the pool
                const uint32_t bytes = npg * 2 * (JT_PAGE_SIZE * 128);  // both CTAs' halves
                if (kw) {
                    // K: this CTA's 64 keys (pages 4X..4X+3 of the tile), both
                    // 64-dim chunks; the slot frees once QK of tile jj - nst is done
                    if (jj >= nst && !mbar_wait_warp(&bars->k_empty[st], empty_parity, p.err, abort)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0 && rank == 0) mbar_arrive_expect_tx(&bars->k_full[st], bytes);
                    __syncwarp();
                    if (lane < npg && (lane >> 2) == static_cast<int>(rank)) {
                        const uint32_t lead = cluster_map(&bars->k_full[st], 0);
                        for (int c = 0; c < 2; ++c)
                            tma_load_4d_pair(sK + st * SL::kKHalf + c * SL::kKChunk + (lane & 3) * (JT_PAGE_SIZE * 128),
                                             &tm_k, lead, c * 64, pc.g, 0, pid);
                    }
                    iss = jj + 1;
                    continue;
                }
                // V: this CTA's 64 dims of every key; the slot frees once PV
                // of tile jj - nst is done
                if (jj >= nst && !mbar_wait_warp(&bars->v_empty[st], empty_parity, p.err, abort)) {
                    ok = false;
                    break;
                }
                uint8_t* vt = sV + st * SL::kVHalf;
                if (pc.t0 + j != pc.T - 1) {
                    if (lane == 0 && rank == 0) mbar_arrive_expect_tx(&bars->v_full[st], bytes);
                    __syncwarp();
                    if (lane < npg)
                        tma_load_4d_pair(vt + lane * (JT_PAGE_SIZE * 128), &tm_v, cluster_map(&bars->v_full[st], 0),
                                         static_cast<int>(rank) * 64, pc.g, 0, pid);
                } else {
                    // the unit's final tile: each CTA lands its half on its
                    // own barrier, zeroes the rows past the last needed slot
                    // (stale or foreign data: P is 0 there but 0 * NaN would
                    // not be) and reports to the leader's v_last; the
                    // leader's v_full phase of this tile completes empty
                    if (lane == 0) {
                        if (rank == 0) mbar_arrive(&bars->v_full[st]);
                        mbar_arrive_expect_tx(&bars->v_own[st], npg * (JT_PAGE_SIZE * 128));
                    }
                    __syncwarp();
                    if (lane < npg)
                        tma_load_4d(vt + lane * (JT_PAGE_SIZE * 128), &tm_v, &bars->v_own[st],
                                    static_cast<int>(rank) * 64, pc.g, 0, pid);
                    if (!mbar_wait_warp(&bars->v_own[st], vo[st] & 1, p.err, abort)) {
                        ok = false;
                        break;
                    }
                    ++vo[st];
                    const int n16 = (kTileN - nvalid) * 8;  // 16-byte pieces
                    for (int idx = lane; idx < n16; idx += 32)
                        reinterpret_cast<uint4*>(vt + (nvalid + (idx >> 3)) * 128)[idx & 7] = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(cluster_map(&bars->v_last[st], 0));
                }
                iss = jj + 1;
            }
            if (!ok) break;
            ++npc;
        }
        // on abort: the leader lets the copies it counted land before the
        // pair exits (the peer's copies report to the leader's barriers)
        if (*abort && rank == 0) {
            uint64_t* full = kw ? bars->k_full : bars->v_full;
            for (int j = max(0, iss - nst); j < iss; ++j) mbar_wait(&full[j % nst], (j / nst) & 1, p.err, nullptr);
            if (kw && q_pending > 0) mbar_wait(&bars->q_full, (q_pending - 1) & 1, p.err, nullptr);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA
        if (rank == 0) {
            const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), SL::kVHalf, 1024);
            Walker w;
            w.init(p, bars, work);
            Piece pc;
            int jj = 0, npc = 0;
            int vl[kPairVStages] = {0, 0, 0, 0};
            bool ok = true;
            while (ok && w.next(p, pc)) {
                ok = mbar_wait_warp(&bars->q_full, npc & 1, p.err, abort);
                const int j0 = jj;
                int issued = 0;  // QKs of this piece issued
                // QK of the piece's next tile; block: wait for its K, else
                // return false when K has not landed yet
                auto qk_next = [&](bool block) -> bool {
                    const int t = j0 + issued, st = t % kPairKStages;
                    const uint32_t par = (t / kPairKStages) & 1;
                    if (block) {
                        if (!mbar_wait_warp(&bars->k_full[st], par, p.err, abort)) {
                            ok = false;
                            return false;
                        }
                    } else if (!__all_sync(0xFFFFFFFFu, mbar_try_wait(&bars->k_full[st], par))) {
                        return false;
                    }
                    tc_fence_after();
                    issue_qk_pair(tmem + 128 * (t % 3), dq0, dk0 + st * (SL::kKHalf >> 4));
                    commit_pair_warp(&bars->s_full[t % 3]);
                    commit_pair_warp(&bars->k_empty[st]);
                    if (++issued == pc.nt) commit_pair_warp(&bars->q_empty);  // the piece's last QK
                    return true;
                };
                while (ok && issued < min(3, pc.nt)) qk_next(true);
                for (int j = 0; ok && j < pc.nt; ++j, ++jj) {
                    const int st = jj % kPairVStages, b = jj % 3;
                    const bool unit_final = pc.t0 + j == pc.T - 1;
                    ok = mbar_wait_warp(&bars->p_full[b], (jj / 3) & 1, p.err, abort);
                    if (ok)
                        ok = unit_final ? mbar_wait_warp(&bars->v_last[st], vl[st] & 1, p.err, abort)
                                        : mbar_wait_warp(&bars->v_full[st], (jj / kPairVStages) & 1, p.err, abort);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv_pair(tmem + 384, tmem + 128 * b, dv0 + st * (SL::kVHalf >> 4), j > 0);
                    commit_pair_warp(&bars->o_done[b]);
                    commit_pair_warp(&bars->v_empty[st]);
                    if (unit_final) ++vl[st];
                    // S(j mod 3) is free for QK(j + 3) once PV(j) is issued.
                    // QK(j + 1) must be on its way before P(j + 1) is awaited;
                    // later QKs go now only if their K has landed, so that a
                    // late K never holds back the next PV
                    while (ok && issued < min(j + 4, pc.nt))
                        if (!qk_next(issued > j + 1 ? false : true)) break;
                }
                ++npc;
            }
            commit_pair_warp(&bars->mma_final);
        }
        // both CTAs: every MMA of the pair has completed before TMEM is released
        mbar_wait_warp(&bars->mma_final, 0, p.err, nullptr);
    } else {
        // ------------------------------------------- softmax of this CTA's tile
        const int x = static_cast<int>(rank);
        const int r = tid;  // query row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tO = tmem + 384 + lane_off;
        const float sl2 = p.scale_log2;
        uint8_t* stage = smem + SL::kStage + warp * 4096;
        const uint32_t lead_p[3] = {cluster_map(&bars->p_full[0], 0), cluster_map(&bars->p_full[1], 0),
                                    cluster_map(&bars->p_full[2], 0)};
        Walker w;
        w.init(p, bars, work);
        Piece pc;
        int cnt = 0;  // tiles of this work slot so far (the pair's global tile count)
        // the tile's four softmax warps meet (bounded; one phase of msync
        // per meeting, and no warp can be a meeting ahead of another).  A
        // merge meets exactly twice, so meeting i of it completes a phase
        // of parity i.
        auto sync4 = [&](int i) -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->msync[x]);
            return mbar_wait_warp(&bars->msync[x], static_cast<uint32_t>(i), p.err, abort);
        };
        bool ok = true;
        while (ok && w.next(p, pc)) {
            const bool active = (2 * pc.mp + x) * npt < pc.s.B;  // this CTA's query tile exists
            const int L = pc.s.L;
            const int n_end = min(pc.s.B, (2 * pc.mp + 2) * npt);
            const int node = (2 * pc.mp + x) * npt + r / p.G;
            const int head = pc.g * p.G + r % p.G;
            const bool valid_row = node < n_end;
            uint32_t a[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                a[k] = valid_row ? p.anc[static_cast<long long>(pc.s.off + node) * 8 + k] : 0u;
#ifdef JT_CHECKS
            if (valid_row) {  // a node's set holds the node itself and only nodes before it
                bool ok_set = true;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int lo = 32 * k;
                    const uint32_t allowed =
                        node >= lo + 31 ? 0xFFFFFFFFu : (node < lo ? 0u : (2u << (node - lo)) - 1u);
                    if (a[k] & ~allowed) ok_set = false;
                    if (node >= lo && node < lo + 32 && !((a[k] >> (node - lo)) & 1u)) ok_set = false;
                }
                JT_DCHECK(ok_set, p.err);
            }
#endif
            float m_run = -INFINITY, l_run = 0.0f;
            for (int j = 0; j < pc.nt; ++j, ++cnt) {
                const int b = cnt % 3;
                const uint32_t tS = tmem + 128 * b + lane_off;
                if (!mbar_wait_warp(&bars->s_full[b], (cnt / 3) & 1, p.err, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (active) {
                    const int slot0 = (pc.t0 + j) * kTileN;
                    SRow sr;
                    load_srow(tS, sr);
                    if (slot0 + kTileN > L) mask_srow(sr, a, slot0 - L);  // tiles inside the prefix need no mask
                    const float mx = max_srow8(sr);
                    const float mx_s = mx * sl2;
                    bool resc = false;
                    float factor = 1.0f;
                    if (mx_s > m_run + kPairRescaleLog2 || m_run == -INFINITY) {
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
                        // O holds PV(cnt - 1) before it is rescaled
                        if (!mbar_wait_warp(&bars->o_done[(cnt - 1) % 3], ((cnt - 1) / 3) & 1, p.err, abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        {
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
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(lead_p[b]);
            }
            if (!ok || !active) continue;
            // epilogue of the piece (after the last piece the combine may be
            // scheduled; it waits for this grid): PV(cnt - 1), the piece's
            // last, has completed
            if (w.remaining <= 0) pdl_trigger();
            if (!mbar_wait_warp(&bars->o_done[(cnt - 1) % 3], ((cnt - 1) / 3) & 1, p.err, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            piece_output<D>(p, pc, bars, work, x, r, lane, node, head, valid_row, tO, stage, m_run, l_run, sync4);
            // O has been read (tcgen05.wait::ld) before this thread releases
            // P of the next piece's first tile, whose PV overwrites O
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no copy, arrive or MMA of the pair targets either CTA any more
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

// Split mode: merge the key splits of every unit cut into more than one.
// Grid (units, 32): blockIdx.y picks 8 of the unit's 256 query rows, one
// warp per row; lane k holds split k's (m, l), each lane D/32 columns of O.
constexpr int kCombineThreads = 256;
constexpr int kCombineRowBlocks = 2 * kTileM / (kCombineThreads / 32);

template <int D>
__global__ void __launch_bounds__(kCombineThreads)
    tree_attn_combine_kernel(const AttnParams p) {
    constexpr int kCols = D / 32;
    pdl_wait();  // the partials are complete and visible
    const int u = blockIdx.x;
    const int b = u / (p.Hkv * p.npairs);
    const int rem = u % (p.Hkv * p.npairs);
    const int g = rem / p.npairs, mp = rem % p.npairs;
    if (b >= p.nseq) return;
    const SeqInfo s = load_seq(p, b);
    if (mp >= s.np) return;
    const int T = unit_tiles(s, mp, p.npt);
    const int tps = split_tiles(T, p.splits);
    const int nsp = (T + tps - 1) / tps;  // non-empty splits
    if (nsp <= 1) return;                 // the whole unit was one split: written directly
    const int row = blockIdx.y * (kCombineThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int x = row / kTileM, r = row % kTileM;
    if (x == 1 && (2 * mp + 1) * p.npt >= s.B) return;  // tile B absent
    const int node = (2 * mp + x) * p.npt + r / p.G;
    if (node >= min(s.B, (2 * mp + 2) * p.npt)) return;
    const int head = g * p.G + r % p.G;
    auto prow = [&](int k) {  // partial row of split k (slot 2 * CTA)
        return (static_cast<long long>(2 * (u * p.splits + k)) * 2 + x) * kTileM + r;
    };
    // lane k: split k's running max and sum (nsp <= 32)
    const float2 ml = (lane < nsp) ? p.part_ml[prow(lane)] : make_float2(-INFINITY, 0.0f);
    float M = ml.x;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    const float w = (ml.x == -INFINITY) ? 0.0f : exp2f(ml.x - M);
    float lsum = w * ml.y;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o);
    float acc[kCols];
#pragma unroll
    for (int q = 0; q < kCols; ++q) acc[q] = 0.0f;
    for (int k0 = 0; k0 < nsp; k0 += 8) {  // eight splits' loads in flight
        float v[8][kCols];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = k0 + i;
            const float* po = p.part_o + prow(k < nsp ? k : 0) * D + lane * kCols;
#pragma unroll
            for (int q = 0; q < kCols; ++q) v[i][q] = (k < nsp) ? po[q] : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float wk = __shfl_sync(0xFFFFFFFFu, w, (k0 + i) & 31);
            if (k0 + i < nsp)
#pragma unroll
                for (int q = 0; q < kCols; ++q) acc[q] += wk * v[i][q];
        }
    }
    const float inv = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;
    const long long rowid = static_cast<long long>(s.off + node) * p.Hq + head;
    __nv_bfloat16* dst = p.out + rowid * D + lane * kCols;
#pragma unroll
    for (int q = 0; q < kCols; q += 2)
        *reinterpret_cast<uint32_t*>(dst + q) = pack_bf16x2(acc[q] * inv, acc[q + 1] * inv);
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

// Whether a D = 128 call runs the CTA-pair kernel.  By default when every
// (sequence, KV head) has one query-tile pair at max_tree (npairs == 1):
// then both kernels read each K/V byte once and the pair kernel spends two
// SMs on each unit.  With several pairs per head the pairs of one head share
// their K/V through L2, which the single-SM kernel's twice as many work
// slots keep better (measured on the serving and verify-step batches).  The
// environment variable JT_ATTN_KERNEL = "pair" or "single" overrides the
// choice; D = 64 always runs the single-SM kernel.
static bool pair_kernel_selected(int npairs) {
    const char* v = std::getenv("JT_ATTN_KERNEL");
    if (v && std::strcmp(v, "pair") == 0) return true;
    if (v && std::strcmp(v, "single") == 0) return false;
    return npairs == 1;
}

// Work slots of the CTA-pair kernel on the current device: the clusters of
// two CTAs that can be resident at once (one CTA per SM).
static int pair_work_slots() {
    static PerDeviceCache cache;
    return cache.get([] {
        const int fallback = device_sm_count() / 2;
        if (cudaFuncSetAttribute(tree_attn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairSmem::kAlloc) != cudaSuccess)
            return fallback;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * std::max(1, fallback));
        cfg.blockDim = dim3(kPairThreads);
        cfg.dynamicSmemBytes = PairSmem::kAlloc;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tree_attn_pair_kernel, &cfg) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            return fallback;
        }
        return n;
    });
}

AttnPlan attn_plan(int nseq, int Hkv, int Hq, int D, int max_tree, int max_pages, int dtype) {
    AttnPlan pl;
    const int G = Hq / Hkv;
    pl.rows_per_tile_nodes = kTileM / G;
    pl.mtiles = (max_tree + pl.rows_per_tile_nodes - 1) / pl.rows_per_tile_nodes;
    pl.grid = 0;
    pl.work = 0;
    pl.pair = 0;
    pl.nseq = nseq;
    pl.npairs = (pl.mtiles + 1) / 2;
    pl.splits = 0;
    if (dtype == JT_DTYPE_BF16) {
        pl.pair = (D == 128 && pair_kernel_selected(pl.npairs)) ? 1 : 0;
        // one work slot per SM (single-SM kernel) or per resident CTA pair,
        // every one the same tile count
        const int slots = pl.pair ? pair_work_slots() : device_sm_count();
        pl.work = slots;
        // Few units (at most half the slots): split mode, each unit's keys
        // split over slots / units work slots (at most one split per two key
        // tiles) and merged by the combine kernel.
        const long long units = static_cast<long long>(nseq) * Hkv * pl.npairs;
        const int tmax = (max_pages * JT_PAGE_SIZE + kTileN - 1) / kTileN;
        if (units > 0 && 2 * units <= slots) {
            int sp = static_cast<int>(slots / units);
            sp = std::min(sp, std::max(1, tmax / 2));
            sp = std::min(sp, 32);
            if (sp >= 2) {
                pl.splits = sp;
                pl.work = static_cast<int>(units) * sp;
            }
        }
        pl.grid = pl.pair ? 2 * pl.work : pl.work;
    }
    return pl;
}

// Workspace of the bf16 path after the header: the merge counts of cut
// units (two per work slot; like the header they must be zero before the
// workspace's first use, and stay valid across calls), the plan (T_total, P,
// the first global tile of each sequence), then two partial slots per work
// slot.
static size_t attn_cnt_bytes(const AttnPlan& p) { return align_up(static_cast<size_t>(p.work) * 2 * 8); }
static size_t attn_plan_bytes(const AttnPlan& p) { return align_up(static_cast<size_t>(p.nseq + 3) * sizeof(int)); }
static size_t attn_ml_bytes(const AttnPlan& p) {
    return align_up(static_cast<size_t>(2) * p.work * 2 * kTileM * sizeof(float2));
}

size_t attn_workspace_bytes(const AttnPlan& p, int total_nodes, int Hq, int D) {
    (void)total_nodes;
    (void)Hq;
    size_t b = kWsHeader;
    if (p.grid > 0)
        b += attn_cnt_bytes(p) + attn_plan_bytes(p) + attn_ml_bytes(p) +
             align_up(static_cast<size_t>(2) * p.work * 2 * kTileM * D * sizeof(float));
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
    if (plan.grid < 1) return cudaErrorInvalidValue;
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
    char* w = ws_parts;
    prm.merge_cnt = reinterpret_cast<unsigned long long*>(w);
    w += attn_cnt_bytes(plan);
    prm.plan = reinterpret_cast<int*>(w);
    w += attn_plan_bytes(plan);
    prm.part_ml = reinterpret_cast<float2*>(w);
    w += attn_ml_bytes(plan);
    prm.part_o = reinterpret_cast<float*>(w);
    prm.tickets = &reinterpret_cast<WsHeader*>(err)->tickets;
    prm.err = err;
    prm.max_pages = max_pages;
    prm.num_pages = num_pages;
    prm.nseq = nseq;
    prm.total_nodes = total_nodes;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = G;
    prm.npt = plan.rows_per_tile_nodes;
    prm.splits = plan.splits;
    prm.npairs = plan.npairs;
    prm.scale_log2 = scale * 1.4426950408889634f;

    cudaError_t e;
    if (plan.pair) {
        if (D != 128) return cudaErrorInvalidValue;
        static PerDeviceCache attr;  // the shared-memory opt-in is per device
        const cudaError_t ea = static_cast<cudaError_t>(attr.get([] {
            return static_cast<int>(cudaFuncSetAttribute(
                tree_attn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PairSmem::kAlloc));
        }));
        if (ea != cudaSuccess) return ea;
        e = launch_kernel_pdl(tree_attn_pair_kernel, dim3(plan.grid), dim3(kPairThreads), PairSmem::kAlloc, st, tq,
                              tk, tv, prm);
    } else {
        using SL = SmemLayout<D>;
        static PerDeviceCache attr;
        const cudaError_t ea = static_cast<cudaError_t>(attr.get([] {
            return static_cast<int>(cudaFuncSetAttribute(tree_attn_tc_kernel<D>,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SL::kAlloc));
        }));
        if (ea != cudaSuccess) return ea;
        e = launch_kernel_pdl(tree_attn_tc_kernel<D>, dim3(plan.grid), dim3(kAttnThreads), SL::kAlloc, st, tq, tk,
                              tv, prm);
    }
    if (e != cudaSuccess || plan.splits == 0) return e;
    return launch_kernel_pdl(tree_attn_combine_kernel<D>, dim3(plan.work / plan.splits, kCombineRowBlocks),
                             dim3(kCombineThreads), 0, st, prm);
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
