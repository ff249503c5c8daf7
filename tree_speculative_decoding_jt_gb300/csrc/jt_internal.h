// jt_internal.h -- declarations shared between the host API (jt_api.cu) and
// the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "../../include/jt.h"

// NVTX ranges around every extern "C" entry point, compiled in with
// -DJT_NVTX (header-only NVTX v3: nothing is linked, and the ranges cost a
// branch when no profiler is attached); compiled out by default.
#ifdef JT_NVTX
#include <nvtx3/nvToolsExt.h>
namespace jt {
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace jt
#define JT_RANGE(name) ::jt::NvtxRange jt_nvtx_range_(name)
#else
#define JT_RANGE(name) ((void)0)
#endif

namespace jt {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

// Workspace header (first kAlign bytes of every workspace).
struct WsHeader {
    uint32_t err;                // device error flags (DEVERR_*)
    uint32_t reserved;
    unsigned long long tickets;  // attention: CTA arrivals over all calls (call number = tickets / grid)
};
constexpr size_t kWsHeader = kAlign;

// tree_build.cu
// ent: room for the entropy partials of the mixed build
size_t topw_workspace_bytes(long long rows, long long V, int W, bool ent = false);
cudaError_t tree_topw_launch(const float* z, long long rows, long long V, int W, int32_t* tok,
                             double* lp, double* lse, char* ws_parts, cudaStream_t st);
cudaError_t tree_build_launch(const float* z, const int32_t* root_token, const int32_t* tree_off,
                              int nseq, int total_nodes, int N, int W, long long V, double alpha,
                              int32_t* parent, int32_t* token, int32_t* depth, uint32_t* anc, char* ws_parts,
                              uint32_t* err, cudaStream_t st);
// w_cap / n_cap: optional per-sequence width and depth caps (nullptr = none)
cudaError_t tree_expand_launch(const int32_t* tok, const double* lp, const int32_t* root_token,
                               const int32_t* tree_off, const int32_t* w_cap, const int32_t* n_cap, int nseq,
                               int total_nodes, int N, int W, int32_t* parent, int32_t* token, int32_t* depth,
                               uint32_t* anc, uint32_t* err, cudaStream_t st);
cudaError_t tree_policy_launch(const double* lp, int nseq, int N, int W, const int32_t* accept_len,
                               const jt_policy_params& prm, int32_t* budget_state, double* acc_ema,
                               int32_t* tree_off, int32_t* w_cap, int32_t* n_cap, uint32_t* err,
                               cudaStream_t st);
cudaError_t tree_build_adaptive_launch(const float* z, const int32_t* root_token, int nseq, int capacity, int N,
                                       int W, long long V, const int32_t* accept_len, const jt_policy_params& prm,
                                       int32_t* budget_state, double* acc_ema, int32_t* tree_off, int32_t* w_cap,
                                       int32_t* n_cap, int32_t* parent, int32_t* token, int32_t* depth,
                                       uint32_t* anc, char* ws_parts, uint32_t* err, cudaStream_t st);

// verify_accept.cu
size_t accept_workspace_bytes(int nseq, int total_nodes);
cudaError_t verify_accept_launch(const float* z, const int32_t* parent, const int32_t* token,
                                 const int32_t* tree_off, int nseq, int N, long long V,
                                 int total_nodes, int rule, double log_t, int32_t* accept_len,
                                 int32_t* path, int32_t* bonus, char* ws, cudaStream_t st);

// verify_stochastic.cu
cudaError_t verify_stochastic_launch(const float* z, const float* zd, const int32_t* parent,
                                     const int32_t* token, const int32_t* tree_off, int nseq, int N,
                                     long long V, int total_nodes, const double* u_accept,
                                     const double* u_bonus, int32_t* accept_len, int32_t* path,
                                     int32_t* bonus, char* ws, cudaStream_t st);

// tree_attn.cu / tree_attn_f32.cu
struct AttnPlan {
    int grid;        // CTAs of the bf16 kernel (0 on the fp32 path)
    int work;        // work slots: one per CTA, or one per CTA pair (pair != 0)
    int pair;        // the CTA-pair kernel (D = 128): two CTAs per work slot
    int nseq;
    int mtiles;      // row tiles per (sequence, kv head) at max_tree
    int rows_per_tile_nodes;  // tree nodes per 128-row tile (128 / G)
    int splits;      // > 0: split mode, one work slot per (unit, key split); 0: equal tile ranges per slot
    int npairs;      // query-tile pairs per (sequence, KV head) at max_tree
};
AttnPlan attn_plan(int nseq, int Hkv, int Hq, int D, int max_tree, int max_pages, int dtype);
size_t attn_workspace_bytes(const AttnPlan& p, int total_nodes, int Hq, int D);
cudaError_t tree_attn_bf16_launch(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, int max_pages, int num_pages,
                                  const int32_t* prefix_len, const int32_t* tree_off,
                                  const uint32_t* anc, int nseq, int total_nodes, int Hq, int Hkv,
                                  int D, float scale, void* out, float* lse, const AttnPlan& plan,
                                  char* ws_parts, uint32_t* err, cudaStream_t st);
cudaError_t tree_attn_f32_launch(const float* q, const float* k_cache, const float* v_cache,
                                 const int32_t* block_table, int max_pages, int num_pages,
                                 const int32_t* prefix_len, const int32_t* tree_off,
                                 const uint32_t* anc, int nseq, int total_nodes, int Hq, int Hkv,
                                 int D, float scale, float* out, float* lse, uint32_t* err,
                                 cudaStream_t st);

// jt_selftest.cu
cudaError_t selftest_wait_timeout_launch(uint32_t* err, cudaStream_t st);

int device_sm_count();

// One-time set-up remembered per device.  Kernel attributes
// (cudaFuncSetAttribute) and occupancy answers belong to the device that was
// current when they were set or asked, so a process that drives several
// devices must redo them on each; get() runs `compute` the first time the
// current device asks (per key) and returns the stored value afterwards.
// Thread-safe.  Where no device can be named the value is computed afresh.
constexpr int kMaxDevices = 64;
class PerDeviceCache {
  public:
    template <typename F>
    int get(F compute, long long key = 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return compute();
        std::lock_guard<std::mutex> lk(mu_);
        Slot& s = slot_[dev];
        if (!s.set || s.key != key) {
            s.val = compute();
            s.key = key;
            s.set = true;
        }
        return s.val;
    }

  private:
    struct Slot {
        bool set = false;
        long long key = 0;
        int val = 0;
    };
    std::mutex mu_;
    Slot slot_[kMaxDevices];
};

}  // namespace jt
