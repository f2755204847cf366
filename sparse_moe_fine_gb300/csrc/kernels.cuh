// Internal launch interfaces between the ABI layer and the kernel files.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace usaf {

constexpr int PERM_CHUNK = 256;

// ---------------------------------------------------------------- routing
struct RouteWs {
  float* logits;        // [T,E] when the caller gives no logits_out
  int32_t* chunk_hist;  // [nchunks, E]
  void* wr3;            // [E, 3H] bf16 split of the router weight (tensor-core logits)
};
void route_ws_layout(const usaf_moe_shape& s, Carver& c, RouteWs& w);
usaf_status route_launch(const usaf_moe_shape& s, const void* x, usaf_dtype xdt, const float* wr,
                         const float* logits_in, float* logits_out, int renorm,
                         const usaf_routing& rt, RouteWs& w, uint32_t* dev_status,
                         cudaStream_t st);

// ---------------------------------------------------------------- expert forward / backward
struct FwdWs {
  float* y_acc;  // [T,H] fp32 accumulator of the routing-weighted combine
  int32_t* plan; // [E+1] prefix of token tiles per expert (tensor-core path)
  float* wperm;  // [R_cap] routing weight per permuted row
};
struct BwdWs {
  float* dw;          // [T*k] when the caller gives no dw_slot
  float* dw_part;     // [4 * ceil(I / 128)][T*k] per-tile partial sums of dw (tensor-core path)
  float* dl;          // [T*k] dlogit at the selected experts (renorm = 1)
  float* dl_perm;     // [R_cap] the same in permuted row order
  float* dlogit;      // [T,E] dense dlogit (renorm = 0)
  void* dh;           // dh^T [2I, R_cap] of dtype
  float* dx_acc;      // [T,H]
  float* gvec;        // [R_cap, I] (fp32 path only)
  int32_t* plan;      // [E+1] prefix of token tiles per expert (tensor-core path)
  float* wperm;       // [R_cap] routing weight per permuted row
  void* dy_perm;      // dy^T [H, R_cap]: dy in permuted order, feature-major
  float* g_part;      // [token tiles][H] router-gradient partial sums (tensor-core path)
};
void fwd_ws_layout(const usaf_moe_shape& s, usaf_dtype dt, Carver& c, FwdWs& w);
void bwd_ws_layout(const usaf_moe_shape& s, usaf_dtype dt, int64_t K, Carver& c, BwdWs& w);

// Tokens per tensor-core tile at most; the per-expert tile plan (written by the gathers) counts
// ceil(padded rows / TC_TOKEN_TILE) tiles per expert.
constexpr int TC_TOKEN_TILE = 256;

struct MoeArgs {
  usaf_moe_shape s;
  usaf_dtype dt;
  int64_t R_cap;
  const void* x;
  const float* w_router;
  const void* w_gate_up;
  const void* w_down;
  usaf_routing rt;
  int32_t* plan;  // token-tile prefix written by tc_plan (tensor-core path)
  float* wperm;   // [R_cap] routing weight of each permuted row (0 in padding), by the gather
  uint32_t* status;  // device status word of the call (may be null): bounded waits that give up
};

// The masked-gradient plan of an active set (built by usaf_masked_plan_build): the experts whose
// active density makes a dense tensor-core tile cheaper than per-entry dot products, and for
// those the first active entry of every row. row_ptr per expert: gate_up rows 0 .. 2I (2I + 1
// values, the last the end of the expert's gate_up entries), then down rows 0 .. H.
struct MaskedPlan {
  const int32_t* n_dense;     // device: number of listed experts
  const int32_t* dense_list;  // [E]
  const int32_t* dense_flag;  // [E] 1 for listed experts
  const int64_t* row_ptr;     // [E][rp_stride]
  int64_t rp_stride;          // 2I + H + 2
};
size_t masked_plan_bytes(const usaf_moe_shape& s);
MaskedPlan masked_plan_layout(const usaf_moe_shape& s, void* base);
usaf_status masked_plan_build_launch(const usaf_moe_shape& s, const int64_t* act, int64_t K,
                                     int64_t thr_count, void* plan, cudaStream_t st);

// weights_ready (may be null): the kernels that read the expert weights wait for it; the token
// gather before them does not
// forward stages (usaf_moe_fwd_stage)
constexpr int FWD_GATHER = 1, FWD_GATE_UP = 2, FWD_DOWN = 4, FWD_ALL = 7;
usaf_status moe_fwd_launch(const MoeArgs& a, void* x_perm, void* h, void* wa, void* y, FwdWs& w,
                           cudaEvent_t weights_ready, cudaEvent_t down_ready, int stages,
                           cudaStream_t st);
// plan / n_dense: the masked-gradient plan of act_idx and its number of dense experts as the
// host read it (0: every entry by the sparse kernel, plan unused)
usaf_status moe_bwd_launch(const MoeArgs& a, int renorm, const float* logits, const void* x_perm,
                           const void* h, const void* wa, const void* dy, const int64_t* act_idx,
                           int64_t K, float* g_act, float* g_router, void* dx, float* dw_slot,
                           float* g_dense, int accumulate, uint32_t* dev_status, BwdWs& w,
                           cudaStream_t st, const MaskedPlan* plan = nullptr, int64_t n_dense = 0);
usaf_status moe_wgrad_dense_launch(const MoeArgs& a, const void* x_perm, const void* wa,
                                   float* g_dense, int accumulate, BwdWs& w, cudaStream_t st);

// tensor-core (tcgen05) grouped GEMM stages, bf16 only
bool tc_shape_ok(const usaf_moe_shape& s);
usaf_status tc_router_logits(const usaf_moe_shape& s, const void* x, const float* wr, void* wr3,
                             float* logits, uint32_t* status, cudaStream_t st);
usaf_status tc_fwd_gate_up(const MoeArgs& a, const void* xT, void* hT, void* waT,
                           cudaStream_t st);
usaf_status tc_fwd_down(const MoeArgs& a, const void* wa, float* y_acc, cudaStream_t st);
// dw_part [4 * ceil(I / 128)][T*k]: one partial of dw per (M tile, row quarter, slot)
usaf_status tc_bwd_gvec(const MoeArgs& a, const void* dyT, const void* hT, void* dhT,
                        float* dw_part, cudaStream_t st);
// The tensor map of a feature-major token array [features, R_cap] (bf16) in boxes of 64 tokens x
// 64 features, 128-byte swizzle: the GEMMs' token operand, and the gather's TMA store target.
bool tc_token_map(CUtensorMap* m, const void* base, uint64_t features, uint64_t R_cap);
// dl_perm (may be null): dlogit per permuted row; with it the router's share of dx (renormalised
// routing) is added in the epilogue
usaf_status tc_bwd_dx(const MoeArgs& a, const void* dh, float* dx_acc, const float* dl_perm,
                      cudaStream_t st);
// dense expert weight gradient g[e] (a_rows x b_rows, fp32) = aT . bT^T over each expert's tokens
usaf_status tc_wgrad_dense(const MoeArgs& a, const void* aT, int64_t a_rows, const void* bT,
                           int64_t b_rows, float* g, int accumulate, cudaStream_t st);
// the gradient at the active entries of the plan's dense experts: tensor 0 gate_up, 1 down
usaf_status tc_wgrad_gather(const MoeArgs& a, const void* aT, int64_t a_rows, const void* bT,
                            int64_t b_rows, const MaskedPlan& plan, int tensor, const int64_t* act,
                            float* g_act, int accumulate, cudaStream_t st);
// one CTA whose bounded wait runs out on purpose (see usaf_diag_bounded_wait)
usaf_status diag_wait_launch(int64_t limit_cycles, uint32_t* status, cudaStream_t st);


// ---------------------------------------------------------------- optimizer
usaf_status nonfinite_scan_launch(const float* g, int64_t n, uint32_t* dev_status,
                                  cudaStream_t st);
usaf_status adam_launch(int64_t n, const int64_t* idx, const float* g, float* p, float* m,
                        float* v, void* w0, int64_t n0, void* w1, usaf_dtype wdt, double lr,
                        double b1, double b2, double eps, int64_t step, int skip,
                        uint32_t* dev_status, cudaStream_t st);
// USAF_DEV_BAD_INDEX when idx[0..K) is not strictly ascending inside [0, N)
usaf_status validate_launch(const int64_t* idx, int64_t K, int64_t N, uint32_t* dev_status,
                            cudaStream_t st);

// ---------------------------------------------------------------- selection / RigL
size_t select_ws_bytes(int64_t N, int64_t K, bool with_bitmap);
usaf_status importance_select_launch(const float* g, int64_t N, int64_t K, int64_t* out_idx,
                                     uint32_t* dev_status, void* ws, cudaStream_t st);
size_t reselect_ws_bytes(int64_t N, int64_t K);
usaf_status reselect_launch(const float* g, int64_t N, int64_t K, const int64_t* old_idx,
                            int64_t K_old, const float* p_in, const float* m_in,
                            const float* v_in, const void* w0, int64_t n0, const void* w1,
                            usaf_dtype wdt, int64_t* new_idx, float* p_out, float* m_out,
                            float* v_out, int64_t* n_kept, uint32_t* dev_status, void* ws,
                            cudaStream_t st);
// shard primitives of a selection spread over ranks (see usaf_shard_* in usaf.h)
usaf_status shard_hist_launch(const float* g, int64_t n, const uint32_t* excl, uint32_t prefix,
                              int shift, int bits, unsigned long long* hist, cudaStream_t st);
size_t shard_emit_ws_bytes(int64_t n, int64_t count);
usaf_status shard_emit_launch(const float* g, int64_t n, const uint32_t* excl, uint32_t tau,
                              int64_t take_eq, int64_t count, int64_t base, int64_t* out,
                              uint32_t* dev_status, void* ws, cudaStream_t st);
usaf_status bitmap_range_launch(const int64_t* idx, int64_t K, int64_t lo, int64_t n,
                                uint32_t* bm, cudaStream_t st);
size_t rigl_ws_bytes(int64_t N, int64_t K, int64_t D);
usaf_status rigl_launch(const float* g, int64_t N, const int64_t* act_idx, int64_t K, int64_t D,
                        const float* p_in, const float* m_in, const float* v_in, const void* w0,
                        int64_t n0, const void* w1, usaf_dtype wdt, int64_t* new_idx,
                        float* p_out, float* m_out, float* v_out, int64_t* n_swapped,
                        uint32_t* dev_status, void* ws, cudaStream_t st,
                        const int64_t* grown_in = nullptr);
size_t select_and_swap_ws_bytes(int64_t N, int64_t Ksel, int64_t K, int64_t D);
usaf_status select_and_swap_launch(const float* g, int64_t N, int64_t Ksel, int64_t* sel_idx,
                                   const int64_t* act_idx, int64_t K, int64_t D,
                                   const float* p_in, const float* m_in, const float* v_in,
                                   const void* w0, int64_t n0, const void* w1, usaf_dtype wdt,
                                   int64_t* new_idx, float* p_out, float* m_out, float* v_out,
                                   int64_t* n_swapped, uint32_t* dev_status, void* ws,
                                   cudaStream_t st);
usaf_status reselect_carry_launch(const int64_t* new_idx, int64_t K, int64_t N,
                                  const int64_t* old_idx, int64_t K_old, const float* p_in,
                                  const float* m_in, const float* v_in, const void* w0, int64_t n0,
                                  const void* w1, usaf_dtype wdt, float* p_out, float* m_out,
                                  float* v_out, int64_t* n_kept, uint32_t* dev_status, void* ws,
                                  cudaStream_t st);
size_t reselect_carry_ws_bytes();

}  // namespace usaf
