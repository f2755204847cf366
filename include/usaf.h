/*
 * usaf.h - C ABI of the GB300 (sm_103a) hot path of USAF sparse MoE fine-tuning.
 *
 * One MoE layer's train step, as the USAF README describes it: the router is trained in full
 * ("The router is leverage" paragraph), 0.5% of the native expert weights, picked by gradient
 * magnitude ("Not all weights matter" paragraph), are trained in place with Adam state kept only
 * for them (A100 operations table: "SparseAdam (26M)"), and the active set is reselected
 * RigL-style every 50 steps ("Sparsity adapts" paragraph; RESELECT_EVERY in the environment
 * variable table). The fused expert layouts gate_up_proj [E, 2I, H] and down_proj [E, H, I] and the
 * act(gate) * up epilogue are the ones stated on the experts4bit-qlora page ("The abstraction that
 * fails, and what replaces it" section, and its epilogue-contract bullet).
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless a comment says "host".
 *    The library allocates no device memory: scratch comes from a caller-provided workspace whose
 *    size the matching *_workspace_size() query returns (a host-only computation).
 *  - Tensors are dense and row-major. Element types are given by usaf_dtype.
 *  - `stream` is a cudaStream_t passed as void*. Every call only enqueues work on that stream and
 *    never synchronises the host. Calls keep no state between them and are thread-safe.
 *  - Host-side argument checks run before anything is enqueued; a failed check returns
 *    USAF_ERR_INVALID_ARG (or USAF_ERR_UNSUPPORTED / USAF_ERR_WORKSPACE) and enqueues nothing.
 *    A failed kernel launch returns USAF_ERR_CUDA. Conditions that only the device can see
 *    (non-finite gradients, a selection that had to take the exact multi-pass path, a bounded
 *    wait that gave up, an active-set index out of range) are OR-ed as bits into the caller's
 *    `dev_status` word (device memory, may be NULL); no kernel traps.
 *  - With the environment variable USAF_DEBUG=1 set when a call is made, every call that reads
 *    an active set first runs usaf_validate_active on it (one extra kernel per call).
 *  - Flat expert-weight index f (int64): f < N_gu = E*2I*H addresses gate_up_proj row-major,
 *    N_gu <= f < N = E*3*I*H addresses down_proj row-major at f - N_gu. Active sets are sorted
 *    ascending and free of duplicates.
 */
#ifndef USAF_H
#define USAF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define USAF_ABI_VERSION 2

/* Each expert's rows in the permuted (expert-sorted) order start at a multiple of this. */
#define USAF_ROW_ALIGN 16

typedef enum {
  USAF_OK = 0,
  USAF_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad enum, aliasing that is not allowed */
  USAF_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle (see each call) */
  USAF_ERR_WORKSPACE = 3,   /* workspace pointer NULL or smaller than the query says */
  USAF_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a kernel launch failed */
  USAF_ERR_TIMEOUT = 5      /* not returned by any call: timeouts are device status bits */
} usaf_status;

typedef enum { USAF_F32 = 0, USAF_BF16 = 1 } usaf_dtype;

/* Bits OR-ed into *dev_status by the device. */
#define USAF_DEV_NONFINITE 1u       /* a gradient (or selection key) was NaN or Inf */
#define USAF_DEV_SELECT_EXACT_PATH 2u /* informational: the sampled one-pass selection fell back
                                       * to the exact multi-pass radix select */
#define USAF_DEV_TIMEOUT 4u         /* a tensor-core kernel's pipeline wait gave up after about
                                     * two seconds; that kernel's outputs are incomplete (the
                                     * router kernel then writes none of the affected logits) */
#define USAF_DEV_BAD_INDEX 8u       /* an active-set index was out of range, out of order or
                                     * repeated; kernels skip such entries, never address them */
/* The bits after which usaf_sparse_adam_step with skip_if_nonfinite updates nothing. */
#define USAF_DEV_SKIP_MASK (USAF_DEV_NONFINITE | USAF_DEV_TIMEOUT | USAF_DEV_BAD_INDEX)

/* MoE layer dimensions: T tokens, H hidden size, E experts, k experts per token, I expert
 * intermediate size. */
typedef struct {
  int64_t T, H, E, k, I;
} usaf_moe_shape;

/* Routing tables written by usaf_route_topk and read by usaf_moe_fwd / usaf_moe_bwd_sparse.
 * R = T*k routed slots; slot s = t*k + j is the j-th expert of token t.
 * The permuted order lists, for e = 0..E-1, the slots routed to e in ascending token order;
 * expert e's segment starts at row expert_offset[e] (a multiple of USAF_ROW_ALIGN) and its
 * rows past expert_count[e] up to the next offset are padding rows (perm_tok = 0, perm_slot = -1).
 * R_cap = usaf_routed_rows_capacity(shape) is the number of rows every permuted array holds. */
typedef struct {
  int32_t* topk_idx;      /* [T*k]   expert of each slot, in descending-logit order per token   */
  float* topk_w;          /* [T*k]   routing weight of each slot                                */
  int32_t* expert_count;  /* [E]     tokens routed to each expert                               */
  int32_t* expert_offset; /* [E+1]   first permuted row of each expert; [E] = padded total rows */
  int32_t* perm_tok;      /* [R_cap] token of each permuted row                                 */
  int32_t* perm_slot;     /* [R_cap] slot of each permuted row, -1 for padding                  */
  int32_t* slot_row;      /* [T*k]   permuted row of each slot                                  */
} usaf_routing;

int usaf_abi_version(void);
const char* usaf_status_string(usaf_status s); /* host string, static storage */

/* Rows every permuted array (perm_tok, perm_slot, saved activations) must hold:
 * T*k + E*(USAF_ROW_ALIGN-1) rounded up to 256, plus 256 rows of read-ahead slack. Host only. */
int64_t usaf_routed_rows_capacity(const usaf_moe_shape* shape);

/* ---------------------------------------------------------------------------------------------
 * usaf_route_topk - router logits, top-k with renormalised softmax weights, token permutation.
 * Router logits logits[t,e] = sum_h x[t,h] * w_router[e,h] (fp32 arithmetic, x upcast exactly).
 * Per token the k experts with the largest fp32 logits are taken, ties to the lower expert index,
 * in descending order. renorm=1: w_j = softmax over the k selected logits (equal to softmax over
 * all E, top-k, renormalised); renorm=0: w_j = softmax over all E at the selected experts.
 * The router is the gating network the USAF README trains in full ("The router is leverage").
 *   x          [T,H] of x_dtype (USAF_F32 or USAF_BF16); ignored when logits_in != NULL
 *   w_router   [E,H] fp32; ignored when logits_in != NULL
 *   logits_in  [T,E] fp32 or NULL: use these logits instead of computing them
 *   logits_out [T,E] fp32 or NULL: where computed logits are written
 *   rt         routing tables (all seven arrays required)
 *   dev_status gets USAF_DEV_TIMEOUT if the tensor-core logits kernel gave up a wait (its logits
 *              are then not written and the routing of the affected tokens is meaningless); may
 *              be NULL
 * Limits: 1 <= k <= E <= 1024, k <= 32, T*k < 2^31. Errors: INVALID_ARG, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
size_t usaf_route_topk_workspace_size(const usaf_moe_shape* shape);
usaf_status usaf_route_topk(const usaf_moe_shape* shape, const void* x, usaf_dtype x_dtype,
                            const float* w_router, const float* logits_in, float* logits_out,
                            int renorm, const usaf_routing* rt, uint32_t* dev_status, void* ws,
                            size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_route_topk_noalloc - usaf_route_topk for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists for deployments in which the routing
 * call site must not reach any allocator: servers whose device-memory pool is fixed once at
 * start-up, code invoked from inside another runtime's memory manager (where allocating again
 * would recurse or deadlock), and embedded targets that forbid dynamic device allocation after
 * initialisation. Such callers cannot size and pass a workspace, so this call takes none.
 * Same inputs, outputs and results as usaf_route_topk, except that logits_in or logits_out must
 * be given (the logits are never kept in scratch).
 * Scratch: a fixed device array of USAF_NOALLOC_SCRATCH_BYTES inside the library, which every
 * GPU that loads the library holds until the process exits. It needs ceil(T*k/256)*E*4 bytes
 * (rounded up to 256), plus 6*E*H bytes for the bf16 split of the router weight when the
 * tensor-core logits path runs (logits_in NULL, x bf16, H and I multiples of 64); a call needing
 * more is refused with USAF_ERR_WORKSPACE before anything is enqueued. The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture. All calls share the one array and leave their scratch in it;
 * every byte a call reads from it was written earlier by the same call, so nothing needs
 * clearing, but calls whose work overlaps on the GPU (other streams, other host threads) race
 * on it and must be serialised by the caller. No cudaMalloc, cudaFree or allocating library
 * routine is called. Errors: INVALID_ARG, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
#define USAF_NOALLOC_SCRATCH_BYTES (4u << 20)
usaf_status usaf_route_topk_noalloc(const usaf_moe_shape* shape, const void* x,
                                    usaf_dtype x_dtype, const float* w_router,
                                    const float* logits_in, float* logits_out, int renorm,
                                    const usaf_routing* rt, uint32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_moe_fwd - grouped SwiGLU expert forward over the permuted rows.
 * For every routed slot (t, j) with expert e: h = gate_up_proj[e] . x[t]  (2I values; the first I
 * rows of gate_up_proj[e] are the gate, the last I the up projection), A = silu(gate) * up,
 * y = down_proj[e] . A, and Y[t] = sum_j w[t,j] * y_j. Layouts per the experts4bit-qlora page
 * (gate_up_proj [E,2I,H], down_proj [E,H,I]); act(gate)*up per its epilogue-contract bullet.
 *   dtype        USAF_BF16: x, weights, saved activations and y are bf16, accumulation fp32, on
 *                tcgen05 tensor cores (needs H % 64 == 0, I % 64 == 0).
 *                USAF_F32: everything fp32 on CUDA cores (any sizes).
 *   x            [T,H];  w_gate_up [E,2I,H];  w_down [E,H,I]
 *   x_perm_save  [H,R_cap]  out: x in permuted row order, feature-major (kept for the backward)
 *   h_save       [2I,R_cap] out: gate|up pre-activations, feature-major: element (j, row) is
 *                feature j (gate for j < I, up for j >= I) of permuted row `row`
 *   wa_save      [I,R_cap]  out: w * A per permuted row, feature-major (0 in padding rows)
 *   y            [T,H]      out
 *   dev_status   gets USAF_DEV_TIMEOUT if a tensor-core kernel gave up a wait (may be NULL)
 * Errors: INVALID_ARG, UNSUPPORTED (bf16 shape limits; also any dtype with
 * max(2I,H) * R_cap >= 2^31 * (16 / element size), the range of the 32-bit vector indices into the
 * feature-major rows), WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
size_t usaf_moe_fwd_workspace_size(const usaf_moe_shape* shape, usaf_dtype dtype);
usaf_status usaf_moe_fwd(const usaf_moe_shape* shape, usaf_dtype dtype, const void* x,
                         const void* w_gate_up, const void* w_down, const usaf_routing* rt,
                         void* x_perm_save, void* h_save, void* wa_save, void* y,
                         uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* usaf_moe_fwd_wait - usaf_moe_fwd whose reads of the expert weights wait for a CUDA event.
 * weights_ready is a cudaEvent_t (NULL: no wait, the same as usaf_moe_fwd), typically recorded
 * by the caller on another stream after an optimizer update of w_gate_up / w_down. The token
 * gather into x_perm_save, which reads only x and the routing tables, is enqueued before the
 * wait and so overlaps that update; everything after it on `stream` is ordered after the event.
 * Same results and errors as usaf_moe_fwd. */
usaf_status usaf_moe_fwd_wait(const usaf_moe_shape* shape, usaf_dtype dtype, const void* x,
                              const void* w_gate_up, const void* w_down, const usaf_routing* rt,
                              void* x_perm_save, void* h_save, void* wa_save, void* y,
                              void* weights_ready, uint32_t* dev_status, void* ws,
                              size_t ws_bytes, void* stream);

/* usaf_moe_fwd_wait2 - usaf_moe_fwd_wait with one event per weight tensor: the gate_up GEMM waits
 * for gate_up_ready, the down GEMM for down_ready (either may be NULL), so an optimizer update of
 * w_down (issued after that of w_gate_up, on another stream) overlaps the gate_up GEMM. Same
 * results and errors as usaf_moe_fwd. */
usaf_status usaf_moe_fwd_wait2(const usaf_moe_shape* shape, usaf_dtype dtype, const void* x,
                               const void* w_gate_up, const void* w_down, const usaf_routing* rt,
                               void* x_perm_save, void* h_save, void* wa_save, void* y,
                               void* gate_up_ready, void* down_ready, uint32_t* dev_status,
                               void* ws, size_t ws_bytes, void* stream);

/* usaf_moe_fwd_stage - the stages of usaf_moe_fwd run on their own, for callers that order other
 * work between them (one CUDA graph per stage, say, with waits for a weight update between their
 * replays). stages is a bit set: 1 the token gather into x_perm_save (it also clears the combine
 * accumulator and writes the tile plan, in ws), 2 the gate_up GEMM + SwiGLU (h_save, wa_save),
 * 4 the down GEMM and the combine into y; 7 is usaf_moe_fwd. A later stage reads what the earlier
 * ones left in x_perm_save, h_save, wa_save and ws: run them in order, on one stream, with the
 * same routing and workspace. fp32 layers run stages 2 and 4 only together (UNSUPPORTED
 * otherwise). Errors: INVALID_ARG (stages outside 1..7), the errors of usaf_moe_fwd. */
usaf_status usaf_moe_fwd_stage(const usaf_moe_shape* shape, usaf_dtype dtype, const void* x,
                               const void* w_gate_up, const void* w_down, const usaf_routing* rt,
                               void* x_perm_save, void* h_save, void* wa_save, void* y,
                               int stages, uint32_t* dev_status, void* ws, size_t ws_bytes,
                               void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_moe_bwd_sparse - sparse backward of the layer for upstream gradient dy = dL/dY.
 * Per slot: gvec = down_proj[e]^T dy[t], dw = <gvec, A>, dA = w*gvec, dgate = dA*up*silu'(gate),
 * dup = dA*silu(gate). Router: dlogit[t,e_j] = w_j*(dw_j - sum_i w_i dw_i) (renorm=1; renorm=0
 * uses the all-E softmax form), g_router = dlogit^T x. dx = sum_j gate_up_proj[e_j]^T dh_j +
 * dlogit . w_router. Expert weight gradients are formed only at the active set
 * (news article, key differences: inside each expert that fires, only part of its weights is
 * trained; README, A100 operations table: the backward row, counted over the trained 26M):
 *   g_act[a] = sum over rows of expert e of dh[row, r] * x[tok, c]         (gate_up entry e,r,c)
 *   g_act[a] = sum over rows of expert e of dy[tok, r] * w * A[row, c]      (down entry e,r,c)
 * Experts that received no token get zero gradient.
 *   renorm       must match the routing call; logits [T,E] fp32 needed only when renorm == 0
 *   x_perm_save, h_save, wa_save   as written by usaf_moe_fwd with the same routing
 *   dy           [T,H] of dtype
 *   act_idx      [K] sorted flat indices (int64), 0 <= K <= N
 *   g_act        [K] fp32 out;  g_router [E,H] fp32 out
 *   dx           [T,H] of dtype out, or NULL to skip the input gradient
 *   dw_slot      [T*k] fp32 out (dL/dw per slot), or NULL
 *   dev_status   gets USAF_DEV_NONFINITE if any produced gradient is NaN/Inf, USAF_DEV_TIMEOUT if
 *                a tensor-core kernel gave up a wait, USAF_DEV_BAD_INDEX if an active index does
 *                not address an expert weight (that entry's g_act is left 0) (may be NULL)
 * bf16 layers with renorm = 1 form g_router on a side stream of the library (one per calling
 * thread and device, created by usaf_moe_bwd_workspace_size or by an uncaptured call and kept for
 * the thread's life), forked from `stream` after dlogit and joined back before the call returns:
 * the call's work as a whole stays ordered on `stream`, and in a stream capture it becomes two
 * branches of the graph. A call captured on a thread that has no side stream yet runs it in line.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
size_t usaf_moe_bwd_workspace_size(const usaf_moe_shape* shape, usaf_dtype dtype, int64_t K);
usaf_status usaf_moe_bwd_sparse(const usaf_moe_shape* shape, usaf_dtype dtype, int renorm,
                                const void* x, const float* w_router, const void* w_gate_up,
                                const void* w_down, const usaf_routing* rt, const float* logits,
                                const void* x_perm_save, const void* h_save, const void* wa_save,
                                const void* dy, const int64_t* act_idx, int64_t K, float* g_act,
                                float* g_router, void* dx, float* dw_slot, uint32_t* dev_status,
                                void* ws, size_t ws_bytes, void* stream);

/* Byte offset inside the backward workspace of dlogit at the selected experts: after a
 * usaf_moe_bwd_sparse* call with renorm = 1, ws + offset holds [T*k] fp32 values in slot order
 * (slot t*k + j: dL/dlogit[t, topk_idx[t*k + j]]; every other expert's dlogit is 0). A read-only
 * view for checking the router backward; -1 for an invalid shape. Host only. */
int64_t usaf_moe_bwd_dlogit_offset(const usaf_moe_shape* shape, usaf_dtype dtype, int64_t K);

/* ---------------------------------------------------------------------------------------------
 * usaf_moe_bwd_sparse_accumulate - usaf_moe_bwd_sparse for one micro-batch of a step that
 * accumulates gradients over several (USAF README environment table: MICROBATCH): g_act and
 * g_router are added to instead of overwritten; dx and dw_slot are this micro-batch's own, as
 * in usaf_moe_bwd_sparse. Same arguments, workspace and errors as usaf_moe_bwd_sparse.
 * ------------------------------------------------------------------------------------------- */
usaf_status usaf_moe_bwd_sparse_accumulate(
    const usaf_moe_shape* shape, usaf_dtype dtype, int renorm, const void* x,
    const float* w_router, const void* w_gate_up, const void* w_down, const usaf_routing* rt,
    const float* logits, const void* x_perm_save, const void* h_save, const void* wa_save,
    const void* dy, const int64_t* act_idx, int64_t K, float* g_act, float* g_router, void* dx,
    float* dw_slot, uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Masked-gradient plan of an active set. The sparse backward forms each active entry's gradient
 * as a dot product over its expert's routed tokens (usaf_moe_bwd_sparse). Where the active set
 * is dense inside an expert (importance selection concentrates on some experts; the skewed
 * workload puts 80% of the set on 16 of 128 experts), a dense tensor-core tile of that expert's
 * gradient, read out at the active entries only, costs less. The plan lists those experts and,
 * for each, the first active entry of every weight row. It depends only on the active set and
 * the shape: build it when the set changes (README, "Sparsity adapts": every 50 steps).
 *   usaf_masked_plan_size   bytes of the plan buffer for this shape (host only)
 *   usaf_masked_plan_build  dense_density: an expert is listed when its active entries (both
 *                           tensors) are at least dense_density * 3*I*H (> 0; 1 lists none).
 *                           plan [usaf_masked_plan_size] device buffer, 256-byte aligned.
 *                           After the stream has run the build, the plan's first 8 bytes hold
 *                           the number of listed experts as an int64, for the caller to read.
 * Errors: INVALID_ARG, CUDA.
 * ------------------------------------------------------------------------------------------- */
size_t usaf_masked_plan_size(const usaf_moe_shape* shape);
usaf_status usaf_masked_plan_build(const usaf_moe_shape* shape, const int64_t* act_idx, int64_t K,
                                   double dense_density, void* plan, size_t plan_bytes,
                                   void* stream);

/* usaf_moe_bwd_sparse_planned - usaf_moe_bwd_sparse (accumulate = 0) or
 * usaf_moe_bwd_sparse_accumulate (accumulate = 1) with a masked-gradient plan of act_idx: the
 * listed experts' active entries are read out of dense bf16 tensor-core tiles (fp32
 * accumulation), every other entry as before. n_dense is the count the caller read from the
 * plan's first 8 bytes; with n_dense = 0 the plan is not read (may be NULL) and the call is the
 * plain sparse backward. fp32 layers ignore the plan. Same results (within the bf16 bound),
 * workspace and errors as usaf_moe_bwd_sparse. */
usaf_status usaf_moe_bwd_sparse_planned(
    const usaf_moe_shape* shape, usaf_dtype dtype, int renorm, const void* x,
    const float* w_router, const void* w_gate_up, const void* w_down, const usaf_routing* rt,
    const float* logits, const void* x_perm_save, const void* h_save, const void* wa_save,
    const void* dy, const int64_t* act_idx, int64_t K, float* g_act, float* g_router, void* dx,
    float* dw_slot, int accumulate, const void* plan, int64_t n_dense, uint32_t* dev_status,
    void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_moe_bwd_dense - the same backward as usaf_moe_bwd_sparse (dh, dw, router gradient, dx),
 * with the expert weight gradient formed densely for the importance phase (USAF README: the
 * weights to train are the 0.5% with the largest gradient magnitude, found by a dense gradient
 * pass; A100 operations table: "RigL dense pass ~60 s" over the accumulated gradient):
 *   g_dense[f] = dL/dW at every flat index f (gate_up [E,2I,H] row-major, then down [E,H,I])
 *   gate_up entry (e, r, c) = sum over rows of expert e of dh[row, r] * x[tok, c];
 *   down entry (e, r, c)    = sum over rows of expert e of dy[tok, r] * w * A[row, c];
 * experts without tokens give 0.
 *   g_dense     [N] fp32, 16-byte aligned; accumulate = 1 adds into it and into g_router
 *               (micro-batch accumulation), 0 overwrites both
 *   the other arguments and the workspace (usaf_moe_bwd_workspace_size with K = 0) as for
 *   usaf_moe_bwd_sparse
 * bf16 layers form g_dense on tensor cores (fp32 accumulation; stores or adds by TMA); fp32
 * layers on CUDA cores. Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
usaf_status usaf_moe_bwd_dense(const usaf_moe_shape* shape, usaf_dtype dtype, int renorm,
                               const void* x, const float* w_router, const void* w_gate_up,
                               const void* w_down, const usaf_routing* rt, const float* logits,
                               const void* x_perm_save, const void* h_save, const void* wa_save,
                               const void* dy, float* g_dense, int accumulate, float* g_router,
                               void* dx, float* dw_slot, uint32_t* dev_status, void* ws,
                               size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_moe_wgrad_dense - the dense expert weight gradient of usaf_moe_bwd_dense alone, for a
 * micro-batch whose backward already ran (the importance phase's dense pass on a step that also
 * trains: README, "Sparsity adapts"; A100 operations table, "RigL dense pass"). It reads the dh
 * and the permuted dy that the preceding usaf_moe_bwd_sparse* or usaf_moe_bwd_dense call left in
 * its workspace: pass that same workspace, with the same shape, dtype and routing, on the same
 * stream and with no other backward call in between; gvec, the router gradient and dx are not
 * recomputed.
 *   x_perm_save, wa_save   as written by usaf_moe_fwd with that routing
 *   g_dense     [N] fp32, 16-byte aligned; accumulate = 1 adds into it, 0 overwrites
 *   dev_status  gets USAF_DEV_TIMEOUT if a tensor-core kernel gave up a wait (may be NULL)
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
usaf_status usaf_moe_wgrad_dense(const usaf_moe_shape* shape, usaf_dtype dtype,
                                 const usaf_routing* rt, const void* x_perm_save,
                                 const void* wa_save, float* g_dense, int accumulate,
                                 uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_sparse_adam_step - fused gather / Adam update / scatter over n entries (the README's
 * "SparseAdam (26M)" optimizer, torch.optim.SparseAdam semantics, no weight decay):
 *   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*g^2;
 *   p -= lr*sqrt(1-b2^step)/(1-b1^step) * m/(sqrt(v)+eps)
 * then the dense weight at the entry's flat index receives p (rounded to nearest-even for bf16).
 *   idx          [n] flat indices, or NULL for the dense identity 0..n-1
 *   g, p, m, v   [n] fp32 (p is the fp32 master copy of the trained entries; p, m, v in place)
 *   w_seg0       dense weights holding flat indices [0, n_seg0); w_seg1 holds [n_seg0, ...) and
 *                may be NULL when every index is below n_seg0; both of w_dtype
 *   lr, beta1, beta2, eps  host scalars; 1-b1, 1-b2 and the bias-corrected step size are formed
 *                in double on the host and passed to the kernel as fp32
 *   step         1-based step count
 *   skip_if_nonfinite  1: the entry point first scans g, and no entry is updated when this
 *                scan or an earlier call found a non-finite gradient, or an earlier call timed
 *                out or saw a bad active index (any bit of USAF_DEV_SKIP_MASK already set in
 *                *dev_status, e.g. by usaf_moe_bwd_sparse) (the README's NaN step skip);
 *                2: the same without the scan, for a gradient the caller has scanned whole with
 *                usaf_scan_nonfinite before updating it in parts (so that a non-finite entry in
 *                any part skips every part); 0: no check
 *   dev_status   with USAF_DEV_BAD_INDEX already set, no entry is updated whatever
 *                skip_if_nonfinite says (the indices would address memory outside the weights)
 * Errors: INVALID_ARG, CUDA.
 * ------------------------------------------------------------------------------------------- */
usaf_status usaf_sparse_adam_step(int64_t n, const int64_t* idx, const float* g, float* p,
                                  float* m, float* v, void* w_seg0, int64_t n_seg0, void* w_seg1,
                                  usaf_dtype w_dtype, double lr, double beta1, double beta2,
                                  double eps, int64_t step, int skip_if_nonfinite,
                                  uint32_t* dev_status, void* stream);

/* usaf_scan_nonfinite - sets USAF_DEV_NONFINITE in *dev_status when any of g[0, n) is NaN or
 * infinite (the scan of usaf_sparse_adam_step's skip_if_nonfinite = 1, on its own).
 * Errors: INVALID_ARG (n < 0, g NULL with n > 0, dev_status NULL), CUDA. */
usaf_status usaf_scan_nonfinite(const float* g, int64_t n, uint32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_importance_select - the importance phase of the USAF README ("Not all weights matter":
 * the 0.5% of weights with the highest gradient magnitude). Exact top-K of |g| over N entries,
 * ordered by (|g| descending, index ascending); the K winners are written sorted ascending.
 * |g| is compared as its fp32 bit pattern with the sign cleared.
 *   g        [N] fp32 dense gradient
 *   out_idx  [K] int64 out
 * Limits: 1 <= K <= N < 2^32. Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
size_t usaf_importance_select_workspace_size(int64_t N, int64_t K);
usaf_status usaf_importance_select(const float* g, int64_t N, int64_t K, int64_t* out_idx,
                                   uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_rigl_swap - RigL reselection of the active set (USAF README, "Sparsity adapts"):
 * drop the D active entries with the smallest |p| (ties: lower flat index dropped first), grow
 * the D inactive entries (not in the old set) with the largest |g| (ties: lower flat index
 * first). new_idx = (act_idx minus dropped) union grown, sorted. Kept entries carry p, m, v
 * unchanged; grown entries start with p = the dense weight value and m = v = 0.
 *   g          [N] fp32 dense gradient;  act_idx [K] sorted
 *   p_in, m_in, v_in   [K] fp32 state aligned with act_idx
 *   w_seg0/n_seg0/w_seg1/w_dtype   dense weights, as for usaf_sparse_adam_step
 *   new_idx, p_out, m_out, v_out   [K] out; must not overlap the inputs
 *   n_swapped  [1] int64 out: number of entries of act_idx not in new_idx (= D)
 * The drop selection runs on a private stream forked from and joined back to `stream` (created
 * and released inside the call), so it overlaps the pass over g; the call's work as a whole is
 * still ordered on `stream`.
 * Limits: 0 <= D <= K, D <= N - K, N < 2^32. Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
size_t usaf_rigl_swap_workspace_size(int64_t N, int64_t K, int64_t D);
usaf_status usaf_rigl_swap(const float* g, int64_t N, const int64_t* act_idx, int64_t K,
                           int64_t D, const float* p_in, const float* m_in, const float* v_in,
                           const void* w_seg0, int64_t n_seg0, const void* w_seg1,
                           usaf_dtype w_dtype, int64_t* new_idx, float* p_out, float* m_out,
                           float* v_out, int64_t* n_swapped, uint32_t* dev_status, void* ws,
                           size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_select_and_swap - the importance selection and the RigL swap of one dense gradient from
 * one pass over g (USAF README, "Not all weights matter" and "Sparsity adapts"): sel_idx gets
 * exactly what usaf_importance_select(g, N, K_sel) writes, and new_idx, p_out, m_out, v_out and
 * n_swapped exactly what usaf_rigl_swap(g, N, act_idx, K, D, ...) writes. Both selections are
 * found among one set of candidates compacted in a single read of g; where either selection would
 * not take the sampled path (small N, K_sel or D a large part of N, D = 0), the call runs the two
 * selections one after the other instead (same results).
 *   g          [N] fp32 dense gradient
 *   sel_idx    [K_sel] int64 out, sorted ascending; must not overlap the other outputs or inputs
 *   the rest   as for usaf_rigl_swap
 * Limits: 1 <= K_sel <= N; 0 <= D <= K, D <= N - K; N < 2^32.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
size_t usaf_select_and_swap_workspace_size(int64_t N, int64_t K_sel, int64_t K, int64_t D);
usaf_status usaf_select_and_swap(const float* g, int64_t N, int64_t K_sel, int64_t* sel_idx,
                                 const int64_t* act_idx, int64_t K, int64_t D, const float* p_in,
                                 const float* m_in, const float* v_in, const void* w_seg0,
                                 int64_t n_seg0, const void* w_seg1, usaf_dtype w_dtype,
                                 int64_t* new_idx, float* p_out, float* m_out, float* v_out,
                                 int64_t* n_swapped, uint32_t* dev_status, void* ws,
                                 size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_reselect_full - reselection by re-ranking (USAF README, "Sparsity adapts": the active set
 * is chosen again from fresh gradient magnitudes, with the large turnover the README reports at
 * the first reselections): new_idx = the K entries with the largest |g| (ties: lower flat index
 * first), sorted, exactly as usaf_importance_select. Entries that were in old_idx carry their
 * p, m, v; entries new to the set start with p = the dense weight value and m = v = 0.
 *   g            [N] fp32 dense gradient
 *   old_idx      [K_old] sorted previous active set; p_in, m_in, v_in [K_old] aligned with it
 *   w_seg0/n_seg0/w_seg1/w_dtype   dense weights, as for usaf_sparse_adam_step
 *   new_idx, p_out, m_out, v_out   [K] out; must not overlap the inputs
 *   n_kept       [1] int64 out: entries of new_idx that were in old_idx
 * Limits: 0 <= K, K_old <= N < 2^32. Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
size_t usaf_reselect_full_workspace_size(int64_t N, int64_t K);
usaf_status usaf_reselect_full(const float* g, int64_t N, int64_t K, const int64_t* old_idx,
                               int64_t K_old, const float* p_in, const float* m_in,
                               const float* v_in, const void* w_seg0, int64_t n_seg0,
                               const void* w_seg1, usaf_dtype w_dtype, int64_t* new_idx,
                               float* p_out, float* m_out, float* v_out, int64_t* n_kept,
                               uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Selection spread over data-parallel ranks (the importance pass of the README's DataParallel
 * mode, "Multi-GPU (DataParallel)"; every rank holds the same weights and active set). After a
 * reduce-scatter of the dense gradient each rank holds a contiguous part g[0, n) of it, at global
 * offset `base`. The top-K of |g| over all parts (ties to the lower global index) is found by
 * digit rounds: each rank forms the digit histogram of its part, the histograms are summed over
 * the ranks, and every rank picks the same digit. A rank's own histograms also give its counts
 * above and at the final threshold; the tie quota is split in rank order, and each rank emits its
 * winners, which an all-gather concatenates into the sorted set. The exchanges and the digit
 * picks are the caller's (see sparse_moe_fine_gb300/dist_select.py); these calls are the per-part
 * kernels. Keys are |g| as the fp32 bit pattern with the sign cleared. excl (may be NULL): n-bit
 * bitmap of excluded entries of the part (RigL's grow set excludes the active set), from
 * usaf_active_bitmap.
 *   usaf_shard_key_histogram  hist[d] += keys whose bits above shift+bits equal prefix's, by the
 *                             digit d of `bits` bits at `shift` (1 <= bits <= 11,
 *                             shift + bits <= 31); hist [2^bits]
 *   usaf_shard_emit           out[0 .. gt + take_eq) = base + i for the part's keys > tau and its
 *                             first take_eq keys == tau, ascending; count = gt + eq of the part
 *                             (sizes the compaction; any value gives the same result: a
 *                             compaction region that overflows sends the part to the exact
 *                             whole-part pass and sets USAF_DEV_SELECT_EXACT_PATH)
 *   usaf_active_bitmap        bitmap [ceil(n/32)] words: bit i set when lo + i is in idx[0, K)
 * Limits: 0 <= n < 2^32. Errors: INVALID_ARG, WORKSPACE, CUDA.
 * ------------------------------------------------------------------------------------------- */
usaf_status usaf_shard_key_histogram(const float* g, int64_t n, const uint32_t* excl,
                                     uint32_t prefix, int shift, int bits,
                                     unsigned long long* hist, void* stream);
size_t usaf_shard_emit_workspace_size(int64_t n, int64_t count);
usaf_status usaf_shard_emit(const float* g, int64_t n, const uint32_t* excl, uint32_t tau,
                            int64_t take_eq, int64_t count, int64_t base, int64_t* out,
                            uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);
usaf_status usaf_active_bitmap(const int64_t* idx, int64_t K, int64_t lo, int64_t n,
                               uint32_t* bitmap, void* stream);

/* usaf_rigl_apply - usaf_rigl_swap with the grow set given (grown [D], sorted, disjoint from
 * act_idx, in [0, N); chosen across ranks): the drop selection and the merge, state as
 * usaf_rigl_swap.
 * usaf_reselect_carry - the state carry of usaf_reselect_full for a given new set new_idx [K]
 * (sorted, in [0, N)).
 * N is the number of expert weight entries (w_seg1 holds N - n_seg0). A given entry outside
 * [0, N) is not read from the weights: it gets p = 0 and sets USAF_DEV_BAD_INDEX in dev_status
 * (may be NULL); with USAF_DEBUG=1 the given sets are validated as by usaf_validate_active.
 * Workspace: usaf_rigl_apply_workspace_size(K, D), usaf_reselect_carry_workspace_size().
 * Errors: INVALID_ARG, WORKSPACE, CUDA. */
size_t usaf_rigl_apply_workspace_size(int64_t K, int64_t D);
usaf_status usaf_rigl_apply(const int64_t* act_idx, int64_t K, int64_t N, int64_t D,
                            const int64_t* grown,
                            const float* p_in, const float* m_in, const float* v_in,
                            const void* w_seg0, int64_t n_seg0, const void* w_seg1,
                            usaf_dtype w_dtype, int64_t* new_idx, float* p_out, float* m_out,
                            float* v_out, int64_t* n_swapped, uint32_t* dev_status, void* ws,
                            size_t ws_bytes, void* stream);
size_t usaf_reselect_carry_workspace_size(void);
usaf_status usaf_reselect_carry(const int64_t* new_idx, int64_t K, int64_t N,
                                const int64_t* old_idx, int64_t K_old, const float* p_in,
                                const float* m_in, const float* v_in, const void* w_seg0,
                                int64_t n_seg0, const void* w_seg1, usaf_dtype w_dtype,
                                float* p_out, float* m_out, float* v_out, int64_t* n_kept,
                                uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_validate_active - checks an active set against the contract every call above assumes
 * (USAF README, "Not all weights matter": the trained subset is a set of expert weights, here a
 * sorted list of flat indices): 0 <= idx[i] < N, and idx[i-1] < idx[i] (ascending, no repeats).
 * One kernel reads idx[0..K) and nothing else; any violation sets USAF_DEV_BAD_INDEX in
 * *dev_status (required). The host learns of it by reading the word after the stream has run it.
 * Limits: 0 <= K, 1 <= N. Errors: INVALID_ARG, CUDA.
 * ------------------------------------------------------------------------------------------- */
usaf_status usaf_validate_active(const int64_t* idx, int64_t K, int64_t N, uint32_t* dev_status,
                                 void* stream);

/* ---------------------------------------------------------------------------------------------
 * usaf_diag_bounded_wait - exercises the failure path of the tensor-core kernels' bounded waits
 * without any GPU fault. The pages have no counterpart; it exists so a test can show that a wait
 * that runs out is reported and leaves the context usable. One CTA allocates tensor memory,
 * initialises an mbarrier that nothing ever arrives on, and waits on it with the same bounded
 * wait the GEMM kernels use, limited to limit_cycles SM clock cycles; when the wait gives up it
 * sets USAF_DEV_TIMEOUT in *dev_status (required), drains its (empty) MMA pipeline with the same
 * deadline-bounded drain, frees the tensor memory and returns.
 * Limits: 1 <= limit_cycles <= 2^32 (about two seconds). Errors: INVALID_ARG, CUDA.
 * ------------------------------------------------------------------------------------------- */
usaf_status usaf_diag_bounded_wait(int64_t limit_cycles, uint32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Kernel timing trace (host side, off by default). While enabled, every kernel launch of the hot
 * path is bracketed by two CUDA events recorded on its stream, so per-kernel device time can be
 * read without a profiler. usaf_trace_enable(1) clears earlier records; usaf_trace_summary
 * waits for the recorded events, then fills up to `cap` entries (one per kernel name, in order
 * of first launch) and returns how many names were seen, or -1 on a CUDA error. The trace times
 * launches issued directly; keep it off while capturing calls into a CUDA graph, since events
 * recorded during a capture mark graph dependencies and are never timed.
 * ------------------------------------------------------------------------------------------- */
typedef struct {
  char name[48];
  int64_t launches;
  double total_ms;
} usaf_trace_entry;

usaf_status usaf_trace_enable(int on);
int usaf_trace_summary(usaf_trace_entry* out, int cap);

/* Number of kernel launches the library has issued since it was loaded (all threads). A caller
 * can difference two readings to count the device work behind a sequence of calls. A call
 * captured into a CUDA graph counts its launches once, at capture; replays of the graph add
 * nothing, so a caller that replays graphs counts their kernels itself. */
int64_t usaf_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* USAF_H */
