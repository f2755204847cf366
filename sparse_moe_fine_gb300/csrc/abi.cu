// The extern "C" entry points declared in include/usaf.h: argument checks, workspace carving,
// and the launch sequence of each call. Everything here is host code; the arithmetic is in the
// kernel files.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.cuh"

namespace usaf {

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // clear the sticky-free error of a machine without a GPU
    return 152;
  }
  return n;
}

// ------------------------------------------------------------------ per-thread side stream
namespace {
struct SideSlot {
  bool made = false;
  SideStream ss{};
};
thread_local SideSlot t_side[16];

bool make_side(SideSlot& sl) {
  if (cudaStreamCreateWithFlags(&sl.ss.s, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&sl.ss.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&sl.ss.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  sl.made = true;
  return true;
}

SideSlot* side_slot() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) {
    cudaGetLastError();
    return nullptr;
  }
  return &t_side[dev];
}
}  // namespace

void side_stream_setup() {
  SideSlot* sl = side_slot();
  if (sl && !sl->made) make_side(*sl);
}

bool side_stream(SideStream& out, cudaStream_t st) {
  SideSlot* sl = side_slot();
  if (!sl) return false;
  if (!sl->made) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (cs != cudaStreamCaptureStatusNone || !make_side(*sl)) return false;
  }
  out = sl->ss;
  return true;
}

// ------------------------------------------------------------------ kernel timing trace
namespace {
struct TraceRec {
  std::string name;
  cudaEvent_t a, b;
};
std::atomic<bool> g_trace{false};
std::mutex g_trace_mu;
std::vector<TraceRec> g_recs;
std::vector<cudaEvent_t> g_pool;
thread_local std::vector<size_t> t_open;

cudaEvent_t pool_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
void recycle_locked() {
  for (auto& r : g_recs) {
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
}
}  // namespace

bool trace_on() { return g_trace.load(std::memory_order_relaxed); }

static std::atomic<long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void trace_begin(const char* name, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  TraceRec r{name, pool_event(), pool_event()};
  cudaEventRecord(r.a, st);
  t_open.push_back(g_recs.size());
  g_recs.push_back(r);
}

void trace_end(cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (t_open.empty()) return;
  const size_t i = t_open.back();
  t_open.pop_back();
  if (i < g_recs.size()) cudaEventRecord(g_recs[i].b, st);
}

void route_ws_layout(const usaf_moe_shape& s, Carver& c, RouteWs& w) {
  w.logits = c.take<float>(s.T * s.E);
  w.chunk_hist = c.take<int32_t>(ceil_div(s.T * s.k, PERM_CHUNK) * s.E);
  w.wr3 = c.take<char>(s.E * 3 * s.H * 2);
}

static bool shape_ok(const usaf_moe_shape* s) {
  if (!s) return false;
  if (s->T < 1 || s->H < 1 || s->E < 1 || s->k < 1 || s->I < 1) return false;
  if (s->k > s->E || s->E > 1024 || s->k > 32) return false;
  if (s->T * s->k >= (int64_t(1) << 31) - 65536) return false;
  if (s->E * 3 * s->I * s->H >= (int64_t(1) << 40)) return false;
  return true;
}

static bool routing_ok(const usaf_routing* r) {
  return r && r->topk_idx && r->topk_w && r->expert_count && r->expert_offset && r->perm_tok &&
         r->perm_slot && r->slot_row;
}

static bool dtype_ok(usaf_dtype d) { return d == USAF_F32 || d == USAF_BF16; }

// USAF_DEBUG=1 in the environment: calls that read an active set validate it first.
static bool debug_on() {
  const char* v = std::getenv("USAF_DEBUG");
  return v && v[0] == '1';
}
static usaf_status debug_validate(const int64_t* idx, int64_t K, int64_t N, uint32_t* dev_status,
                                  void* stream) {
  if (!debug_on() || !idx || K <= 0 || !dev_status) return USAF_OK;
  return validate_launch(idx, K, N, dev_status, static_cast<cudaStream_t>(stream));
}

}  // namespace usaf

using namespace usaf;

extern "C" {

int usaf_abi_version(void) { return USAF_ABI_VERSION; }

int64_t usaf_launch_count(void) { return (int64_t)g_launches.load(); }

usaf_status usaf_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  recycle_locked();
  t_open.clear();
  g_trace.store(on != 0);
  return USAF_OK;
}

int usaf_trace_summary(usaf_trace_entry* out, int cap) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  std::vector<std::string> names;
  std::vector<int64_t> cnt;
  std::vector<double> ms;
  for (auto& r : g_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return -1;
    size_t k = 0;
    while (k < names.size() && names[k] != r.name) ++k;
    if (k == names.size()) {
      names.push_back(r.name);
      cnt.push_back(0);
      ms.push_back(0.0);
    }
    cnt[k] += 1;
    ms[k] += t;
  }
  for (size_t k = 0; k < names.size() && (int)k < cap && out; ++k) {
    std::memset(out[k].name, 0, sizeof(out[k].name));
    std::strncpy(out[k].name, names[k].c_str(), sizeof(out[k].name) - 1);
    out[k].launches = cnt[k];
    out[k].total_ms = ms[k];
  }
  return (int)names.size();
}

const char* usaf_status_string(usaf_status s) {
  switch (s) {
    case USAF_OK: return "ok";
    case USAF_ERR_INVALID_ARG: return "invalid argument";
    case USAF_ERR_UNSUPPORTED: return "unsupported shape or type";
    case USAF_ERR_WORKSPACE: return "workspace missing or too small";
    case USAF_ERR_CUDA: return "CUDA error";
    case USAF_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int64_t usaf_routed_rows_capacity(const usaf_moe_shape* s) {
  if (!shape_ok(s)) return -1;
  return round_up(s->T * s->k + s->E * (USAF_ROW_ALIGN - 1), 256) + 256;
}

size_t usaf_route_topk_workspace_size(const usaf_moe_shape* s) {
  if (!shape_ok(s)) return 0;
  Carver c(nullptr);
  RouteWs w;
  route_ws_layout(*s, c, w);
  return c.size();
}

usaf_status usaf_route_topk(const usaf_moe_shape* s, const void* x, usaf_dtype x_dtype,
                            const float* w_router, const float* logits_in, float* logits_out,
                            int renorm, const usaf_routing* rt, uint32_t* dev_status, void* ws,
                            size_t ws_bytes, void* stream) {
  if (!shape_ok(s) || !routing_ok(rt)) return USAF_ERR_INVALID_ARG;
  if (!logits_in && (!x || !w_router || !dtype_ok(x_dtype))) return USAF_ERR_INVALID_ARG;
  if (renorm != 0 && renorm != 1) return USAF_ERR_INVALID_ARG;
  const size_t need = usaf_route_topk_workspace_size(s);
  if (!ws || ws_bytes < need) return USAF_ERR_WORKSPACE;
  Carver c(ws);
  RouteWs w;
  route_ws_layout(*s, c, w);
  return route_launch(*s, x, x_dtype, w_router, logits_in, logits_out, renorm, *rt, w,
                      dev_status, static_cast<cudaStream_t>(stream));
}

size_t usaf_moe_fwd_workspace_size(const usaf_moe_shape* s, usaf_dtype dt) {
  if (!shape_ok(s) || !dtype_ok(dt)) return 0;
  Carver c(nullptr);
  FwdWs w;
  fwd_ws_layout(*s, dt, c, w);
  return c.size();
}

static usaf_status fill_args(MoeArgs& a, const usaf_moe_shape* s, usaf_dtype dt, const void* x,
                             const float* wr, const void* wgu, const void* wd,
                             const usaf_routing* rt) {
  if (!shape_ok(s) || !dtype_ok(dt) || !routing_ok(rt) || !x || !wgu || !wd)
    return USAF_ERR_INVALID_ARG;
  if (dt == USAF_BF16 && !tc_shape_ok(*s)) return USAF_ERR_UNSUPPORTED;
  // feature-major rows are addressed by 32-bit 16-byte-vector indices
  const int64_t vw = dt == USAF_BF16 ? 8 : 4;
  if (std::max<int64_t>(2 * s->I, s->H) * usaf_routed_rows_capacity(s) / vw >= INT32_MAX)
    return USAF_ERR_UNSUPPORTED;
  a.s = *s;
  a.dt = dt;
  a.R_cap = usaf_routed_rows_capacity(s);
  a.x = x;
  a.w_router = wr;
  a.w_gate_up = wgu;
  a.w_down = wd;
  a.rt = *rt;
  return USAF_OK;
}

static usaf_status moe_fwd_entry(const usaf_moe_shape* s, usaf_dtype dt, const void* x,
                                 const void* w_gate_up, const void* w_down,
                                 const usaf_routing* rt, void* x_perm_save, void* h_save,
                                 void* wa_save, void* y, void* gate_up_ready, void* down_ready,
                                 int stages, uint32_t* dev_status, void* ws, size_t ws_bytes,
                                 void* stream) {
  MoeArgs a{};
  USAF_TRY(fill_args(a, s, dt, x, nullptr, w_gate_up, w_down, rt));
  a.status = dev_status;
  if (!x_perm_save || !h_save || !wa_save || !y) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_moe_fwd_workspace_size(s, dt)) return USAF_ERR_WORKSPACE;
  Carver c(ws);
  FwdWs w;
  fwd_ws_layout(*s, dt, c, w);
  return moe_fwd_launch(a, x_perm_save, h_save, wa_save, y, w,
                        static_cast<cudaEvent_t>(gate_up_ready),
                        static_cast<cudaEvent_t>(down_ready), stages,
                        static_cast<cudaStream_t>(stream));
}

usaf_status usaf_moe_fwd_wait2(const usaf_moe_shape* s, usaf_dtype dt, const void* x,
                               const void* w_gate_up, const void* w_down, const usaf_routing* rt,
                               void* x_perm_save, void* h_save, void* wa_save, void* y,
                               void* gate_up_ready, void* down_ready, uint32_t* dev_status,
                               void* ws, size_t ws_bytes, void* stream) {
  return moe_fwd_entry(s, dt, x, w_gate_up, w_down, rt, x_perm_save, h_save, wa_save, y,
                       gate_up_ready, down_ready, FWD_ALL, dev_status, ws, ws_bytes, stream);
}

usaf_status usaf_moe_fwd_stage(const usaf_moe_shape* s, usaf_dtype dt, const void* x,
                               const void* w_gate_up, const void* w_down, const usaf_routing* rt,
                               void* x_perm_save, void* h_save, void* wa_save, void* y,
                               int stages, uint32_t* dev_status, void* ws, size_t ws_bytes,
                               void* stream) {
  if (stages < 1 || stages > FWD_ALL) return USAF_ERR_INVALID_ARG;
  return moe_fwd_entry(s, dt, x, w_gate_up, w_down, rt, x_perm_save, h_save, wa_save, y, nullptr,
                       nullptr, stages, dev_status, ws, ws_bytes, stream);
}

usaf_status usaf_moe_fwd_wait(const usaf_moe_shape* s, usaf_dtype dt, const void* x,
                              const void* w_gate_up, const void* w_down, const usaf_routing* rt,
                              void* x_perm_save, void* h_save, void* wa_save, void* y,
                              void* weights_ready, uint32_t* dev_status, void* ws,
                              size_t ws_bytes, void* stream) {
  return usaf_moe_fwd_wait2(s, dt, x, w_gate_up, w_down, rt, x_perm_save, h_save, wa_save, y,
                            weights_ready, nullptr, dev_status, ws, ws_bytes, stream);
}

usaf_status usaf_moe_fwd(const usaf_moe_shape* s, usaf_dtype dt, const void* x,
                         const void* w_gate_up, const void* w_down, const usaf_routing* rt,
                         void* x_perm_save, void* h_save, void* wa_save, void* y,
                         uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  return usaf_moe_fwd_wait(s, dt, x, w_gate_up, w_down, rt, x_perm_save, h_save, wa_save, y,
                           nullptr, dev_status, ws, ws_bytes, stream);
}

size_t usaf_moe_bwd_workspace_size(const usaf_moe_shape* s, usaf_dtype dt, int64_t K) {
  if (!shape_ok(s) || !dtype_ok(dt) || K < 0) return 0;
  side_stream_setup();  // a host-only call: the backward's side stream is created here
  Carver c(nullptr);
  BwdWs w;
  bwd_ws_layout(*s, dt, K, c, w);
  return c.size();
}

int64_t usaf_moe_bwd_dlogit_offset(const usaf_moe_shape* s, usaf_dtype dt, int64_t K) {
  if (!shape_ok(s) || !dtype_ok(dt) || K < 0) return -1;
  Carver c(reinterpret_cast<void*>(uintptr_t(256)));  // a nonzero base: offsets, not sizes
  BwdWs w;
  bwd_ws_layout(*s, dt, K, c, w);
  return (int64_t)(reinterpret_cast<char*>(w.dl) - reinterpret_cast<char*>(uintptr_t(256)));
}

usaf_status usaf_moe_bwd_sparse(const usaf_moe_shape* s, usaf_dtype dt, int renorm,
                                const void* x, const float* w_router, const void* w_gate_up,
                                const void* w_down, const usaf_routing* rt, const float* logits,
                                const void* x_perm_save, const void* h_save, const void* wa_save,
                                const void* dy, const int64_t* act_idx, int64_t K, float* g_act,
                                float* g_router, void* dx, float* dw_slot, uint32_t* dev_status,
                                void* ws, size_t ws_bytes, void* stream) {
  MoeArgs a{};
  USAF_TRY(fill_args(a, s, dt, x, w_router, w_gate_up, w_down, rt));
  a.status = dev_status;
  if (renorm != 0 && renorm != 1) return USAF_ERR_INVALID_ARG;
  if (!w_router || !x_perm_save || !h_save || !wa_save || !dy || !g_router)
    return USAF_ERR_INVALID_ARG;
  if (renorm == 0 && !logits) return USAF_ERR_INVALID_ARG;
  const int64_t N = s->E * 3 * s->I * s->H;
  if (K < 0 || K > N || (K > 0 && (!act_idx || !g_act))) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_moe_bwd_workspace_size(s, dt, K)) return USAF_ERR_WORKSPACE;
  USAF_TRY(debug_validate(act_idx, K, N, dev_status, stream));
  Carver c(ws);
  BwdWs w;
  bwd_ws_layout(*s, dt, K, c, w);
  return moe_bwd_launch(a, renorm, logits, x_perm_save, h_save, wa_save, dy, act_idx, K, g_act,
                        g_router, dx, dw_slot, nullptr, 0, dev_status, w,
                        static_cast<cudaStream_t>(stream));
}

usaf_status usaf_moe_bwd_sparse_accumulate(
    const usaf_moe_shape* s, usaf_dtype dt, int renorm, const void* x, const float* w_router,
    const void* w_gate_up, const void* w_down, const usaf_routing* rt, const float* logits,
    const void* x_perm_save, const void* h_save, const void* wa_save, const void* dy,
    const int64_t* act_idx, int64_t K, float* g_act, float* g_router, void* dx, float* dw_slot,
    uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  MoeArgs a{};
  USAF_TRY(fill_args(a, s, dt, x, w_router, w_gate_up, w_down, rt));
  a.status = dev_status;
  if (renorm != 0 && renorm != 1) return USAF_ERR_INVALID_ARG;
  if (!w_router || !x_perm_save || !h_save || !wa_save || !dy || !g_router)
    return USAF_ERR_INVALID_ARG;
  if (renorm == 0 && !logits) return USAF_ERR_INVALID_ARG;
  const int64_t N = s->E * 3 * s->I * s->H;
  if (K < 0 || K > N || (K > 0 && (!act_idx || !g_act))) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_moe_bwd_workspace_size(s, dt, K)) return USAF_ERR_WORKSPACE;
  USAF_TRY(debug_validate(act_idx, K, N, dev_status, stream));
  Carver c(ws);
  BwdWs w;
  bwd_ws_layout(*s, dt, K, c, w);
  return moe_bwd_launch(a, renorm, logits, x_perm_save, h_save, wa_save, dy, act_idx, K, g_act,
                        g_router, dx, dw_slot, nullptr, 1, dev_status, w,
                        static_cast<cudaStream_t>(stream));
}

size_t usaf_masked_plan_size(const usaf_moe_shape* s) {
  if (!shape_ok(s)) return 0;
  return masked_plan_bytes(*s);
}

usaf_status usaf_masked_plan_build(const usaf_moe_shape* s, const int64_t* act_idx, int64_t K,
                                   double dense_density, void* plan, size_t plan_bytes,
                                   void* stream) {
  if (!shape_ok(s) || !plan || K < 0 || (K > 0 && !act_idx)) return USAF_ERR_INVALID_ARG;
  if (!(dense_density > 0.0)) return USAF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(plan) & 255) != 0) return USAF_ERR_INVALID_ARG;
  if (K > s->E * 3 * s->I * s->H) return USAF_ERR_INVALID_ARG;
  if (plan_bytes < masked_plan_bytes(*s)) return USAF_ERR_WORKSPACE;
  const double thr = std::ceil(dense_density * (double)(3 * s->I * s->H));
  const int64_t thr_count = thr > 9.0e18 ? INT64_MAX : std::max<int64_t>(1, (int64_t)thr);
  return masked_plan_build_launch(*s, act_idx, K, thr_count, plan,
                                  static_cast<cudaStream_t>(stream));
}

usaf_status usaf_moe_bwd_sparse_planned(
    const usaf_moe_shape* s, usaf_dtype dt, int renorm, const void* x, const float* w_router,
    const void* w_gate_up, const void* w_down, const usaf_routing* rt, const float* logits,
    const void* x_perm_save, const void* h_save, const void* wa_save, const void* dy,
    const int64_t* act_idx, int64_t K, float* g_act, float* g_router, void* dx, float* dw_slot,
    int accumulate, const void* plan, int64_t n_dense, uint32_t* dev_status, void* ws,
    size_t ws_bytes, void* stream) {
  MoeArgs a{};
  USAF_TRY(fill_args(a, s, dt, x, w_router, w_gate_up, w_down, rt));
  a.status = dev_status;
  if (renorm != 0 && renorm != 1) return USAF_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return USAF_ERR_INVALID_ARG;
  if (!w_router || !x_perm_save || !h_save || !wa_save || !dy || !g_router)
    return USAF_ERR_INVALID_ARG;
  if (renorm == 0 && !logits) return USAF_ERR_INVALID_ARG;
  const int64_t N = s->E * 3 * s->I * s->H;
  if (K < 0 || K > N || (K > 0 && (!act_idx || !g_act))) return USAF_ERR_INVALID_ARG;
  if (n_dense < 0 || n_dense > s->E || (n_dense > 0 && !plan)) return USAF_ERR_INVALID_ARG;
  if (plan && (reinterpret_cast<uintptr_t>(plan) & 255) != 0) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_moe_bwd_workspace_size(s, dt, K)) return USAF_ERR_WORKSPACE;
  USAF_TRY(debug_validate(act_idx, K, N, dev_status, stream));
  Carver c(ws);
  BwdWs w;
  bwd_ws_layout(*s, dt, K, c, w);
  MaskedPlan mp{};
  if (n_dense > 0) mp = masked_plan_layout(*s, const_cast<void*>(plan));
  return moe_bwd_launch(a, renorm, logits, x_perm_save, h_save, wa_save, dy, act_idx, K, g_act,
                        g_router, dx, dw_slot, nullptr, accumulate, dev_status, w,
                        static_cast<cudaStream_t>(stream), n_dense > 0 ? &mp : nullptr,
                        n_dense);
}

usaf_status usaf_moe_bwd_dense(const usaf_moe_shape* s, usaf_dtype dt, int renorm, const void* x,
                               const float* w_router, const void* w_gate_up, const void* w_down,
                               const usaf_routing* rt, const float* logits,
                               const void* x_perm_save, const void* h_save, const void* wa_save,
                               const void* dy, float* g_dense, int accumulate, float* g_router,
                               void* dx, float* dw_slot, uint32_t* dev_status, void* ws,
                               size_t ws_bytes, void* stream) {
  MoeArgs a{};
  USAF_TRY(fill_args(a, s, dt, x, w_router, w_gate_up, w_down, rt));
  a.status = dev_status;
  if (renorm != 0 && renorm != 1) return USAF_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return USAF_ERR_INVALID_ARG;
  if (!w_router || !x_perm_save || !h_save || !wa_save || !dy || !g_router || !g_dense)
    return USAF_ERR_INVALID_ARG;
  if (renorm == 0 && !logits) return USAF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(g_dense) & 15) != 0) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_moe_bwd_workspace_size(s, dt, 0)) return USAF_ERR_WORKSPACE;
  Carver c(ws);
  BwdWs w;
  bwd_ws_layout(*s, dt, 0, c, w);
  return moe_bwd_launch(a, renorm, logits, x_perm_save, h_save, wa_save, dy, nullptr, 0, nullptr,
                        g_router, dx, dw_slot, g_dense, accumulate, dev_status, w,
                        static_cast<cudaStream_t>(stream));
}

usaf_status usaf_moe_wgrad_dense(const usaf_moe_shape* s, usaf_dtype dt, const usaf_routing* rt,
                                 const void* x_perm_save, const void* wa_save, float* g_dense,
                                 int accumulate, uint32_t* dev_status, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (!shape_ok(s) || !dtype_ok(dt) || !routing_ok(rt)) return USAF_ERR_INVALID_ARG;
  if (dt == USAF_BF16 && !tc_shape_ok(*s)) return USAF_ERR_UNSUPPORTED;
  if (!x_perm_save || !wa_save || !g_dense) return USAF_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return USAF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(g_dense) & 15) != 0) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_moe_bwd_workspace_size(s, dt, 0)) return USAF_ERR_WORKSPACE;
  MoeArgs a{};
  a.s = *s;
  a.dt = dt;
  a.R_cap = usaf_routed_rows_capacity(s);
  a.rt = *rt;
  a.status = dev_status;
  Carver c(ws);
  BwdWs w;
  bwd_ws_layout(*s, dt, 0, c, w);
  return moe_wgrad_dense_launch(a, x_perm_save, wa_save, g_dense, accumulate, w,
                                static_cast<cudaStream_t>(stream));
}

usaf_status usaf_sparse_adam_step(int64_t n, const int64_t* idx, const float* g, float* p,
                                  float* m, float* v, void* w_seg0, int64_t n_seg0, void* w_seg1,
                                  usaf_dtype w_dtype, double lr, double beta1, double beta2,
                                  double eps, int64_t step, int skip_if_nonfinite,
                                  uint32_t* dev_status, void* stream) {
  if (n < 0 || step < 1 || !dtype_ok(w_dtype) || n_seg0 < 0) return USAF_ERR_INVALID_ARG;
  if (n > 0 && (!g || !p || !m || !v || !w_seg0)) return USAF_ERR_INVALID_ARG;
  if (!idx && n > n_seg0) return USAF_ERR_INVALID_ARG;
  if (skip_if_nonfinite < 0 || skip_if_nonfinite > 2) return USAF_ERR_INVALID_ARG;
  if (skip_if_nonfinite && !dev_status) return USAF_ERR_INVALID_ARG;
  if (!(beta1 >= 0.0 && beta1 < 1.0 && beta2 >= 0.0 && beta2 < 1.0 && eps >= 0.0))
    return USAF_ERR_INVALID_ARG;
  // the set's bound is not known here: only order and sign are checked (N = INT64_MAX)
  USAF_TRY(debug_validate(idx, n, INT64_MAX, dev_status, stream));
  return adam_launch(n, idx, g, p, m, v, w_seg0, n_seg0, w_seg1, w_dtype, lr, beta1, beta2, eps,
                     step, skip_if_nonfinite, dev_status, static_cast<cudaStream_t>(stream));
}

usaf_status usaf_scan_nonfinite(const float* g, int64_t n, uint32_t* dev_status, void* stream) {
  if (n < 0 || (n > 0 && !g) || !dev_status) return USAF_ERR_INVALID_ARG;
  return nonfinite_scan_launch(g, n, dev_status, static_cast<cudaStream_t>(stream));
}

size_t usaf_importance_select_workspace_size(int64_t N, int64_t K) {
  if (N < 1 || K < 1 || K > N || N >= (int64_t(1) << 32)) return 0;
  return select_ws_bytes(N, K, false);
}

usaf_status usaf_importance_select(const float* g, int64_t N, int64_t K, int64_t* out_idx,
                                   uint32_t* dev_status, void* ws, size_t ws_bytes,
                                   void* stream) {
  if (!g || !out_idx || N < 1 || K < 1 || K > N) return USAF_ERR_INVALID_ARG;
  if (N >= (int64_t(1) << 32)) return USAF_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < usaf_importance_select_workspace_size(N, K)) return USAF_ERR_WORKSPACE;
  return importance_select_launch(g, N, K, out_idx, dev_status, ws,
                                  static_cast<cudaStream_t>(stream));
}

size_t usaf_rigl_swap_workspace_size(int64_t N, int64_t K, int64_t D) {
  if (N < 1 || K < 0 || K > N || D < 0 || D > K || D > N - K || N >= (int64_t(1) << 32))
    return 0;
  return rigl_ws_bytes(N, K, D);
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

usaf_status usaf_rigl_swap(const float* g, int64_t N, const int64_t* act_idx, int64_t K,
                           int64_t D, const float* p_in, const float* m_in, const float* v_in,
                           const void* w_seg0, int64_t n_seg0, const void* w_seg1,
                           usaf_dtype w_dtype, int64_t* new_idx, float* p_out, float* m_out,
                           float* v_out, int64_t* n_swapped, uint32_t* dev_status, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!g || N < 1 || K < 0 || K > N || D < 0 || D > K || D > N - K || !n_swapped)
    return USAF_ERR_INVALID_ARG;
  if (!dtype_ok(w_dtype) || n_seg0 < 0) return USAF_ERR_INVALID_ARG;
  if (K > 0 && (!act_idx || !p_in || !m_in || !v_in || !new_idx || !p_out || !m_out || !v_out))
    return USAF_ERR_INVALID_ARG;
  if (D > 0 && (!w_seg0 || (N > n_seg0 && !w_seg1))) return USAF_ERR_INVALID_ARG;
  if (N >= (int64_t(1) << 32)) return USAF_ERR_UNSUPPORTED;
  const size_t kb = size_t(K) * 4;
  const void* ins[4] = {p_in, m_in, v_in, act_idx};
  const size_t insz[4] = {kb, kb, kb, size_t(K) * 8};
  const void* outs[4] = {p_out, m_out, v_out, new_idx};
  const size_t outsz[4] = {kb, kb, kb, size_t(K) * 8};
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j)
      if (overlaps(ins[i], insz[i], outs[j], outsz[j])) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_rigl_swap_workspace_size(N, K, D)) return USAF_ERR_WORKSPACE;
  USAF_TRY(debug_validate(act_idx, K, N, dev_status, stream));
  return rigl_launch(g, N, act_idx, K, D, p_in, m_in, v_in, w_seg0, n_seg0, w_seg1, w_dtype,
                     new_idx, p_out, m_out, v_out, n_swapped, dev_status, ws,
                     static_cast<cudaStream_t>(stream));
}

size_t usaf_select_and_swap_workspace_size(int64_t N, int64_t K_sel, int64_t K, int64_t D) {
  if (usaf_rigl_swap_workspace_size(N, K, D) == 0 || K_sel < 1 || K_sel > N) return 0;
  return select_and_swap_ws_bytes(N, K_sel, K, D);
}

usaf_status usaf_select_and_swap(const float* g, int64_t N, int64_t K_sel, int64_t* sel_idx,
                                 const int64_t* act_idx, int64_t K, int64_t D, const float* p_in,
                                 const float* m_in, const float* v_in, const void* w_seg0,
                                 int64_t n_seg0, const void* w_seg1, usaf_dtype w_dtype,
                                 int64_t* new_idx, float* p_out, float* m_out, float* v_out,
                                 int64_t* n_swapped, uint32_t* dev_status, void* ws,
                                 size_t ws_bytes, void* stream) {
  if (!g || N < 1 || K < 0 || K > N || D < 0 || D > K || D > N - K || !n_swapped)
    return USAF_ERR_INVALID_ARG;
  if (K_sel < 1 || K_sel > N || !sel_idx) return USAF_ERR_INVALID_ARG;
  if (!dtype_ok(w_dtype) || n_seg0 < 0) return USAF_ERR_INVALID_ARG;
  if (K > 0 && (!act_idx || !p_in || !m_in || !v_in || !new_idx || !p_out || !m_out || !v_out))
    return USAF_ERR_INVALID_ARG;
  if (D > 0 && (!w_seg0 || (N > n_seg0 && !w_seg1))) return USAF_ERR_INVALID_ARG;
  if (N >= (int64_t(1) << 32)) return USAF_ERR_UNSUPPORTED;
  const size_t kb = size_t(K) * 4;
  const void* ins[5] = {p_in, m_in, v_in, act_idx, g};
  const size_t insz[5] = {kb, kb, kb, size_t(K) * 8, size_t(N) * 4};
  const void* outs[5] = {p_out, m_out, v_out, new_idx, sel_idx};
  const size_t outsz[5] = {kb, kb, kb, size_t(K) * 8, size_t(K_sel) * 8};
  for (int i = 0; i < 5; ++i)
    for (int j = 0; j < 5; ++j)
      if (overlaps(ins[i], insz[i], outs[j], outsz[j])) return USAF_ERR_INVALID_ARG;
  for (int j = 0; j < 4; ++j)
    if (overlaps(sel_idx, size_t(K_sel) * 8, outs[j], outsz[j])) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_select_and_swap_workspace_size(N, K_sel, K, D))
    return USAF_ERR_WORKSPACE;
  USAF_TRY(debug_validate(act_idx, K, N, dev_status, stream));
  return select_and_swap_launch(g, N, K_sel, sel_idx, act_idx, K, D, p_in, m_in, v_in, w_seg0,
                                n_seg0, w_seg1, w_dtype, new_idx, p_out, m_out, v_out, n_swapped,
                                dev_status, ws, static_cast<cudaStream_t>(stream));
}

size_t usaf_reselect_full_workspace_size(int64_t N, int64_t K) {
  if (N < 1 || K < 0 || K > N || N >= (int64_t(1) << 32)) return 0;
  return reselect_ws_bytes(N, K);
}

usaf_status usaf_reselect_full(const float* g, int64_t N, int64_t K, const int64_t* old_idx,
                               int64_t K_old, const float* p_in, const float* m_in,
                               const float* v_in, const void* w_seg0, int64_t n_seg0,
                               const void* w_seg1, usaf_dtype w_dtype, int64_t* new_idx,
                               float* p_out, float* m_out, float* v_out, int64_t* n_kept,
                               uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  if (!g || N < 1 || K < 0 || K > N || K_old < 0 || K_old > N || !n_kept)
    return USAF_ERR_INVALID_ARG;
  if (!dtype_ok(w_dtype) || n_seg0 < 0) return USAF_ERR_INVALID_ARG;
  if (K_old > 0 && (!old_idx || !p_in || !m_in || !v_in)) return USAF_ERR_INVALID_ARG;
  if (K > 0 && (!new_idx || !p_out || !m_out || !v_out || !w_seg0 || (N > n_seg0 && !w_seg1)))
    return USAF_ERR_INVALID_ARG;
  if (N >= (int64_t(1) << 32)) return USAF_ERR_UNSUPPORTED;
  const void* ins[4] = {p_in, m_in, v_in, old_idx};
  const size_t insz[4] = {size_t(K_old) * 4, size_t(K_old) * 4, size_t(K_old) * 4,
                          size_t(K_old) * 8};
  const void* outs[4] = {p_out, m_out, v_out, new_idx};
  const size_t outsz[4] = {size_t(K) * 4, size_t(K) * 4, size_t(K) * 4, size_t(K) * 8};
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j)
      if (overlaps(ins[i], insz[i], outs[j], outsz[j])) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_reselect_full_workspace_size(N, K)) return USAF_ERR_WORKSPACE;
  USAF_TRY(debug_validate(old_idx, K_old, N, dev_status, stream));
  return reselect_launch(g, N, K, old_idx, K_old, p_in, m_in, v_in, w_seg0, n_seg0, w_seg1,
                         w_dtype, new_idx, p_out, m_out, v_out, n_kept, dev_status, ws,
                         static_cast<cudaStream_t>(stream));
}

usaf_status usaf_shard_key_histogram(const float* g, int64_t n, const uint32_t* excl,
                                     uint32_t prefix, int shift, int bits,
                                     unsigned long long* hist, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || (n > 0 && !g) || !hist) return USAF_ERR_INVALID_ARG;
  if (bits < 1 || bits > 11 || shift < 0 || shift + bits > 31) return USAF_ERR_INVALID_ARG;
  return shard_hist_launch(g, n, excl, prefix, shift, bits, hist,
                           static_cast<cudaStream_t>(stream));
}

size_t usaf_shard_emit_workspace_size(int64_t n, int64_t count) {
  if (n < 0 || n >= (int64_t(1) << 32) || count < 0) return 0;
  return shard_emit_ws_bytes(n, count);
}

usaf_status usaf_shard_emit(const float* g, int64_t n, const uint32_t* excl, uint32_t tau,
                            int64_t take_eq, int64_t count, int64_t base, int64_t* out,
                            uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || (n > 0 && (!g || !out)) || take_eq < 0 ||
      take_eq > n || count < 0 || base < 0)
    return USAF_ERR_INVALID_ARG;
  if (n > 0 && (!ws || ws_bytes < shard_emit_ws_bytes(n, count))) return USAF_ERR_WORKSPACE;
  return shard_emit_launch(g, n, excl, tau, take_eq, count, base, out, dev_status, ws,
                           static_cast<cudaStream_t>(stream));
}

usaf_status usaf_active_bitmap(const int64_t* idx, int64_t K, int64_t lo, int64_t n,
                               uint32_t* bitmap, void* stream) {
  if (K < 0 || (K > 0 && !idx) || n < 1 || !bitmap || lo < 0) return USAF_ERR_INVALID_ARG;
  return bitmap_range_launch(idx, K, lo, n, bitmap, static_cast<cudaStream_t>(stream));
}

size_t usaf_rigl_apply_workspace_size(int64_t K, int64_t D) {
  if (K < 0 || D < 0 || D > K) return 0;
  Carver c(nullptr);
  c.take<int64_t>(D);
  c.take<int64_t>(D);
  c.take<char>(select_ws_bytes(K > 0 ? K : 1, D > 0 ? D : 1, false));
  return c.size();
}

usaf_status usaf_rigl_apply(const int64_t* act_idx, int64_t K, int64_t N, int64_t D,
                            const int64_t* grown,
                            const float* p_in, const float* m_in, const float* v_in,
                            const void* w_seg0, int64_t n_seg0, const void* w_seg1,
                            usaf_dtype w_dtype, int64_t* new_idx, float* p_out, float* m_out,
                            float* v_out, int64_t* n_swapped, uint32_t* dev_status, void* ws,
                            size_t ws_bytes, void* stream) {
  if (K < 0 || D < 0 || D > K || K > N || !n_swapped || !dtype_ok(w_dtype) || n_seg0 < 0 ||
      n_seg0 > N)
    return USAF_ERR_INVALID_ARG;
  if (K > 0 && (!act_idx || !p_in || !m_in || !v_in || !new_idx || !p_out || !m_out || !v_out))
    return USAF_ERR_INVALID_ARG;
  if (D > 0 && (!grown || !w_seg0 || (N > n_seg0 && !w_seg1))) return USAF_ERR_INVALID_ARG;
  const size_t kb = size_t(K) * 4;
  const void* ins[4] = {p_in, m_in, v_in, act_idx};
  const size_t insz[4] = {kb, kb, kb, size_t(K) * 8};
  const void* outs[4] = {p_out, m_out, v_out, new_idx};
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j)
      if (overlaps(ins[i], insz[i], outs[j], insz[j])) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < usaf_rigl_apply_workspace_size(K, D)) return USAF_ERR_WORKSPACE;
  USAF_TRY(debug_validate(act_idx, K, N, dev_status, stream));
  USAF_TRY(debug_validate(grown, D, N, dev_status, stream));
  return rigl_launch(nullptr, N, act_idx, K, D, p_in, m_in, v_in, w_seg0, n_seg0, w_seg1,
                     w_dtype, new_idx, p_out, m_out, v_out, n_swapped, dev_status, ws,
                     static_cast<cudaStream_t>(stream), D > 0 ? grown : act_idx);
}

size_t usaf_reselect_carry_workspace_size(void) { return reselect_carry_ws_bytes(); }

usaf_status usaf_reselect_carry(const int64_t* new_idx, int64_t K, int64_t N,
                                const int64_t* old_idx, int64_t K_old, const float* p_in,
                                const float* m_in, const float* v_in, const void* w_seg0,
                                int64_t n_seg0, const void* w_seg1, usaf_dtype w_dtype,
                                float* p_out, float* m_out, float* v_out, int64_t* n_kept,
                                uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  if (K < 0 || K_old < 0 || K > N || K_old > N || !n_kept || !dtype_ok(w_dtype) || n_seg0 < 0 ||
      n_seg0 > N)
    return USAF_ERR_INVALID_ARG;
  if (K > 0 && (!new_idx || !p_out || !m_out || !v_out || !w_seg0 || (N > n_seg0 && !w_seg1)))
    return USAF_ERR_INVALID_ARG;
  if (K_old > 0 && (!old_idx || !p_in || !m_in || !v_in)) return USAF_ERR_INVALID_ARG;
  if (!ws || ws_bytes < reselect_carry_ws_bytes()) return USAF_ERR_WORKSPACE;
  USAF_TRY(debug_validate(new_idx, K, N, dev_status, stream));
  return reselect_carry_launch(new_idx, K, N, old_idx, K_old, p_in, m_in, v_in, w_seg0, n_seg0,
                               w_seg1, w_dtype, p_out, m_out, v_out, n_kept, dev_status, ws,
                               static_cast<cudaStream_t>(stream));
}

usaf_status usaf_validate_active(const int64_t* idx, int64_t K, int64_t N, uint32_t* dev_status,
                                 void* stream) {
  if (K < 0 || N < 1 || !dev_status || (K > 0 && !idx)) return USAF_ERR_INVALID_ARG;
  return validate_launch(idx, K, N, dev_status, static_cast<cudaStream_t>(stream));
}

usaf_status usaf_diag_bounded_wait(int64_t limit_cycles, uint32_t* dev_status, void* stream) {
  if (limit_cycles < 1 || limit_cycles > (int64_t(1) << 32) || !dev_status)
    return USAF_ERR_INVALID_ARG;
  return diag_wait_launch(limit_cycles, dev_status, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
