// usaf_route_topk_noalloc: the routing entry point for callers that cannot allocate device
// memory, with its scratch in a fixed array that lives in the library itself.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they route tokens:
// code that runs under a fixed, pre-planned device-memory budget (an inference/training server
// whose pool is sized once at start-up and must not grow), code called back from inside another
// runtime's allocator or memory manager, where allocating again would recurse or deadlock, and
// embedded deployments that forbid dynamic device allocation after initialisation. For them this
// variant takes no workspace argument: its scratch is the file-scope device array below, which
// every GPU that loads the library holds until the process exits.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace usaf {

namespace {

// The scratch: per-chunk expert histograms of the permutation and the bf16 split of the router
// weight for the tensor-core logits.
static __device__ __align__(256) unsigned char g_route_scratch[USAF_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_ptr[MAX_DEVICES] = {};

size_t hist_bytes(const usaf_moe_shape& s) {
  return (size_t)round_up(ceil_div(s.T * s.k, PERM_CHUNK) * s.E * (int64_t)sizeof(int32_t), 256);
}

// The bf16 split of the router weight exists only on the tensor-core logits path, the same
// condition route_launch takes it under.
size_t split_bytes(const usaf_moe_shape& s, const float* logits_in, usaf_dtype x_dtype) {
  const bool tc = !logits_in && x_dtype == USAF_BF16 && tc_shape_ok(s);
  return tc ? (size_t)(s.E * 3 * s.H * 2) : 0;
}

// Device address of the scratch array on the current device, looked up once per device.
usaf_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return USAF_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return USAF_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return USAF_OK;
}

}  // namespace

}  // namespace usaf

using namespace usaf;

extern "C" usaf_status usaf_route_topk_noalloc(const usaf_moe_shape* s, const void* x,
                                               usaf_dtype x_dtype, const float* w_router,
                                               const float* logits_in, float* logits_out,
                                               int renorm, const usaf_routing* rt,
                                               uint32_t* dev_status, void* stream) {
  if (!s || usaf_routed_rows_capacity(s) < 0) return USAF_ERR_INVALID_ARG;
  if (!rt || !rt->topk_idx || !rt->topk_w || !rt->expert_count || !rt->expert_offset ||
      !rt->perm_tok || !rt->perm_slot || !rt->slot_row)
    return USAF_ERR_INVALID_ARG;
  if (!logits_in && !logits_out) return USAF_ERR_INVALID_ARG;  // logits are never scratch here
  if (!logits_in && (!x || !w_router || (x_dtype != USAF_F32 && x_dtype != USAF_BF16)))
    return USAF_ERR_INVALID_ARG;
  if (renorm != 0 && renorm != 1) return USAF_ERR_INVALID_ARG;
  if (hist_bytes(*s) + split_bytes(*s, logits_in, x_dtype) > (size_t)USAF_NOALLOC_SCRATCH_BYTES)
    return USAF_ERR_WORKSPACE;  // the layer needs more scratch than the fixed array holds
  void* base = nullptr;
  USAF_TRY(scratch_address(&base));
  RouteWs w;
  w.logits = nullptr;
  w.chunk_hist = static_cast<int32_t*>(base);
  w.wr3 = static_cast<char*>(base) + hist_bytes(*s);
  return route_launch(*s, x, x_dtype, w_router, logits_in, logits_out, renorm, *rt, w,
                      dev_status, static_cast<cudaStream_t>(stream));
}
