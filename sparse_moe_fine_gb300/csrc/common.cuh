// Shared device/host helpers of the USAF GB300 library (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "usaf.h"

namespace usaf {

void count_launch();

#define USAF_CHECK_LAUNCH()                                        \
  do {                                                             \
    ::usaf::count_launch();                                        \
    cudaError_t e_ = cudaGetLastError();                           \
    if (e_ != cudaSuccess) return USAF_ERR_CUDA;                   \
  } while (0)

#define USAF_TRY(expr)                                             \
  do {                                                             \
    usaf_status s_ = (expr);                                       \
    if (s_ != USAF_OK) return s_;                                  \
  } while (0)

static inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
static inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
// blocks for a grid-stride loop over n elements with 256 threads
static inline unsigned grid_dim_for(int64_t n) {
  int64_t b = ceil_div(n, 256);
  return (unsigned)(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

// ------------------------------------------------------------------------------------------------
// Workspace carving: the same code computes sizes (base == nullptr) and pointers.
// ------------------------------------------------------------------------------------------------
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(int64_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += size_t(count > 0 ? count : 0) * sizeof(T);
    return p;
  }
  size_t size() const { return (off + 255) & ~size_t(255); }
};

// ------------------------------------------------------------------------------------------------
// Element conversions
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ uint32_t abs_key(float v) {
  return __float_as_uint(v) & 0x7FFFFFFFu;
}

__device__ __forceinline__ void flag_status(uint32_t* st, uint32_t bit) {
  if (st) atomicOr(st, bit);
}

// Warp-aggregated status flag: one atomic per warp that saw the condition.
__device__ __forceinline__ void flag_status_warp(uint32_t* st, bool cond, uint32_t bit) {
  unsigned m = __ballot_sync(__activemask(), cond);
  if (m && st && (threadIdx.x & 31) == __ffs(m) - 1) atomicOr(st, bit);
}

__device__ __forceinline__ bool finite_f(float v) { return isfinite(v); }

// Butterfly transpose-reduce across a warp: lane l returns the warp-wide sum of x[l] (31 shuffles
// for 32 sums). x is clobbered.
__device__ __forceinline__ float transpose_reduce32(float (&x)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < off; ++j) {
      const float send = upper ? x[j] : x[j + off];
      const float keep = upper ? x[j + off] : x[j];
      x[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return x[0];
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }
__device__ __forceinline__ float silu_grad_f(float z) {
  float s = 1.0f / (1.0f + expf(-z));
  return s * (1.0f + z * (1.0f - s));
}

int device_sm_count();

// A side stream with a fork and a join event, one per calling thread and device (created once and
// kept for the thread's life), for work that a call runs beside its main stream and joins back
// before it returns. side_stream_setup() creates it from a host-only call; side_stream() hands it
// out, creating it first unless `st` is being captured (then false: run the work on `st`).
struct SideStream {
  cudaStream_t s;
  cudaEvent_t fork, join;
};
void side_stream_setup();
bool side_stream(SideStream& out, cudaStream_t st);

// Optional per-kernel timing: while usaf_trace_enable(1) is in force, a TraceScope records a
// CUDA event pair around the launches inside it.
bool trace_on();
void trace_begin(const char* name, cudaStream_t st);
void trace_end(cudaStream_t st);
struct TraceScope {
  cudaStream_t st;
  bool on;
  TraceScope(const char* name, cudaStream_t s) : st(s), on(trace_on()) {
    if (on) trace_begin(name, st);
  }
  ~TraceScope() {
    if (on) trace_end(st);
  }
};
#define USAF_TRACE(name, st) ::usaf::TraceScope usaf_trace_scope_(name, st)

}  // namespace usaf
