// Grouped SwiGLU expert layer: forward, sparse backward, router backward.
//
// Layouts follow the experts4bit-qlora page ("The abstraction that fails, and what replaces it"):
// gate_up_proj [E, 2I, H] (first I rows gate, last I rows up) and down_proj [E, H, I]; the
// activation placement act(gate) * up follows its epilogue-contract bullet. The sparse backward
// forms expert weight gradients only at the active set (USAF README, "Not all weights matter";
// news article, key differences: a subset of weights inside each activated expert).
//
// This file holds the element-wise, gather/scatter and router kernels shared by both element
// types, the CUDA-core grouped GEMMs used for fp32 layers, and the host orchestration. The bf16
// grouped GEMMs run on tcgen05 tensor cores (moe_tc.cu).
#include "common.cuh"
#include "kernels.cuh"

namespace usaf {

// ================================================================================================
// CUDA-core grouped GEMM (fp32 layers). One block computes a 64x64 tile of expert blockIdx.z.
// ================================================================================================
template <typename P>
__global__ void __launch_bounds__(256) simt_gemm_kernel(P p) {
  const int e = blockIdx.z;
  int M, N, K;
  p.dims(e, M, N, K);
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  if (m0 >= M || n0 >= N) return;
  __shared__ float As[16][68];
  __shared__ float Bs[16][68];
  const int tid = threadIdx.x, tm = tid / 16, tn = tid % 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = tid; i < 64 * 16; i += 256) {
      const int r = i % 64, kk = i / 64;
      As[kk][r] = (m0 + r < M && k0 + kk < K) ? p.a(e, m0 + r, k0 + kk) : 0.f;
      Bs[kk][r] = (n0 + r < N && k0 + kk < K) ? p.b(e, k0 + kk, n0 + r) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = As[kk][tm * 4 + i];
        bv[i] = Bs[kk][tn * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + tm * 4 + i, n = n0 + tn * 4 + j;
      if (m < M && n < N) p.store(e, m, n, acc[i][j]);
    }
}

// S4 (CUDA cores): h[n, row] = sum_k x_perm[row, k] * gate_up[e, n, k]  (h feature-major)
template <typename T>
struct ProbGateUp {
  const T* xp;
  const T* wgu;
  T* h;
  const int32_t* cnt;
  const int32_t* off;
  int H, I2;
  int64_t rcap;
  __device__ void dims(int e, int& M, int& N, int& K) const {
    M = cnt[e];
    N = I2;
    K = H;
  }
  __device__ float a(int e, int m, int k) const {
    return to_f32(xp[(int64_t)(off[e] + m) * H + k]);
  }
  __device__ float b(int e, int k, int n) const {
    return to_f32(wgu[((int64_t)e * I2 + n) * H + k]);
  }
  __device__ void store(int e, int m, int n, float v) const {
    h[(int64_t)n * rcap + off[e] + m] = from_f32<T>(v);
  }
};

// S5 (CUDA cores): y_acc[tok, n] += sum_k wa[row, k] * down[e, n, k]
template <typename T>
struct ProbDown {
  const T* wa;
  const T* wd;
  float* yacc;
  const int32_t* cnt;
  const int32_t* off;
  const int32_t* ptok;
  int H, I;
  __device__ void dims(int e, int& M, int& N, int& K) const {
    M = cnt[e];
    N = H;
    K = I;
  }
  __device__ float a(int e, int m, int k) const {
    return to_f32(wa[(int64_t)(off[e] + m) * I + k]);
  }
  __device__ float b(int e, int k, int n) const {
    return to_f32(wd[((int64_t)e * H + n) * I + k]);
  }
  __device__ void store(int e, int m, int n, float v) const {
    atomicAdd(&yacc[(int64_t)ptok[off[e] + m] * H + n], v);
  }
};

// S6 (CUDA cores): gvec[row, n] = sum_k dy[tok, k] * down[e, k, n]
template <typename T>
struct ProbGvec {
  const T* dy;
  const T* wd;
  float* gvec;
  const int32_t* cnt;
  const int32_t* off;
  const int32_t* ptok;
  int H, I;
  __device__ void dims(int e, int& M, int& N, int& K) const {
    M = cnt[e];
    N = I;
    K = H;
  }
  __device__ float a(int e, int m, int k) const {
    return to_f32(dy[(int64_t)ptok[off[e] + m] * H + k]);
  }
  __device__ float b(int e, int k, int n) const {
    return to_f32(wd[((int64_t)e * H + k) * I + n]);
  }
  __device__ void store(int e, int m, int n, float v) const {
    gvec[(int64_t)(off[e] + m) * I + n] = v;
  }
};

// S8 (CUDA cores): dx_acc[tok, n] += sum_k dh[row, k] * gate_up[e, k, n]
template <typename T>
struct ProbDx {
  const T* dh;
  const T* wgu;
  float* dxacc;
  const int32_t* cnt;
  const int32_t* off;
  const int32_t* ptok;
  int H, I2;
  __device__ void dims(int e, int& M, int& N, int& K) const {
    M = cnt[e];
    N = H;
    K = I2;
  }
  __device__ float a(int e, int m, int k) const {
    return to_f32(dh[(int64_t)(off[e] + m) * I2 + k]);
  }
  __device__ float b(int e, int k, int n) const {
    return to_f32(wgu[((int64_t)e * I2 + k) * H + n]);
  }
  __device__ void store(int e, int m, int n, float v) const {
    atomicAdd(&dxacc[(int64_t)ptok[off[e] + m] * H + n], v);
  }
};

// SwiGLU after S4 on CUDA cores: wa[row, j] = w * silu(gate) * up (0 in padding rows).
template <typename T>
__global__ void swiglu_fwd_rows_kernel(const T* __restrict__ h, const int32_t* __restrict__ pslot,
                                       const float* __restrict__ topk_w,
                                       const int32_t* __restrict__ off_end, int I, int64_t rcap,
                                       T* __restrict__ wa) {
  const int64_t row = blockIdx.x;
  if (row >= *off_end) return;
  const int slot = pslot[row];
  const float w = slot >= 0 ? topk_w[slot] : 0.f;
  for (int j = threadIdx.x; j < I; j += blockDim.x) {
    float g = to_f32(h[j * rcap + row]), u = to_f32(h[(I + j) * rcap + row]);
    wa[row * I + j] = from_f32<T>(slot >= 0 ? w * silu_f(g) * u : 0.f);
  }
}

// SwiGLU backward after S6 on CUDA cores: dw, dh per permuted row.
template <typename T>
__global__ void swiglu_bwd_rows_kernel(const float* __restrict__ gvec, const T* __restrict__ h,
                                       const int32_t* __restrict__ pslot,
                                       const float* __restrict__ topk_w,
                                       const int32_t* __restrict__ off_end, int I, int64_t rcap,
                                       T* __restrict__ dh, float* __restrict__ dw) {
  const int64_t row = blockIdx.x;
  if (row >= *off_end) return;
  const int slot = pslot[row];
  __shared__ float red[32];
  if (slot < 0) {
    for (int j = threadIdx.x; j < 2 * I; j += blockDim.x) dh[row * 2 * I + j] = from_f32<T>(0.f);
    return;
  }
  const float w = topk_w[slot];
  float part = 0.f;
  for (int j = threadIdx.x; j < I; j += blockDim.x) {
    float g = to_f32(h[j * rcap + row]), u = to_f32(h[(I + j) * rcap + row]);
    float gv = gvec[row * I + j];
    float sg = silu_f(g);
    part = fmaf(gv, sg * u, part);
    float dA = w * gv;
    dh[row * 2 * I + j] = from_f32<T>(dA * u * silu_grad_f(g));
    dh[row * 2 * I + I + j] = from_f32<T>(dA * sg);
  }
  for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    dw[slot] = s;
  }
}

// Masked expert gradient on CUDA cores: one thread per active entry (fp32 layers).
template <typename T>
__global__ void masked_wgrad_simt_kernel(const int64_t* __restrict__ act_idx, int64_t K,
                                         const T* __restrict__ xp, const T* __restrict__ dy,
                                         const T* __restrict__ dh, const T* __restrict__ wa,
                                         const int32_t* __restrict__ cnt,
                                         const int32_t* __restrict__ off,
                                         const int32_t* __restrict__ ptok, int H, int I,
                                         int64_t Ngu, float* __restrict__ g_act,
                                         uint32_t* dev_status) {
  const int64_t a = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  bool bad = false;
  if (a < K) {
    const int64_t f = act_idx[a];
    float acc = 0.f;
    if (f < Ngu) {
      const int e = (int)(f / ((int64_t)2 * I * H));
      const int r = (int)((f / H) % (2 * I));
      const int c = (int)(f % H);
      const int n = cnt[e], o = off[e];
      for (int i = 0; i < n; ++i)
        acc = fmaf(to_f32(dh[(int64_t)(o + i) * 2 * I + r]), to_f32(xp[(int64_t)(o + i) * H + c]),
                   acc);
    } else {
      const int64_t fd = f - Ngu;
      const int e = (int)(fd / ((int64_t)H * I));
      const int r = (int)((fd / I) % H);
      const int c = (int)(fd % I);
      const int n = cnt[e], o = off[e];
      for (int i = 0; i < n; ++i)
        acc = fmaf(to_f32(dy[(int64_t)ptok[o + i] * H + r]), to_f32(wa[(int64_t)(o + i) * I + c]),
                   acc);
    }
    g_act[a] = acc;
    bad = !finite_f(acc);
  }
  flag_status_warp(dev_status, bad, USAF_DEV_NONFINITE);
}

// ================================================================================================
// Shared element-wise kernels
// ================================================================================================

// x_perm[row] = x[perm_tok[row]] for routed rows, 0 for padding and tail rows. One warp per row,
// 16-byte vectors when a row is a whole number of them.
constexpr int GATHER_ROWS = 8;
template <typename T>
__global__ void __launch_bounds__(32 * GATHER_ROWS) gather_rows_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ ptok, const int32_t* __restrict__ pslot,
    const int32_t* __restrict__ off_end, int64_t R_cap, int H, T* __restrict__ xp) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * GATHER_ROWS + (threadIdx.x >> 5);
  if (row >= R_cap) return;
  const bool live = row < *off_end && pslot[row] >= 0;
  const int64_t src = live ? (int64_t)ptok[row] * H : 0;
  if (((H * sizeof(T)) & 15) == 0) {
    const int nv = (int)(H * sizeof(T) / 16);
    const uint4* sp = reinterpret_cast<const uint4*>(x + src);
    uint4* dp = reinterpret_cast<uint4*>(xp + row * H);
#pragma unroll 4
    for (int i = lane; i < nv; i += 32) dp[i] = live ? __ldg(sp + i) : make_uint4(0, 0, 0, 0);
  } else {
    for (int i = lane; i < H; i += 32) xp[row * H + i] = live ? x[src + i] : from_f32<T>(0.f);
  }
}

__global__ void zero_f32_kernel(float* __restrict__ p, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0.f;
}

template <typename T>
__global__ void f32_to_kernel(const float* __restrict__ src, T* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = from_f32<T>(src[i]);
}

// dlogit at the selected experts, renormalised routing: w_j (dw_j - sum_i w_i dw_i).
__global__ void dlogit_sel_kernel(const float* __restrict__ w, const float* __restrict__ dw,
                                  const int32_t* __restrict__ slot_row, int Tn, int k,
                                  float* __restrict__ dl, float* __restrict__ dl_perm) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= Tn) return;
  float s = 0.f;
  for (int j = 0; j < k; ++j) s = fmaf(w[(int64_t)t * k + j], dw[(int64_t)t * k + j], s);
  for (int j = 0; j < k; ++j) {
    const int64_t q = (int64_t)t * k + j;
    const float d = w[q] * (dw[q] - s);
    dl[q] = d;
    dl_perm[slot_row[q]] = d;  // the same value at the slot's permuted row
  }
}

// dense dlogit for softmax-over-all-E routing: p_e (dw_e [e selected] - sum_i p_{e_i} dw_i).
__global__ void dlogit_dense_kernel(const float* __restrict__ logits,
                                    const int32_t* __restrict__ idx,
                                    const float* __restrict__ w, const float* __restrict__ dw,
                                    int Tn, int E, int k, float* __restrict__ dlogit) {
  const int t = blockIdx.x;
  const float* l = logits + (int64_t)t * E;
  __shared__ float red[32];
  __shared__ float sh_mx, sh_sum, sh_s;
  float mx = -INFINITY;
  for (int e = threadIdx.x; e < E; e += blockDim.x) mx = fmaxf(mx, l[e]);
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    sh_mx = m;
  }
  __syncthreads();
  float sum = 0.f;
  for (int e = threadIdx.x; e < E; e += blockDim.x) sum += expf(l[e] - sh_mx);
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s2 = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s2 += red[i];
    sh_sum = s2;
    float s = 0.f;
    for (int j = 0; j < k; ++j) s = fmaf(w[(int64_t)t * k + j], dw[(int64_t)t * k + j], s);
    sh_s = s;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float p = expf(l[e] - sh_mx) / sh_sum;
    float d = 0.f;
    for (int j = 0; j < k; ++j)
      if (idx[(int64_t)t * k + j] == e) d = dw[(int64_t)t * k + j];
    dlogit[(int64_t)t * E + e] = p * (d - sh_s);
  }
}

// g_router[e, h] = sum over the rows routed to e of dl[row] * x_perm[row, h] (renormalised
// routing); each thread owns two adjacent h, rows in order, eight rows in flight.
template <typename T>
__global__ void __launch_bounds__(256) g_router_sel_kernel(
    const T* __restrict__ xp, const float* __restrict__ dl_perm, const int32_t* __restrict__ cnt,
    const int32_t* __restrict__ off, int H, float* __restrict__ g_router, uint32_t* dev_status) {
  const int e = blockIdx.y;
  const int h0 = (blockIdx.x * blockDim.x + threadIdx.x) * 2;
  float a0 = 0.f, a1 = 0.f;
  if (h0 < H) {
    const bool two = h0 + 1 < H;
    const int n = cnt[e], o = off[e];
    const T* base = xp + (int64_t)o * H + h0;
    int i = 0;
    for (; i + 8 <= n; i += 8) {
      float x0[8], x1[8], d[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        x0[u] = to_f32(base[(int64_t)(i + u) * H]);
        x1[u] = two ? to_f32(base[(int64_t)(i + u) * H + 1]) : 0.f;
        d[u] = dl_perm[o + i + u];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        a0 = fmaf(d[u], x0[u], a0);
        a1 = fmaf(d[u], x1[u], a1);
      }
    }
    for (; i < n; ++i) {
      const float d = dl_perm[o + i];
      a0 = fmaf(d, to_f32(base[(int64_t)i * H]), a0);
      if (two) a1 = fmaf(d, to_f32(base[(int64_t)i * H + 1]), a1);
    }
    g_router[(int64_t)e * H + h0] = a0;
    if (two) g_router[(int64_t)e * H + h0 + 1] = a1;
  }
  flag_status_warp(dev_status, h0 < H && (!finite_f(a0) || !finite_f(a1)), USAF_DEV_NONFINITE);
}

// g_router[e, h] = sum_t dlogit[t, e] * x[t, h]   (softmax-over-all-E routing)
template <typename T>
__global__ void g_router_dense_kernel(const T* __restrict__ x, const float* __restrict__ dlogit,
                                      int Tn, int E, int H, float* __restrict__ g_router,
                                      uint32_t* dev_status) {
  const int e = blockIdx.y;
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  float acc = 0.f;
  if (h < H) {
    for (int t = 0; t < Tn; ++t)
      acc = fmaf(dlogit[(int64_t)t * E + e], to_f32(x[(int64_t)t * H + h]), acc);
    g_router[(int64_t)e * H + h] = acc;
  }
  flag_status_warp(dev_status, h < H && !finite_f(acc), USAF_DEV_NONFINITE);
}

// dx[t, h] = dx_acc[t, h] + router term: sum_j dl[t,j] Wr[e_j, h] (renormalised routing) or
// sum_e dlogit[t,e] Wr[e, h]. One token per block, four h per thread.
template <typename T>
__global__ void __launch_bounds__(256) dx_finalize_kernel(
    const float* __restrict__ dx_acc, const float* __restrict__ wr, const int32_t* __restrict__ idx,
    const float* __restrict__ dl, const float* __restrict__ dlogit, int Tn, int H, int E, int k,
    int renorm, T* __restrict__ dx, uint32_t* dev_status) {
  __shared__ float s_d[1024];
  __shared__ int s_e[32];
  const int t = blockIdx.x;
  if (renorm) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      s_d[j] = dl[(int64_t)t * k + j];
      s_e[j] = idx[(int64_t)t * k + j];
    }
  } else {
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_d[e] = dlogit[(int64_t)t * E + e];
  }
  __syncthreads();
  bool bad = false;
  const bool vec = (H & 3) == 0;
  for (int h0 = threadIdx.x * 4; h0 < H; h0 += blockDim.x * 4) {
    float v[4];
    if (vec) {
      const float4 a = *reinterpret_cast<const float4*>(dx_acc + (int64_t)t * H + h0);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = h0 + q < H ? dx_acc[(int64_t)t * H + h0 + q] : 0.f;
    }
    const int nterm = renorm ? k : E;
    for (int j = 0; j < nterm; ++j) {
      const float d = s_d[j];
      const float* wrow = wr + (int64_t)(renorm ? s_e[j] : j) * H + h0;
      if (vec) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(wrow));
        v[0] = fmaf(d, b.x, v[0]); v[1] = fmaf(d, b.y, v[1]);
        v[2] = fmaf(d, b.z, v[2]); v[3] = fmaf(d, b.w, v[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (h0 + q < H) v[q] = fmaf(d, wrow[q], v[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (h0 + q < H) {
        dx[(int64_t)t * H + h0 + q] = from_f32<T>(v[q]);
        bad |= !finite_f(v[q]);
      }
    }
  }
  flag_status_warp(dev_status, bad, USAF_DEV_NONFINITE);
}

// ================================================================================================
// Host orchestration
// ================================================================================================
void fwd_ws_layout(const usaf_moe_shape& s, usaf_dtype dt, Carver& c, FwdWs& w) {
  w.y_acc = c.take<float>(s.T * s.H);
  w.plan = dt == USAF_BF16 ? c.take<int32_t>(s.E + 1) : nullptr;
}

void bwd_ws_layout(const usaf_moe_shape& s, usaf_dtype dt, int64_t K, Carver& c, BwdWs& w) {
  (void)K;
  const int64_t R_cap = usaf_routed_rows_capacity(&s);
  const size_t es = dt == USAF_BF16 ? 2 : 4;
  w.dw = c.take<float>(s.T * s.k);
  w.dl = c.take<float>(s.T * s.k);
  w.dl_perm = c.take<float>(R_cap);
  w.dlogit = c.take<float>(s.T * s.E);
  w.dh = c.take<char>(R_cap * 2 * s.I * (int64_t)es);
  w.dx_acc = c.take<float>(s.T * s.H);
  w.gvec = dt == USAF_F32 ? c.take<float>(R_cap * s.I) : nullptr;
  w.tile_ptr = dt == USAF_BF16 ? c.take<int32_t>(tile_ptr_entries(s)) : nullptr;
  w.plan = dt == USAF_BF16 ? c.take<int32_t>(s.E + 1) : nullptr;
  w.dy_perm = dt == USAF_BF16 ? (void*)c.take<char>(R_cap * s.H * 2) : nullptr;
}


template <typename T>
static usaf_status fwd_simt(const MoeArgs& a, T* xp, T* h, T* wa, float* yacc, cudaStream_t st) {
  USAF_TRACE("simt_fwd", st);
  const auto& s = a.s;
  const int H = (int)s.H, I = (int)s.I, E = (int)s.E;
  const int32_t* cnt = a.rt.expert_count;
  const int32_t* off = a.rt.expert_offset;
  ProbGateUp<T> p1{xp, static_cast<const T*>(a.w_gate_up), h, cnt, off, H, 2 * I, a.R_cap};
  dim3 g1((unsigned)ceil_div(2 * I, 64), (unsigned)ceil_div(s.T, 64), (unsigned)E);
  simt_gemm_kernel<<<g1, 256, 0, st>>>(p1);
  USAF_CHECK_LAUNCH();
  swiglu_fwd_rows_kernel<T><<<(unsigned)a.R_cap, 128, 0, st>>>(h, a.rt.perm_slot, a.rt.topk_w,
                                                               off + E, I, a.R_cap, wa);
  USAF_CHECK_LAUNCH();
  ProbDown<T> p2{wa, static_cast<const T*>(a.w_down), yacc, cnt, off, a.rt.perm_tok, H, I};
  dim3 g2((unsigned)ceil_div(H, 64), (unsigned)ceil_div(s.T, 64), (unsigned)E);
  simt_gemm_kernel<<<g2, 256, 0, st>>>(p2);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

template <typename T>
static usaf_status moe_fwd_t(const MoeArgs& a, T* xp, T* h, T* wa, T* y, FwdWs& w,
                             cudaStream_t st) {
  const auto& s = a.s;
  const int64_t TH = s.T * s.H;
  {
  USAF_TRACE("gather_x", st);
  gather_rows_kernel<T><<<(unsigned)ceil_div(a.R_cap, GATHER_ROWS), 32 * GATHER_ROWS, 0, st>>>(
      static_cast<const T*>(a.x), a.rt.perm_tok, a.rt.perm_slot, a.rt.expert_offset + s.E,
      a.R_cap, (int)s.H, xp);
  USAF_CHECK_LAUNCH();
  zero_f32_kernel<<<grid_dim_for(TH), 256, 0, st>>>(w.y_acc, TH);
  USAF_CHECK_LAUNCH();
  }
  if (a.dt == USAF_BF16) {
    MoeArgs b = a;
    b.plan = w.plan;
    USAF_TRY(tc_plan(b, st));
    USAF_TRY(tc_fwd_gate_up(b, xp, h, wa, st));
    USAF_TRY(tc_fwd_down(b, wa, w.y_acc, st));
  } else {
    USAF_TRY(fwd_simt<T>(a, xp, h, wa, w.y_acc, st));
  }
  USAF_TRACE("combine_finalize", st);
  f32_to_kernel<T><<<grid_dim_for(TH), 256, 0, st>>>(w.y_acc, y, TH);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

usaf_status moe_fwd_launch(const MoeArgs& a, void* x_perm, void* h, void* wa, void* y, FwdWs& w,
                           cudaStream_t st) {
  if (a.dt == USAF_BF16)
    return moe_fwd_t<__nv_bfloat16>(a, static_cast<__nv_bfloat16*>(x_perm),
                                    static_cast<__nv_bfloat16*>(h),
                                    static_cast<__nv_bfloat16*>(wa),
                                    static_cast<__nv_bfloat16*>(y), w, st);
  return moe_fwd_t<float>(a, static_cast<float*>(x_perm), static_cast<float*>(h),
                          static_cast<float*>(wa), static_cast<float*>(y), w, st);
}

// For every weight row (gate_up rows, then down rows) and every 256-column tile of it, the first
// active entry at or after the tile's first column; entry NT of a row is the row's end. The
// actives are sorted, so their (row, tile) positions are too: active a fills the entries between
// its predecessor's position and its own, and the entries after the last active get K.
__device__ __forceinline__ int64_t tile_pos(int64_t f, int64_t Ngu, int64_t n_gu_rows, int H,
                                            int I, int nt_gu, int nt_d) {
  if (f < Ngu) return (f / H) * (nt_gu + 1) + (f % H) / 256;
  const int64_t fd = f - Ngu;
  return n_gu_rows * (nt_gu + 1) + (fd / I) * (nt_d + 1) + (fd % I) / 256;
}

__global__ void tile_ptr_kernel(const int64_t* __restrict__ act, int64_t K, int64_t n_gu_rows,
                                int64_t n_entries, int H, int I, int64_t Ngu, int nt_gu, int nt_d,
                                int32_t* __restrict__ tp) {
  const int64_t tail = K > 0 ? tile_pos(act[K - 1], Ngu, n_gu_rows, H, I, nt_gu, nt_d) + 1 : 0;
  const int64_t n = K > n_entries ? K : n_entries;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < K) {
      const int64_t pos = tile_pos(act[i], Ngu, n_gu_rows, H, I, nt_gu, nt_d);
      const int64_t prev = i > 0 ? tile_pos(act[i - 1], Ngu, n_gu_rows, H, I, nt_gu, nt_d) : -1;
      for (int64_t x = prev + 1; x <= pos; ++x) tp[x] = (int32_t)i;
    }
    if (i >= tail && i < n_entries) tp[i] = (int32_t)K;
  }
}

int64_t tile_ptr_entries(const usaf_moe_shape& s) {
  return s.E * 2 * s.I * (ceil_div(s.H, 256) + 1) + s.E * s.H * (ceil_div(s.I, 256) + 1);
}

template <typename T>
static usaf_status moe_bwd_t(const MoeArgs& a0, int renorm, const float* logits, const T* xp,
                             const T* h, const T* wa, const T* dy, const int64_t* act_idx,
                             int64_t K, float* g_act, float* g_router, T* dx, float* dw_out,
                             uint32_t* dev_status, BwdWs& w, cudaStream_t st) {
  MoeArgs a = a0;
  a.plan = w.plan;
  const auto& s = a.s;
  const int H = (int)s.H, I = (int)s.I, E = (int)s.E, Tn = (int)s.T, k = (int)s.k;
  const int32_t* cnt = a.rt.expert_count;
  const int32_t* off = a.rt.expert_offset;
  const int32_t* ptok = a.rt.perm_tok;
  const int32_t* pslot = a.rt.perm_slot;
  float* dw = dw_out ? dw_out : w.dw;
  T* dh = static_cast<T*>(w.dh);
  T* dyp = static_cast<T*>(w.dy_perm);
  const int64_t Ngu = s.E * 2 * s.I * s.H;

  // S6: gvec, dw, dh
  if (a.dt == USAF_BF16) {
    {
      USAF_TRACE("gather_dy", st);
      gather_rows_kernel<T><<<(unsigned)ceil_div(a.R_cap, GATHER_ROWS), 32 * GATHER_ROWS, 0,
                              st>>>(dy, ptok, pslot, off + E, a.R_cap, H, dyp);
      USAF_CHECK_LAUNCH();
      zero_f32_kernel<<<grid_dim_for(s.T * s.k), 256, 0, st>>>(dw, s.T * s.k);
      USAF_CHECK_LAUNCH();
    }
    USAF_TRY(tc_plan(a, st));
    USAF_TRY(tc_bwd_gvec(a, dyp, h, dh, dw, st));
  } else {
    ProbGvec<T> p{dy, static_cast<const T*>(a.w_down), w.gvec, cnt, off, ptok, H, I};
    dim3 g((unsigned)ceil_div(I, 64), (unsigned)ceil_div(Tn, 64), (unsigned)E);
    simt_gemm_kernel<<<g, 256, 0, st>>>(p);
    USAF_CHECK_LAUNCH();
    swiglu_bwd_rows_kernel<T><<<(unsigned)a.R_cap, 128, 0, st>>>(w.gvec, h, pslot, a.rt.topk_w,
                                                                 off + E, I, a.R_cap, dh, dw);
    USAF_CHECK_LAUNCH();
  }
  // S7: router gradient
  {
  USAF_TRACE("router_bwd", st);
  if (renorm) {
    dlogit_sel_kernel<<<(unsigned)ceil_div(Tn, 128), 128, 0, st>>>(a.rt.topk_w, dw, a.rt.slot_row,
                                                                  Tn, k, w.dl, w.dl_perm);
    USAF_CHECK_LAUNCH();
    g_router_sel_kernel<T><<<dim3((unsigned)ceil_div(ceil_div(H, 2), 256), (unsigned)E), 256, 0,
                             st>>>(xp, w.dl_perm, cnt, off, H, g_router, dev_status);
    USAF_CHECK_LAUNCH();
  } else {
    dlogit_dense_kernel<<<(unsigned)Tn, 128, 0, st>>>(logits, a.rt.topk_idx, a.rt.topk_w, dw, Tn,
                                                      E, k, w.dlogit);
    USAF_CHECK_LAUNCH();
    g_router_dense_kernel<T><<<dim3((unsigned)ceil_div(H, 128), (unsigned)E), 128, 0, st>>>(
        static_cast<const T*>(a.x), w.dlogit, Tn, E, H, g_router, dev_status);
    USAF_CHECK_LAUNCH();
  }
  }
  // S8: dx
  if (dx) {
    {
      USAF_TRACE("dx_zero", st);
      zero_f32_kernel<<<grid_dim_for(s.T * s.H), 256, 0, st>>>(w.dx_acc, s.T * s.H);
      USAF_CHECK_LAUNCH();
    }
    if (a.dt == USAF_BF16) {
      USAF_TRY(tc_bwd_dx(a, dh, w.dx_acc, st));
    } else {
      ProbDx<T> p{dh, static_cast<const T*>(a.w_gate_up), w.dx_acc, cnt, off, ptok, H, 2 * I};
      dim3 g((unsigned)ceil_div(H, 64), (unsigned)ceil_div(Tn, 64), (unsigned)E);
      simt_gemm_kernel<<<g, 256, 0, st>>>(p);
      USAF_CHECK_LAUNCH();
    }
    USAF_TRACE("dx_finalize", st);
    dx_finalize_kernel<T><<<(unsigned)Tn, 256, 0, st>>>(
        w.dx_acc, a.w_router, a.rt.topk_idx, w.dl, w.dlogit, Tn, H, E, k, renorm, dx,
        dev_status);
    USAF_CHECK_LAUNCH();
  }
  // S9, S10: expert weight gradients at the active set
  if (K > 0) {
    if (a.dt == USAF_BF16) {
      const int64_t n_gu_rows = s.E * 2 * s.I, n_rows = n_gu_rows + s.E * s.H;
      {
      USAF_TRACE("wgrad_tile_ptr", st);
      tile_ptr_kernel<<<grid_dim_for(std::max<int64_t>(K, tile_ptr_entries(s))), 256, 0, st>>>(
          act_idx, K, n_gu_rows, tile_ptr_entries(s), H, I, Ngu, (int)ceil_div(H, 256),
          (int)ceil_div(I, 256), w.tile_ptr);
      USAF_CHECK_LAUNCH();
      }
      USAF_TRY(tc_bwd_wgrad(a, xp, dyp, dh, wa, act_idx, K, w.tile_ptr, g_act, dev_status, st));
    } else {
      USAF_TRACE("simt_wgrad", st);
      masked_wgrad_simt_kernel<T><<<(unsigned)ceil_div(K, 128), 128, 0, st>>>(
          act_idx, K, xp, dy, dh, wa, cnt, off, ptok, H, I, Ngu, g_act, dev_status);
      USAF_CHECK_LAUNCH();
    }
  }
  return USAF_OK;
}

usaf_status moe_bwd_launch(const MoeArgs& a, int renorm, const float* logits, const void* x_perm,
                           const void* h, const void* wa, const void* dy, const int64_t* act_idx,
                           int64_t K, float* g_act, float* g_router, void* dx, float* dw_slot,
                           uint32_t* dev_status, BwdWs& w, cudaStream_t st) {
  using B = __nv_bfloat16;
  if (a.dt == USAF_BF16)
    return moe_bwd_t<B>(a, renorm, logits, static_cast<const B*>(x_perm),
                        static_cast<const B*>(h), static_cast<const B*>(wa),
                        static_cast<const B*>(dy), act_idx, K, g_act, g_router,
                        static_cast<B*>(dx), dw_slot, dev_status, w, st);
  return moe_bwd_t<float>(a, renorm, logits, static_cast<const float*>(x_perm),
                          static_cast<const float*>(h), static_cast<const float*>(wa),
                          static_cast<const float*>(dy), act_idx, K, g_act, g_router,
                          static_cast<float*>(dx), dw_slot, dev_status, w, st);
}

}  // namespace usaf
