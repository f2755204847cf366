// Grouped SwiGLU expert layer: forward, sparse backward, router backward.
//
// Layouts follow the experts4bit-qlora page ("The abstraction that fails, and what replaces it"):
// gate_up_proj [E, 2I, H] (first I rows gate, last I rows up) and down_proj [E, H, I]; the
// activation placement act(gate) * up follows its epilogue-contract bullet. The sparse backward
// forms expert weight gradients only at the active set (USAF README, "Not all weights matter";
// news article, key differences: a subset of weights inside each activated expert).
//
// Per-row activations are feature-major: x^T [H, R_cap], h^T [2I, R_cap], (w*A)^T [I, R_cap],
// dy^T [H, R_cap], dh^T [2I, R_cap], each row one feature over the permuted rows, so an expert's
// tokens are contiguous. The masked weight gradient is then, for every active entry, one dot
// product of two contiguous token vectors (a sampled dense-dense product on CUDA cores).
//
// This file holds the gathers, the masked-gradient and router kernels shared by both element
// types, the CUDA-core grouped GEMMs used for fp32 layers, and the host orchestration. The bf16
// grouped GEMMs run on tcgen05 tensor cores (moe_tc.cu).
#include <algorithm>

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

// The fp32 GEMMs: M = the expert's tokens, N = features. Feature-major operands are read at
// X[k * rcap + off[e] + m].
// S4: h^T[n, row] = sum_k x^T[k, row] * gate_up[e, n, k]
template <typename T>
struct ProbGateUp {
  const T* xT;
  const T* wgu;
  T* hT;
  const int32_t* cnt;
  const int32_t* off;
  int H, I2;
  int64_t rcap;
  __device__ void dims(int e, int& M, int& N, int& K) const {
    M = cnt[e];
    N = I2;
    K = H;
  }
  __device__ float a(int e, int m, int k) const { return to_f32(xT[(int64_t)k * rcap + off[e] + m]); }
  __device__ float b(int e, int k, int n) const {
    return to_f32(wgu[((int64_t)e * I2 + n) * H + k]);
  }
  __device__ void store(int e, int m, int n, float v) const {
    hT[(int64_t)n * rcap + off[e] + m] = from_f32<T>(v);
  }
};

// S5: y_acc[tok, n] += sum_k (wA)^T[k, row] * down[e, n, k]
template <typename T>
struct ProbDown {
  const T* waT;
  const T* wd;
  float* yacc;
  const int32_t* cnt;
  const int32_t* off;
  const int32_t* ptok;
  int H, I;
  int64_t rcap;
  __device__ void dims(int e, int& M, int& N, int& K) const {
    M = cnt[e];
    N = H;
    K = I;
  }
  __device__ float a(int e, int m, int k) const { return to_f32(waT[(int64_t)k * rcap + off[e] + m]); }
  __device__ float b(int e, int k, int n) const { return to_f32(wd[((int64_t)e * H + n) * I + k]); }
  __device__ void store(int e, int m, int n, float v) const {
    atomicAdd(&yacc[(int64_t)ptok[off[e] + m] * H + n], v);
  }
};

// S6: gvec[row, n] = sum_k dy^T[k, row] * down[e, k, n]
template <typename T>
struct ProbGvec {
  const T* dyT;
  const T* wd;
  float* gvec;
  const int32_t* cnt;
  const int32_t* off;
  int H, I;
  int64_t rcap;
  __device__ void dims(int e, int& M, int& N, int& K) const {
    M = cnt[e];
    N = I;
    K = H;
  }
  __device__ float a(int e, int m, int k) const { return to_f32(dyT[(int64_t)k * rcap + off[e] + m]); }
  __device__ float b(int e, int k, int n) const { return to_f32(wd[((int64_t)e * H + k) * I + n]); }
  __device__ void store(int e, int m, int n, float v) const {
    gvec[(int64_t)(off[e] + m) * I + n] = v;
  }
};

// S8: dx_acc[tok, n] += sum_k dh^T[k, row] * gate_up[e, k, n]
template <typename T>
struct ProbDx {
  const T* dhT;
  const T* wgu;
  float* dxacc;
  const int32_t* cnt;
  const int32_t* off;
  const int32_t* ptok;
  int H, I2;
  int64_t rcap;
  __device__ void dims(int e, int& M, int& N, int& K) const {
    M = cnt[e];
    N = H;
    K = I2;
  }
  __device__ float a(int e, int m, int k) const { return to_f32(dhT[(int64_t)k * rcap + off[e] + m]); }
  __device__ float b(int e, int k, int n) const {
    return to_f32(wgu[((int64_t)e * I2 + k) * H + n]);
  }
  __device__ void store(int e, int m, int n, float v) const {
    atomicAdd(&dxacc[(int64_t)ptok[off[e] + m] * H + n], v);
  }
};

// SwiGLU after S4 on CUDA cores: (wA)^T[j, row] = w * silu(gate) * up (0 in padding rows).
template <typename T>
__global__ void swiglu_fwd_rows_kernel(const T* __restrict__ hT, const int32_t* __restrict__ pslot,
                                       const float* __restrict__ topk_w,
                                       const int32_t* __restrict__ off_end, int I, int64_t rcap,
                                       T* __restrict__ waT) {
  const int64_t row = blockIdx.x;
  if (row >= *off_end) return;
  const int slot = pslot[row];
  const float w = slot >= 0 ? topk_w[slot] : 0.f;
  for (int j = threadIdx.x; j < I; j += blockDim.x) {
    const float g = to_f32(hT[j * rcap + row]), u = to_f32(hT[(I + j) * rcap + row]);
    waT[j * rcap + row] = from_f32<T>(slot >= 0 ? w * silu_f(g) * u : 0.f);
  }
}

// SwiGLU backward after S6 on CUDA cores: dw per slot and dh^T per permuted row.
template <typename T>
__global__ void swiglu_bwd_rows_kernel(const float* __restrict__ gvec, const T* __restrict__ hT,
                                       const int32_t* __restrict__ pslot,
                                       const float* __restrict__ topk_w,
                                       const int32_t* __restrict__ off_end, int I, int64_t rcap,
                                       T* __restrict__ dhT, float* __restrict__ dw) {
  const int64_t row = blockIdx.x;
  if (row >= *off_end) return;
  const int slot = pslot[row];
  __shared__ float red[32];
  if (slot < 0) {
    for (int j = threadIdx.x; j < 2 * I; j += blockDim.x) dhT[j * rcap + row] = from_f32<T>(0.f);
    return;
  }
  const float w = topk_w[slot];
  float part = 0.f;
  for (int j = threadIdx.x; j < I; j += blockDim.x) {
    const float g = to_f32(hT[j * rcap + row]), u = to_f32(hT[(I + j) * rcap + row]);
    const float gv = gvec[row * I + j];
    const float sg = silu_f(g);
    part = fmaf(gv, sg * u, part);
    const float dA = w * gv;
    dhT[j * rcap + row] = from_f32<T>(dA * u * silu_grad_f(g));
    dhT[(I + j) * rcap + row] = from_f32<T>(dA * sg);
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

// ================================================================================================
// Gathers, masked gradient, router
// ================================================================================================

// Side duties of a gather launch, so that they need no launch of their own: zero up to two fp32
// buffers (16-byte aligned), and in block (0, 0) write the tensor-core tile plan (per expert
// ceil(padded rows / TC_TOKEN_TILE), exclusive prefix over experts, E <= 1024).
struct GatherExtra {
  float* z0;
  int64_t n0;
  float* z1;
  int64_t n1;
  const int32_t* off;
  int E;
  int32_t* plan;
};

// z[0..n) = 0, shared by all blocks of the grid: grid-stride float4 stores (scalar ones when z is
// off a 16-byte boundary)
__device__ void zero_slice(float* z, int64_t n) {
  if (!z || n == 0) return;
  const int64_t nb = (int64_t)gridDim.x * gridDim.y, b = (int64_t)blockIdx.y * gridDim.x + blockIdx.x;
  const int64_t stride = nb * blockDim.x, i0 = b * blockDim.x + threadIdx.x;
  if ((reinterpret_cast<uintptr_t>(z) & 15) != 0) {
    for (int64_t i = i0; i < n; i += stride) z[i] = 0.f;
    return;
  }
  const int64_t n4 = n >> 2;
  float4* z4 = reinterpret_cast<float4*>(z);
  for (int64_t i = i0; i < n4; i += stride) z4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (b == 0 && threadIdx.x < (n & 3)) z[(n4 << 2) + threadIdx.x] = 0.f;
}

__device__ void tile_plan(const int32_t* __restrict__ off, int E, int32_t* __restrict__ plan) {
  __shared__ int32_t wsum[32];
  constexpr int PER = 4;  // experts per thread (256 threads, E <= 1024)
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int32_t n[PER], tot = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = threadIdx.x * PER + j;
    n[j] = e < E ? (off[e + 1] - off[e] + TC_TOKEN_TILE - 1) / TC_TOKEN_TILE : 0;
    tot += n[j];
  }
  int32_t v = tot;
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) wsum[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int32_t w = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  int32_t run = v - tot + (wid > 0 ? wsum[wid - 1] : 0);
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = threadIdx.x * PER + j;
    if (e < E) plan[e] = run;
    run += n[j];
    if (e == E - 1) plan[E] = run;
  }
}

// Gather-transpose: xT[h, row] = x[perm_tok[row], h] for routed rows, 0 for padding and tail
// rows. A block moves a 128-row x 64-feature tile through shared memory with 16-byte accesses, so
// each feature row of xT receives 256 contiguous bytes (bf16).
constexpr int GT_ROWS = 128;
template <typename T>
__global__ void __launch_bounds__(256, 8) gather_transpose_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ ptok, const int32_t* __restrict__ pslot,
    const int32_t* __restrict__ off_end, int64_t R_cap, int H, T* __restrict__ xT,
    const float* __restrict__ topk_w, float* __restrict__ wperm, GatherExtra ex) {
  constexpr int VW = 16 / sizeof(T);  // elements per 16-byte vector
  // feature f's row of the tile is rotated by (f / VW) * VW columns: the column writes of the
  // load phase then fall in distinct banks, and the 16-byte reads of the store phase stay aligned
  __shared__ __align__(16) T tile[64 * GT_ROWS];
  const int64_t r0 = (int64_t)blockIdx.x * GT_ROWS;
  const int h0 = blockIdx.y * 64;
  const int64_t end = *off_end;
  const bool vec = (H % VW) == 0;
  for (int v = threadIdx.x; v < GT_ROWS * (64 / VW); v += blockDim.x) {
    const int r = v / (64 / VW), f = (v % (64 / VW)) * VW;
    const int64_t row = r0 + r;
    const bool live = row < R_cap && row < end && pslot[row] >= 0;
    const int64_t src = live ? (int64_t)ptok[row] * H : 0;
    alignas(16) T buf[VW];
    if (vec && h0 + f + VW <= H) {
      const uint4 u = live ? __ldg(reinterpret_cast<const uint4*>(x + src + h0 + f))
                           : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(buf) = u;
    } else {
#pragma unroll
      for (int q = 0; q < VW; ++q)
        buf[q] = (live && h0 + f + q < H) ? x[src + h0 + f + q] : from_f32<T>(0.f);
    }
    // feature f + q goes to row f + q of the tile, rotated by f columns (f is a multiple of VW)
    T* dst = &tile[f * GT_ROWS + ((r + f) & (GT_ROWS - 1))];
#pragma unroll
    for (int q = 0; q < VW; ++q) dst[q * GT_ROWS] = buf[q];
  }
  zero_slice(ex.z0, ex.n0);
  zero_slice(ex.z1, ex.n1);
  if (ex.plan && blockIdx.x == 0 && blockIdx.y == 0) tile_plan(ex.off, ex.E, ex.plan);
  if (wperm && blockIdx.y == 0) {
    for (int r = threadIdx.x; r < GT_ROWS; r += blockDim.x) {
      const int64_t row = r0 + r;
      if (row >= R_cap) break;
      const int sl = row < end ? pslot[row] : -1;
      wperm[row] = sl >= 0 ? topk_w[sl] : 0.f;
    }
  }
  __syncthreads();
  for (int v = threadIdx.x; v < 64 * (GT_ROWS / VW); v += blockDim.x) {
    const int f = v / (GT_ROWS / VW), r = (v % (GT_ROWS / VW)) * VW;
    if (h0 + f >= H || r0 + r >= R_cap) continue;
    *reinterpret_cast<uint4*>(xT + (int64_t)(h0 + f) * R_cap + r0 + r) =
        *reinterpret_cast<const uint4*>(&tile[f * GT_ROWS + ((r + (f / VW) * VW) & (GT_ROWS - 1))]);
  }
}

// Gather-transpose of bf16 rows: a block takes 256 permuted rows x 64 features and writes the
// transposed tile with four TMA stores of 64 tokens x 64 features (128-byte swizzled boxes). Lane
// l of warp w takes the eight rows 32 w + 8 (l / 8) .. + 8 and the eight features 8 (l % 8) .. + 8,
// so each load instruction reads 128 contiguous bytes of four rows; it transposes its 8 x 8 block
// in registers (one byte permute per output word) and puts each feature's eight tokens into the
// box. In the box, 16-byte chunk c of feature row f sits at chunk c ^ (f % 8); lane l writes its
// eight feature rows starting from row l % 8 of its eight, so the eight lanes that share a token
// chunk write eight different chunk positions and every store is conflict-free. H a multiple of
// 64, R_cap of 256. Side duties as in gather_transpose_kernel.
constexpr int GR_ROWS = 256;
constexpr int GR_SMEM = 4 * 8192 + 1024;  // four boxes, and room to align them to 1 KB
__global__ void __launch_bounds__(256) gather_transpose_bf16_kernel(
    const __grid_constant__ CUtensorMap tm_out, const __nv_bfloat16* __restrict__ x,
    const int32_t* __restrict__ ptok, const int32_t* __restrict__ pslot,
    const int32_t* __restrict__ off_end, int64_t R_cap, int H, const float* __restrict__ topk_w,
    float* __restrict__ wperm, GatherExtra ex) {
  extern __shared__ uint8_t gr_raw[];
  uint8_t* tile = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gr_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int tl = wid * 32 + (lane >> 3) * 8;  // first row within the block's 256
  const int fl = (lane & 7) * 8;              // first feature within the block's 64
  const int64_t r0 = (int64_t)blockIdx.x * GR_ROWS + tl;
  const int f0 = blockIdx.y * 64 + fl;
  const int64_t end = *off_end;
  int tok[8];
  bool live[8];
  {
    const int4 t0 = *reinterpret_cast<const int4*>(ptok + r0);
    const int4 t1 = *reinterpret_cast<const int4*>(ptok + r0 + 4);
    const int4 s0 = *reinterpret_cast<const int4*>(pslot + r0);
    const int4 s1 = *reinterpret_cast<const int4*>(pslot + r0 + 4);
    const int tt[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
    const int ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      live[i] = r0 + i < end && ss[i] >= 0;
      tok[i] = tt[i];
    }
  }
  uint32_t a[8][4];  // a[i][w]: row i, features 2w and 2w+1
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 v = live[i]
                        ? __ldg(reinterpret_cast<const uint4*>(x + (int64_t)tok[i] * H + f0))
                        : make_uint4(0, 0, 0, 0);
    a[i][0] = v.x;
    a[i][1] = v.y;
    a[i][2] = v.z;
    a[i][3] = v.w;
  }
  zero_slice(ex.z0, ex.n0);
  zero_slice(ex.z1, ex.n1);
  if (ex.plan && blockIdx.x == 0 && blockIdx.y == 0) tile_plan(ex.off, ex.E, ex.plan);
  if (wperm && blockIdx.y == 0) {
    for (int r = threadIdx.x; r < GR_ROWS; r += blockDim.x) {
      const int64_t row = (int64_t)blockIdx.x * GR_ROWS + r;
      const int sl = row < end ? pslot[row] : -1;
      wperm[row] = sl >= 0 ? topk_w[sl] : 0.f;
    }
  }
  // out[j]: feature fl + j, the eight rows' tokens; feature 2w takes the low halves of word w of
  // rows 2u, 2u+1 and feature 2w+1 the high halves
  uint4 out[8];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    out[2 * w].x = __byte_perm(a[0][w], a[1][w], 0x5410);
    out[2 * w].y = __byte_perm(a[2][w], a[3][w], 0x5410);
    out[2 * w].z = __byte_perm(a[4][w], a[5][w], 0x5410);
    out[2 * w].w = __byte_perm(a[6][w], a[7][w], 0x5410);
    out[2 * w + 1].x = __byte_perm(a[0][w], a[1][w], 0x7632);
    out[2 * w + 1].y = __byte_perm(a[2][w], a[3][w], 0x7632);
    out[2 * w + 1].z = __byte_perm(a[4][w], a[5][w], 0x7632);
    out[2 * w + 1].w = __byte_perm(a[6][w], a[7][w], 0x7632);
  }
  // rotate by rot = lane % 8 (three conditional rotations): out[k] becomes feature fl + (k + rot) % 8
  const int rot = lane & 7;
#pragma unroll
  for (int sh = 1; sh < 8; sh <<= 1) {
    if (rot & sh) {
      uint4 t[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) t[k] = out[(k + sh) & 7];
#pragma unroll
      for (int k = 0; k < 8; ++k) out[k] = t[k];
    }
  }
  uint8_t* bx = tile + (tl >> 6) * 8192;
  const int c = (tl & 63) >> 3;  // this thread's 16-byte token chunk within the box's rows
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int fk = (k + rot) & 7;  // = f % 8
    *reinterpret_cast<uint4*>(bx + (fl + fk) * 128 + ((c ^ fk) << 4)) = out[k];
  }
  // the tile is complete in shared memory: make it visible to the copy engine and store it
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t src = static_cast<uint32_t>(__cvta_generic_to_shared(tile));
    for (int b = 0; b < 4; ++b)
      asm volatile(
          "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
              reinterpret_cast<uint64_t>(&tm_out)),
          "r"((int)(blockIdx.x * GR_ROWS + b * 64)), "r"((int)(blockIdx.y * 64)),
          "r"(src + b * 8192)
          : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // written before the block ends
  }
}

// The masked-gradient dot products. The bf16 products use the mixed-precision FMA (bf16 sources,
// fp32 addend and result, sm_100 and later): the product of two bf16 values is exact in fp32, so
// each step equals an fp32 FMA of the widened values and no unpacking is needed.
// c + a.lo * b.lo, then + a.hi * b.hi, for two bf16 pairs a and b
__device__ __forceinline__ float fma_bf16_pair(uint32_t a, uint32_t b, float c) {
  unsigned short al, ah, bl, bh;
  asm("mov.b32 {%0, %1}, %2;" : "=h"(al), "=h"(ah) : "r"(a));
  asm("mov.b32 {%0, %1}, %2;" : "=h"(bl), "=h"(bh) : "r"(b));
  asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(c) : "h"(al), "h"(bl));
  asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(c) : "h"(ah), "h"(bh));
  return c;
}
// s + the dot product of two 16-byte vectors (8 bf16 or 4 fp32), accumulated in fp32
template <typename T>
__device__ __forceinline__ float dot_acc(const uint4& a, const uint4& b, float s);
template <>
__device__ __forceinline__ float dot_acc<__nv_bfloat16>(const uint4& a, const uint4& b, float s) {
  s = fma_bf16_pair(a.x, b.x, s);
  s = fma_bf16_pair(a.y, b.y, s);
  s = fma_bf16_pair(a.z, b.z, s);
  return fma_bf16_pair(a.w, b.w, s);
}
template <>
__device__ __forceinline__ float dot_acc<float>(const uint4& a, const uint4& b, float s) {
  s = fmaf(__uint_as_float(a.x), __uint_as_float(b.x), s);
  s = fmaf(__uint_as_float(a.y), __uint_as_float(b.y), s);
  s = fmaf(__uint_as_float(a.z), __uint_as_float(b.z), s);
  return fmaf(__uint_as_float(a.w), __uint_as_float(b.w), s);
}

// Butterfly transpose-reduce of G values across a warp (G = 2, 4, 8 or 16): every lane l returns
// the warp-wide sum of x[l % G] (G - 1 + log2(32 / G) shuffles). x is clobbered.
template <int G>
__device__ __forceinline__ float transpose_reduce(float (&x)[G], int lane) {
#pragma unroll
  for (int off = G / 2; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < off; ++j) {
      const float send = upper ? x[j] : x[j + off];
      const float keep = upper ? x[j + off] : x[j];
      x[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = x[0];
#pragma unroll
  for (int o = G; o < 32; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

// One 16-byte vector of a row operand held for repeated dot products against other vectors.
template <typename T>
struct RowVec {
  uint4 r;
  __device__ __forceinline__ void set(const uint4& a) { r = a; }
  __device__ __forceinline__ float dot_acc(const uint4& b, float s) const {
    return ::usaf::dot_acc<T>(r, b, s);
  }
};

// Number of sorted active entries below flat index n (the gate_up entries): a 32-way search by
// one warp, about five dependent loads for millions of entries.
__device__ __forceinline__ int64_t count_below(const int64_t* __restrict__ act, int64_t K,
                                               int64_t n, int lane) {
  int64_t lo = 0, hi = K;  // act[i] < n for i < lo, act[i] >= n for i >= hi
  while (hi - lo > 32) {
    const int64_t step = (hi - lo + 31) / 32;
    const int64_t i = lo + (int64_t)lane * step;
    const int c = __popc(__ballot_sync(0xffffffffu, i < hi && act[i] < n));
    if (c == 0) {  // act[lo] >= n
      hi = lo;
      break;
    }
    // probes j < c are below n; probe c is not (or lies past hi)
    const int64_t nhi = lo + (int64_t)c * step;
    lo += (int64_t)(c - 1) * step + 1;
    hi = nhi < hi ? nhi : hi;
  }
  const int64_t i = lo + lane;
  return lo + __popc(__ballot_sync(0xffffffffu, i < hi && act[i] < n));
}

// S9/S10 masked weight gradient as a sampled dense-dense product on CUDA cores. The gate_up and
// the down entries are cut separately into batches of 32 consecutive active entries; for a batch
// the warp's lane l decodes entry l into the two feature-major rows whose dot product over the
// expert's routed tokens is that entry's gradient:
//   gate_up entry (e, j, c):  g = sum_t dh^T[j, o_e + t] * x^T[c, o_e + t]
//   down entry (e, h, c):     g = sum_t dy^T[h, o_e + t] * (wA)^T[c, o_e + t]
// The 32 entries are then taken in groups of SD_G.
// - Full passes: the warp walks the group's entries together, lane l reading 16-byte vector l of
//   both rows (a pass covers 32 vectors, 256 bf16 tokens), four entries' loads in flight before
//   their FMAs. The row vector is loaded only where the weight row changes. The number of passes
//   is the group's smallest vector count rounded to the nearest multiple of 32. When every entry
//   has a vector for every lane the pass runs unguarded; otherwise lanes past an entry's last
//   vector re-read that vector (an in-bounds address) and keep their partial sum unchanged.
// - Vectors past the full passes go to 32 / SD_G lanes per entry, which take entry i's remaining
//   vectors in turn and combine with shuffles.
// A butterfly transpose of the SD_G per-lane partial sums then leaves entry i's total in lane i.
constexpr int SD_WARPS = 8;
constexpr int SD_BLOCKS_PER_SM = 4;
constexpr int SD_G = 16;    // entries per group
constexpr int SD_RING = 6;  // entries whose vectors are in flight through a warp's ring
constexpr int SD_RING_BYTES = SD_WARPS * SD_RING * 2 * 512;  // a slot: b vector, a vector

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// wait until at most n of this thread's committed groups are pending (n a small constant after
// unrolling)
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
  }
}
template <typename T, bool RING>
__global__ void __launch_bounds__(SD_WARPS * 32, SD_BLOCKS_PER_SM) sddmm_kernel(
    const int64_t* __restrict__ act, int64_t K, const int32_t* __restrict__ cnt,
    const int32_t* __restrict__ off, int E, int H, int I, int64_t Ngu, int64_t rcap,
    const T* __restrict__ dhT, const T* __restrict__ xT, const T* __restrict__ dyT,
    const T* __restrict__ waT, float* __restrict__ g_act, int accumulate, uint32_t* dev_status,
    const int32_t* __restrict__ dense_flag) {
  constexpr int VW = 16 / sizeof(T);
  constexpr uint32_t FULL = 0xffffffffu;
  // per entry: a-row vector, b-row vector, vector count, last vector (0 when there is none)
  __shared__ int4 meta[SD_WARPS][32];
  extern __shared__ __align__(16) uint8_t sd_ring[];  // SD_RING_BYTES
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, il = lane % SD_G;
  const int64_t kgu = count_below(act, K, Ngu, lane);
  const int64_t nb_gu = (kgu + 31) / 32, nb = nb_gu + (K - kgu + 31) / 32;
  bool bad = false, badidx = false;
  uint32_t skipm = 0;  // entries of the batch left to the dense tile kernel (not stored here)
  for (int64_t bt = (int64_t)blockIdx.x * SD_WARPS + wid; bt < nb;
       bt += (int64_t)gridDim.x * SD_WARPS) {
    const bool gu = bt < nb_gu;
    const int64_t b0 = gu ? 32 * bt : kgu + 32 * (bt - nb_gu);
    const int64_t lim = gu ? kgu : K;
    const uint4* A = reinterpret_cast<const uint4*>(gu ? dhT : dyT);
    const uint4* Bm = reinterpret_cast<const uint4*>(gu ? xT : waT);
    {
      const int64_t q = b0 + lane;
      int4 md = make_int4(0, 0, 0, 0);
      const int64_t f = q < lim ? (gu ? act[q] : act[q] - Ngu) : 0;
      // an index outside its tensor (out of range, or an unsorted set split at the wrong place)
      // is flagged and gets a zero gradient; it is never decoded into addresses
      const bool inr = f >= 0 && f < (gu ? Ngu : (int64_t)E * H * I);
      badidx |= q < lim && !inr;
      bool mine_dense = false;  // the entry's expert is formed by the dense tile kernel
      if (q < lim && inr && dense_flag) {
        const int64_t per = gu ? (int64_t)2 * I * H : (int64_t)H * I;
        mine_dense = dense_flag[(int)(f / per)] != 0;
      }
      skipm = __ballot_sync(FULL, mine_dense);
      if (q < lim && inr && !mine_dense) {
        const int64_t wcols = gu ? H : I, wrows = gu ? 2 * I : H;
        int64_t col, arow;
        int e;
        if ((uint64_t)f <= 0xFFFFFFFFull) {  // 32-bit divisions where the flat index allows
          const uint32_t r32 = (uint32_t)f / (uint32_t)wcols;
          const uint32_t e32 = r32 / (uint32_t)wrows;
          col = (int64_t)((uint32_t)f - r32 * (uint32_t)wcols);
          e = (int)e32;
          arow = (int64_t)(r32 - e32 * (uint32_t)wrows);
        } else {
          const int64_t row = f / wcols;
          col = f - row * wcols;
          e = (int)(row / wrows);
          arow = row - (int64_t)e * wrows;
        }
        const int64_t o = off[e];
        const int nv = (cnt[e] + VW - 1) / VW;
        if (nv > 0) {
          md.x = (int)((arow * rcap + o) / VW);
          md.y = (int)((col * rcap + o) / VW);
          md.z = nv;
          md.w = nv - 1;
        }
      }
      meta[wid][lane] = md;
    }
    __syncwarp();
    for (int hf = 0; hf < 32 / SD_G; ++hf) {
      const int4* mh = &meta[wid][SD_G * hf];
      const int4 mine = mh[il];
      const uint32_t nvl = (uint32_t)mine.z;
      const uint32_t nmin = __reduce_min_sync(FULL, nvl);
      const uint32_t passes = (nmin + 16u) / 32u;
      const uint32_t vrest = 32u * passes;  // first vector left to the lane pairs
      const bool filled = nmin >= vrest;    // every entry has a vector for every lane of a pass
      // bit i: entry i loads its row vector (a new weight row, or a new vector on every pass)
      const bool fl = il == 0 || passes > 1 || mine.x != mh[il == 0 ? 0 : il - 1].x;
      const uint32_t fresh = __ballot_sync(FULL, fl) & ((1u << SD_G) - 1u);
      float part[SD_G];
#pragma unroll
      for (int i = 0; i < SD_G; ++i) part[i] = 0.f;
      if constexpr (RING) {
        if (passes > 0) {
          // Each entry's vectors come through a per-warp ring of SD_RING slots by cp.async, so
          // the loads of the next SD_RING entries are in flight while one entry's products run
          // (no registers are held for them). A lane copies, and reads back, only its own vector.
          uint8_t* ring = sd_ring + (size_t)wid * SD_RING * 2 * 512 + lane * 16;
          RowVec<T> rowv;
          for (uint32_t p = 0; p < passes; ++p) {
            const uint32_t v = p * 32u + (uint32_t)lane;
            auto issue = [&](int i) {
              const int4 m = mh[i];
              const uint32_t vv = filled ? v : min(v, (uint32_t)m.w);  // in bounds
              uint8_t* slot = ring + (i % SD_RING) * 1024;
              cp_async16(slot, Bm + ((uint32_t)m.y + vv));
              if (fresh & (1u << i)) cp_async16(slot + 512, A + ((uint32_t)m.x + vv));
              cp_async_commit();
            };
#pragma unroll
            for (int i = 0; i < SD_RING; ++i) issue(i);
#pragma unroll
            for (int i = 0; i < SD_G; ++i) {
              // groups committed after entry i's: min(SD_G, i + SD_RING) - (i + 1)
              cp_async_wait_dyn(min(SD_G, i + SD_RING) - (i + 1));
              const uint8_t* slot = ring + (i % SD_RING) * 1024;
              const uint4 bv = *reinterpret_cast<const uint4*>(slot);
              if (fresh & (1u << i)) rowv.set(*reinterpret_cast<const uint4*>(slot + 512));
              const float d = rowv.dot_acc(bv, part[i]);
              if (filled || v < (uint32_t)mh[i].z) part[i] = d;
              if (i + SD_RING < SD_G) issue(i + SD_RING);
            }
          }
        }
      } else if (passes > 0) {
        // Long rows (thousands of tokens per expert): the walk takes U entries at a time through
        // all their passes, their loads in flight together (registers).
        constexpr int U = 2;
        RowVec<T> rowv;
#pragma unroll
        for (int i0 = 0; i0 < SD_G; i0 += U) {
          for (uint32_t p = 0; p < passes; ++p) {
            const uint32_t v = p * 32u + (uint32_t)lane;
            uint4 av[U], bv[U];
            if (filled) {
#pragma unroll
              for (int u = 0; u < U; ++u) {
                const int4 m = mh[i0 + u];
                if (fresh & (1u << (i0 + u))) av[u] = __ldg(A + ((uint32_t)m.x + v));
                bv[u] = __ldg(Bm + ((uint32_t)m.y + v));
              }
#pragma unroll
              for (int u = 0; u < U; ++u) {
                if (fresh & (1u << (i0 + u))) rowv.set(av[u]);
                part[i0 + u] = rowv.dot_acc(bv[u], part[i0 + u]);
              }
            } else {
              uint32_t ok = 0;  // bit u: entry i0 + u has vector v
#pragma unroll
              for (int u = 0; u < U; ++u) {
                const int4 m = mh[i0 + u];
                ok |= (uint32_t)(v < (uint32_t)m.z) << u;
                const uint32_t vv = min(v, (uint32_t)m.w);
                if (fresh & (1u << (i0 + u))) av[u] = __ldg(A + ((uint32_t)m.x + vv));
                bv[u] = __ldg(Bm + ((uint32_t)m.y + vv));
              }
#pragma unroll
              for (int u = 0; u < U; ++u) {
                if (fresh & (1u << (i0 + u))) rowv.set(av[u]);
                const float d = rowv.dot_acc(bv[u], part[i0 + u]);
                if (ok & (1u << u)) part[i0 + u] = d;
              }
            }
          }
        }
      }
      float rem = 0.f;
      if (__any_sync(FULL, nvl > vrest)) {
        constexpr int LP = 32 / SD_G;  // lanes per entry
        const int4 m = mh[lane / LP];
        const uint32_t nr = (uint32_t)m.z > vrest ? (uint32_t)m.z - vrest : 0u;
        const uint32_t vend = vrest + __reduce_max_sync(FULL, nr);
        float s = 0.f;
        for (uint32_t v = vrest + (uint32_t)(lane % LP); v < vend; v += LP) {
          const uint32_t vv = min(v, (uint32_t)m.w);
          const float d = dot_acc<T>(__ldg(A + ((uint32_t)m.x + vv)),
                                     __ldg(Bm + ((uint32_t)m.y + vv)), s);
          if (v < (uint32_t)m.z) s = d;
        }
#pragma unroll
        for (int o = 1; o < LP; o <<= 1) s += __shfl_xor_sync(FULL, s, o);
        rem = __shfl_sync(FULL, s, LP * il);  // entry il's remainder, from lane LP il
      }
      const float gsum = transpose_reduce<SD_G>(part, lane) + rem;
      const int64_t q = b0 + SD_G * hf + lane;
      if (lane < SD_G && q < lim && !((skipm >> (SD_G * hf + lane)) & 1u)) {
        const float gv = accumulate ? g_act[q] + gsum : gsum;
        g_act[q] = gv;
        bad |= !finite_f(gv);
      }
    }
    __syncwarp();  // the next batch rewrites meta
  }
  flag_status_warp(dev_status, bad, USAF_DEV_NONFINITE);
  flag_status_warp(dev_status, badidx, USAF_DEV_BAD_INDEX);
}

// g_router[e, h] = sum over the rows routed to e of dl[row] * x[tok(row), h] (renormalised
// routing), read from the token-major x, whose rows stay in L2 while the eight experts of each
// token read them. On the tensor-core path (g_router_part_kernel):
// block (features, t) takes token tile t of the tensor-core tile plan (at most 256 rows of one
// expert, the experts' rows split in equal 16-row multiples) and 32 x VW features (one 16-byte
// vector per lane); its eight warps take contiguous eighths of the tile's rows with four rows'
// loads in flight, and the eight sums are added in warp order. A crowded expert is spread over as
// many blocks as it has tiles, each writing its sums to part[t][h]; g_router_reduce_kernel then
// adds them in tile order. An expert of one tile is written directly, one of none gets zeros from
// the reduction. The result does not depend on scheduling.
template <typename T>
__global__ void __launch_bounds__(256) g_router_part_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ ptok, const float* __restrict__ dl_perm,
    const int32_t* __restrict__ cnt, const int32_t* __restrict__ off,
    const int32_t* __restrict__ plan, int E, int H, float* __restrict__ part,
    float* __restrict__ g_router, int accumulate, uint32_t* dev_status) {
  constexpr int VW = 16 / sizeof(T);
  constexpr int FB = 32 * VW;  // features per block
  __shared__ float sp[8][FB];
  const int t = blockIdx.y;
  if (t >= plan[E]) return;  // the grid covers the most tiles any routing can have
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int lo = 0, hi = E;  // the tile's expert: the last e with plan[e] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (plan[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int e = lo;
  const int nts = plan[e + 1] - plan[e], npad = off[e + 1] - off[e];
  const int base = ((npad + nts - 1) / nts + 15) / 16 * 16;
  const int row0 = off[e] + (t - plan[e]) * base;
  const int rend = min(row0 + base, off[e] + cnt[e]);  // routed rows only (not the padding)
  const int n = max(0, rend - row0);
  const int r0 = row0 + (int)((int64_t)n * wid / 8), r1 = row0 + (int)((int64_t)n * (wid + 1) / 8);
  const int h = blockIdx.x * FB + lane * VW;
  const bool vec = (H % VW) == 0;
  struct Vec {
    float f[VW];
  };
  float acc[VW];
#pragma unroll
  for (int q = 0; q < VW; ++q) acc[q] = 0.f;
  auto load = [&](int tk) {
    alignas(16) T buf[VW];
    if (vec && h < H) {
      *reinterpret_cast<uint4*>(buf) = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)tk * H + h));
    } else {
#pragma unroll
      for (int q = 0; q < VW; ++q)
        buf[q] = h + q < H ? x[(int64_t)tk * H + h + q] : from_f32<T>(0.f);
    }
    Vec v;
#pragma unroll
    for (int q = 0; q < VW; ++q) v.f[q] = to_f32(buf[q]);
    return v;
  };
  int r = r0;
  for (; r + 4 <= r1; r += 4) {
    Vec v[4];
    float d[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      d[u] = dl_perm[r + u];
      v[u] = load(ptok[r + u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int q = 0; q < VW; ++q) acc[q] = fmaf(d[u], v[u].f[q], acc[q]);
  }
  for (; r < r1; ++r) {
    const float d = dl_perm[r];
    const Vec v = load(ptok[r]);
#pragma unroll
    for (int q = 0; q < VW; ++q) acc[q] = fmaf(d, v.f[q], acc[q]);
  }
#pragma unroll
  for (int q = 0; q < VW; ++q) sp[wid][lane * VW + q] = acc[q];
  __syncthreads();
  bool bad = false;
  const int c = threadIdx.x;  // FB <= blockDim.x: one feature per thread
  const int hh = blockIdx.x * FB + c;
  float sum = 0.f;
  if (c < FB) {
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += sp[w][c];
  }
  if (nts > 1) {
    if (c < FB && hh < H) part[(int64_t)t * H + hh] = sum;
    return;
  }
  if (c < FB && hh < H) {
    const int64_t u = (int64_t)e * H + hh;
    const float gv = accumulate ? g_router[u] + sum : sum;
    g_router[u] = gv;
    bad = !finite_f(gv);
  }
  flag_status_warp(dev_status, bad, USAF_DEV_NONFINITE);
}

// g_router rows of the experts with several tiles (their partial sums in tile order) and of the
// experts with none (zeros); the rows of one-tile experts are already written.
__global__ void g_router_reduce_kernel(const float* __restrict__ part,
                                       const int32_t* __restrict__ plan, int E, int H,
                                       float* __restrict__ g_router, int accumulate,
                                       uint32_t* dev_status) {
  bool bad = false;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < (int64_t)E * H;
       u += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(u / H), h = (int)(u - (int64_t)e * H);
    const int t0 = plan[e], t1 = plan[e + 1];
    if (t1 - t0 == 1) continue;
    float sum = 0.f;
    for (int t = t0; t < t1; ++t) sum += part[(int64_t)t * H + h];
    const float gv = accumulate ? g_router[u] + sum : sum;
    g_router[u] = gv;
    bad |= !finite_f(gv);
  }
  flag_status_warp(dev_status, bad, USAF_DEV_NONFINITE);
}

// The same sum for layers without the tile plan (fp32 layers): one block per expert and 32 x VW
// features, its eight warps over contiguous eighths of all the expert's rows.
template <typename T>
__global__ void __launch_bounds__(256) g_router_sel_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ ptok, const float* __restrict__ dl_perm,
    const int32_t* __restrict__ cnt, const int32_t* __restrict__ off, int H,
    float* __restrict__ g_router, int accumulate, uint32_t* dev_status) {
  constexpr int VW = 16 / sizeof(T);
  constexpr int FB = 32 * VW;
  __shared__ float sp[8][FB];
  const int e = blockIdx.y, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int h = blockIdx.x * FB + lane * VW;
  const int o = off[e], n = cnt[e];
  const int r0 = o + (int)((int64_t)n * wid / 8), r1 = o + (int)((int64_t)n * (wid + 1) / 8);
  float acc[VW];
#pragma unroll
  for (int q = 0; q < VW; ++q) acc[q] = 0.f;
  for (int r = r0; r < r1; ++r) {
    const float d = dl_perm[r];
    const int64_t xr = (int64_t)ptok[r] * H;
#pragma unroll
    for (int q = 0; q < VW; ++q)
      if (h + q < H) acc[q] = fmaf(d, to_f32(x[xr + h + q]), acc[q]);
  }
#pragma unroll
  for (int q = 0; q < VW; ++q) sp[wid][lane * VW + q] = acc[q];
  __syncthreads();
  bool bad = false;
  for (int c = threadIdx.x; c < FB; c += blockDim.x) {
    const int hh = blockIdx.x * FB + c;
    if (hh >= H) continue;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += sp[w][c];
    const int64_t u = (int64_t)e * H + hh;
    const float gv = accumulate ? g_router[u] + sum : sum;
    g_router[u] = gv;
    bad |= !finite_f(gv);
  }
  flag_status_warp(dev_status, bad, USAF_DEV_NONFINITE);
}


template <typename T>
__global__ void f32_to_kernel(const float* __restrict__ src, T* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = from_f32<T>(src[i]);
}

// dw[q] = the sum of slot q's nparts partials (one per M tile and row quarter of the gvec GEMM),
// in a fixed order with four loads in flight: dw does not depend on which tile finished first.
__global__ void __launch_bounds__(256) dw_reduce_kernel(const float* __restrict__ part, int nparts,
                                                        int64_t n_slots, float* __restrict__ dw) {
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n_slots;
       q += (int64_t)gridDim.x * blockDim.x) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int i = 0;
    for (; i + 4 <= nparts; i += 4) {
      a0 += part[(int64_t)i * n_slots + q];
      a1 += part[(int64_t)(i + 1) * n_slots + q];
      a2 += part[(int64_t)(i + 2) * n_slots + q];
      a3 += part[(int64_t)(i + 3) * n_slots + q];
    }
    for (; i < nparts; ++i) a0 += part[(int64_t)i * n_slots + q];
    dw[q] = (a0 + a1) + (a2 + a3);
  }
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
  __shared__ float s_dw[32];
  if (threadIdx.x < k) s_dw[threadIdx.x] = dw[(int64_t)t * k + threadIdx.x];
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
    for (int j = 0; j < k; ++j) s = fmaf(w[(int64_t)t * k + j], s_dw[j], s);
    sh_s = s;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float p = expf(l[e] - sh_mx) / sh_sum;
    float d = 0.f;
    for (int j = 0; j < k; ++j)
      if (idx[(int64_t)t * k + j] == e) d = s_dw[j];
    dlogit[(int64_t)t * E + e] = p * (d - sh_s);
  }
}

// g_router[e, h] = sum over the rows routed to e of dl[row] * x_perm[row, h] (renormalised
// routing); each thread owns two adjacent h, rows in order, eight rows in flight.
template <typename T>
__global__ void g_router_dense_kernel(const T* __restrict__ x, const float* __restrict__ dlogit,
                                      int Tn, int E, int H, float* __restrict__ g_router,
                                      int accumulate, uint32_t* dev_status) {
  const int e = blockIdx.y;
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  float acc = 0.f;
  if (h < H) {
    for (int t = 0; t < Tn; ++t)
      acc = fmaf(dlogit[(int64_t)t * E + e], to_f32(x[(int64_t)t * H + h]), acc);
    if (accumulate) acc += g_router[(int64_t)e * H + h];
    g_router[(int64_t)e * H + h] = acc;
  }
  flag_status_warp(dev_status, h < H && !finite_f(acc), USAF_DEV_NONFINITE);
}

// dx[t, h] = dx_acc[t, h] + router term: sum_j dl[t,j] Wr[e_j, h] (renormalised routing) or
// sum_e dlogit[t,e] Wr[e, h]; router_term = 0 when the dx GEMM's epilogue already added it. One
// token per block, four h per thread.
template <typename T>
__global__ void __launch_bounds__(256) dx_finalize_kernel(
    const float* __restrict__ dx_acc, const float* __restrict__ wr, const int32_t* __restrict__ idx,
    const float* __restrict__ dl, const float* __restrict__ dlogit, int Tn, int H, int E, int k,
    int renorm, int router_term, T* __restrict__ dx, uint32_t* dev_status) {
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
    const int nterm = !router_term ? 0 : renorm ? k : E;
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
  w.wperm = c.take<float>(usaf_routed_rows_capacity(&s));
}

void bwd_ws_layout(const usaf_moe_shape& s, usaf_dtype dt, int64_t K, Carver& c, BwdWs& w) {
  (void)K;
  const int64_t R_cap = usaf_routed_rows_capacity(&s);
  const size_t es = dt == USAF_BF16 ? 2 : 4;
  w.dw = c.take<float>(s.T * s.k);
  w.dw_part = dt == USAF_BF16 ? c.take<float>(4 * ceil_div(s.I, 128) * s.T * s.k) : nullptr;
  w.dl = c.take<float>(s.T * s.k);
  w.dl_perm = c.take<float>(R_cap);
  w.dlogit = c.take<float>(s.T * s.E);
  w.dh = c.take<char>(R_cap * 2 * s.I * (int64_t)es);
  w.dx_acc = c.take<float>(s.T * s.H);
  w.gvec = dt == USAF_F32 ? c.take<float>(R_cap * s.I) : nullptr;
  w.plan = dt == USAF_BF16 ? c.take<int32_t>(s.E + 1) : nullptr;
  w.wperm = c.take<float>(R_cap);
  w.dy_perm = c.take<char>(R_cap * s.H * (int64_t)es);
  w.g_part = dt == USAF_BF16 ? c.take<float>((ceil_div(R_cap, TC_TOKEN_TILE) + s.E) * s.H)
                             : nullptr;
}

template <typename T>
static usaf_status gather_t(const MoeArgs& a, const T* src, T* dstT, cudaStream_t st,
                           GatherExtra ex) {
  if constexpr (sizeof(T) == 2) {
    const auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    CUtensorMap tm;
    if (a.s.H % 64 == 0 && a.R_cap % GR_ROWS == 0 && al16(src) && al16(dstT) &&
        al16(a.rt.perm_tok) && al16(a.rt.perm_slot) && tc_token_map(&tm, dstT, a.s.H, a.R_cap)) {
      static bool attr_done = false;
      if (!attr_done) {
        if (cudaFuncSetAttribute(gather_transpose_bf16_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 GR_SMEM) != cudaSuccess)
          return USAF_ERR_CUDA;
        attr_done = true;
      }
      const dim3 grid((unsigned)(a.R_cap / GR_ROWS), (unsigned)(a.s.H / 64));
      gather_transpose_bf16_kernel<<<grid, 256, GR_SMEM, st>>>(
          tm, src, a.rt.perm_tok, a.rt.perm_slot, a.rt.expert_offset + a.s.E, a.R_cap,
          (int)a.s.H, a.rt.topk_w, a.wperm, ex);
      USAF_CHECK_LAUNCH();
      return USAF_OK;
    }
  }
  const dim3 grid((unsigned)ceil_div(a.R_cap, GT_ROWS), (unsigned)ceil_div(a.s.H, 64));
  gather_transpose_kernel<T><<<grid, 256, 0, st>>>(src, a.rt.perm_tok, a.rt.perm_slot,
                                                   a.rt.expert_offset + a.s.E, a.R_cap,
                                                   (int)a.s.H, dstT, a.rt.topk_w, a.wperm, ex);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

template <typename T>
static usaf_status fwd_simt(const MoeArgs& a, T* xT, T* hT, T* waT, float* yacc, cudaStream_t st) {
  USAF_TRACE("simt_fwd", st);
  const auto& s = a.s;
  const int H = (int)s.H, I = (int)s.I, E = (int)s.E;
  const int32_t* cnt = a.rt.expert_count;
  const int32_t* off = a.rt.expert_offset;
  ProbGateUp<T> p1{xT, static_cast<const T*>(a.w_gate_up), hT, cnt, off, H, 2 * I, a.R_cap};
  dim3 g1((unsigned)ceil_div(2 * I, 64), (unsigned)ceil_div(s.T, 64), (unsigned)E);
  simt_gemm_kernel<<<g1, 256, 0, st>>>(p1);
  USAF_CHECK_LAUNCH();
  swiglu_fwd_rows_kernel<T><<<(unsigned)a.R_cap, 128, 0, st>>>(hT, a.rt.perm_slot, a.rt.topk_w,
                                                               off + E, I, a.R_cap, waT);
  USAF_CHECK_LAUNCH();
  ProbDown<T> p2{waT, static_cast<const T*>(a.w_down), yacc, cnt, off, a.rt.perm_tok, H, I,
                 a.R_cap};
  dim3 g2((unsigned)ceil_div(H, 64), (unsigned)ceil_div(s.T, 64), (unsigned)E);
  simt_gemm_kernel<<<g2, 256, 0, st>>>(p2);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

// Make `st` wait for `ev` (NULL: no wait).
static usaf_status wait_event(cudaStream_t st, cudaEvent_t ev) {
  if (!ev) return USAF_OK;
  return cudaStreamWaitEvent(st, ev, 0) == cudaSuccess ? USAF_OK : USAF_ERR_CUDA;
}

// The forward's stages (FWD_* bits): the token gather (which also clears the combine accumulator
// and writes the tile plan), the gate_up GEMM, the down GEMM with the combine into y.
template <typename T>
static usaf_status moe_fwd_t(const MoeArgs& a, T* xT, T* hT, T* waT, T* y, FwdWs& w,
                             cudaEvent_t weights_ready, cudaEvent_t down_ready, int stages,
                             cudaStream_t st) {
  const auto& s = a.s;
  const int64_t TH = s.T * s.H;
  MoeArgs aw = a;
  aw.wperm = w.wperm;
  if (a.dt != USAF_BF16 && (stages & (FWD_GATE_UP | FWD_DOWN)) != 0 &&
      (stages & (FWD_GATE_UP | FWD_DOWN)) != (FWD_GATE_UP | FWD_DOWN))
    return USAF_ERR_UNSUPPORTED;  // the fp32 layers' GEMMs run as one stage
  if (stages & FWD_GATHER) {
    USAF_TRACE("gather_x", st);
    const GatherExtra ex{w.y_acc, TH, nullptr, 0, a.rt.expert_offset, (int)s.E,
                         a.dt == USAF_BF16 ? w.plan : nullptr};
    USAF_TRY(gather_t<T>(aw, static_cast<const T*>(a.x), xT, st, ex));
  }
  // the expert weights are read from here on: wait for their last update only now (gate_up's
  // before its GEMM, down_proj's before the down GEMM)
  if (a.dt == USAF_BF16) {
    MoeArgs b = aw;
    b.plan = w.plan;
    if (stages & FWD_GATE_UP) {
      USAF_TRY(wait_event(st, weights_ready));
      USAF_TRY(tc_fwd_gate_up(b, xT, hT, waT, st));
    }
    if (stages & FWD_DOWN) {
      USAF_TRY(wait_event(st, down_ready));
      USAF_TRY(tc_fwd_down(b, waT, w.y_acc, st));
    }
  } else if (stages & FWD_GATE_UP) {
    USAF_TRY(wait_event(st, weights_ready));
    USAF_TRY(wait_event(st, down_ready));
    USAF_TRY(fwd_simt<T>(a, xT, hT, waT, w.y_acc, st));
  }
  if (stages & FWD_DOWN) {
    USAF_TRACE("combine_finalize", st);
    f32_to_kernel<T><<<grid_dim_for(TH), 256, 0, st>>>(w.y_acc, y, TH);
    USAF_CHECK_LAUNCH();
  }
  return USAF_OK;
}

usaf_status moe_fwd_launch(const MoeArgs& a, void* x_perm, void* h, void* wa, void* y, FwdWs& w,
                           cudaEvent_t weights_ready, cudaEvent_t down_ready, int stages,
                           cudaStream_t st) {
  if (a.dt == USAF_BF16)
    return moe_fwd_t<__nv_bfloat16>(a, static_cast<__nv_bfloat16*>(x_perm),
                                    static_cast<__nv_bfloat16*>(h),
                                    static_cast<__nv_bfloat16*>(wa),
                                    static_cast<__nv_bfloat16*>(y), w, weights_ready, down_ready,
                                    stages, st);
  return moe_fwd_t<float>(a, static_cast<float*>(x_perm), static_cast<float*>(h),
                          static_cast<float*>(wa), static_cast<float*>(y), w, weights_ready,
                          down_ready, stages, st);
}

// Dense expert weight gradient on CUDA cores (fp32 layers): one thread per entry of
// g[e] (a_rows x b_rows), summing over the expert's routed tokens.
template <typename T>
__global__ void dense_wgrad_simt_kernel(const T* __restrict__ aT, int64_t a_rows,
                                        const T* __restrict__ bT, int64_t b_rows,
                                        const int32_t* __restrict__ off, int E, int64_t rcap,
                                        float* __restrict__ g, int accumulate) {
  const int64_t per = a_rows * b_rows, n = (int64_t)E * per;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / per);
    const int64_t rc = i - (int64_t)e * per, r = rc / b_rows, c = rc - r * b_rows;
    const int o = off[e], np = off[e + 1] - o;
    const T* ar = aT + r * rcap + o;
    const T* br = bT + c * rcap + o;
    float acc = 0.f;
    for (int t = 0; t < np; ++t) acc = fmaf(to_f32(ar[t]), to_f32(br[t]), acc);
    g[i] = accumulate ? g[i] + acc : acc;
  }
}

template <typename T>
static usaf_status moe_bwd_t(const MoeArgs& a0, int renorm, const float* logits, const T* xT,
                             const T* hT, const T* waT, const T* dy, const int64_t* act_idx,
                             int64_t K, float* g_act, float* g_router, T* dx, float* dw_out,
                             float* g_dense, int accumulate, uint32_t* dev_status, BwdWs& w,
                             cudaStream_t st, const MaskedPlan* plan, int64_t n_dense) {
  MoeArgs a = a0;
  a.plan = w.plan;
  a.wperm = w.wperm;
  const auto& s = a.s;
  const int H = (int)s.H, I = (int)s.I, E = (int)s.E, Tn = (int)s.T, k = (int)s.k;
  const int32_t* cnt = a.rt.expert_count;
  const int32_t* off = a.rt.expert_offset;
  const int32_t* pslot = a.rt.perm_slot;
  float* dw = dw_out ? dw_out : w.dw;
  T* dhT = static_cast<T*>(w.dh);
  T* dyT = static_cast<T*>(w.dy_perm);
  const int64_t Ngu = s.E * 2 * s.I * s.H;
  SideStream side{};
  bool forked = false;  // the router gradient runs beside dx and the masked gradient

  // S6: gvec, dw, dh
  {
    USAF_TRACE("gather_dy", st);
    // also zeroes the dx accumulator and writes the tile plan
    const GatherExtra ex{dx ? w.dx_acc : nullptr, dx ? s.T * s.H : 0, nullptr, 0,
                         a.rt.expert_offset, (int)s.E, a.dt == USAF_BF16 ? w.plan : nullptr};
    USAF_TRY(gather_t<T>(a, dy, dyT, st, ex));
  }
  if (a.dt == USAF_BF16) {
    USAF_TRY(tc_bwd_gvec(a, dyT, hT, dhT, w.dw_part, st));
  } else {
    USAF_TRACE("simt_gvec", st);
    ProbGvec<T> p{dyT, static_cast<const T*>(a.w_down), w.gvec, cnt, off, H, I, a.R_cap};
    dim3 g((unsigned)ceil_div(I, 64), (unsigned)ceil_div(Tn, 64), (unsigned)E);
    simt_gemm_kernel<<<g, 256, 0, st>>>(p);
    USAF_CHECK_LAUNCH();
    swiglu_bwd_rows_kernel<T><<<(unsigned)a.R_cap, 128, 0, st>>>(w.gvec, hT, pslot, a.rt.topk_w,
                                                                 off + E, I, a.R_cap, dhT, dw);
    USAF_CHECK_LAUNCH();
  }
  // S7: router gradient (on the tensor-core path dw is first summed from its tile partials)
  {
    USAF_TRACE("router_bwd", st);
    if (a.dt == USAF_BF16) {
      const int nparts = 4 * (int)ceil_div(s.I, 128);
      dw_reduce_kernel<<<grid_dim_for(s.T * s.k), 256, 0, st>>>(w.dw_part, nparts, s.T * s.k,
                                                               dw);
      USAF_CHECK_LAUNCH();
    }
    if (renorm) {
      dlogit_sel_kernel<<<(unsigned)ceil_div(Tn, 128), 128, 0, st>>>(
          a.rt.topk_w, dw, a.rt.slot_row, Tn, k, w.dl, w.dl_perm);
      USAF_CHECK_LAUNCH();
      constexpr int FB = 32 * (16 / (int)sizeof(T));
      if (a.dt == USAF_BF16) {
        // g_router needs only dl (dx's epilogue reads dl too, nothing reads g_router before the
        // call returns): it runs on a side stream beside dx and the masked gradient, forked here
        // and joined back at the end of the call (two branches of a captured graph)
        forked = side_stream(side, st);
        if (forked && (cudaEventRecord(side.fork, st) != cudaSuccess ||
                       cudaStreamWaitEvent(side.s, side.fork, 0) != cudaSuccess))
          return USAF_ERR_CUDA;
        const cudaStream_t rs = forked ? side.s : st;
        USAF_TRACE("router_grad", rs);
        // token tiles of at most 256 rows: ceil(R_cap / 256) + E bounds their count
        const unsigned ntile = (unsigned)(ceil_div(a.R_cap, TC_TOKEN_TILE) + E);
        g_router_part_kernel<T><<<dim3((unsigned)ceil_div(H, FB), ntile), 256, 0, rs>>>(
            static_cast<const T*>(a.x), a.rt.perm_tok, w.dl_perm, cnt, off, w.plan, E, H,
            w.g_part, g_router, accumulate, dev_status);
        USAF_CHECK_LAUNCH();
        g_router_reduce_kernel<<<grid_dim_for((int64_t)E * H), 256, 0, rs>>>(
            w.g_part, w.plan, E, H, g_router, accumulate, dev_status);
      } else {
        g_router_sel_kernel<T><<<dim3((unsigned)ceil_div(H, FB), (unsigned)E), 256, 0, st>>>(
            static_cast<const T*>(a.x), a.rt.perm_tok, w.dl_perm, cnt, off, H, g_router,
            accumulate, dev_status);
      }
      USAF_CHECK_LAUNCH();
    } else {
      dlogit_dense_kernel<<<(unsigned)Tn, 128, 0, st>>>(logits, a.rt.topk_idx, a.rt.topk_w, dw,
                                                        Tn, E, k, w.dlogit);
      USAF_CHECK_LAUNCH();
      g_router_dense_kernel<T><<<dim3((unsigned)ceil_div(H, 128), (unsigned)E), 128, 0, st>>>(
          static_cast<const T*>(a.x), w.dlogit, Tn, E, H, g_router, accumulate, dev_status);
      USAF_CHECK_LAUNCH();
    }
  }
  // S8: dx
  // with renormalised routing the tensor-core dx epilogue adds the router's share itself
  const bool rterm_in_gemm = a.dt == USAF_BF16 && renorm &&
                             (reinterpret_cast<uintptr_t>(a.w_router) & 15) == 0;
  if (dx) {
    if (a.dt == USAF_BF16) {
      USAF_TRY(tc_bwd_dx(a, dhT, w.dx_acc, rterm_in_gemm ? w.dl_perm : nullptr, st));
    } else {
      USAF_TRACE("simt_dx", st);
      ProbDx<T> p{dhT, static_cast<const T*>(a.w_gate_up), w.dx_acc, cnt, off, a.rt.perm_tok,
                  H, 2 * I, a.R_cap};
      dim3 g((unsigned)ceil_div(H, 64), (unsigned)ceil_div(Tn, 64), (unsigned)E);
      simt_gemm_kernel<<<g, 256, 0, st>>>(p);
      USAF_CHECK_LAUNCH();
    }
    USAF_TRACE("dx_finalize", st);
    dx_finalize_kernel<T><<<(unsigned)Tn, 256, 0, st>>>(w.dx_acc, a.w_router, a.rt.topk_idx, w.dl,
                                                        w.dlogit, Tn, H, E, k, renorm,
                                                        rterm_in_gemm ? 0 : 1, dx, dev_status);
    USAF_CHECK_LAUNCH();
  }
  // S9, S10: expert weight gradients at the active set
  if (K > 0) {
    const bool use_plan = plan && n_dense > 0 && a.dt == USAF_BF16;
    {
      USAF_TRACE("wgrad_sddmm", st);
      const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(K, SD_WARPS * 32),
                                                          device_sm_count() * SD_BLOCKS_PER_SM);
      // the cp.async ring where experts hold up to about a thousand routed rows on average;
      // the register walk where rows run to thousands of tokens (there the ring's restart per
      // 256-token pass costs more than it hides)
      if ((int64_t)s.T * s.k <= (int64_t)1024 * E) {
        static bool ring_attr = false;  // the ring plus the static metadata exceed 48 KB
        if (!ring_attr) {
          if (cudaFuncSetAttribute(sddmm_kernel<T, true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   SD_RING_BYTES) != cudaSuccess)
            return USAF_ERR_CUDA;
          ring_attr = true;
        }
        sddmm_kernel<T, true><<<blocks, SD_WARPS * 32, SD_RING_BYTES, st>>>(
            act_idx, K, cnt, off, E, H, I, Ngu, a.R_cap, dhT, xT, dyT, waT, g_act, accumulate,
            dev_status, use_plan ? plan->dense_flag : nullptr);
      } else {
        sddmm_kernel<T, false><<<blocks, SD_WARPS * 32, 0, st>>>(
            act_idx, K, cnt, off, E, H, I, Ngu, a.R_cap, dhT, xT, dyT, waT, g_act, accumulate,
            dev_status, use_plan ? plan->dense_flag : nullptr);
      }
      USAF_CHECK_LAUNCH();
    }
    if (use_plan) {
      // the experts whose active density makes a dense tile cheaper: tensor-core tiles, the
      // accumulator written at the active entries only
      USAF_TRY(tc_wgrad_gather(a, dhT, 2 * I, xT, H, *plan, 0, act_idx, g_act, accumulate, st));
      USAF_TRY(tc_wgrad_gather(a, dyT, H, waT, I, *plan, 1, act_idx, g_act, accumulate, st));
    }
  }
  // dense expert weight gradients (importance phase)
  if (g_dense) {
    if (a.dt == USAF_BF16) {
      USAF_TRY(tc_wgrad_dense(a, dhT, 2 * I, xT, H, g_dense, accumulate, st));
      USAF_TRY(tc_wgrad_dense(a, dyT, H, waT, I, g_dense + Ngu, accumulate, st));
    } else {
      USAF_TRACE("simt_wgrad_dense", st);
      dense_wgrad_simt_kernel<T><<<grid_dim_for(Ngu), 256, 0, st>>>(
          dhT, 2 * I, xT, H, off, E, a.R_cap, g_dense, accumulate);
      USAF_CHECK_LAUNCH();
      dense_wgrad_simt_kernel<T><<<grid_dim_for(Ngu / 2), 256, 0, st>>>(
          dyT, H, waT, I, off, E, a.R_cap, g_dense + Ngu, accumulate);
      USAF_CHECK_LAUNCH();
    }
  }
  if (forked && (cudaEventRecord(side.join, side.s) != cudaSuccess ||
                 cudaStreamWaitEvent(st, side.join, 0) != cudaSuccess))
    return USAF_ERR_CUDA;
  return USAF_OK;
}

// The dense expert weight gradient alone, from the dh^T and dy^T that the preceding backward call
// left in the same workspace (the importance phase's dense pass after a sparse backward).
usaf_status moe_wgrad_dense_launch(const MoeArgs& a0, const void* x_perm, const void* wa,
                                   float* g_dense, int accumulate, BwdWs& w, cudaStream_t st) {
  MoeArgs a = a0;
  a.plan = w.plan;
  a.wperm = w.wperm;
  const auto& s = a.s;
  const int H = (int)s.H, I = (int)s.I, E = (int)s.E;
  const int64_t Ngu = s.E * 2 * s.I * s.H;
  if (a.dt == USAF_BF16) {
    using T = __nv_bfloat16;
    const T* dhT = static_cast<const T*>(w.dh);
    const T* dyT = static_cast<const T*>(w.dy_perm);
    USAF_TRY(tc_wgrad_dense(a, dhT, 2 * I, x_perm, H, g_dense, accumulate, st));
    USAF_TRY(tc_wgrad_dense(a, dyT, H, wa, I, g_dense + Ngu, accumulate, st));
    return USAF_OK;
  }
  USAF_TRACE("simt_wgrad_dense", st);
  const float* dhT = static_cast<const float*>(w.dh);
  const float* dyT = static_cast<const float*>(w.dy_perm);
  const int32_t* off = a.rt.expert_offset;
  dense_wgrad_simt_kernel<float><<<grid_dim_for(Ngu), 256, 0, st>>>(
      dhT, 2 * I, static_cast<const float*>(x_perm), H, off, E, a.R_cap, g_dense, accumulate);
  USAF_CHECK_LAUNCH();
  dense_wgrad_simt_kernel<float><<<grid_dim_for(Ngu / 2), 256, 0, st>>>(
      dyT, H, static_cast<const float*>(wa), I, off, E, a.R_cap, g_dense + Ngu, accumulate);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

usaf_status moe_bwd_launch(const MoeArgs& a, int renorm, const float* logits, const void* x_perm,
                           const void* h, const void* wa, const void* dy, const int64_t* act_idx,
                           int64_t K, float* g_act, float* g_router, void* dx, float* dw_slot,
                           float* g_dense, int accumulate, uint32_t* dev_status, BwdWs& w,
                           cudaStream_t st, const MaskedPlan* plan, int64_t n_dense) {
  using B = __nv_bfloat16;
  if (a.dt == USAF_BF16)
    return moe_bwd_t<B>(a, renorm, logits, static_cast<const B*>(x_perm),
                        static_cast<const B*>(h), static_cast<const B*>(wa),
                        static_cast<const B*>(dy), act_idx, K, g_act, g_router,
                        static_cast<B*>(dx), dw_slot, g_dense, accumulate, dev_status, w, st,
                        plan, n_dense);
  return moe_bwd_t<float>(a, renorm, logits, static_cast<const float*>(x_perm),
                          static_cast<const float*>(h), static_cast<const float*>(wa),
                          static_cast<const float*>(dy), act_idx, K, g_act, g_router,
                          static_cast<float*>(dx), dw_slot, g_dense, accumulate, dev_status, w,
                          st, nullptr, 0);
}

// ================================================================================================
// Masked-gradient plan of an active set
// ================================================================================================
size_t masked_plan_bytes(const usaf_moe_shape& s) {
  Carver c(nullptr);
  c.take<int64_t>(4);
  c.take<int32_t>(s.E);
  c.take<int32_t>(s.E);
  c.take<int64_t>(s.E * (2 * s.I + s.H + 2));
  return c.size();
}

MaskedPlan masked_plan_layout(const usaf_moe_shape& s, void* base) {
  Carver c(base);
  MaskedPlan p{};
  int64_t* head = c.take<int64_t>(4);
  p.dense_list = c.take<int32_t>(s.E);
  p.dense_flag = c.take<int32_t>(s.E);
  p.row_ptr = c.take<int64_t>(s.E * (2 * s.I + s.H + 2));
  p.n_dense = reinterpret_cast<const int32_t*>(head + 1);  // head[0]: the same count as int64
  p.rp_stride = 2 * s.I + s.H + 2;
  return p;
}

__device__ __forceinline__ int64_t lower_bound_act(const int64_t* a, int64_t lo, int64_t hi,
                                                   int64_t key) {
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// One block, one thread per expert (E <= 1024): the expert's active entries in both tensors; an
// expert with at least thr_count of them is listed (in expert order) for the dense tile kernel.
__global__ void __launch_bounds__(1024) plan_experts_kernel(const int64_t* __restrict__ act,
                                                            int64_t K, int E, int H, int I,
                                                            int64_t thr_count, int64_t* head,
                                                            int32_t* dense_list,
                                                            int32_t* dense_flag) {
  __shared__ int32_t wsum[32];
  const int e = threadIdx.x, lane = e & 31, wid = e >> 5;
  int32_t dense = 0;
  if (e < E) {
    const int64_t pgu = (int64_t)2 * I * H, pd = (int64_t)H * I, Ngu = (int64_t)E * pgu;
    const int64_t a0 = lower_bound_act(act, 0, K, (int64_t)e * pgu);
    const int64_t a1 = lower_bound_act(act, a0, K, (int64_t)(e + 1) * pgu);
    const int64_t b0 = lower_bound_act(act, 0, K, Ngu + (int64_t)e * pd);
    const int64_t b1 = lower_bound_act(act, b0, K, Ngu + (int64_t)(e + 1) * pd);
    dense = (a1 - a0) + (b1 - b0) >= thr_count ? 1 : 0;
    dense_flag[e] = dense;
  }
  int32_t x = dense;
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int32_t v = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    wsum[lane] = v;
  }
  __syncthreads();
  const int32_t before = x - dense + (wid > 0 ? wsum[wid - 1] : 0);
  if (dense) dense_list[before] = e;
  if (e == (int)blockDim.x - 1) {
    const int32_t total = wsum[(blockDim.x >> 5) - 1];
    head[0] = total;
    reinterpret_cast<int32_t*>(head + 1)[0] = total;
  }
}

// First active entry of every row of the listed experts (gate_up rows 0 .. 2I, down rows 0 .. H).
__global__ void plan_rows_kernel(const int64_t* __restrict__ act, int64_t K, int E, int H, int I,
                                 const int32_t* __restrict__ dense_flag, int64_t stride,
                                 int64_t* __restrict__ row_ptr) {
  const int e = blockIdx.y;
  if (!dense_flag[e]) return;
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= stride) return;
  const int64_t pgu = (int64_t)2 * I * H, pd = (int64_t)H * I, Ngu = (int64_t)E * pgu;
  const int64_t f = r <= 2 * I ? (int64_t)e * pgu + r * H
                               : Ngu + (int64_t)e * pd + (r - (2 * I + 1)) * I;
  row_ptr[(int64_t)e * stride + r] = lower_bound_act(act, 0, K, f);
}

usaf_status masked_plan_build_launch(const usaf_moe_shape& s, const int64_t* act, int64_t K,
                                     int64_t thr_count, void* plan, cudaStream_t st) {
  USAF_TRACE("masked_plan", st);
  const MaskedPlan p = masked_plan_layout(s, plan);
  int64_t* head = static_cast<int64_t*>(plan);
  plan_experts_kernel<<<1, 1024, 0, st>>>(act, K, (int)s.E, (int)s.H, (int)s.I, thr_count, head,
                                          const_cast<int32_t*>(p.dense_list),
                                          const_cast<int32_t*>(p.dense_flag));
  USAF_CHECK_LAUNCH();
  const dim3 grid((unsigned)ceil_div(p.rp_stride, 256), (unsigned)s.E);
  plan_rows_kernel<<<grid, 256, 0, st>>>(act, K, (int)s.E, (int)s.H, (int)s.I, p.dense_flag,
                                         p.rp_stride, const_cast<int64_t*>(p.row_ptr));
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

}  // namespace usaf
