// Routing: router logits, warp-shuffle top-k with renormalised softmax weights, and the
// deterministic counting-sort permutation into padded per-expert segments.
//
// The router is the gating network the USAF README trains in full ("The router is leverage").
// The routing rule (softmax over experts, top-k, renormalise) is the Qwen3-MoE gating of the
// model the README benchmarks; the pages do not spell it out.
#include "common.cuh"
#include "kernels.cuh"

namespace usaf {

// ------------------------------------------------------------------------------------------------
// S1: logits[t,e] = sum_h x[t,h] * Wr[e,h]  (fp32 FFMA, x upcast exactly)
// Tile: 64 tokens x 64 experts per block, 256 threads, each thread 4 tokens x 4 experts; the
// k-major shared tiles are read as float4, two vector loads per 16 FMAs.
// ------------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) router_logits_kernel(const T* __restrict__ x,
                                                            const float* __restrict__ wr,
                                                            float* __restrict__ logits, int Tn,
                                                            int H, int E) {
  constexpr int BT = 64, BE = 64, BK = 32, LD = 68;
  __shared__ __align__(16) float xs[BK][LD];
  __shared__ __align__(16) float ws[BK][LD];
  const int t0 = blockIdx.y * BT, e0 = blockIdx.x * BE;
  const int tid = threadIdx.x;
  const int tr = tid / 16;  // tokens tr*4 .. +3
  const int ec = tid % 16;  // experts ec*4 .. +3
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += BK) {
    for (int i = tid; i < BT * BK; i += 256) {
      const int tt = i / BK, kk = i % BK;
      const int t = t0 + tt, k = k0 + kk;
      xs[kk][tt] = (t < Tn && k < H) ? to_f32(x[(int64_t)t * H + k]) : 0.f;
    }
    for (int i = tid; i < BE * BK; i += 256) {
      const int ee = i / BK, kk = i % BK;
      const int e = e0 + ee, k = k0 + kk;
      ws[kk][ee] = (e < E && k < H) ? wr[(int64_t)e * H + k] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[kk][tr * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&ws[kk][ec * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + tr * 4 + i;
    if (t >= Tn) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + ec * 4 + j;
      if (e < E) logits[(int64_t)t * E + e] = acc[i][j];
    }
  }
}

// ------------------------------------------------------------------------------------------------
// S2: one warp per token. k rounds of a warp argmax over the logits not yet taken; order is
// (logit descending, expert ascending) with floating-point comparison (so -0 == +0). Lane l
// holds the token's logits l, l + 32, ... in registers (NL of them), with a bit mask of the ones
// taken; lane j keeps the j-th selection.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

template <int NL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int Tn,
                                                   int E, int k, int renorm,
                                                   int32_t* __restrict__ topk_idx,
                                                   float* __restrict__ topk_w) {
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x % 32;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= Tn) return;
  const float* row = logits + (int64_t)t * E;
  float v[NL];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < NL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
    if (e < E) mx = fmaxf(mx, v[i]);
  }
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
  uint32_t taken = 0;  // bit i: logit lane + 32 i is selected
  float my_l = 0.f;    // lane j < k: the j-th selected logit and its expert
  int my_e = 0;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, be)) {
        bv = v[i];
        be = e;
      }
    }
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(FULL, bv, o);
      const int oe = __shfl_xor_sync(FULL, be, o);
      if (better(ov, oe, bv, be)) {
        bv = ov;
        be = oe;
      }
    }
    // every lane holds the same winner now
    if (be == 0x7fffffff) be = 0;  // only if all remaining logits are NaN
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_l = bv;
      my_e = be;
    }
  }
  const float ref = __shfl_sync(FULL, my_l, 0);
  float denom = 0.f;
  if (renorm) {
    for (int j = 0; j < k; ++j) denom += expf(__shfl_sync(FULL, my_l, j) - ref);
  } else {
#pragma unroll
    for (int i = 0; i < NL; ++i)
      if (lane + 32 * i < E) denom += expf(v[i] - mx);
    for (int o = 16; o; o >>= 1) denom += __shfl_xor_sync(FULL, denom, o);
  }
  if (lane < k) {
    const float num = renorm ? expf(my_l - ref) : expf(my_l - mx);
    topk_idx[(int64_t)t * k + lane] = my_e;
    topk_w[(int64_t)t * k + lane] = num / denom;
  }
}

// ------------------------------------------------------------------------------------------------
// S3: counting sort of the R = T*k slots by expert; within an expert, ascending slot (= token).
// Chunks of PERM_CHUNK consecutive slots: per-chunk histograms, one scan, one ordered fill.
// ------------------------------------------------------------------------------------------------
__global__ void perm_count_kernel(const int32_t* __restrict__ topk_idx, int64_t R, int E,
                                  int32_t* __restrict__ chunk_hist) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t s0 = (int64_t)blockIdx.x * PERM_CHUNK;
  for (int64_t s = s0 + threadIdx.x; s < min(R, s0 + PERM_CHUNK); s += blockDim.x)
    atomicAdd(&hist[topk_idx[s]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_hist[(int64_t)blockIdx.x * E + e] = hist[e];
}

// One block of 1024 threads: per expert totals and per-chunk bases, then padded offsets.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ chunk_hist,
                                                         int nchunks, int E,
                                                         int32_t* __restrict__ expert_count,
                                                         int32_t* __restrict__ expert_offset) {
  __shared__ int32_t padded[1024];
  __shared__ int32_t warp_sums[32];
  const int e = threadIdx.x;
  int32_t total = 0;
  if (e < E) {
    // 16 chunks' counts are loaded before any base is written back, so the column costs
    // nchunks / 16 load latencies instead of nchunks
    constexpr int UNR = 16;
    for (int b0 = 0; b0 < nchunks; b0 += UNR) {
      int32_t c[UNR];
#pragma unroll
      for (int j = 0; j < UNR; ++j)
        c[j] = b0 + j < nchunks ? chunk_hist[(int64_t)(b0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < UNR; ++j) {
        if (b0 + j < nchunks) chunk_hist[(int64_t)(b0 + j) * E + e] = total;  // exclusive base
        total += c[j];
      }
    }
    expert_count[e] = total;
  }
  int32_t pad = (e < E) ? (int32_t)((total + USAF_ROW_ALIGN - 1) / USAF_ROW_ALIGN * USAF_ROW_ALIGN)
                        : 0;
  // block exclusive scan of pad
  const int lane = e & 31, wid = e >> 5;
  int32_t v = pad;
  for (int o = 1; o < 32; o <<= 1) {
    int32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int32_t w = warp_sums[lane];
    for (int o = 1; o < 32; o <<= 1) {
      int32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  int32_t incl = v + (wid > 0 ? warp_sums[wid - 1] : 0);
  padded[e] = incl - pad;
  __syncthreads();
  if (e < E) expert_offset[e] = padded[e];
  if (e == E - 1) expert_offset[E] = incl;
}

// One warp per chunk: ranks within the chunk by __match_any_sync, in slot order.
__global__ void __launch_bounds__(32) perm_fill_kernel(const int32_t* __restrict__ topk_idx,
                                                       int64_t R, int E, int k,
                                                       const int32_t* __restrict__ chunk_base,
                                                       const int32_t* __restrict__ expert_offset,
                                                       int32_t* __restrict__ perm_tok,
                                                       int32_t* __restrict__ perm_slot,
                                                       int32_t* __restrict__ slot_row) {
  extern __shared__ int32_t cnt[];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32)
    cnt[e] = expert_offset[e] + chunk_base[(int64_t)blockIdx.x * E + e];
  __syncwarp();
  const int64_t s0 = (int64_t)blockIdx.x * PERM_CHUNK;
  const int64_t s1 = min(R, s0 + PERM_CHUNK);
  // the chunk's experts, all loaded before the ranking walk (unique dummies for idle lanes)
  constexpr int NPASS = PERM_CHUNK / 32;
  int ev[NPASS];
#pragma unroll
  for (int i = 0; i < NPASS; ++i) {
    const int64_t s = s0 + 32 * i + lane;
    ev[i] = s < s1 ? topk_idx[s] : -1 - lane;
  }
#pragma unroll
  for (int i = 0; i < NPASS; ++i) {
    const int64_t s = s0 + 32 * i + lane;
    const bool ok = s < s1;
    const int e = ev[i];
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1));
    const int pos = ok ? cnt[e] + rank : 0;
    __syncwarp();
    if (ok && rank == 0) cnt[e] += __popc(peers);
    __syncwarp();
    if (ok) {
      perm_tok[pos] = (int32_t)(s / k);
      perm_slot[pos] = (int32_t)s;
      slot_row[s] = pos;
    }
  }
}

// Padding rows of each segment and the tail up to R_cap: perm_tok = 0, perm_slot = -1.
__global__ void perm_pad_kernel(const int32_t* __restrict__ expert_count,
                                const int32_t* __restrict__ expert_offset, int E, int64_t R_cap,
                                int32_t* __restrict__ perm_tok, int32_t* __restrict__ perm_slot) {
  const int e = blockIdx.x;
  int64_t lo, hi;
  if (e < E) {
    lo = expert_offset[e] + expert_count[e];
    hi = expert_offset[e + 1];
  } else {
    lo = expert_offset[E];
    hi = R_cap;
  }
  for (int64_t r = lo + threadIdx.x; r < hi; r += blockDim.x) {
    perm_tok[r] = 0;
    perm_slot[r] = -1;
  }
}

usaf_status route_launch(const usaf_moe_shape& s, const void* x, usaf_dtype xdt,
                         const float* wr, const float* logits_in, float* logits_out, int renorm,
                         const usaf_routing& rt, RouteWs& w, uint32_t* dev_status,
                         cudaStream_t st) {
  const int Tn = (int)s.T, H = (int)s.H, E = (int)s.E, k = (int)s.k;
  const int64_t R = s.T * s.k;
  const float* logits = logits_in;
  if (!logits_in && xdt == USAF_BF16 && tc_shape_ok(s)) {
    // bf16 tokens: three bf16 tensor-core products of the split fp32 router weight
    float* out = logits_out ? logits_out : w.logits;
    USAF_TRY(tc_router_logits(s, x, wr, w.wr3, out, dev_status, st));
    logits = out;
  } else if (!logits_in) {
    USAF_TRACE("route_logits", st);
    float* out = logits_out ? logits_out : w.logits;
    dim3 grid((unsigned)ceil_div(E, 64), (unsigned)ceil_div(Tn, 64));
    if (xdt == USAF_BF16)
      router_logits_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
          static_cast<const __nv_bfloat16*>(x), wr, out, Tn, H, E);
    else
      router_logits_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x), wr, out,
                                                        Tn, H, E);
    USAF_CHECK_LAUNCH();
    logits = out;
  }
  {
    USAF_TRACE("route_topk", st);
    const int warps = 8;
    const dim3 grid((unsigned)ceil_div(Tn, warps));
    const int nl = (E + 31) / 32;  // logits per lane (E <= 1024)
    if (nl <= 1)
      topk_kernel<1><<<grid, warps * 32, 0, st>>>(logits, Tn, E, k, renorm, rt.topk_idx, rt.topk_w);
    else if (nl <= 2)
      topk_kernel<2><<<grid, warps * 32, 0, st>>>(logits, Tn, E, k, renorm, rt.topk_idx, rt.topk_w);
    else if (nl <= 4)
      topk_kernel<4><<<grid, warps * 32, 0, st>>>(logits, Tn, E, k, renorm, rt.topk_idx, rt.topk_w);
    else if (nl <= 8)
      topk_kernel<8><<<grid, warps * 32, 0, st>>>(logits, Tn, E, k, renorm, rt.topk_idx, rt.topk_w);
    else if (nl <= 16)
      topk_kernel<16><<<grid, warps * 32, 0, st>>>(logits, Tn, E, k, renorm, rt.topk_idx,
                                                    rt.topk_w);
    else
      topk_kernel<32><<<grid, warps * 32, 0, st>>>(logits, Tn, E, k, renorm, rt.topk_idx,
                                                    rt.topk_w);
    USAF_CHECK_LAUNCH();
  }
  USAF_TRACE("route_permute", st);
  const int nchunks = (int)ceil_div(R, PERM_CHUNK);
  perm_count_kernel<<<nchunks, 256, E * sizeof(int32_t), st>>>(rt.topk_idx, R, E, w.chunk_hist);
  USAF_CHECK_LAUNCH();
  perm_scan_kernel<<<1, 1024, 0, st>>>(w.chunk_hist, nchunks, E, rt.expert_count,
                                       rt.expert_offset);
  USAF_CHECK_LAUNCH();
  perm_fill_kernel<<<nchunks, 32, E * sizeof(int32_t), st>>>(
      rt.topk_idx, R, E, k, w.chunk_hist, rt.expert_offset, rt.perm_tok, rt.perm_slot,
      rt.slot_row);
  USAF_CHECK_LAUNCH();
  perm_pad_kernel<<<E + 1, 256, 0, st>>>(rt.expert_count, rt.expert_offset, E,
                                         usaf_routed_rows_capacity(&s), rt.perm_tok,
                                         rt.perm_slot);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

}  // namespace usaf
