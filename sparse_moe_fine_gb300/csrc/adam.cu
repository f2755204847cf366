// Fused SparseAdam: gather the active entries' state, update, scatter the new weight.
//
// USAF README, A100 operations table: the optimizer is SparseAdam over the trained entries (the
// 0.5% expert subset plus the router), with Adam state kept only for them (news article, key
// differences). The update is torch.optim.SparseAdam's (eps added to the uncorrected sqrt(v),
// bias corrections folded into the step size). Steps with a non-finite gradient are skipped
// (README results table, "Steps skipped (NaN)").
#include "common.cuh"
#include "kernels.cuh"

namespace usaf {

__global__ void nonfinite_scan_kernel(const float* __restrict__ g, int64_t n,
                                      uint32_t* dev_status) {
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    bad |= !finite_f(g[i]);
  flag_status_warp(dev_status, bad, USAF_DEV_NONFINITE);
}

template <typename W>
__device__ __forceinline__ void adam_one(int64_t i, float gi, float& pi, float& mi, float& vi,
                                         const int64_t* __restrict__ idx, W* __restrict__ w0,
                                         int64_t n0, W* __restrict__ w1, float b1, float b2,
                                         float om_b1, float om_b2, float eps, float step_size) {
  mi = fmaf(b1, mi, om_b1 * gi);
  vi = fmaf(b2, vi, om_b2 * gi * gi);
  pi = pi - step_size * (mi / (sqrtf(vi) + eps));
  const int64_t f = idx ? idx[i] : i;
  if (f < n0) w0[f] = from_f32<W>(pi);
  else w1[f - n0] = from_f32<W>(pi);
}

// Four consecutive entries per thread with 16-byte loads and stores of g, p, m, v (all four
// arrays 16-byte aligned), the rest one by one.
template <typename W>
__global__ void __launch_bounds__(256) adam_kernel(int64_t n, const int64_t* __restrict__ idx,
                                                   const float* __restrict__ g,
                                                   float* __restrict__ p, float* __restrict__ m,
                                                   float* __restrict__ v, W* __restrict__ w0,
                                                   int64_t n0, W* __restrict__ w1, float b1,
                                                   float b2, float om_b1, float om_b2, float eps,
                                                   float step_size, int skip, int vec,
                                                   const uint32_t* dev_status) {
  if (dev_status) {
    const uint32_t st = *(volatile const uint32_t*)dev_status;
    if ((st & USAF_DEV_BAD_INDEX) || (skip && (st & USAF_DEV_SKIP_MASK))) return;
  }
  const int64_t n4 = vec ? n / 4 : 0;
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4;
       q += (int64_t)gridDim.x * blockDim.x) {
    const float4 g4 = reinterpret_cast<const float4*>(g)[q];
    float4 p4 = reinterpret_cast<const float4*>(p)[q];
    float4 m4 = reinterpret_cast<const float4*>(m)[q];
    float4 v4 = reinterpret_cast<const float4*>(v)[q];
    const int64_t i = 4 * q;
    adam_one(i, g4.x, p4.x, m4.x, v4.x, idx, w0, n0, w1, b1, b2, om_b1, om_b2, eps, step_size);
    adam_one(i + 1, g4.y, p4.y, m4.y, v4.y, idx, w0, n0, w1, b1, b2, om_b1, om_b2, eps, step_size);
    adam_one(i + 2, g4.z, p4.z, m4.z, v4.z, idx, w0, n0, w1, b1, b2, om_b1, om_b2, eps, step_size);
    adam_one(i + 3, g4.w, p4.w, m4.w, v4.w, idx, w0, n0, w1, b1, b2, om_b1, om_b2, eps, step_size);
    reinterpret_cast<float4*>(p)[q] = p4;
    reinterpret_cast<float4*>(m)[q] = m4;
    reinterpret_cast<float4*>(v)[q] = v4;
  }
  for (int64_t i = 4 * n4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float pi = p[i], mi = m[i], vi = v[i];
    adam_one(i, g[i], pi, mi, vi, idx, w0, n0, w1, b1, b2, om_b1, om_b2, eps, step_size);
    p[i] = pi;
    m[i] = mi;
    v[i] = vi;
  }
}

// Active-set contract: 0 <= idx[i] < N and idx[i - 1] < idx[i]. Reads idx only.
__global__ void validate_active_kernel(const int64_t* __restrict__ idx, int64_t K, int64_t N,
                                       uint32_t* dev_status) {
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < K;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t f = idx[i];
    bad |= f < 0 || f >= N || (i > 0 && idx[i - 1] >= f);
  }
  flag_status_warp(dev_status, bad, USAF_DEV_BAD_INDEX);
}

usaf_status validate_launch(const int64_t* idx, int64_t K, int64_t N, uint32_t* dev_status,
                            cudaStream_t st) {
  if (K == 0) return USAF_OK;
  USAF_TRACE("validate_active", st);
  validate_active_kernel<<<grid_dim_for(K), 256, 0, st>>>(idx, K, N, dev_status);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

usaf_status nonfinite_scan_launch(const float* g, int64_t n, uint32_t* dev_status,
                                  cudaStream_t st) {
  if (n == 0) return USAF_OK;
  USAF_TRACE("nonfinite_scan", st);
  const int64_t blocks = std::min<int64_t>(ceil_div(n, 256), device_sm_count() * 8);
  nonfinite_scan_kernel<<<(unsigned)blocks, 256, 0, st>>>(g, n, dev_status);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

usaf_status adam_launch(int64_t n, const int64_t* idx, const float* g, float* p, float* m,
                        float* v, void* w0, int64_t n0, void* w1, usaf_dtype wdt, double lr,
                        double b1, double b2, double eps, int64_t step, int skip,
                        uint32_t* dev_status, cudaStream_t st) {
  if (n == 0) return USAF_OK;
  USAF_TRACE("sparse_adam", st);
  const int threads = 256;
  int64_t blocks = ceil_div(n, threads);
  const int cap = device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  const auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  const int vec = al(g) && al(p) && al(m) && al(v) ? 1 : 0;
  const int64_t ublocks = std::max<int64_t>(1, ceil_div(vec ? ceil_div(n, 4) : n, threads));
  if (skip == 1) {  // 2: the caller scanned (usaf_scan_nonfinite); only the status is checked
    nonfinite_scan_kernel<<<(unsigned)blocks, threads, 0, st>>>(g, n, dev_status);
    USAF_CHECK_LAUNCH();
  }
  // bias corrections in double on the host, as one fp32 step size
  const double bc1 = 1.0 - std::pow(b1, (double)step);
  const double bc2 = 1.0 - std::pow(b2, (double)step);
  const float step_size = (float)(lr * std::sqrt(bc2) / bc1);
  const float om_b1 = (float)(1.0 - b1), om_b2 = (float)(1.0 - b2);
  const float b1f = (float)b1, b2f = (float)b2, epsf = (float)eps;
  if (wdt == USAF_BF16)
    adam_kernel<__nv_bfloat16><<<(unsigned)ublocks, threads, 0, st>>>(
        n, idx, g, p, m, v, static_cast<__nv_bfloat16*>(w0), n0,
        static_cast<__nv_bfloat16*>(w1), b1f, b2f, om_b1, om_b2, epsf, step_size, skip, vec,
        dev_status);
  else
    adam_kernel<float><<<(unsigned)ublocks, threads, 0, st>>>(
        n, idx, g, p, m, v, static_cast<float*>(w0), n0, static_cast<float*>(w1), b1f, b2f, om_b1,
        om_b2, epsf, step_size, skip, vec, dev_status);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

}  // namespace usaf
