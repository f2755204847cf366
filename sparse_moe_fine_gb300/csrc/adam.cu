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
__global__ void __launch_bounds__(256) adam_kernel(int64_t n, const int64_t* __restrict__ idx,
                                                   const float* __restrict__ g,
                                                   float* __restrict__ p, float* __restrict__ m,
                                                   float* __restrict__ v, W* __restrict__ w0,
                                                   int64_t n0, W* __restrict__ w1, float b1,
                                                   float b2, float om_b1, float om_b2, float eps,
                                                   float step_size, int skip,
                                                   const uint32_t* dev_status) {
  if (skip && dev_status && (*(volatile const uint32_t*)dev_status & USAF_DEV_NONFINITE)) return;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float gi = g[i];
    const float mi = fmaf(b1, m[i], om_b1 * gi);
    const float vi = fmaf(b2, v[i], om_b2 * gi * gi);
    const float pi = p[i] - step_size * (mi / (sqrtf(vi) + eps));
    m[i] = mi;
    v[i] = vi;
    p[i] = pi;
    const int64_t f = idx ? idx[i] : i;
    if (f < n0) w0[f] = from_f32<W>(pi);
    else w1[f - n0] = from_f32<W>(pi);
  }
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
  if (skip) {
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
    adam_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, st>>>(
        n, idx, g, p, m, v, static_cast<__nv_bfloat16*>(w0), n0,
        static_cast<__nv_bfloat16*>(w1), b1f, b2f, om_b1, om_b2, epsf, step_size, skip, dev_status);
  else
    adam_kernel<float><<<(unsigned)blocks, threads, 0, st>>>(
        n, idx, g, p, m, v, static_cast<float*>(w0), n0, static_cast<float*>(w1), b1f, b2f, om_b1,
        om_b2, epsf, step_size, skip, dev_status);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

}  // namespace usaf
