// Exact top-K selection by magnitude (the importance phase) and RigL drop/grow.
//
// USAF README: "Not all weights matter" (the importance phase keeps the 0.5% of weights with the
// highest gradient magnitude) and "Sparsity adapts" (every 50 steps RigL swaps active weights that
// contribute little for inactive ones with large gradients). Order: key descending, flat index
// ascending among equal keys; the key of |g| is its fp32 bit pattern with the sign cleared.
//
// Fast path, one read of g: 131,072 strided samples give a candidate threshold tau0 a safe margin
// below the K-th largest key; one coalesced pass compacts every (key, index) with key >= tau0 into
// per-warp regions in index order and counts the candidates' first radix digit; the remaining
// digit rounds and the ordered count, scan and write then run on the candidates only (one warp per
// region). If a region overflows or fewer than K candidates exist, the same kernels run on the
// full array instead (exact multi-pass path); the choice is taken on the device, so the launch
// sequence is fixed and needs no host synchronisation. RigL's grow selection is the same with an
// exclusion bitmap of the active set; the selection and the swap of one importance pass can share
// one pass over g (usaf_select_and_swap).
#include "common.cuh"
#include "kernels.cuh"

namespace usaf {

namespace {

constexpr int SEL_THREADS = 256;
constexpr int COMPACT_WARPS = 8;  // warps per block of the compacting pass, one region each
constexpr int ROUND_THREADS = 256;  // radix rounds: eight blocks per SM, parts taken in turn
constexpr int SAMPLE_S = 131072;  // strided samples of the keys for the threshold
constexpr int TAU_BLOCKS = 32;    // blocks of the threshold's second digit round
// radix rounds over the 31-bit key, most significant digit first: bits 30..23, 22..15, 14..7, 6..0
__host__ __device__ constexpr int round_shift(int r) { return r == 0 ? 23 : r == 1 ? 15 : r == 2 ? 7 : 0; }
__host__ __device__ constexpr int round_bits(int r) { return r == 3 ? 7 : 8; }
// the selection's own radix rounds: 8 bits (the exponent), 8, 8 and 7 bits (256-bin histograms,
// so each block adds at most 256 bins into the global one)
constexpr int SEL_ROUNDS = 4;
constexpr int MAX_BINS = 256;
__host__ __device__ constexpr int sel_shift(int r) {
  return r == 0 ? 23 : r == 1 ? 15 : r == 2 ? 7 : 0;
}
__host__ __device__ constexpr int sel_bits(int r) { return r == 3 ? 7 : 8; }

struct SelCtrl {
  uint32_t tau0;
  uint32_t mode;  // 0 full array, 1 candidate regions, 2 drop keys from |p|
  uint32_t overflow;
  uint32_t ticket;
  unsigned long long total;
  uint32_t prefix;  // radix state: the K-th key's bits found so far
  uint32_t k_rem;   // rank still to find among keys matching prefix
  uint32_t hist[MAX_BINS];
  unsigned long long n_swapped;
  uint32_t r0_done;  // the first radix digit was taken from the compacting pass's histogram
};

// Where block b's part of the source lives.
struct Src {
  const float* g;          // modes 0, 2
  const uint32_t* excl;    // mode 0: bitmap of excluded indices, or null
  int64_t n;               // modes 0, 2: element count
  int64_t L;               // modes 0, 2: elements per block (multiple of 4)
  const uint32_t* ckeys;   // mode 1
  const uint32_t* cids;
  const uint32_t* ccnt;
  int64_t cap;
  int drop;                // 1: keys are complemented |p| (mode 2 source)
  int skip_tagged;         // mode 1: candidates whose key carries bit 31 (an excluded entry of a
                           // shared candidate set) are not part of this selection
  int G;                   // parts (regions)
  int64_t base;            // modes 0, 2: added to the element index an ordered write emits
};

struct SelPlan {
  int G;            // blocks (= regions)
  int64_t L;        // elements per block on the full array
  int64_t cap;      // region capacity
  int q;            // sample rank for tau0 (0: no sampling)
  bool sampling;
};

struct SelWs {
  SelCtrl* ctrl;
  uint32_t* ckeys;
  uint32_t* cids;
  uint32_t* ccnt;
  uint32_t* blk_gt;
  uint32_t* blk_eq;
  uint32_t* base_gt;
  uint32_t* base_eq;
  uint32_t* samples;  // [SAMPLE_S] sampled keys (sampled path)
  uint32_t* bhist;    // [SAMPLE_BLOCKS][256] first-digit histograms of the samples, per block
  uint32_t* bhist2;   // [TAU_BLOCKS][256] second-digit histograms of the threshold, per block
};

SelPlan make_plan(int64_t N, int64_t K) {
  SelPlan p{};
  const int64_t sms = device_sm_count();
  p.sampling = N >= (int64_t)4 * 1024 * 1024 && K * 16 <= N;
  if (p.sampling) {
    const double q = std::ceil((double)SAMPLE_S * (double)K / (double)N);
    const double qq = q + 5.0 * std::sqrt(q) + 16.0;  // 5 sigma above the expected rank
    p.q = (int)std::min<double>(qq, SAMPLE_S);
    if (p.q >= SAMPLE_S / 8) p.sampling = false;
  }
  if (p.sampling) {
    // one candidate region per warp of the compacting pass (COMPACT_WARPS per block), at least
    // 4096 entries each, up to 32 per SM: a part of a few tens of millions of entries still fills
    // every SM with warps
    int64_t G = std::min<int64_t>(ceil_div(N, 4096), sms * 32);
    G = round_up(G < 1 ? 1 : G, COMPACT_WARPS);
    p.G = (int)G;
    p.L = round_up(ceil_div(N, G), 1024);
    const double mean = (double)p.L * (double)p.q / SAMPLE_S;
    p.cap = round_up((int64_t)(mean * 1.5 + 8.0 * std::sqrt(mean)) + 256, 256);
  } else {
    // exact path: regions of at least 4096 entries, up to eight blocks per SM (a selection over
    // the K values of |p| still fills the GPU)
    int64_t G = ceil_div(N, 4096);
    if (G > sms * 8) G = sms * 8;
    if (G < 1) G = 1;
    p.G = (int)G;
    p.L = round_up(ceil_div(N, G), 1024);
    p.q = 0;
    p.cap = 0;
  }
  return p;
}

void sel_layout(const SelPlan& p, Carver& c, SelWs& w) {
  w.ctrl = c.take<SelCtrl>(1);
  w.ckeys = c.take<uint32_t>(p.G * p.cap);
  w.cids = c.take<uint32_t>(p.G * p.cap);
  w.ccnt = c.take<uint32_t>(p.G);
  w.blk_gt = c.take<uint32_t>(p.G);
  w.blk_eq = c.take<uint32_t>(p.G);
  w.base_gt = c.take<uint32_t>(p.G);
  w.base_eq = c.take<uint32_t>(p.G);
  w.samples = p.sampling ? c.take<uint32_t>(SAMPLE_S) : nullptr;
  w.bhist = p.sampling ? c.take<uint32_t>(SAMPLE_S / 1024 * 256) : nullptr;
  w.bhist2 = p.sampling ? c.take<uint32_t>(TAU_BLOCKS * 256) : nullptr;
}

// ------------------------------------------------------------------------------------------------
// block-level helpers
// ------------------------------------------------------------------------------------------------
// Exclusive scan of one value per thread over the block; returns the prefix, *total the sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* total) {
  __shared__ uint32_t wsum[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint32_t x = v;
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) wsum[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = lane < nw ? wsum[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    wsum[lane] = s;
  }
  __syncthreads();
  const uint32_t before = (wid > 0 ? wsum[wid - 1] : 0) + x - v;
  *total = wsum[nw - 1];
  __syncthreads();
  return before;
}

__device__ __forceinline__ bool excluded(const uint32_t* excl, int64_t i) {
  return excl && ((excl[i >> 5] >> (i & 31)) & 1u);
}

// key of element i of a modes-0/2 source
__device__ __forceinline__ uint32_t src_key(const Src& s, int64_t i) {
  const uint32_t k = abs_key(s.g[i]);
  return s.drop ? (~k & 0x7FFFFFFFu) : k;
}

// Visit block b's part in index order, blockDim elements per step: f(key, id, valid).
template <class F>
__device__ __forceinline__ void for_part(const Src& s, int mode, int b, F f) {
  if (mode == 1) {
    const int64_t n = s.ccnt[b];
    const uint32_t* kk = s.ckeys + (int64_t)b * s.cap;
    const uint32_t* ii = s.cids + (int64_t)b * s.cap;
    for (int64_t j0 = 0; j0 < n; j0 += blockDim.x) {
      const int64_t j = j0 + threadIdx.x;
      const uint32_t kj = j < n ? kk[j] : 0u;
      const bool ok = j < n && !(s.skip_tagged && (kj >> 31));
      f(kj & 0x7FFFFFFFu, ok ? s.base + (int64_t)ii[j] : 0, ok);
    }
  } else {
    const int64_t lo = (int64_t)b * s.L;
    const int64_t hi = min(s.n, lo + s.L);
    for (int64_t i0 = lo; i0 < hi; i0 += blockDim.x) {
      const int64_t i = i0 + threadIdx.x;
      const bool ok = i < hi && !(mode == 0 && excluded(s.excl, i));
      f(ok ? src_key(s, i) : 0u, s.base + i, ok);
    }
  }
}

// ------------------------------------------------------------------------------------------------
// kernels
// ------------------------------------------------------------------------------------------------
// Clear a control block for a selection of K, by one block.
__device__ __forceinline__ void ctrl_init_block(SelCtrl* c, int64_t K) {
  for (int i = threadIdx.x; i < MAX_BINS; i += blockDim.x) c->hist[i] = 0;
  if (threadIdx.x == 0) {
    c->tau0 = 0;
    c->mode = 0;
    c->overflow = 0;
    c->ticket = 0;
    c->total = 0;
    c->prefix = 0;
    c->k_rem = (uint32_t)K;
    c->n_swapped = 0;
    c->r0_done = 0;
  }
}

__global__ void sel_init_kernel(SelCtrl* c, int64_t K, uint32_t* ccnt, int G) {
  ctrl_init_block(c, K);
  for (int i = threadIdx.x; i < G; i += blockDim.x) ccnt[i] = 0;
}

// The digit of one radix round from a 256-bin histogram (digits above dmask empty), by warp 0:
// the largest d whose bins above d hold fewer than *krem keys and whose bins from d up hold at
// least *krem; *krem becomes the rank still to find among the keys with digit d. Lane l owns
// bins 255 - 8l .. 248 - 8l; a warp scan gives each lane the keys above its bins.
__device__ __forceinline__ void pick_digit_warp(const uint32_t* hist, uint32_t* krem_io,
                                                uint32_t* prefix_io, int shift) {
  const int lane = threadIdx.x & 31;
  const uint32_t krem = *krem_io;
  uint32_t bins[8], mine = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    bins[j] = hist[255 - 8 * lane - j];
    mine += bins[j];
  }
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t above = incl - mine;
  const unsigned hit = __ballot_sync(0xffffffffu, above < krem && krem <= incl);
  int d = 0;
  uint32_t cum = 0;
  if (hit) {
    const int src = __ffs(hit) - 1;
    if (lane == src) {
      cum = above;
      d = 255 - 8 * lane - 7;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (cum + bins[j] >= krem) {
          d = 255 - 8 * lane - j;
          break;
        }
        cum += bins[j];
      }
    }
    d = __shfl_sync(0xffffffffu, d, src);
    cum = __shfl_sync(0xffffffffu, cum, src);
  } else {
    // krem above the total (cannot happen for a rank inside the sample): digit 0
    cum = __shfl_sync(0xffffffffu, incl, 31) - hist[0];
  }
  if (lane == 0) {
    *krem_io = krem - cum;
    *prefix_io |= (uint32_t)d << shift;
  }
}

// The SAMPLE_S strided samples of the keys (0 where excluded), 1024 per block so that the random
// reads of g spread over SAMPLE_BLOCKS SMs; each block also writes the histogram of its samples'
// first digit (bits 30..23). With samples_all (two selections sharing one pass), the same
// positions' keys and their histogram are also written without the exclusion. Block 0 also
// clears the control blocks (c for the samples, c_all for samples_all) and the region counts.
constexpr int SAMPLE_BLOCKS = SAMPLE_S / 1024;
__global__ void __launch_bounds__(1024) sel_sample_kernel(
    const float* __restrict__ g, int64_t N, const uint32_t* __restrict__ excl,
    uint32_t* __restrict__ samples, uint32_t* __restrict__ bhist,
    uint32_t* __restrict__ samples_all, uint32_t* __restrict__ bhist_all, SelCtrl* c, int64_t K,
    SelCtrl* c_all, int64_t K_all, uint32_t* ccnt, int G) {
  __shared__ uint32_t h[256], ha[256];
  if (threadIdx.x < 256) {
    h[threadIdx.x] = 0;
    ha[threadIdx.x] = 0;
  }
  if (blockIdx.x == 0) {
    ctrl_init_block(c, K);
    if (c_all) ctrl_init_block(c_all, K_all);
    for (int i = threadIdx.x; i < G; i += blockDim.x) ccnt[i] = 0;
  }
  __syncthreads();
  const int i = blockIdx.x * 1024 + threadIdx.x;
  const int64_t pos = (int64_t)(((unsigned long long)i * (unsigned long long)N) / SAMPLE_S);
  const uint32_t k = abs_key(g[pos]);
  const uint32_t ks = excluded(excl, pos) ? 0u : k;
  samples[i] = ks;
  atomicAdd(&h[ks >> sel_shift(0)], 1u);
  if (samples_all) {
    samples_all[i] = k;
    atomicAdd(&ha[k >> sel_shift(0)], 1u);
  }
  __syncthreads();
  if (threadIdx.x < 256) {
    bhist[blockIdx.x * 256 + threadIdx.x] = h[threadIdx.x];
    if (samples_all) bhist_all[blockIdx.x * 256 + threadIdx.x] = ha[threadIdx.x];
  }
}

// One selection's threshold job: its samples, their per-block histograms, the second round's
// per-block histograms, the sample rank and the control block.
struct TauJob {
  const uint32_t* samples;
  const uint32_t* bhist;
  uint32_t* bhist2;
  int q;
  SelCtrl* c;
};

// The threshold of the sampled path: the top 16 bits of the q-th largest sample (1-based), found
// in two digit rounds by TAU_BLOCKS blocks of 1024 threads per selection (blocks [TAU_BLOCKS j,
// TAU_BLOCKS (j + 1)) take job j). Every block sums the sample blocks' first-digit histograms
// (four threads per bin, 32 histograms each) and picks the first digit; each then counts the
// second digit of the samples of its own slice that carry the first, and the last block to finish
// sums those counts and picks the second. tau0 := the two digits (the lower edge of the sample
// quantile's bin).
constexpr int TAU_THREADS = 1024;
__global__ void __launch_bounds__(TAU_THREADS) sel_sample_tau_kernel(TauJob j0, TauJob j1) {
  constexpr int PARTS = TAU_THREADS / 256;
  __shared__ uint32_t part[PARTS][256];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_krem;
  __shared__ bool last;
  const bool second = blockIdx.x >= TAU_BLOCKS;
  const TauJob& jb = second ? j1 : j0;
  const int bid = (int)blockIdx.x - (second ? TAU_BLOCKS : 0);
  SelCtrl* c = jb.c;
  const int wid = threadIdx.x >> 5, bin = threadIdx.x & 255, pr = threadIdx.x >> 8;
  {
    constexpr int PER_PART = SAMPLE_BLOCKS / PARTS;
    uint32_t t = 0;
#pragma unroll
    for (int b = 0; b < PER_PART; ++b) t += __ldg(jb.bhist + (pr * PER_PART + b) * 256 + bin);
    part[pr][bin] = t;
  }
  if (threadIdx.x == 0) {
    s_prefix = 0;
    s_krem = (uint32_t)jb.q;
  }
  __syncthreads();
  if (threadIdx.x < 256) {
    uint32_t t = 0;
#pragma unroll
    for (int r = 0; r < PARTS; ++r) t += part[r][threadIdx.x];
    hist[threadIdx.x] = t;
  }
  __syncthreads();
  if (wid == 0) pick_digit_warp(hist, &s_krem, &s_prefix, round_shift(0));
  __syncthreads();
  const uint32_t d0 = s_prefix >> round_shift(0);
  if (threadIdx.x < 256) hist[threadIdx.x] = 0;
  __syncthreads();
  constexpr int PER = SAMPLE_S / TAU_BLOCKS / TAU_THREADS;
  uint32_t key[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j)
    key[j] = __ldg(jb.samples + (bid * PER + j) * TAU_THREADS + threadIdx.x);
#pragma unroll
  for (int j = 0; j < PER; ++j)
    if ((key[j] >> round_shift(0)) == d0) atomicAdd(&hist[(key[j] >> round_shift(1)) & 255u], 1u);
  __syncthreads();
  if (threadIdx.x < 256) jb.bhist2[bid * 256 + threadIdx.x] = hist[threadIdx.x];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&c->ticket, 1u) == TAU_BLOCKS - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x < 256) {
    uint32_t t = 0;
#pragma unroll
    for (int b = 0; b < TAU_BLOCKS; ++b) t += __ldcg(jb.bhist2 + b * 256 + threadIdx.x);
    hist[threadIdx.x] = t;
  }
  __syncthreads();
  if (wid == 0) pick_digit_warp(hist, &s_krem, &s_prefix, round_shift(1));
  __syncthreads();
  if (threadIdx.x == 0) {
    c->tau0 = s_prefix;
    c->ticket = 0;
  }
}

// The one pass over g: every warp compacts the (key, index) pairs with key >= tau0 (and not
// excluded) of its own contiguous part of g into its own region, in index order. A step is 512
// elements, taken as 16 rows of 32: lane l holds element 32 r + l of row r, so one ballot per row
// gives each lane with a candidate its place (the candidates of lower lanes of the row) and the
// region stays in index order without a scan. The next step's loads are issued before the current
// one is examined; a row is examined only when some lane of its 128-element group holds a key at
// or above tau0 (the groups of the sampled path mostly hold none or one).
// The exclusion bitmap (EX != EX_NONE) streams beside g: the 16 words of a step (parts start on
// multiples of 1024) are loaded one step ahead by lanes 0-15, and row r's word, whose bit l is
// lane l's element, is shuffled out only for rows with a candidate.
// EX_TAG (two selections from one pass, `c` without and `cg` with the exclusion): the threshold
// is the lower of the two tau0 and excluded entries stay candidates with bit 31 of their stored
// key set; the first-digit histogram and count of the excluded ones are kept apart, and `cg`
// receives the differences (the non-excluded candidates').
enum { EX_NONE = 0, EX_SKIP = 1, EX_TAG = 2 };

// max of a and b, NaN when either is NaN (max.NaN)
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
template <int EX>
__global__ void __launch_bounds__(COMPACT_WARPS * 32) sel_compact_kernel(
    const float* __restrict__ g, int64_t N, int64_t L, const uint32_t* __restrict__ excl,
    int64_t cap, uint32_t* __restrict__ ckeys, uint32_t* __restrict__ cids,
    uint32_t* __restrict__ ccnt, SelCtrl* c, SelCtrl* cg, uint32_t* dev_status) {
  constexpr bool TAG = EX == EX_TAG;
  constexpr int UN = 4;  // groups of 4 rows per step
  constexpr int STEP = 128 * UN;
  __shared__ uint32_t dhist[256];  // first radix digit (bits 30..23) of this block's candidates
  __shared__ uint32_t dhist_x[TAG ? 256 : 1];  // the same over the excluded ones
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    dhist[i] = 0;
    if (TAG) dhist_x[i] = 0;
  }
  __syncthreads();
  const uint32_t tau0 = TAG ? min(c->tau0, cg->tau0) : c->tau0;
  // a group is examined when some |x| >= tau0 as floats, or is NaN: a superset of the groups
  // holding a key >= tau0 (a threshold in the NaN range tests against +inf; the exact integer key
  // test follows). Every non-finite element's group is examined, so the flag is set there.
  const float tau_f = __uint_as_float(min(tau0, 0x7F800000u));
  const int lane = threadIdx.x & 31;
  const uint32_t below = (1u << lane) - 1u;
  const int64_t r = (int64_t)blockIdx.x * COMPACT_WARPS + (threadIdx.x >> 5);
  const int64_t lo = r * L;
  const int64_t hi = min(N, lo + L);
  uint32_t* rk = ckeys + r * cap;
  uint32_t* ri = cids + r * cap;
  uint32_t count = 0, count_x = 0, kmax = 0;  // kmax: largest key of the examined groups
  bool over = false;
  // lane l < 16: the bitmap word of elements [t + 32 l, t + 32 l + 32) (words past hi are not read)
  auto load_bw = [&](int64_t t) -> uint32_t {
    return EX != EX_NONE && lane < 16 && t + lane * 32 < hi ? __ldg(excl + (t >> 5) + lane) : 0u;
  };
  // the 16 rows of the step at t (zeros past hi)
  auto load_step = [&](int64_t t, float (&v)[UN][4]) {
    if (t + STEP <= hi) {
#pragma unroll
      for (int u = 0; u < UN; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j) v[u][j] = __ldg(g + t + u * 128 + j * 32 + lane);
    } else {
#pragma unroll
      for (int u = 0; u < UN; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t i = t + u * 128 + j * 32 + lane;
          v[u][j] = i < hi ? __ldg(g + i) : 0.f;
        }
    }
  };
  float nxt[UN][4];
  load_step(lo, nxt);
  uint32_t bw_nxt = load_bw(lo);
  for (int64_t t0 = lo; t0 < hi; t0 += STEP) {
    float cur[UN][4];
#pragma unroll
    for (int u = 0; u < UN; ++u)
#pragma unroll
      for (int j = 0; j < 4; ++j) cur[u][j] = nxt[u][j];
    const uint32_t bw = bw_nxt;
    if (t0 + STEP < hi) {
      load_step(t0 + STEP, nxt);
      bw_nxt = load_bw(t0 + STEP);
    }
    const bool full = t0 + STEP <= hi;  // no range tests
#pragma unroll
    for (int u = 0; u < UN; ++u) {
      const float f4 = max_nan(max_nan(fabsf(cur[u][0]), fabsf(cur[u][1])),
                               max_nan(fabsf(cur[u][2]), fabsf(cur[u][3])));
      if (!__any_sync(0xffffffffu, !(f4 < tau_f))) continue;  // elements past hi read as 0
      const uint32_t key[4] = {abs_key(cur[u][0]), abs_key(cur[u][1]), abs_key(cur[u][2]),
                               abs_key(cur[u][3])};
      kmax = max(kmax, max(max(key[0], key[1]), max(key[2], key[3])));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t i = t0 + u * 128 + j * 32 + lane;
        uint32_t b = __ballot_sync(0xffffffffu, key[j] >= tau0 && (full || i < hi));
        if (!b) continue;
        uint32_t word = 0;  // bit l: lane l's element is excluded
        if (EX != EX_NONE) word = __shfl_sync(0xffffffffu, bw, u * 4 + j);
        if (EX == EX_SKIP) {
          b &= ~word;
          if (!b) continue;
        }
        if ((b >> lane) & 1u) {
          const uint32_t pos = count + __popc(b & below);
          const bool ex = TAG && ((word >> lane) & 1u);
          if (pos < cap) {
            rk[pos] = key[j] | (ex ? 0x80000000u : 0u);
            ri[pos] = (uint32_t)i;
          } else {
            over = true;
          }
          atomicAdd(&dhist[key[j] >> sel_shift(0)], 1u);
          if (ex) atomicAdd(&dhist_x[key[j] >> sel_shift(0)], 1u);
        }
        count += __popc(b);
        if (TAG) count_x += __popc(b & word);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    if (dhist[i]) atomicAdd(&c->hist[i], dhist[i]);
    if (TAG && dhist[i] - dhist_x[i]) atomicAdd(&cg->hist[i], dhist[i] - dhist_x[i]);
  }
  if (lane == 0 && lo < N) {
    ccnt[r] = count < cap ? count : (uint32_t)cap;
    atomicAdd(&c->total, (unsigned long long)count);
    if (TAG) atomicAdd(&cg->total, (unsigned long long)(count - count_x));
  }
  if (over) c->overflow = 1;
  if (TAG && over) cg->overflow = 1;
  flag_status_warp(dev_status, kmax >= 0x7F800000u, USAF_DEV_NONFINITE);
}

// One block of 256 threads: the candidate path or the exact path, and on the candidate path the
// first radix digit from the histogram the compacting pass built (so the first round is skipped).
__device__ __forceinline__ void decide_body(SelCtrl* c, int64_t K, int sampling,
                                            uint32_t* dev_status) {
  __shared__ uint32_t h[256];
  __shared__ bool ok;
  if (threadIdx.x == 0) {
    ok = sampling && !c->overflow && c->total >= (unsigned long long)K;
    c->mode = ok ? 1u : 0u;
    if (sampling && !ok) flag_status(dev_status, USAF_DEV_SELECT_EXACT_PATH);
  }
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    h[i] = reinterpret_cast<volatile uint32_t*>(c->hist)[i];
    c->hist[i] = 0;
  }
  __syncthreads();
  if (ok && threadIdx.x < 32) {
    __shared__ uint32_t s_krem, s_prefix;
    if (threadIdx.x == 0) {
      s_krem = c->k_rem;
      s_prefix = 0;
    }
    __syncwarp();
    pick_digit_warp(h, &s_krem, &s_prefix, sel_shift(0));
    __syncwarp();
    if (threadIdx.x == 0) {
      c->k_rem = s_krem;
      c->prefix = s_prefix;
      c->r0_done = 1;
    }
  }
}

__global__ void sel_decide_kernel(SelCtrl* c, int64_t K, int sampling, uint32_t* dev_status) {
  decide_body(c, K, sampling, dev_status);
}

// Two selections over one candidate set: block b decides selection b.
__global__ void sel_decide2_kernel(SelCtrl* c0, int64_t K0, SelCtrl* c1, int64_t K1,
                                   uint32_t* dev_status) {
  if (blockIdx.x == 0)
    decide_body(c0, K0, 1, dev_status);
  else
    decide_body(c1, K1, 1, dev_status);
}

// One radix round over the source (digits of up to 12 bits). Each block counts the digits of the
// keys that match the prefix found so far into a shared histogram and adds it to the global one;
// the last block to finish picks the digit with a block-wide scan from the top. The first round's
// digits (the exponent) fall in few bins, so a warp adds equal digits once; later rounds' digits
// are spread out and each key adds its own.
__device__ __forceinline__ void round_body(const Src& s, SelCtrl* c, int shift, int bits,
                                           int fixed_mode, int bid, int nblk) {
  __shared__ uint32_t hist[MAX_BINS];
  __shared__ bool last;
  __shared__ int pick;
  if (shift == sel_shift(0) && c->r0_done) return;  // taken during the compacting pass
  const int mode = fixed_mode >= 0 ? fixed_mode : (int)c->mode;
  const int nb = 1 << bits;
  const uint32_t dmask = (uint32_t)nb - 1;
  const int hs = shift + bits;
  const uint32_t prefix = c->prefix;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const bool first = shift == sel_shift(0);  // exponent digits: few bins, aggregate per warp
  for (int b = bid; b < s.G; b += nblk)
  for_part(s, mode, b, [&](uint32_t key, int64_t, bool ok) {
    const bool m = ok && (hs >= 32 || (key >> hs) == (prefix >> hs));
    const int d = (int)((key >> shift) & dmask);
    if (first) {
      const unsigned peers = __match_any_sync(0xffffffffu, m ? d : -1 - (int)(threadIdx.x & 31));
      if (m && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
    } else if (m) {
      atomicAdd(&hist[d], 1u);
    }
  });
  __syncthreads();
  for (int i = threadIdx.x; i < nb; i += blockDim.x)
    if (hist[i]) atomicAdd(&c->hist[i], hist[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&c->ticket, 1u) == (uint32_t)nblk - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    hist[i] = reinterpret_cast<volatile uint32_t*>(c->hist)[i];
    c->hist[i] = 0;
  }
  if (threadIdx.x == 0) pick = 0;
  __syncthreads();
  // thread t owns the per = nb / blockDim bins just below the (t)-th slice from the top
  const int per = (nb + blockDim.x - 1) / blockDim.x;
  const int hi = nb - 1 - threadIdx.x * per;  // highest digit of this thread's slice
  uint32_t mine = 0;
  for (int j = 0; j < per && hi - j >= 0; ++j) mine += hist[hi - j];
  uint32_t tot;
  const uint32_t above = block_excl_scan(mine, &tot);  // keys in the slices above this one
  const uint32_t krem = c->k_rem;
  if (above < krem && krem <= above + mine) {
    uint32_t cum = above;
    int d = hi;
    for (int j = 0; j < per && hi - j >= 0; ++j) {
      d = hi - j;
      if (cum + hist[d] >= krem) break;
      cum += hist[d];
    }
    pick = d;
    c->k_rem = krem - cum;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    c->prefix = prefix | ((uint32_t)pick << shift);
    c->ticket = 0;
  }
}

__global__ void __launch_bounds__(ROUND_THREADS) sel_round_kernel(Src s, SelCtrl* c, int shift,
                                                                int bits, int fixed_mode) {
  round_body(s, c, shift, bits, fixed_mode, blockIdx.x, gridDim.x);
}

// One round of two selections over one candidate set: the first half of the blocks runs
// selection 0, the second half selection 1.
__global__ void __launch_bounds__(ROUND_THREADS) sel_round2_kernel(Src s0, SelCtrl* c0, Src s1,
                                                                 SelCtrl* c1, int shift,
                                                                 int bits) {
  const int half = (int)gridDim.x / 2;
  if ((int)blockIdx.x < half)
    round_body(s0, c0, shift, bits, -1, blockIdx.x, half);
  else
    round_body(s1, c1, shift, bits, -1, blockIdx.x - half, gridDim.x - half);

}

// Per block: elements strictly above tau and equal to tau.
__global__ void __launch_bounds__(SEL_THREADS) sel_count_kernel(Src s, const SelCtrl* c,
                                                                uint32_t* blk_gt, uint32_t* blk_eq,
                                                                int fixed_mode) {
  const int mode = fixed_mode >= 0 ? fixed_mode : (int)c->mode;
  const uint32_t tau = c->prefix;
  uint32_t gt = 0, eq = 0;
  for_part(s, mode, blockIdx.x, [&](uint32_t key, int64_t, bool ok) {
    gt += ok && key > tau;
    eq += ok && key == tau;
  });
  uint32_t tg, te;
  block_excl_scan(gt, &tg);
  block_excl_scan(eq, &te);
  if (threadIdx.x == 0) {
    blk_gt[blockIdx.x] = tg;
    blk_eq[blockIdx.x] = te;
  }
}

__device__ __forceinline__ void scan_body(const uint32_t* blk_gt, const uint32_t* blk_eq, int G,
                                          uint32_t* base_gt, uint32_t* base_eq) {
  uint32_t run_gt = 0, run_eq = 0;
  for (int c0 = 0; c0 < G; c0 += blockDim.x) {
    const int i = c0 + threadIdx.x;
    const uint32_t a = i < G ? blk_gt[i] : 0, b = i < G ? blk_eq[i] : 0;
    uint32_t ta, tb;
    const uint32_t pa = block_excl_scan(a, &ta);
    const uint32_t pb = block_excl_scan(b, &tb);
    if (i < G) {
      base_gt[i] = run_gt + pa;
      base_eq[i] = run_eq + pb;
    }
    run_gt += ta;
    run_eq += tb;
  }
}

__global__ void __launch_bounds__(1024) sel_scan_kernel(const uint32_t* blk_gt,
                                                        const uint32_t* blk_eq, int G,
                                                        uint32_t* base_gt, uint32_t* base_eq) {
  scan_body(blk_gt, blk_eq, G, base_gt, base_eq);
}

// Ordered write: selected = key > tau, or key == tau among the first need_eq such (by index).
__global__ void __launch_bounds__(SEL_THREADS) sel_write_kernel(Src s, const SelCtrl* c,
                                                                const uint32_t* base_gt,
                                                                const uint32_t* base_eq,
                                                                int64_t* __restrict__ out,
                                                                int fixed_mode) {
  const int mode = fixed_mode >= 0 ? fixed_mode : (int)c->mode;
  const uint32_t tau = c->prefix;
  const uint32_t need = c->k_rem;
  uint32_t gt_run = base_gt[blockIdx.x], eq_run = base_eq[blockIdx.x];
  for_part(s, mode, blockIdx.x, [&](uint32_t key, int64_t id, bool ok) {
    const uint32_t isgt = ok && key > tau, iseq = ok && key == tau;
    uint32_t tg, te;
    const uint32_t pg = gt_run + block_excl_scan(isgt, &tg);
    const uint32_t pe = eq_run + block_excl_scan(iseq, &te);
    if (isgt || (iseq && pe < need)) out[pg + min(pe, need)] = id;
    gt_run += tg;
    eq_run += te;
  });
}

// The same count and ordered write with one warp per region (the sampled path, where a region
// holds about a thousand candidates): ranks come from ballots, so no block barrier is needed.
// Mode 0 (a region overflowed, the whole array) walks the region's elements 128 at a time.
template <typename F>
__device__ __forceinline__ void for_region_warp(const Src& s, int mode, int b, int lane, F f) {
  if (mode == 1) {
    const int64_t n = s.ccnt[b];
    const uint32_t* kk = s.ckeys + (int64_t)b * s.cap;
    const uint32_t* ii = s.cids + (int64_t)b * s.cap;
    for (int64_t j0 = 0; j0 < n; j0 += 32) {
      const int64_t j = j0 + lane;
      const uint32_t kj = j < n ? kk[j] : 0u;
      const bool ok = j < n && !(s.skip_tagged && (kj >> 31));
      f(kj & 0x7FFFFFFFu, ok ? s.base + (int64_t)ii[j] : 0, ok);
    }
  } else {
    const int64_t lo = (int64_t)b * s.L;
    const int64_t hi = min(s.n, lo + s.L);
    for (int64_t i0 = lo; i0 < hi; i0 += 128) {
      uint32_t key[4];
      bool ok[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + u * 32 + lane;
        ok[u] = i < hi && !(mode == 0 && excluded(s.excl, i));
        key[u] = ok[u] ? src_key(s, i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) f(key[u], s.base + i0 + u * 32 + lane, ok[u]);
    }
  }
}

__device__ __forceinline__ void count_warp_body(const Src& s, const SelCtrl* c, uint32_t* blk_gt,
                                                uint32_t* blk_eq, int b) {
  const int lane = threadIdx.x & 31;
  if (b >= s.G) return;
  const int mode = (int)c->mode;
  const uint32_t tau = c->prefix;
  uint32_t gt = 0, eq = 0;
  for_region_warp(s, mode, b, lane, [&](uint32_t key, int64_t, bool ok) {
    gt += __popc(__ballot_sync(0xffffffffu, ok && key > tau));
    eq += __popc(__ballot_sync(0xffffffffu, ok && key == tau));
  });
  if (lane == 0) {
    blk_gt[b] = gt;
    blk_eq[b] = eq;
  }
}

__global__ void __launch_bounds__(256) sel_count_warp_kernel(Src s, const SelCtrl* c,
                                                            uint32_t* blk_gt, uint32_t* blk_eq) {
  count_warp_body(s, c, blk_gt, blk_eq, blockIdx.x * 8 + (threadIdx.x >> 5));
}

__device__ __forceinline__ void write_warp_body(const Src& s, const SelCtrl* c,
                                                const uint32_t* base_gt, const uint32_t* base_eq,
                                                int64_t* __restrict__ out, int b) {
  const int lane = threadIdx.x & 31;
  if (b >= s.G) return;
  const int mode = (int)c->mode;
  const uint32_t tau = c->prefix;
  const uint32_t need = c->k_rem;
  const uint32_t below = (1u << lane) - 1u;
  uint32_t gt_run = base_gt[b], eq_run = base_eq[b];
  for_region_warp(s, mode, b, lane, [&](uint32_t key, int64_t id, bool ok) {
    const bool isgt = ok && key > tau, iseq = ok && key == tau;
    const uint32_t mg = __ballot_sync(0xffffffffu, isgt);
    const uint32_t me = __ballot_sync(0xffffffffu, iseq);
    const uint32_t pg = gt_run + __popc(mg & below), pe = eq_run + __popc(me & below);
    if (isgt || (iseq && pe < need)) out[pg + min(pe, need)] = id;
    gt_run += __popc(mg);
    eq_run += __popc(me);
  });
}

__global__ void __launch_bounds__(256) sel_write_warp_kernel(Src s, const SelCtrl* c,
                                                            const uint32_t* base_gt,
                                                            const uint32_t* base_eq,
                                                            int64_t* __restrict__ out) {
  write_warp_body(s, c, base_gt, base_eq, out, blockIdx.x * 8 + (threadIdx.x >> 5));
}

// The ordered write's arrays of one selection.
struct WriteJob {
  Src s;
  const SelCtrl* c;
  uint32_t *blk_gt, *blk_eq, *base_gt, *base_eq;
  int64_t* out;
};

// Count, scan and write of two selections over one candidate set: the first nb blocks (or, for
// the scan, block 0) take job 0, the rest job 1.
__global__ void __launch_bounds__(256) sel_count_warp2_kernel(WriteJob j0, WriteJob j1, int nb) {
  const bool second = (int)blockIdx.x >= nb;
  const WriteJob& j = second ? j1 : j0;
  count_warp_body(j.s, j.c, j.blk_gt, j.blk_eq, ((int)blockIdx.x - (second ? nb : 0)) * 8 +
                                                    (int)(threadIdx.x >> 5));
}

__global__ void __launch_bounds__(256) sel_write_warp2_kernel(WriteJob j0, WriteJob j1, int nb) {
  const bool second = (int)blockIdx.x >= nb;
  const WriteJob& j = second ? j1 : j0;
  write_warp_body(j.s, j.c, j.base_gt, j.base_eq, j.out,
                  ((int)blockIdx.x - (second ? nb : 0)) * 8 + (int)(threadIdx.x >> 5));
}

__global__ void __launch_bounds__(1024) sel_scan2_kernel(WriteJob j0, WriteJob j1, int G) {
  const WriteJob& j = blockIdx.x ? j1 : j0;
  scan_body(j.blk_gt, j.blk_eq, G, j.base_gt, j.base_eq);
}

__global__ void bitmap_zero_kernel(uint32_t* bm, int64_t words) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x)
    bm[i] = 0;
}

// Indices outside [0, N) are skipped and flagged (the set violates its contract).
__global__ void bitmap_set_kernel(const int64_t* __restrict__ idx, int64_t K, int64_t N,
                                  uint32_t* bm, uint32_t* dev_status) {
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < K;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t f = idx[i];
    if (f < 0 || f >= N) {
      bad = true;
      continue;
    }
    atomicOr(&bm[f >> 5], 1u << (f & 31));
  }
  flag_status_warp(dev_status, bad, USAF_DEV_BAD_INDEX);
}

// Count, scan and ordered write of the selected entries: one warp per region on the sampled
// path (the mode taken on the device), one block per region otherwise.
usaf_status ordered_write(const SelPlan& p, const SelWs& w, const Src& s, int64_t* out, int fm,
                          bool warp_regions, cudaStream_t st) {
  if (warp_regions) {
    const unsigned nb = (unsigned)ceil_div(p.G, 8);
    sel_count_warp_kernel<<<nb, 256, 0, st>>>(s, w.ctrl, w.blk_gt, w.blk_eq);
    USAF_CHECK_LAUNCH();
    sel_scan_kernel<<<1, 1024, 0, st>>>(w.blk_gt, w.blk_eq, p.G, w.base_gt, w.base_eq);
    USAF_CHECK_LAUNCH();
    sel_write_warp_kernel<<<nb, 256, 0, st>>>(s, w.ctrl, w.base_gt, w.base_eq, out);
    USAF_CHECK_LAUNCH();
    return USAF_OK;
  }
  sel_count_kernel<<<p.G, SEL_THREADS, 0, st>>>(s, w.ctrl, w.blk_gt, w.blk_eq, fm);
  USAF_CHECK_LAUNCH();
  sel_scan_kernel<<<1, 1024, 0, st>>>(w.blk_gt, w.blk_eq, p.G, w.base_gt, w.base_eq);
  USAF_CHECK_LAUNCH();
  sel_write_kernel<<<p.G, SEL_THREADS, 0, st>>>(s, w.ctrl, w.base_gt, w.base_eq, out, fm);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

// The same for two selections over one candidate set (the warp-per-region form), in one launch
// per stage.
usaf_status ordered_write2(const SelPlan& p, const SelWs& w0, const Src& s0, int64_t* out0,
                           const SelWs& w1, const Src& s1, int64_t* out1, cudaStream_t st) {
  const WriteJob j0{s0, w0.ctrl, w0.blk_gt, w0.blk_eq, w0.base_gt, w0.base_eq, out0};
  const WriteJob j1{s1, w1.ctrl, w1.blk_gt, w1.blk_eq, w1.base_gt, w1.base_eq, out1};
  const int nb = (int)ceil_div(p.G, 8);
  sel_count_warp2_kernel<<<2 * nb, 256, 0, st>>>(j0, j1, nb);
  USAF_CHECK_LAUNCH();
  sel_scan2_kernel<<<2, 1024, 0, st>>>(j0, j1, p.G);
  USAF_CHECK_LAUNCH();
  sel_write_warp2_kernel<<<2 * nb, 256, 0, st>>>(j0, j1, nb);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

// The fixed sequence of launches that selects the top-K of `s` (see file comment).
usaf_status run_select(const SelPlan& p, const SelWs& w, Src s, int64_t K, int64_t* out,
                       uint32_t* dev_status, bool fixed_drop, cudaStream_t st) {
  if (p.sampling && !fixed_drop) {
    {
      USAF_TRACE("select_sample", st);
      sel_sample_kernel<<<SAMPLE_BLOCKS, 1024, 0, st>>>(s.g, s.n, s.excl, w.samples, w.bhist,
                                                         nullptr, nullptr, w.ctrl, K, nullptr, 0,
                                                         w.ccnt, p.G);
      USAF_CHECK_LAUNCH();
      const TauJob job{w.samples, w.bhist, w.bhist2, p.q, w.ctrl};
      sel_sample_tau_kernel<<<TAU_BLOCKS, TAU_THREADS, 0, st>>>(job, job);
      USAF_CHECK_LAUNCH();
    }
    USAF_TRACE("select_compact", st);
    if (s.excl)
      sel_compact_kernel<EX_SKIP><<<p.G / COMPACT_WARPS, COMPACT_WARPS * 32, 0, st>>>(
          s.g, s.n, p.L, s.excl, p.cap, w.ckeys, w.cids, w.ccnt, w.ctrl, nullptr,
          dev_status);
    else
      sel_compact_kernel<EX_NONE><<<p.G / COMPACT_WARPS, COMPACT_WARPS * 32, 0, st>>>(
          s.g, s.n, p.L, nullptr, p.cap, w.ckeys, w.cids, w.ccnt, w.ctrl, nullptr,
          dev_status);
    USAF_CHECK_LAUNCH();
  } else {
    USAF_TRACE("select_init", st);
    sel_init_kernel<<<1, 256, 0, st>>>(w.ctrl, K, w.ccnt, p.G);
    USAF_CHECK_LAUNCH();
  }
  sel_decide_kernel<<<1, 256, 0, st>>>(w.ctrl, K, p.sampling && !fixed_drop ? 1 : 0, dev_status);
  USAF_CHECK_LAUNCH();
  s.ckeys = w.ckeys;
  s.cids = w.cids;
  s.ccnt = w.ccnt;
  s.cap = p.cap;
  const int fm = fixed_drop ? 2 : -1;
  s.G = p.G;
  const int rgrid = (int)std::min<int64_t>(p.G, device_sm_count() * 8);
  {
    USAF_TRACE("select_radix", st);
    for (int r = 0; r < SEL_ROUNDS; ++r) {
      sel_round_kernel<<<rgrid, ROUND_THREADS, 0, st>>>(s, w.ctrl, sel_shift(r), sel_bits(r), fm);
      USAF_CHECK_LAUNCH();
    }
  }
  USAF_TRACE("select_write", st);
  return ordered_write(p, w, s, out, fm, p.sampling && !fixed_drop, st);
}

// Entries of the sorted a[0, n) below key, found by one warp with 32 probes per step (about four
// dependent loads for a million entries instead of twenty); every lane gets the result.
__device__ __forceinline__ int64_t lower_bound_warp(const int64_t* a, int64_t n, int64_t key) {
  const int lane = threadIdx.x & 31;
  int64_t lo = 0, hi = n;  // a[i] < key for i < lo, a[i] >= key for i >= hi
  while (hi - lo > 32) {
    const int64_t step = (hi - lo + 31) / 32;
    const int64_t i = lo + (int64_t)lane * step;
    const int c = __popc(__ballot_sync(0xffffffffu, i < hi && a[i] < key));
    if (c == 0) {
      hi = lo;
      break;
    }
    const int64_t nhi = lo + (int64_t)c * step;
    lo += (int64_t)(c - 1) * step + 1;
    hi = nhi < hi ? nhi : hi;
  }
  const int64_t i = lo + lane;
  return lo + __popc(__ballot_sync(0xffffffffu, i < hi && a[i] < key));
}

__device__ __forceinline__ int64_t lower_bound_i64(const int64_t* a, int64_t n, int64_t key) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Merge of the kept and grown entries by tiles of the old set: block b takes act[s0, s1) (MG_TILE
// entries). One search each gives the dropped positions inside the tile and the grown entries that
// fall between act[s0] and act[s1] (block 0 also takes those below act[0], the last block those
// above act[K-1]). A kept entry's new position is (kept entries before it) + (grown entries below
// it); a grown entry's is (its index among the grown) + (kept entries below it). Inside the tile
// the kept ranks come from block scans over rounds of consecutive entries (thread t takes entries
// t, t + MG_THREADS, ..., so the reads of p, m, v and the writes of the new set are coalesced),
// and the searches run over the tile in shared memory or over the tile's own range of the grown
// list, so no per-entry search crosses the whole set.
constexpr int MG_TILE = 1024;
constexpr int MG_THREADS = 256;
constexpr int MG_GROWN = 1024;  // grown entries of a tile's range kept in shared memory
template <typename W>
__global__ void __launch_bounds__(MG_THREADS) rigl_merge_tile_kernel(
    const int64_t* __restrict__ act, int64_t K, const int64_t* __restrict__ dpos,
    const int64_t* __restrict__ grown, int64_t D, const float* __restrict__ p_in,
    const float* __restrict__ m_in, const float* __restrict__ v_in, const W* __restrict__ w0,
    int64_t n0, const W* __restrict__ w1, int64_t* __restrict__ new_idx,
    float* __restrict__ p_out, float* __restrict__ m_out, float* __restrict__ v_out, SelCtrl* c,
    int64_t N, uint32_t* dev_status) {
  constexpr int PER = MG_TILE / MG_THREADS;
  __shared__ int64_t sh_act[MG_TILE];
  __shared__ uint32_t sh_keep[MG_TILE + 1];  // exclusive kept ranks inside the tile
  __shared__ int64_t sh_grown[MG_GROWN];      // the tile's range of the grown list, if it fits
  __shared__ int64_t sh_rng[4];               // d0, d1, g0, g1
  const int64_t s0 = (int64_t)blockIdx.x * MG_TILE;
  const int64_t s1 = min(K, s0 + MG_TILE);
  const int n = (int)(s1 - s0);
  const bool last = s1 == K;
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the four boundary searches, one warp each
  if (wid < 4) {
    int64_t r;
    if (wid == 0) r = lower_bound_warp(dpos, D, s0);
    else if (wid == 1) r = lower_bound_warp(dpos, D, s1);
    else if (wid == 2) r = blockIdx.x == 0 ? 0 : lower_bound_warp(grown, D, act[s0]);
    else r = last ? D : lower_bound_warp(grown, D, act[s1]);
    if (lane == 0) sh_rng[wid] = r;
  }
  for (int i = threadIdx.x; i < n; i += MG_THREADS) {
    sh_act[i] = act[s0 + i];
    sh_keep[i] = 1;
  }
  __syncthreads();
  const int64_t d0 = sh_rng[0], d1 = sh_rng[1], g0 = sh_rng[2], g1 = sh_rng[3];
  const bool g_in_smem = g1 - g0 <= MG_GROWN;
  if (g_in_smem)
    for (int64_t j = g0 + threadIdx.x; j < g1; j += MG_THREADS) sh_grown[j - g0] = grown[j];
  for (int64_t j = d0 + threadIdx.x; j < d1; j += MG_THREADS) sh_keep[dpos[j] - s0] = 0;
  __syncthreads();
  // exclusive ranks of the kept entries, in rounds of MG_THREADS consecutive entries (entry
  // u MG_THREADS + t to thread t), so every global access below is coalesced
  uint32_t f[PER];
  uint32_t run = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int i = u * MG_THREADS + threadIdx.x;
    f[u] = i < n ? sh_keep[i] : 0u;
    uint32_t tot;
    const uint32_t r = run + block_excl_scan(f[u], &tot);
    if (i < n) sh_keep[i] = r;  // each thread rewrites only the entry it read
    run += tot;
  }
  if (threadIdx.x == 0) sh_keep[n] = run;
  __syncthreads();
  const int64_t kept_before = s0 - d0;
  // kept entries
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int i = u * MG_THREADS + threadIdx.x;
    if (i >= n || !f[u]) continue;
    const int64_t fi = sh_act[i];
    int64_t below;  // grown entries of the tile's range below fi
    if (g_in_smem) {
      int lo = 0, hi = (int)(g1 - g0);
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sh_grown[mid] < fi) lo = mid + 1;
        else hi = mid;
      }
      below = lo;
    } else {
      below = lower_bound_i64(grown + g0, g1 - g0, fi);
    }
    const int64_t pos = kept_before + sh_keep[i] + g0 + below;
    if (pos >= K) continue;  // only an unsorted act_idx gets here
    new_idx[pos] = fi;
    p_out[pos] = p_in[s0 + i];
    m_out[pos] = m_in[s0 + i];
    v_out[pos] = v_in[s0 + i];
  }
  // grown entries of the tile's range (a given grow set is range-checked before its weight is
  // read: an entry outside [0, N) gets p = 0 and sets USAF_DEV_BAD_INDEX)
  bool bad = false;
  for (int64_t j = g0 + threadIdx.x; j < g1; j += MG_THREADS) {
    const int64_t fj = g_in_smem ? sh_grown[j - g0] : grown[j];
    int lo = 0, hi = n;  // kept-or-dropped tile entries below fj
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sh_act[mid] < fj) lo = mid + 1;
      else hi = mid;
    }
    const int64_t pos = kept_before + sh_keep[lo] + j;
    if (pos < 0 || pos >= K) continue;  // only an unsorted act_idx gets here
    const bool ok = fj >= 0 && fj < N;
    bad |= !ok;
    new_idx[pos] = fj;
    p_out[pos] = ok ? to_f32(fj < n0 ? w0[fj] : w1[fj - n0]) : 0.f;
    m_out[pos] = 0.f;
    v_out[pos] = 0.f;
  }
  flag_status_warp(dev_status, bad, USAF_DEV_BAD_INDEX);
  if (threadIdx.x == 0 && d1 > d0) atomicAdd(&c->n_swapped, (unsigned long long)(d1 - d0));
}

// Full reselection: entry t of the new set carries (p, m, v) from the old set when its flat index
// is there (binary search), else starts from the dense weight with zero moments.
template <typename W>
__global__ void reselect_carry_kernel(const int64_t* __restrict__ new_idx, int64_t K,
                                      const int64_t* __restrict__ old_idx, int64_t K_old,
                                      const float* __restrict__ p_in, const float* __restrict__ m_in,
                                      const float* __restrict__ v_in, const W* __restrict__ w0,
                                      int64_t n0, const W* __restrict__ w1, float* __restrict__ p_out,
                                      float* __restrict__ m_out, float* __restrict__ v_out,
                                      SelCtrl* c, int64_t N, uint32_t* dev_status) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  bool kept = false, bad = false;
  if (t < K) {
    const int64_t f = new_idx[t];
    const int64_t s = lower_bound_i64(old_idx, K_old, f);
    kept = s < K_old && old_idx[s] == f;
    if (kept) {
      p_out[t] = p_in[s];
      m_out[t] = m_in[s];
      v_out[t] = v_in[s];
    } else {
      bad = f < 0 || f >= N;  // a given set is range-checked before its weight is read
      p_out[t] = bad ? 0.f : to_f32(f < n0 ? w0[f] : w1[f - n0]);
      m_out[t] = 0.f;
      v_out[t] = 0.f;
    }
  }
  flag_status_warp(dev_status, bad, USAF_DEV_BAD_INDEX);
  const unsigned n = __popc(__ballot_sync(0xffffffffu, kept));
  if ((threadIdx.x & 31) == 0 && n) atomicAdd(&c->n_swapped, (unsigned long long)n);
}

__global__ void rigl_finish_kernel(const SelCtrl* c, int64_t* n_swapped) {
  if (threadIdx.x == 0) *n_swapped = (int64_t)c->n_swapped;
}

}  // namespace

size_t select_ws_bytes(int64_t N, int64_t K, bool with_bitmap) {
  const SelPlan p = make_plan(N, K);
  Carver c(nullptr);
  SelWs w;
  sel_layout(p, c, w);
  if (with_bitmap) c.take<uint32_t>(ceil_div(N, 32));
  return c.size();
}

usaf_status importance_select_launch(const float* g, int64_t N, int64_t K, int64_t* out_idx,
                                     uint32_t* dev_status, void* ws, cudaStream_t st) {
  const SelPlan p = make_plan(N, K);
  Carver c(ws);
  SelWs w;
  sel_layout(p, c, w);
  Src s{};
  s.g = g;
  s.n = N;
  s.L = p.L;
  s.excl = nullptr;
  s.drop = 0;
  return run_select(p, w, s, K, out_idx, dev_status, false, st);
}

size_t rigl_ws_bytes(int64_t N, int64_t K, int64_t D) {
  Carver c(nullptr);
  c.take<int64_t>(D);  // dropped positions
  c.take<int64_t>(D);  // grown indices
  c.take<char>(select_ws_bytes(K > 0 ? K : 1, D > 0 ? D : 1, false));
  c.take<char>(select_ws_bytes(N, D > 0 ? D : 1, true));
  return c.size();
}

namespace {

// The arguments of a RigL swap that the drop selection and the merge use.
struct RiglIo {
  int64_t N, K, D;
  const int64_t* act_idx;
  const float *p_in, *m_in, *v_in;
  const void *w0, *w1;
  int64_t n0;
  usaf_dtype wdt;
  int64_t* new_idx;
  float *p_out, *m_out, *v_out;
  int64_t* n_swapped;
  uint32_t* dev_status;
};

// Drop selection (the D smallest |p| among the K actives: complemented keys, exact path), the
// grow selection that `grow` issues on `st` (when given: the drop selection then runs on a stream
// of its own, forked from and joined back to `st`, so that its chain of small launches overlaps
// the pass over g), and the merge of the kept and grown entries.
template <class GrowFn>
usaf_status rigl_swap_around(const RiglIo& io, int64_t* dpos, const int64_t* grown, char* ws_drop,
                             bool has_grow, GrowFn grow, cudaStream_t st) {
  const int64_t Ks = io.K > 0 ? io.K : 1, Ds = io.D > 0 ? io.D : 1;
  const SelPlan pd = make_plan(Ks, Ds);
  Carver cd(ws_drop);
  SelWs wd;
  sel_layout(pd, cd, wd);
  Src sd{};
  sd.g = io.p_in;
  sd.n = io.K;
  sd.L = pd.L;
  sd.drop = 1;
  if (io.D <= 0) {
    sel_init_kernel<<<1, 256, 0, st>>>(wd.ctrl, 0, wd.ccnt, pd.G);
    USAF_CHECK_LAUNCH();
  } else if (!has_grow) {
    USAF_TRY(run_select(pd, wd, sd, io.D, dpos, io.dev_status, true, st));
  } else {
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    auto release = [&]() {
      if (fork) cudaEventDestroy(fork);
      if (join) cudaEventDestroy(join);
      if (side) cudaStreamDestroy(side);  // its work still completes
    };
    if (cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventRecord(fork, st) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess) {
      release();
      return USAF_ERR_CUDA;
    }
    const usaf_status sdrop = run_select(pd, wd, sd, io.D, dpos, io.dev_status, true, side);
    if (sdrop != USAF_OK || cudaEventRecord(join, side) != cudaSuccess) {
      release();
      return sdrop != USAF_OK ? sdrop : USAF_ERR_CUDA;
    }
    const usaf_status sgrow = grow();
    const bool joined = cudaStreamWaitEvent(st, join, 0) == cudaSuccess;
    release();
    if (sgrow != USAF_OK) return sgrow;
    if (!joined) return USAF_ERR_CUDA;
  }
  USAF_TRACE("rigl_merge", st);
  if (io.K > 0) {
    const unsigned nb = (unsigned)ceil_div(io.K, MG_TILE);
    if (io.wdt == USAF_BF16)
      rigl_merge_tile_kernel<__nv_bfloat16><<<nb, MG_THREADS, 0, st>>>(
          io.act_idx, io.K, dpos, grown, io.D, io.p_in, io.m_in, io.v_in,
          static_cast<const __nv_bfloat16*>(io.w0), io.n0,
          static_cast<const __nv_bfloat16*>(io.w1), io.new_idx, io.p_out, io.m_out, io.v_out,
          wd.ctrl, io.N, io.dev_status);
    else
      rigl_merge_tile_kernel<float><<<nb, MG_THREADS, 0, st>>>(
          io.act_idx, io.K, dpos, grown, io.D, io.p_in, io.m_in, io.v_in,
          static_cast<const float*>(io.w0), io.n0, static_cast<const float*>(io.w1), io.new_idx,
          io.p_out, io.m_out, io.v_out, wd.ctrl, io.N, io.dev_status);
    USAF_CHECK_LAUNCH();
  }
  rigl_finish_kernel<<<1, 32, 0, st>>>(wd.ctrl, io.n_swapped);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

// The bitmap of the active set (excluded from the grow selection).
usaf_status active_bitmap(const int64_t* act_idx, int64_t K, int64_t N, uint32_t* bitmap,
                          uint32_t* dev_status, cudaStream_t st) {
  USAF_TRACE("rigl_bitmap", st);
  const int64_t words = ceil_div(N, 32);
  bitmap_zero_kernel<<<grid_dim_for(words), 256, 0, st>>>(bitmap, words);
  USAF_CHECK_LAUNCH();
  if (K > 0) {
    bitmap_set_kernel<<<grid_dim_for(K), 256, 0, st>>>(act_idx, K, N, bitmap, dev_status);
    USAF_CHECK_LAUNCH();
  }
  return USAF_OK;
}

}  // namespace

usaf_status rigl_launch(const float* g, int64_t N, const int64_t* act_idx, int64_t K, int64_t D,
                        const float* p_in, const float* m_in, const float* v_in, const void* w0,
                        int64_t n0, const void* w1, usaf_dtype wdt, int64_t* new_idx,
                        float* p_out, float* m_out, float* v_out, int64_t* n_swapped,
                        uint32_t* dev_status, void* ws, cudaStream_t st,
                        const int64_t* grown_in) {
  Carver c(ws);
  int64_t* dpos = c.take<int64_t>(D);
  int64_t* grown = c.take<int64_t>(D);
  const int64_t Ks = K > 0 ? K : 1, Ds = D > 0 ? D : 1;
  char* ws_drop = c.take<char>(select_ws_bytes(Ks, Ds, false));
  const RiglIo io{N, K, D, act_idx, p_in, m_in, v_in, w0, w1, n0, wdt, new_idx, p_out,
                  m_out, v_out, n_swapped, dev_status};
  // the grow set is given (chosen across ranks): drop selection and merge only
  if (grown_in) return rigl_swap_around(io, dpos, grown_in, ws_drop, false, [] { return USAF_OK; }, st);
  char* ws_grow = c.take<char>(select_ws_bytes(N, Ds, true));
  // grow: the D largest |g| outside the active set (sampled path with an exclusion bitmap)
  auto grow = [&]() -> usaf_status {
    const SelPlan pg = make_plan(N, Ds);
    Carver cg(ws_grow);
    SelWs wg;
    sel_layout(pg, cg, wg);
    uint32_t* bitmap = cg.take<uint32_t>(ceil_div(N, 32));
    USAF_TRY(active_bitmap(act_idx, K, N, bitmap, dev_status, st));
    Src sg{};
    sg.g = g;
    sg.n = N;
    sg.L = pg.L;
    sg.excl = bitmap;
    sg.drop = 0;
    return run_select(pg, wg, sg, D, grown, dev_status, false, st);
  };
  return rigl_swap_around(io, dpos, grown, ws_drop, D > 0, grow, st);
}

// ------------------------------------------------------------------------------------------------
// Importance selection and RigL swap from one pass over g. The top-K_sel of |g| and the grow set
// (the D largest |g| outside the active set) are both found among one set of candidates: the
// samples give each selection its own tau0, one compacting pass keeps every key at or above the
// lower of the two (excluded entries tagged by bit 31 of their stored key), and each selection then
// runs its radix rounds and ordered write over the shared candidates (the grow selection skips the
// tagged ones). Results equal the two separate calls'.
// ------------------------------------------------------------------------------------------------
namespace {

struct FusedPlan {
  SelPlan p;      // regions, capacity: the candidates of both selections
  int q_sel, q_grow;
  bool ok;        // both selections take the sampled path
};

FusedPlan make_fused_plan(int64_t N, int64_t Ksel, int64_t K, int64_t D) {
  FusedPlan f{};
  if (D <= 0 || Ksel <= 0) return f;
  const SelPlan a = make_plan(N, Ksel), b = make_plan(N, D);
  // the keys at or above the selection's tau0 are about K_sel; those at or above the grow's are
  // about D outside the active set plus at most the K active ones: the regions are sized for the
  // larger count (an overflow still only sends both selections to the exact path)
  f.p = make_plan(N, std::max(Ksel, K + D));
  f.q_sel = a.q;
  f.q_grow = b.q;
  f.ok = a.sampling && b.sampling && f.p.sampling;
  return f;
}

void fused_layout(const FusedPlan& f, Carver& c, SelWs& ws, SelWs& wg) {
  sel_layout(f.p, c, ws);
  wg = ws;
  wg.ctrl = c.take<SelCtrl>(1);
  wg.blk_gt = c.take<uint32_t>(f.p.G);
  wg.blk_eq = c.take<uint32_t>(f.p.G);
  wg.base_gt = c.take<uint32_t>(f.p.G);
  wg.base_eq = c.take<uint32_t>(f.p.G);
  wg.samples = c.take<uint32_t>(SAMPLE_S);
  wg.bhist = c.take<uint32_t>(SAMPLE_S / 1024 * 256);
  wg.bhist2 = c.take<uint32_t>(TAU_BLOCKS * 256);
}

}  // namespace

size_t select_and_swap_ws_bytes(int64_t N, int64_t Ksel, int64_t K, int64_t D) {
  const FusedPlan f = make_fused_plan(N, Ksel, K, D);
  Carver c(nullptr);
  if (!f.ok) {
    c.take<char>(select_ws_bytes(N, Ksel, false));
    c.take<char>(rigl_ws_bytes(N, K, D));
    return c.size();
  }
  c.take<int64_t>(D);
  c.take<int64_t>(D);
  c.take<char>(select_ws_bytes(K > 0 ? K : 1, D, false));
  SelWs a, b;
  fused_layout(f, c, a, b);
  c.take<uint32_t>(ceil_div(N, 32));
  return c.size();
}

usaf_status select_and_swap_launch(const float* g, int64_t N, int64_t Ksel, int64_t* sel_idx,
                                   const int64_t* act_idx, int64_t K, int64_t D,
                                   const float* p_in, const float* m_in, const float* v_in,
                                   const void* w0, int64_t n0, const void* w1, usaf_dtype wdt,
                                   int64_t* new_idx, float* p_out, float* m_out, float* v_out,
                                   int64_t* n_swapped, uint32_t* dev_status, void* ws,
                                   cudaStream_t st) {
  const FusedPlan f = make_fused_plan(N, Ksel, K, D);
  Carver c(ws);
  if (!f.ok) {
    // a selection on the exact path (small N, or K_sel or D a large part of N): the two calls
    char* ws_sel = c.take<char>(select_ws_bytes(N, Ksel, false));
    char* ws_rigl = c.take<char>(rigl_ws_bytes(N, K, D));
    USAF_TRY(importance_select_launch(g, N, Ksel, sel_idx, dev_status, ws_sel, st));
    return rigl_launch(g, N, act_idx, K, D, p_in, m_in, v_in, w0, n0, w1, wdt, new_idx, p_out,
                       m_out, v_out, n_swapped, dev_status, ws_rigl, st);
  }
  int64_t* dpos = c.take<int64_t>(D);
  int64_t* grown = c.take<int64_t>(D);
  char* ws_drop = c.take<char>(select_ws_bytes(K > 0 ? K : 1, D, false));
  SelWs w1s, w2s;
  fused_layout(f, c, w1s, w2s);
  uint32_t* bitmap = c.take<uint32_t>(ceil_div(N, 32));
  const RiglIo io{N, K, D, act_idx, p_in, m_in, v_in, w0, w1, n0, wdt, new_idx, p_out,
                  m_out, v_out, n_swapped, dev_status};
  const SelPlan& p = f.p;
  auto both = [&]() -> usaf_status {
    USAF_TRY(active_bitmap(act_idx, K, N, bitmap, dev_status, st));
    {
      USAF_TRACE("select_sample", st);
      sel_sample_kernel<<<SAMPLE_BLOCKS, 1024, 0, st>>>(g, N, bitmap, w2s.samples, w2s.bhist,
                                                         w1s.samples, w1s.bhist, w2s.ctrl, D,
                                                         w1s.ctrl, Ksel, w1s.ccnt, p.G);
      USAF_CHECK_LAUNCH();
      const TauJob js{w1s.samples, w1s.bhist, w1s.bhist2, f.q_sel, w1s.ctrl};
      const TauJob jg{w2s.samples, w2s.bhist, w2s.bhist2, f.q_grow, w2s.ctrl};
      sel_sample_tau_kernel<<<2 * TAU_BLOCKS, TAU_THREADS, 0, st>>>(js, jg);
      USAF_CHECK_LAUNCH();
    }
    {
      USAF_TRACE("select_compact", st);
      sel_compact_kernel<EX_TAG><<<p.G / COMPACT_WARPS, COMPACT_WARPS * 32, 0, st>>>(
          g, N, p.L, bitmap, p.cap, w1s.ckeys, w1s.cids, w1s.ccnt, w1s.ctrl, w2s.ctrl, dev_status);
      USAF_CHECK_LAUNCH();
    }
    sel_decide2_kernel<<<2, 256, 0, st>>>(w1s.ctrl, Ksel, w2s.ctrl, D, dev_status);
    USAF_CHECK_LAUNCH();
    Src ss{};
    ss.g = g;
    ss.n = N;
    ss.L = p.L;
    ss.ckeys = w1s.ckeys;
    ss.cids = w1s.cids;
    ss.ccnt = w1s.ccnt;
    ss.cap = p.cap;
    ss.G = p.G;
    Src sg = ss;
    sg.excl = bitmap;
    sg.skip_tagged = 1;
    const int rgrid = (int)std::min<int64_t>(p.G, device_sm_count() * 8);
    {
      USAF_TRACE("select_radix", st);
      for (int r = 0; r < SEL_ROUNDS; ++r) {
        sel_round2_kernel<<<2 * rgrid, ROUND_THREADS, 0, st>>>(ss, w1s.ctrl, sg, w2s.ctrl,
                                                               sel_shift(r), sel_bits(r));
        USAF_CHECK_LAUNCH();
      }
    }
    USAF_TRACE("select_write", st);
    return ordered_write2(p, w1s, ss, sel_idx, w2s, sg, grown, st);
  };
  return rigl_swap_around(io, dpos, grown, ws_drop, true, both, st);
}

// ------------------------------------------------------------------------------------------------
// Shard primitives of a selection spread over several ranks (each rank holds a contiguous part of
// the keys): digit histograms, counts at a threshold, and the ordered emission of a part's winners.
// The rounds, the digit picks and the exchanges between ranks run on the host.
// ------------------------------------------------------------------------------------------------
namespace {
constexpr int SH_THREADS = 256;
constexpr int SH_MAX_BITS = 11;

// hist[d] += keys of g[0, n) (not excluded) whose bits above shift + bits equal prefix's, by the
// digit of `bits` bits at `shift`. Digits of up to 8 bits go to per-warp shared histograms (the
// first round, where every key lands in a few bins); wider digits to one per-block histogram (the
// later rounds, where the prefix test lets few keys through). One global add per block and bin.
template <bool PER_WARP>
__global__ void __launch_bounds__(SH_THREADS) shard_hist_kernel(
    const float* __restrict__ g, int64_t n, const uint32_t* __restrict__ excl, uint32_t prefix,
    int shift, int bits, unsigned long long* hist) {
  constexpr int WB = 257;                                      // per-warp bins, padded
  constexpr int WORDS = PER_WARP ? (SH_THREADS / 32) * WB : (1 << SH_MAX_BITS);
  __shared__ uint32_t sh[WORDS];
  for (int i = threadIdx.x; i < WORDS; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  uint32_t* hw = PER_WARP ? sh + (threadIdx.x >> 5) * WB : sh;
  const uint32_t dmask = (1u << bits) - 1;
  const int hs = shift + bits;
  auto add = [&](uint32_t k, int64_t i) {
    if (excluded(excl, i)) return;
    if (hs >= 32 || (k >> hs) == (prefix >> hs)) atomicAdd(&hw[(k >> shift) & dmask], 1u);
  };
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t done = 0;
  if ((reinterpret_cast<uintptr_t>(g) & 15) == 0) {  // 16-byte loads over the aligned body
    const int64_t n4 = n >> 2;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    for (int64_t q = tid; q < n4; q += stride) {
      const float4 v = __ldg(g4 + q);
      add(abs_key(v.x), 4 * q);
      add(abs_key(v.y), 4 * q + 1);
      add(abs_key(v.z), 4 * q + 2);
      add(abs_key(v.w), 4 * q + 3);
    }
    done = n4 << 2;
  }
  for (int64_t i = done + tid; i < n; i += stride) add(abs_key(g[i]), i);
  __syncthreads();
  for (int d = threadIdx.x; d <= (int)dmask; d += blockDim.x) {
    uint32_t t = 0;
    if (PER_WARP)
      for (int w = 0; w < SH_THREADS / 32; ++w) t += sh[w * WB + d];
    else
      t = sh[d];
    if (t) atomicAdd(&hist[d], (unsigned long long)t);
  }
}

// Control block of an emission at a known threshold: candidates are the keys >= tau.
__global__ void shard_emit_init_kernel(SelCtrl* c, uint32_t tau, uint32_t take_eq, uint32_t* ccnt,
                                       int G) {
  for (int i = threadIdx.x; i < MAX_BINS; i += blockDim.x) c->hist[i] = 0;
  for (int i = threadIdx.x; i < G; i += blockDim.x) ccnt[i] = 0;
  if (threadIdx.x == 0) {
    c->tau0 = tau;
    c->prefix = tau;
    c->k_rem = take_eq;
    c->mode = 0;
    c->overflow = 0;
    c->total = 0;
    c->ticket = 0;
  }
}

// The candidate path unless a region overflowed (then the whole part, in order, reported as
// USAF_DEV_SELECT_EXACT_PATH)
__global__ void shard_emit_decide_kernel(SelCtrl* c, uint32_t* dev_status) {
  if (threadIdx.x == 0) {
    c->mode = c->overflow ? 0u : 1u;
    if (c->overflow) flag_status(dev_status, USAF_DEV_SELECT_EXACT_PATH);
  }
}

__global__ void bitmap_range_kernel(const int64_t* __restrict__ idx, int64_t K, int64_t lo,
                                    int64_t n, uint32_t* bm) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < K;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t f = idx[i] - lo;
    if (f >= 0 && f < n) atomicOr(&bm[f >> 5], 1u << (f & 31));
  }
}
}  // namespace

usaf_status shard_hist_launch(const float* g, int64_t n, const uint32_t* excl, uint32_t prefix,
                              int shift, int bits, unsigned long long* hist, cudaStream_t st) {
  if (n == 0) return USAF_OK;
  USAF_TRACE("shard_hist", st);
  const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(n, 4 * SH_THREADS),
                                                    (int64_t)device_sm_count() * 8);
  if (bits <= 8)
    shard_hist_kernel<true><<<grid, SH_THREADS, 0, st>>>(g, n, excl, prefix, shift, bits, hist);
  else
    shard_hist_kernel<false><<<grid, SH_THREADS, 0, st>>>(g, n, excl, prefix, shift, bits, hist);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

size_t shard_emit_ws_bytes(int64_t n, int64_t count) {
  const int64_t ns = n > 0 ? n : 1;
  SelPlan p = make_plan(ns, count > 0 ? count : 1);
  Carver c(nullptr);
  SelWs w;
  sel_layout(p, c, w);
  return c.size();
}

// The part's winners in index order: keys > tau, then the first take_eq keys == tau. `count` is
// the number of keys >= tau in the part (from the count step); it sizes the candidate regions of
// one compacting pass at threshold tau, after which the ordered write runs over the candidates
// (over the whole part if a region overflowed).
usaf_status shard_emit_launch(const float* g, int64_t n, const uint32_t* excl, uint32_t tau,
                              int64_t take_eq, int64_t count, int64_t base, int64_t* out,
                              uint32_t* dev_status, void* ws, cudaStream_t st) {
  if (n == 0) return USAF_OK;
  USAF_TRACE("shard_emit", st);
  const SelPlan p = make_plan(n, count > 0 ? count : 1);
  Carver c(ws);
  SelWs w;
  sel_layout(p, c, w);
  shard_emit_init_kernel<<<1, 256, 0, st>>>(w.ctrl, tau, (uint32_t)take_eq, w.ccnt, p.G);
  USAF_CHECK_LAUNCH();
  Src s{};
  s.g = g;
  s.n = n;
  s.L = p.L;
  s.excl = excl;
  s.drop = 0;
  s.G = p.G;
  s.base = base;
  int fm = 0;
  if (p.sampling) {
    if (excl)
      sel_compact_kernel<EX_SKIP><<<p.G / COMPACT_WARPS, COMPACT_WARPS * 32, 0, st>>>(
          g, n, p.L, excl, p.cap, w.ckeys, w.cids, w.ccnt, w.ctrl, nullptr, dev_status);
    else
      sel_compact_kernel<EX_NONE><<<p.G / COMPACT_WARPS, COMPACT_WARPS * 32, 0, st>>>(
          g, n, p.L, nullptr, p.cap, w.ckeys, w.cids, w.ccnt, w.ctrl, nullptr,
          dev_status);
    USAF_CHECK_LAUNCH();
    shard_emit_decide_kernel<<<1, 32, 0, st>>>(w.ctrl, dev_status);
    USAF_CHECK_LAUNCH();
    s.ckeys = w.ckeys;
    s.cids = w.cids;
    s.ccnt = w.ccnt;
    s.cap = p.cap;
    fm = -1;
  }
  return ordered_write(p, w, s, out, fm, p.sampling, st);
}

usaf_status bitmap_range_launch(const int64_t* idx, int64_t K, int64_t lo, int64_t n,
                                uint32_t* bm, cudaStream_t st) {
  const int64_t words = ceil_div(n, 32);
  bitmap_zero_kernel<<<grid_dim_for(words), 256, 0, st>>>(bm, words);
  USAF_CHECK_LAUNCH();
  if (K > 0) {
    bitmap_range_kernel<<<grid_dim_for(K), 256, 0, st>>>(idx, K, lo, n, bm);
    USAF_CHECK_LAUNCH();
  }
  return USAF_OK;
}

size_t reselect_ws_bytes(int64_t N, int64_t K) { return select_ws_bytes(N, K > 0 ? K : 1, false); }

// The state carry of a full reselection for a new set chosen elsewhere (across ranks).
usaf_status reselect_carry_launch(const int64_t* new_idx, int64_t K, int64_t N,
                                  const int64_t* old_idx, int64_t K_old, const float* p_in,
                                  const float* m_in, const float* v_in, const void* w0, int64_t n0,
                                  const void* w1, usaf_dtype wdt, float* p_out, float* m_out,
                                  float* v_out, int64_t* n_kept, uint32_t* dev_status, void* ws,
                                  cudaStream_t st) {
  Carver c(ws);
  SelCtrl* ctrl = c.take<SelCtrl>(1);
  uint32_t* ccnt = c.take<uint32_t>(1);
  sel_init_kernel<<<1, 256, 0, st>>>(ctrl, 0, ccnt, 1);
  USAF_CHECK_LAUNCH();
  if (K > 0) {
    USAF_TRACE("reselect_carry", st);
    if (wdt == USAF_BF16)
      reselect_carry_kernel<__nv_bfloat16><<<(unsigned)ceil_div(K, 256), 256, 0, st>>>(
          new_idx, K, old_idx, K_old, p_in, m_in, v_in, static_cast<const __nv_bfloat16*>(w0),
          n0, static_cast<const __nv_bfloat16*>(w1), p_out, m_out, v_out, ctrl, N, dev_status);
    else
      reselect_carry_kernel<float><<<(unsigned)ceil_div(K, 256), 256, 0, st>>>(
          new_idx, K, old_idx, K_old, p_in, m_in, v_in, static_cast<const float*>(w0), n0,
          static_cast<const float*>(w1), p_out, m_out, v_out, ctrl, N, dev_status);
    USAF_CHECK_LAUNCH();
  }
  rigl_finish_kernel<<<1, 32, 0, st>>>(ctrl, n_kept);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}
size_t reselect_carry_ws_bytes() {
  Carver c(nullptr);
  c.take<SelCtrl>(1);
  c.take<uint32_t>(1);
  return c.size();
}

usaf_status reselect_launch(const float* g, int64_t N, int64_t K, const int64_t* old_idx,
                            int64_t K_old, const float* p_in, const float* m_in,
                            const float* v_in, const void* w0, int64_t n0, const void* w1,
                            usaf_dtype wdt, int64_t* new_idx, float* p_out, float* m_out,
                            float* v_out, int64_t* n_kept, uint32_t* dev_status, void* ws,
                            cudaStream_t st) {
  const int64_t Ks = K > 0 ? K : 1;
  const SelPlan p = make_plan(N, Ks);
  Carver c(ws);
  SelWs w;
  sel_layout(p, c, w);
  if (K > 0) {
    Src s{};
    s.g = g;
    s.n = N;
    s.L = p.L;
    s.excl = nullptr;
    s.drop = 0;
    USAF_TRY(run_select(p, w, s, K, new_idx, dev_status, false, st));
    USAF_TRACE("reselect_carry", st);
    if (wdt == USAF_BF16)
      reselect_carry_kernel<__nv_bfloat16><<<(unsigned)ceil_div(K, 256), 256, 0, st>>>(
          new_idx, K, old_idx, K_old, p_in, m_in, v_in, static_cast<const __nv_bfloat16*>(w0),
          n0, static_cast<const __nv_bfloat16*>(w1), p_out, m_out, v_out, w.ctrl, N,
          dev_status);
    else
      reselect_carry_kernel<float><<<(unsigned)ceil_div(K, 256), 256, 0, st>>>(
          new_idx, K, old_idx, K_old, p_in, m_in, v_in, static_cast<const float*>(w0), n0,
          static_cast<const float*>(w1), p_out, m_out, v_out, w.ctrl, N, dev_status);
    USAF_CHECK_LAUNCH();
  } else {
    sel_init_kernel<<<1, 256, 0, st>>>(w.ctrl, 0, w.ccnt, p.G);
    USAF_CHECK_LAUNCH();
  }
  rigl_finish_kernel<<<1, 32, 0, st>>>(w.ctrl, n_kept);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

}  // namespace usaf
