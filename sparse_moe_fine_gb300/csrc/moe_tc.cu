// bf16 grouped expert GEMMs on 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM),
// fed by TMA (cp.async.bulk.tensor) through a 4-stage mbarrier pipeline. One persistent CTA per SM
// with three roles: warp 0 issues TMA loads, warp 1 issues MMAs (one thread) and owns the TMEM
// allocation, eight epilogue warps run the fused epilogue out of a double-buffered TMEM
// accumulator (two warps per TMEM lane quarter, alternating 32-column chunks).
//
// Every GEMM puts the weight dimension on M (128 rows per tile) and the routed tokens on N
// (16..256 per tile), so an expert's ragged token count only pads to 16. The token operand is
// feature-major (one row per feature, the expert's permuted tokens contiguous) and is loaded as
// the MN-major B operand in boxes of 64 tokens.
//   S4 gate_up: h^T = gate_up[e] x^T     A = gate/up rows interleaved (K-major), B = x^T
//               epilogue: SwiGLU (act(gate)*up, experts4bit-qlora epilogue contract) times the
//               routing weight; writes h^T and (w*A)^T with 16-byte stores
//   S5 down:    y^T = down[e] (wA)^T      epilogue: scatter-add into the fp32 combine buffer
//   S6 gvec:    g^T = down[e]^T dy^T      A = down[e] MN-major; epilogue: SwiGLU backward,
//               dw (routing-weight gradient), dh^T
//   S8 dx:      dx^T = gate_up[e]^T dh^T  A = gate_up[e] MN-major; epilogue: scatter-add
//   router:     logits^T = [Wr_hi|Wr_mid|Wr_lo] [x|x|x]^T, three bf16 parts of the fp32 router
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.cuh"

namespace usaf {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN = TC_TOKEN_TILE;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int B_BOX = 64 * BK * 2;  // one MN-major box: 64 tokens x 64 k
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int TMEM_COLS = 512;
constexpr int MAX_E = 1024;
constexpr int PLAN_BYTES = 8704;  // barriers, TMEM slot, abort flag, plan and offsets (E <= 1024)
constexpr int STAGE_PITCH = 80;   // bytes per row of an epilogue warp's store staging (64 + 16)
constexpr int EPI_STAGE_BYTES = 32 * STAGE_PITCH;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + PLAN_BYTES + EPI_WARPS * EPI_STAGE_BYTES;
static_assert(256 + 2 * (MAX_E + 1) * 4 <= PLAN_BYTES, "plan area");
static_assert(SMEM_BYTES <= 232448, "shared memory of the tensor-core kernel");
constexpr long long TIMEOUT_CYCLES = 1ll << 32;  // about two seconds

enum Var { V_GATEUP = 0, V_DOWN = 1, V_GVEC = 2, V_DX = 3, V_ROUTER = 4 };

struct Params {
  const int32_t* off;
  const int32_t* ptok;
  const int32_t* pslot;
  const float* topk_w;
  const int32_t* plan;
  int E, H, I, T;
  int MT, NT;
  int64_t R_cap;  // row pitch of the feature-major arrays
  __nv_bfloat16* h;       // h^T out (S4)
  __nv_bfloat16* wa;      // (w*A)^T out (S4)
  float* acc_out;         // y_acc (S5), dx_acc (S8) or the router logits
  float* dw_part;         // S6: dw partial sums [4 * MT][n_slots] (row quarter of an M tile)
  int64_t n_slots;        // T * k
  __nv_bfloat16* dh;      // dh^T out (S6)
  const __nv_bfloat16* hin;  // h^T in (S6)
  const float* wperm;        // routing weight per permuted row (0 in padding)
  const float* dl_perm;      // S8 (may be null): dlogit of each permuted row's slot, for the
  const float* w_router;     //   router term dl * Wr[e, :] added in the dx epilogue
  uint32_t* status;
};

// ---------------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false when the phase did not complete within the limit or another role gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          long long limit = TIMEOUT_CYCLES) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) return false;
  }
}
// Drain wait, for work this thread has already issued (TMA copies, MMAs): such work completes
// whatever the other roles do, so the abort flag is not consulted; only the deadline (a clock64
// value shared by all of a role's drain waits) bounds it.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, long long deadline) {
  while (!mbar_try_wait(bar, parity))
    if (clock64() > deadline) return false;
  return true;
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                       int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                       int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: 128-byte swizzle, start address, LBO and SBO in bytes.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of this architecture
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulate, M = 128.
__device__ __forceinline__ uint32_t idesc_bf16(int n, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// ---------------------------------------------------------------------------- tiles
struct Tile {
  int e;
  int m0;     // first M row of the tile (feature / weight row)
  int row0;   // first permuted row (token) of the tile
  int nrows;  // tokens in the tile (multiple of 16)
  int klen;   // K extent
};

template <int VAR>
struct VarTraits {
  static constexpr bool router = VAR == V_ROUTER;
  static constexpr bool a_mn = VAR == V_GVEC || VAR == V_DX;
};
constexpr int ROUTER_BN = 32;  // tokens per router tile: T / 32 tiles keep most SMs busy

__device__ __forceinline__ int upper_bound_i32(const int32_t* a, int n, int v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (a[mid] <= v) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Tile t: (expert, M tile, token tile) with token tiles fastest; experts' token tiles come from
// the plan (a prefix over experts of ceil(padded rows / 256)), split into equal 16-row multiples.
template <int VAR>
__device__ __forceinline__ Tile get_tile(const Params& p, const int32_t* s_plan,
                                         const int32_t* s_off, int t) {
  Tile ti{};
  if constexpr (VarTraits<VAR>::router) {
    const int mt = t / p.NT, nt = t % p.NT;
    ti.m0 = mt * BM;
    ti.row0 = nt * ROUTER_BN;
    ti.nrows = min(ROUTER_BN, (p.T - ti.row0 + 15) / 16 * 16);
    ti.klen = 3 * p.H;
  } else {
    const int e = upper_bound_i32(s_plan, p.E + 1, t / p.MT) - 1;
    const int nts = s_plan[e + 1] - s_plan[e];
    const int local = t - p.MT * s_plan[e];
    const int mt = local / nts, nt = local % nts;
    const int npad = s_off[e + 1] - s_off[e];
    const int base = ((npad + nts - 1) / nts + 15) / 16 * 16;
    ti.e = e;
    ti.m0 = mt * (VAR == V_GATEUP ? 64 : BM);
    ti.row0 = s_off[e] + nt * base;
    ti.nrows = min(base, npad - nt * base);
    ti.klen = (VAR == V_GATEUP || VAR == V_GVEC) ? p.H : (VAR == V_DOWN ? p.I : 2 * p.I);
  }
  return ti;
}

template <int VAR>
__device__ __forceinline__ int total_tiles(const Params& p, const int32_t* s_plan) {
  if constexpr (VarTraits<VAR>::router) return p.MT * p.NT;
  else return p.MT * s_plan[p.E];
}

// ---------------------------------------------------------------------------- epilogues
// Column sums of a 32x32 block held one column per register: after 31 shuffles lane l holds the
// sum over the warp's lanes of column l.
__device__ __forceinline__ float sigmoid_fast(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

// two floats as a bf16 pair, rounded to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 pr = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&pr);
}

// load row[0..32) bf16 as 16 words (two tokens each); 0 beyond ncol or when !ok
__device__ __forceinline__ void load_row32(const __nv_bfloat16* row, bool ok, int ncol,
                                           uint32_t (&w)[16]) {
  const uint4* src = reinterpret_cast<const uint4*>(row);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 a = (ok && q * 8 < ncol) ? __ldg(src + q) : make_uint4(0, 0, 0, 0);
    w[4 * q] = a.x;
    w[4 * q + 1] = a.y;
    w[4 * q + 2] = a.z;
    w[4 * q + 3] = a.w;
  }
}

// Writes up to 32 rows of 32 bf16 tokens (16 words per row, the row held by one lane) with whole
// 32-byte sectors: each lane puts its row (staging row `srow`, or none when srow < 0) into the
// warp's shared staging area, then lane 4r + q writes the q-th 16 bytes of staging rows r, r + 8,
// ... to row_addr(row) (skipped when it returns null). The first `ncol` tokens are written (ncol a
// multiple of 8). The 80-byte pitch keeps both phases free of bank conflicts.
template <class RowAddr>
__device__ __forceinline__ void store_rows_staged(uint8_t* stage, int lane, int srow,
                                                  const uint32_t (&w)[16], int nrows, int ncol,
                                                  RowAddr row_addr) {
  if (srow >= 0) {
    uint4* d = reinterpret_cast<uint4*>(stage + srow * STAGE_PITCH);
#pragma unroll
    for (int q = 0; q < 4; ++q) d[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
  __syncwarp();
  const int r = lane >> 2, q = lane & 3;
#pragma unroll 1
  for (int r0 = 0; r0 < nrows; r0 += 8) {
    const int rr = r0 + r;
    if (rr < nrows && q * 8 < ncol) {
      __nv_bfloat16* dst = row_addr(rr);
      if (dst)
        *reinterpret_cast<uint4*>(dst + q * 8) =
            *reinterpret_cast<const uint4*>(stage + rr * STAGE_PITCH + q * 16);
    }
  }
  __syncwarp();
}

__device__ __forceinline__ float bf_at(const uint32_t (&a)[16], int j) {
  return (j & 1) ? __uint_as_float(a[j >> 1] & 0xFFFF0000u) : __uint_as_float(a[j >> 1] << 16);
}

// Per-warp inputs of a tile's epilogue that do not depend on the accumulator, loaded before the
// warp waits for it: for the warp's chunks c = 0..3 (columns (half + 2c) * 32 + lane) the slot,
// token and routing weight of the column, and for S6 the gate/up values of the first chunk.
struct EpiPre {
  int slot[4];
  int tok[4];
  float w[4];
  uint32_t hg[16], hu[16];
};

template <int VAR>
__device__ __forceinline__ void epi_prefetch(const Params& p, const Tile& ti, int row, int lane,
                                             int half, EpiPre& pre) {
  if constexpr (!VarTraits<VAR>::router) {
    const int nch = (ti.nrows + 31) / 32;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int ch = half + 2 * c;
      const int col = ch * 32 + lane;
      const bool in = ch < nch && col < ti.nrows;
      pre.slot[c] = in ? p.pslot[ti.row0 + col] : -1;
      pre.tok[c] = in && (VAR == V_DOWN || VAR == V_DX) ? p.ptok[ti.row0 + col] : 0;
      pre.w[c] = !in ? 0.f
                 : (VAR == V_GATEUP || VAR == V_GVEC) ? p.wperm[ti.row0 + col]
                 : (VAR == V_DX && p.dl_perm) ? p.dl_perm[ti.row0 + col]
                                               : 0.f;
    }
    if constexpr (VAR == V_GVEC) {
      const int i = ti.m0 + row;
      const int ncol = min(32, ti.nrows - half * 32);
      load_row32(p.hin + (int64_t)i * p.R_cap + ti.row0 + half * 32, i < p.I && half < nch, ncol,
                 pre.hg);
      load_row32(p.hin + (int64_t)(p.I + i) * p.R_cap + ti.row0 + half * 32,
                 i < p.I && half < nch, ncol, pre.hu);
    }
  }
}

template <int VAR>
__device__ __forceinline__ void epilogue(const Params& p, const Tile& ti, uint32_t taddr, int row,
                                         int lane, int half, EpiPre& pre, uint8_t* stage) {
  constexpr unsigned FULL = 0xffffffffu;
  const int H = p.H, I = p.I;
  const int nch = (ti.nrows + 31) / 32;
  if constexpr (VarTraits<VAR>::router) {
    const int e = ti.m0 + row;
    for (int ch = half; ch < nch; ch += 2) {
      float v[32];
      tmem_ld32(taddr + ch * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int tok = ti.row0 + ch * 32 + j;
        if (e < p.E && tok < p.T) p.acc_out[(int64_t)tok * p.E + e] = v[j];
      }
    }
    return;
  }
  uint32_t (&hg)[16] = pre.hg;  // V_GVEC: gate and up of the chunk being processed
  uint32_t (&hu)[16] = pre.hu;
  for (int ch = half; ch < nch; ch += 2) {
    const int cbase = ch * 32;
    // this chunk's column inputs, then the next chunk's moved up
    const int slot = pre.slot[0], tok = pre.tok[0];
    const float wl = pre.w[0];
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      pre.slot[c] = pre.slot[c + 1];
      pre.tok[c] = pre.tok[c + 1];
      pre.w[c] = pre.w[c + 1];
    }
    const int ncol = min(32, ti.nrows - cbase);
    if constexpr (VAR == V_GATEUP) {
      float v[32];
      tmem_ld32(taddr + ch * 32, v);
      const int i = ti.m0 + (row >> 1);
      const int g = row & 1;  // rows alternate gate (even lane) and up (odd lane) of feature i
      const int i0 = ti.m0 + ((row - lane) >> 1);  // feature of the warp's first row pair
      __nv_bfloat16* hbase = p.h + ti.row0 + cbase;
      uint32_t w16[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) w16[t] = pack_bf16x2(v[2 * t], v[2 * t + 1]);
      store_rows_staged(stage, lane, lane, w16, 32, ncol, [&](int rr) {
        return hbase + (int64_t)((rr & 1) * I + i0 + (rr >> 1)) * p.R_cap;
      });
      float wa[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float other = __shfl_xor_sync(FULL, v[j], 1);
        const float gate = g ? other : v[j], up = g ? v[j] : other;
        wa[j] = __shfl_sync(FULL, wl, j) * gate * sigmoid_fast(gate) * up;
      }
      // both lanes of the pair hold w*A of feature i; the even lane's row is stored
#pragma unroll
      for (int t = 0; t < 16; ++t) w16[t] = pack_bf16x2(wa[2 * t], wa[2 * t + 1]);
      __nv_bfloat16* wbase = p.wa + ti.row0 + cbase;
      store_rows_staged(stage, lane, g == 0 ? (lane >> 1) : -1, w16, 16, ncol, [&](int rr) {
        return wbase + (int64_t)(i0 + rr) * p.R_cap;
      });
      (void)i;
    } else if constexpr (VAR == V_DOWN || VAR == V_DX) {
      float v[32];
      tmem_ld32(taddr + ch * 32, v);
      // 4x4 transposes inside each group of four lanes: lane 4a + c then holds column j0 + c for
      // rows 4a .. 4a + 3 and adds them with one 16-byte vector atomic
      const int tokv = slot >= 0 ? tok : -1;  // the column's token, -1 for a padding row
      const int pc = lane & 3;
      const int hq = ti.m0 + row - lane + (lane & ~3);  // first of this lane's four rows
      // S8 with renormalised routing: the router's share of dx, dl of the column's slot times
      // Wr[e, h], joins the same atomic (rows hq .. hq + 3 of the expert's router row)
      const bool rterm = VAR == V_DX && p.dl_perm != nullptr && hq < H;
      const float4 wr4 = rterm ? __ldg(reinterpret_cast<const float4*>(
                                     p.w_router + (int64_t)ti.e * H + hq))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j0 = 0; j0 < 32; j0 += 4) {
        if (j0 >= ncol) break;
        float x0 = v[j0], x1 = v[j0 + 1], x2 = v[j0 + 2], x3 = v[j0 + 3];
        {
          const bool h2 = (pc & 2) != 0;
          const float b0 = __shfl_xor_sync(FULL, h2 ? x0 : x2, 2);
          const float b1 = __shfl_xor_sync(FULL, h2 ? x1 : x3, 2);
          if (h2) {
            x0 = b0;
            x1 = b1;
          } else {
            x2 = b0;
            x3 = b1;
          }
        }
        {
          const bool h1 = (pc & 1) != 0;
          const float d0 = __shfl_xor_sync(FULL, h1 ? x0 : x1, 1);
          const float d1 = __shfl_xor_sync(FULL, h1 ? x2 : x3, 1);
          if (h1) {
            x0 = d0;
            x2 = d1;
          } else {
            x1 = d0;
            x3 = d1;
          }
        }
        const int tj = __shfl_sync(FULL, tokv, j0 + pc);
        if (rterm) {
          const float dj = __shfl_sync(FULL, wl, j0 + pc);
          x0 = fmaf(dj, wr4.x, x0);
          x1 = fmaf(dj, wr4.y, x1);
          x2 = fmaf(dj, wr4.z, x2);
          x3 = fmaf(dj, wr4.w, x3);
        }
        if (tj >= 0 && hq < H)
          atomicAdd(reinterpret_cast<float4*>(&p.acc_out[(int64_t)tj * H + hq]),
                    make_float4(x0, x1, x2, x3));
      }
    } else {  // V_GVEC: SwiGLU backward, dh^T and the routing-weight gradient dw
      const int i = ti.m0 + row;
      const bool iv = i < I;
      uint32_t ng[16], nu[16];
      if (ch + 2 < nch) {  // next chunk of gate/up in flight during this one
        const int nc = min(32, ti.nrows - (ch + 2) * 32);
        load_row32(p.hin + (int64_t)i * p.R_cap + ti.row0 + cbase + 64, iv, nc, ng);
        load_row32(p.hin + (int64_t)(I + i) * p.R_cap + ti.row0 + cbase + 64, iv, nc, nu);
      }
      float v[32];
      tmem_ld32(taddr + ch * 32, v);
      uint32_t pg[16], pu[16];  // dgate, dup of two tokens per word
#pragma unroll
      for (int j2 = 0; j2 < 16; ++j2) {
        float dgv[2], duv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int j = 2 * j2 + u;
          const float wj = __shfl_sync(FULL, wl, j);
          const float gt = bf_at(hg, j), ut = bf_at(hu, j);
          const float s = sigmoid_fast(gt);
          const float sg = gt * s;
          const float dA = wj * v[j];
          dgv[u] = dA * ut * s * (1.f + gt * (1.f - s));
          duv[u] = dA * sg;
          v[j] = v[j] * sg * ut;
        }
        pg[j2] = pack_bf16x2(dgv[0], dgv[1]);
        pu[j2] = pack_bf16x2(duv[0], duv[1]);
      }
      {
        const int ib = ti.m0 + row - lane;  // feature of the warp's first row
        __nv_bfloat16* dbase = p.dh + ti.row0 + cbase;
        store_rows_staged(stage, lane, lane, pg, 32, ncol, [&](int rr) -> __nv_bfloat16* {
          return ib + rr < I ? dbase + (int64_t)(ib + rr) * p.R_cap : nullptr;
        });
        store_rows_staged(stage, lane, lane, pu, 32, ncol, [&](int rr) -> __nv_bfloat16* {
          return ib + rr < I ? dbase + (int64_t)(I + ib + rr) * p.R_cap : nullptr;
        });
      }
      // this warp's 32 rows of the tile: one partial per (M tile, row quarter, slot), summed
      // in a fixed order later, so dw does not depend on which tile finished first
      const float dwsum = transpose_reduce32(v, lane);
      if (slot >= 0)
        p.dw_part[((int64_t)(ti.m0 / BM) * 4 + (row >> 5)) * p.n_slots + slot] = dwsum;
      if (ch + 2 < nch) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          hg[j] = ng[j];
          hu[j] = nu[j];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------- the kernel
template <int VAR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain[1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_plan = reinterpret_cast<int32_t*>(smem + STAGES * STAGE_BYTES + 256);
  int32_t* s_off = s_plan + (MAX_E + 1);
  uint8_t* epi_stage = smem + STAGES * STAGE_BYTES + PLAN_BYTES;  // EPI_WARPS x EPI_STAGE_BYTES

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES, tempty0 = tfull0 + 16, drain = tempty0 + 16;

  if constexpr (!VarTraits<VAR>::router) {
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
      s_off[i] = p.off[i];
      s_plan[i] = p.plan[i];
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = total_tiles<VAR>(p, s_plan);
  bool failed = false;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
        const Tile ti = get_tile<VAR>(p, s_plan, s_off, t);
        const int nkb = (ti.klen + BK - 1) / BK;
        const int nbox = VarTraits<VAR>::router ? 0 : (ti.nrows + 63) / 64;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) {
            failed = true;
            break;
          }
          const uint32_t a_dst = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_dst = a_dst + A_BYTES;
          const uint32_t fb = full0 + 8 * stage;
          const int k0 = kb * BK;
          if constexpr (VarTraits<VAR>::router) {
            mbar_expect_tx(fb, A_BYTES + ROUTER_BN * BK * 2);
            tma_2d(a_dst, &tmA, fb, k0, ti.m0);
            tma_2d(b_dst, &tmB, fb, k0 % p.H, ti.row0);  // x, once for each part of Wr
          } else {
            mbar_expect_tx(fb, A_BYTES + nbox * B_BOX);
            if constexpr (VAR == V_GATEUP) {
              tma_4d(a_dst, &tmA, fb, k0, 0, ti.m0, ti.e);
            } else if constexpr (VAR == V_DOWN) {
              tma_2d(a_dst, &tmA, fb, k0, ti.e * p.H + ti.m0);
            } else if constexpr (VAR == V_GVEC) {
              tma_2d(a_dst, &tmA, fb, ti.m0, ti.e * p.H + k0);
              tma_2d(a_dst + 8192, &tmA, fb, ti.m0 + 64, ti.e * p.H + k0);
            } else {  // V_DX
              tma_2d(a_dst, &tmA, fb, ti.m0, ti.e * 2 * p.I + k0);
              tma_2d(a_dst + 8192, &tmA, fb, ti.m0 + 64, ti.e * 2 * p.I + k0);
            }
            // B: feature-major tokens, boxes of 64 tokens x 64 k (MN-major, 8 KB apart)
            for (int q = 0; q < nbox; ++q) tma_2d(b_dst + q * B_BOX, &tmB, fb, ti.row0 + 64 * q, k0);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (failed) {
        *abort_flag = 1;
        flag_status(p.status, USAF_DEV_TIMEOUT);
      }
      // let every issued copy land before the CTA can exit or reuse its shared memory
      const long long deadline = clock64() + TIMEOUT_CYCLES;
      for (int s = 0; s < STAGES && (uint32_t)s < issued; ++s) {
        const uint32_t last = issued - 1 - ((issued - 1 - s) % STAGES);
        mbar_drain(full0 + 8 * s, (last / STAGES) & 1, deadline);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      constexpr bool a_mn = VarTraits<VAR>::a_mn;
      constexpr bool b_mn = !VarTraits<VAR>::router;
      const uint32_t a_step = a_mn ? 2048 : 32, b_step = b_mn ? 2048 : 32;
      const uint32_t a_lbo = a_mn ? 8192 : 16, b_lbo = b_mn ? B_BOX : 16;
      // the operand descriptors of stage 0: a stage or k-step moves only their start-address
      // field (16-byte units, no carry within the CTA's shared memory)
      const uint64_t ad0 = sdesc(smem_u32(smem), a_lbo, 1024);
      const uint64_t bd0 = sdesc(smem_u32(smem) + A_BYTES, b_lbo, 1024);
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
        const Tile ti = get_tile<VAR>(p, s_plan, s_off, t);
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        const uint32_t idesc = idesc_bf16(ti.nrows, a_mn, b_mn);
        const int nkb = (ti.klen + BK - 1) / BK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)((stage * STAGE_BYTES) >> 4);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            umma_bf16(d, ad0 + so + ((ks * a_step) >> 4), bd0 + so + ((ks * b_step) >> 4), idesc,
                      (kb | ks) != 0 ? 1u : 0u);
          umma_commit(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (failed) break;
        umma_commit(tfull0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (failed) {
        *abort_flag = 1;
        flag_status(p.status, USAF_DEV_TIMEOUT);
      }
      // wait for every MMA this thread issued before TMEM is released
      umma_commit(drain);
      mbar_drain(drain, 0, clock64() + TIMEOUT_CYCLES);
    }
  } else {
    // -------------------------------------------------------------- epilogue warps 2..9
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile ti = get_tile<VAR>(p, s_plan, s_off, t);
      EpiPre pre;
      epi_prefetch<VAR>(p, ti, row, lane, half, pre);
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag) ? 1 : 0;
        if (!ok) {
          *abort_flag = 1;
          flag_status(p.status, USAF_DEV_TIMEOUT);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      epilogue<VAR>(p, ti, tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN, row, lane, half,
                    pre, epi_stage + (warp - 2) * EPI_STAGE_BYTES);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------- CTA pairs
// The expert GEMMs on pairs of SMs (tcgen05 cta_group::2): a tile is 256 weight rows by up to 256
// tokens. Each CTA of the pair loads its own 128 weight rows and half of the token tile into its
// shared memory; the pair's MMA (issued by the even CTA) reads both CTAs' halves and leaves each
// CTA's 128 rows x all tokens in that CTA's tensor memory, so each epilogue is the single-CTA one
// over its own rows. A stage is 32 KB per SM instead of 48 KB (the token tile is split, not
// copied), so six stages are in flight instead of four, and the MMA reads 8 KB of shared memory
// per 16-deep step instead of 12 KB.
// - full[s]: in the even CTA only, expecting both CTAs' bytes (the odd CTA's copies signal it);
// - empty[s]: in both CTAs, arrived by the pair's MMA commit (multicast);
// - tfull[a]: in both CTAs, arrived by the MMA commit (multicast) when accumulator a is complete;
// - tempty[a]: in the even CTA, arrived by the 16 epilogue warps of both CTAs.
// Every wait is bounded as in the single-CTA kernel; a role that gives up also raises the other
// CTA's abort flag.
namespace pr {
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;        // this CTA's 128 weight rows
constexpr int B_BYTES = (BN / 2) * BK * 2;  // this CTA's half of the token tile
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + PLAN_BYTES + EPI_WARPS * EPI_STAGE_BYTES;
static_assert(SMEM <= 232448, "shared memory of the CTA-pair kernel");
static_assert(2 * STAGES + 5 <= 30, "barrier area");
}  // namespace pr

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// address of the same shared variable in CTA 0 of the cluster
__device__ __forceinline__ uint32_t map_to_cta0(uint32_t a) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void tma_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_4d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                               uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// arrive on barrier `bar` (same offset) in both CTAs when this thread's MMAs are complete
__device__ __forceinline__ void umma_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void umma_commit_local_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// The epilogue's release of an accumulator buffer to the pair's MMA thread. Relaxed: what the MMA
// must not overtake are this warp's tensor-memory reads, which have completed into registers
// (tcgen05.wait::ld) and are ordered by the tcgen05 fences around the barrier; a release would
// also wait for the warp's global stores and reductions, which nothing on the MMA side reads.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   bar_cluster_addr)
               : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// the other CTA of the pair
__device__ __forceinline__ uint32_t map_to_peer(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank ^ 1u));
  return r;
}

// Instruction descriptor, kind::f16, for the pair's M = 256.
__device__ __forceinline__ uint32_t idesc_bf16_m256(int n, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}

// Pair tile t of CTA `rank`: the pair covers M tiles 2 mt and 2 mt + 1 of the single-CTA plan.
template <int VAR>
__device__ __forceinline__ Tile get_tile_pair(const Params& p, const int32_t* s_plan,
                                              const int32_t* s_off, int t, uint32_t rank) {
  const int MTp = p.MT / 2;
  const int e = upper_bound_i32(s_plan, p.E + 1, t / MTp) - 1;
  const int nts = s_plan[e + 1] - s_plan[e];
  const int local = t - MTp * s_plan[e];
  const int mt = 2 * (local / nts) + (int)rank, nt = local % nts;
  return get_tile<VAR>(p, s_plan, s_off, p.MT * s_plan[e] + mt * nts + nt);
}

template <int VAR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const Params p) {
  static_assert(!VarTraits<VAR>::router, "the router GEMM runs on single CTAs");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pr::STAGES * pr::STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain[1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * pr::STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_plan = reinterpret_cast<int32_t*>(smem + pr::STAGES * pr::STAGE_BYTES + 256);
  int32_t* s_off = s_plan + (MAX_E + 1);
  uint8_t* epi_stage = smem + pr::STAGES * pr::STAGE_BYTES + PLAN_BYTES;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_rank();
  const bool even = rank == 0;
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * pr::STAGES;
  const uint32_t tfull0 = empty0 + 8 * pr::STAGES, tempty0 = tfull0 + 16, drain = tempty0 + 16;
  const uint32_t peer_abort = map_to_peer(smem_u32((const void*)abort_flag), rank);
  auto give_up = [&]() {
    *abort_flag = 1;
    st_cluster_u32(peer_abort, 1u);
    flag_status(p.status, USAF_DEV_TIMEOUT);
  };

  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
    s_off[i] = p.off[i];
    s_plan[i] = p.plan[i];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < pr::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 2 * EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA allocates, together, the same columns in both
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // both CTAs' barriers and abort flags are initialised
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = (p.MT / 2) * s_plan[p.E];
  const int npairs = (int)(gridDim.x / 2), pair0 = (int)(blockIdx.x / 2);
  bool failed = false;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      const uint32_t full_even0 = even ? full0 : map_to_cta0(full0);
      for (int t = pair0; t < total && !failed; t += npairs) {
        const Tile ti = get_tile_pair<VAR>(p, s_plan, s_off, t, rank);
        const int nkb = (ti.klen + BK - 1) / BK;
        const int half = ti.nrows / 2;  // a multiple of 8
        const int nbox = (half + 63) / 64;
        const int tok0 = ti.row0 + (int)rank * half;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) {
            failed = true;
            break;
          }
          const uint32_t a_dst = smem_u32(smem + stage * pr::STAGE_BYTES);
          const uint32_t b_dst = a_dst + pr::A_BYTES;
          const uint32_t fb = full_even0 + 8 * stage;
          const int k0 = kb * BK;
          if (even) mbar_expect_tx(full0 + 8 * stage, 2 * (pr::A_BYTES + nbox * B_BOX));
          if constexpr (VAR == V_GATEUP) {
            tma_4d_pair(a_dst, &tmA, fb, k0, 0, ti.m0, ti.e);
          } else if constexpr (VAR == V_DOWN) {
            tma_2d_pair(a_dst, &tmA, fb, k0, ti.e * p.H + ti.m0);
          } else if constexpr (VAR == V_GVEC) {
            tma_2d_pair(a_dst, &tmA, fb, ti.m0, ti.e * p.H + k0);
            tma_2d_pair(a_dst + 8192, &tmA, fb, ti.m0 + 64, ti.e * p.H + k0);
          } else {  // V_DX
            tma_2d_pair(a_dst, &tmA, fb, ti.m0, ti.e * 2 * p.I + k0);
            tma_2d_pair(a_dst + 8192, &tmA, fb, ti.m0 + 64, ti.e * 2 * p.I + k0);
          }
          for (int q = 0; q < nbox; ++q) tma_2d_pair(b_dst + q * B_BOX, &tmB, fb, tok0 + 64 * q, k0);
          ++issued;
          if (++stage == pr::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (failed) give_up();
      // the even CTA's full barriers complete when both CTAs' copies of a stage have landed
      if (even) {
        const long long deadline = clock64() + TIMEOUT_CYCLES;
        for (int s = 0; s < pr::STAGES && (uint32_t)s < issued; ++s) {
          const uint32_t last = issued - 1 - ((issued - 1 - s) % pr::STAGES);
          mbar_drain(full0 + 8 * s, (last / pr::STAGES) & 1, deadline);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && even) {
      // ------------------------------------------------------------ MMA issuer (even CTA)
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      constexpr bool a_mn = VarTraits<VAR>::a_mn;
      const uint32_t a_step = a_mn ? 2048 : 32, b_step = 2048;
      const uint32_t a_lbo = a_mn ? 8192 : 16, b_lbo = B_BOX;
      const uint64_t ad0 = sdesc(smem_u32(smem), a_lbo, 1024);
      const uint64_t bd0 = sdesc(smem_u32(smem) + pr::A_BYTES, b_lbo, 1024);
      for (int t = pair0; t < total && !failed; t += npairs) {
        const Tile ti = get_tile_pair<VAR>(p, s_plan, s_off, t, rank);
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        const uint32_t idesc = idesc_bf16_m256(ti.nrows, a_mn, true);
        const int nkb = (ti.klen + BK - 1) / BK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)((stage * pr::STAGE_BYTES) >> 4);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            umma_bf16_pair(d, ad0 + so + ((ks * a_step) >> 4), bd0 + so + ((ks * b_step) >> 4),
                           idesc, (kb | ks) != 0 ? 1u : 0u);
          umma_commit_both(empty0 + 8 * stage);
          if (++stage == pr::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (failed) break;
        umma_commit_both(tfull0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (failed) give_up();
      // every MMA this thread issued completes before either CTA releases tensor memory
      umma_commit_local_pair(drain);
      mbar_drain(drain, 0, clock64() + TIMEOUT_CYCLES);
    }
  } else {
    // -------------------------------------------------------------- epilogue warps 2..9
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const uint32_t tempty_even0 = even ? tempty0 : map_to_cta0(tempty0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair0; t < total; t += npairs) {
      const Tile ti = get_tile_pair<VAR>(p, s_plan, s_off, t, rank);
      EpiPre pre;
      epi_prefetch<VAR>(p, ti, row, lane, half, pre);
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag) ? 1 : 0;
        if (!ok) give_up();
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      epilogue<VAR>(p, ti, tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN, row, lane, half,
                    pre, epi_stage + (warp - 2) * EPI_STAGE_BYTES);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_even0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // the pair's MMAs are complete and neither CTA reads the other any more
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------- dense weight gradient
// Dense expert weight gradient for the importance phase (the whole |g| is ranked there):
//   gate_up[e]:  G[j, c] = sum over the expert's tokens of dh^T[j, t] x^T[c, t]      (2I x H)
//   down[e]:     G[h, c] = sum over the expert's tokens of dy^T[h, t] (wA)^T[c, t]   (H x I)
// Both operands are feature-major rows with the tokens contiguous, so both are K-major with
// K = the expert's padded token count (its last k-block issues only the 16-token steps inside
// the expert). A tile is (expert, 128 rows, 256 columns); the fp32 accumulator goes out through a
// per-warp swizzled shared staging buffer and a TMA tensor store, or a TMA add-reduction when the
// gradient accumulates over micro-batches. Padding tokens hold zeros in both operands.
namespace wg {
constexpr int STAGES = 3;
constexpr int A_BYTES = 128 * BK * 2;
constexpr int B_BYTES = 256 * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int OUT_BYTES = 32 * 128;  // one 32 x 32 fp32 box, 128-byte swizzled rows
constexpr int SMEM = STAGES * STAGE_BYTES + EPI_WARPS * 2 * OUT_BYTES + 1024 + 256;
static_assert(SMEM <= 232448, "shared memory of the dense gradient kernel");
}  // namespace wg

struct WgParams {
  const int32_t* off;  // expert offsets of the permuted rows
  int E, M, N;         // rows and columns of one expert's gradient
  int MT, NT;          // tiles per expert along M (128) and N (256)
  int accumulate;      // 1: add into the output (TMA reduce), 0: overwrite (TMA store)
  uint32_t* status;
  // gather form (the gradient is wanted only at the active entries of some experts):
  const int32_t* dlist;   // the experts to form, dlist[0 .. *n_list)
  const int32_t* n_list;
  const int64_t* row_ptr;  // per expert [rp_stride]: first active entry of each row
  int64_t rp_stride;
  int rp_off;              // this tensor's first row in row_ptr (0 gate_up, 2I down)
  const int64_t* act;      // the sorted active set
  int64_t flat0;           // flat index of this tensor's entry (0, 0, 0)
  float* g_act;            // gradient at the active entries
};

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2, int add) {
  if (add)
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::
            "l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// GATHER = true: the tiles of the experts in p.dlist only, and the epilogue writes the
// accumulator at the active entries (g_act) instead of storing the tile: each lane walks its
// row's active entries from row_ptr, the entries of a 32-column chunk taken in column order.
template <bool GATHER>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmO, const WgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* outbuf = smem + wg::STAGES * wg::STAGE_BYTES;  // 1024-aligned: 64 KB, 8 warps x 2
  uint64_t* bars = reinterpret_cast<uint64_t*>(outbuf + EPI_WARPS * 2 * wg::OUT_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * wg::STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * wg::STAGES;
  const uint32_t tfull0 = empty0 + 8 * wg::STAGES, tempty0 = tfull0 + 16, drain = tempty0 + 16;
  if (threadIdx.x == 0) {
    for (int s = 0; s < wg::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int per_e = p.MT * p.NT;
  const int total = (GATHER ? *p.n_list : p.E) * per_e;
  auto expert_of = [&](int t) { return GATHER ? p.dlist[t / per_e] : t / per_e; };
  bool failed = false;
  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
        const int e = expert_of(t), r = t % per_e, mt = r / p.NT, nt = r % p.NT;
        const int o = p.off[e], npad = p.off[e + 1] - o;
        const int nkb = (npad + BK - 1) / BK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) {
            failed = true;
            break;
          }
          const uint32_t a_dst = smem_u32(smem + stage * wg::STAGE_BYTES);
          const uint32_t fb = full0 + 8 * stage;
          mbar_expect_tx(fb, wg::STAGE_BYTES);
          tma_2d(a_dst, &tmA, fb, o + kb * BK, mt * 128);
          tma_2d(a_dst + wg::A_BYTES, &tmB, fb, o + kb * BK, nt * 256);
          ++issued;
          if (++stage == wg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (failed) {
        *abort_flag = 1;
        flag_status(p.status, USAF_DEV_TIMEOUT);
      }
      const long long deadline = clock64() + TIMEOUT_CYCLES;
      for (int s = 0; s < wg::STAGES && (uint32_t)s < issued; ++s) {
        const uint32_t last = issued - 1 - ((issued - 1 - s) % wg::STAGES);
        mbar_drain(full0 + 8 * s, (last / wg::STAGES) & 1, deadline);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      const uint32_t idesc = idesc_bf16(256, false, false);
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
        const int e = expert_of(t);
        const int npad = p.off[e + 1] - p.off[e];
        const int nkb = (npad + BK - 1) / BK;
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * 256;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * wg::STAGE_BYTES);
          const uint32_t b_base = a_base + wg::A_BYTES;
          const int nks = min(BK, npad - kb * BK) / 16;  // 16-token steps inside the expert
          for (int ks = 0; ks < nks; ++ks)
            umma_bf16(d, sdesc(a_base + ks * 32, 16, 1024), sdesc(b_base + ks * 32, 16, 1024),
                      idesc, (kb | ks) != 0 ? 1u : 0u);
          umma_commit(empty0 + 8 * stage);
          if (++stage == wg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (failed) break;
        umma_commit(tfull0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (failed) {
        *abort_flag = 1;
        flag_status(p.status, USAF_DEV_TIMEOUT);
      }
      umma_commit(drain);
      mbar_drain(drain, 0, clock64() + TIMEOUT_CYCLES);
    }
  } else {
    // -------------------------------------------------------------- epilogue warps 2..9
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* ob = outbuf + (warp - 2) * 2 * wg::OUT_BYTES;
    int acc = 0, nstore = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const int e = expert_of(t), r = t % per_e, mt = r / p.NT, nt = r % p.NT;
      const bool empty = p.off[e + 1] == p.off[e];
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag) ? 1 : 0;
        if (!ok) {
          *abort_flag = 1;
          flag_status(p.status, USAF_DEV_TIMEOUT);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256;
      if constexpr (GATHER) {
        // this lane's row of the tile and its active entries, walked chunk by chunk
        const int row = mt * 128 + q * 32 + lane;
        const bool live = row < p.M;
        const int64_t* rp = p.row_ptr + (int64_t)e * p.rp_stride + p.rp_off;
        int64_t ptr = live ? rp[row] : 0, end = live ? rp[row + 1] : 0;
        const int64_t rbase = p.flat0 + ((int64_t)e * p.M + row) * p.N;
        for (int ch = half; ch < 8; ch += 2) {
          const int c0 = nt * 256 + ch * 32;
          if (c0 >= p.N || mt * 128 + q * 32 >= p.M) continue;
          const int64_t fb = rbase + c0;  // flat index of (row, c0)
          while (ptr < end && p.act[ptr] < fb) ++ptr;  // entries of the other half's chunks
          int64_t f = ptr < end ? p.act[ptr] : INT64_MAX;
          if (!__any_sync(0xffffffffu, f < fb + 32)) continue;  // no entry in this chunk
          float v[32];
          if (!empty) {
            tmem_ld32(taddr + ch * 32, v);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (f == fb + j) {
              p.g_act[ptr] = p.accumulate ? p.g_act[ptr] + v[j] : v[j];
              ++ptr;
              f = ptr < end ? p.act[ptr] : INT64_MAX;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
        continue;
      }
      for (int ch = half; ch < 8; ch += 2) {
        const int c0 = nt * 256 + ch * 32;
        const int r0 = mt * 128 + q * 32;
        // boxes starting past the gradient's last row or column are not issued at all
        if (c0 >= p.N || r0 >= p.M || (empty && p.accumulate)) continue;
        float v[32];
        if (!empty) {
          tmem_ld32(taddr + ch * 32, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        uint8_t* buf = ob + (nstore & 1) * wg::OUT_BYTES;
        // the store issued from this buffer two chunks ago must have read it
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncwarp();
        uint4* row = reinterpret_cast<uint4*>(buf + lane * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          row[c ^ (lane & 7)] = make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                                           __float_as_uint(v[4 * c + 2]),
                                           __float_as_uint(v[4 * c + 3]));
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tmO, smem_u32(buf), c0, r0, e, p.accumulate);
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        ++nstore;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// Router weight split for the tensor-core logits: w = hi + mid + lo, each part bf16 and each
// residual exact in fp32, so x . w is carried by three bf16 products with fp32 accumulation.
__global__ void router_split_kernel(const float* __restrict__ wr, int H,
                                    __nv_bfloat16* __restrict__ wr3) {
  // block row e of Wr, two columns per thread (H is a multiple of 64 on this path)
  const int e = blockIdx.y;
  const float* src = wr + (int64_t)e * H;
  __nv_bfloat16* row = wr3 + (int64_t)e * 3 * H;
  for (int k = (blockIdx.x * blockDim.x + threadIdx.x) * 2; k < H; k += gridDim.x * blockDim.x * 2) {
    const float2 w = *reinterpret_cast<const float2*>(src + k);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(w.x, w.y);
    const float2 hf = __bfloat1622float2(hi);
    const float2 r1 = make_float2(w.x - hf.x, w.y - hf.y);
    const __nv_bfloat162 mid = __floats2bfloat162_rn(r1.x, r1.y);
    const float2 mf = __bfloat1622float2(mid);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(r1.x - mf.x, r1.y - mf.y);
    *reinterpret_cast<__nv_bfloat162*>(row + k) = hi;
    *reinterpret_cast<__nv_bfloat162*>(row + H + k) = mid;
    *reinterpret_cast<__nv_bfloat162*>(row + 2 * H + k) = lo;
  }
}

// ---------------------------------------------------------------------------- router, K split
// logits^T tile (128 experts x RK_N tokens) with the 3H / 64 k-blocks cut among the RK_SPLIT CTAs of
// a cluster. A tcgen05 MMA costs about the same at N = 32 as at N = 256, so a long K loop over
// narrow token tiles leaves the tensor pipe mostly idle; here every CTA runs wide MMAs over a
// fraction of the K range. (Clusters of four fit 36 times on a 152-SM part at this shared-memory
// size, clusters of eight only 15 times.) Each CTA leaves its partial tile in its shared memory (the ring, free
// once the MMAs are done); after a cluster barrier CTA r adds the RK_SPLIT partials of tokens
// [r RK_N / RK_SPLIT, (r + 1) RK_N / RK_SPLIT) in split order through distributed shared memory
// and writes those logits.
// The sum order is fixed, so the logits do not depend on timing.
constexpr int RK_SPLIT = 4;                  // CTAs per cluster = K splits
constexpr int RK_N = 128;                    // tokens per tile
constexpr int RK_B_BYTES = RK_N * BK * 2;    // x box: RK_N tokens x 64 k (K-major)
constexpr int RK_STAGE_BYTES = A_BYTES + RK_B_BYTES;
constexpr int RK_STAGES = STAGES * STAGE_BYTES / RK_STAGE_BYTES;  // the ring of the expert GEMMs
static_assert(RK_STAGES >= 2 && (2 * RK_STAGES + 1) * 8 + 8 <= 256, "router ring barriers");
constexpr int RK_EPI_WARPS = 4;
constexpr int RK_THREADS = 64 + 32 * RK_EPI_WARPS;
constexpr int RK_PART_PITCH = BM + 4;        // floats per token row of a partial tile
constexpr int RK_SMEM_BYTES = RK_STAGES * RK_STAGE_BYTES + 1024 + 256;
static_assert(RK_N * RK_PART_PITCH * 4 <= RK_STAGES * RK_STAGE_BYTES, "partial tile in the ring");
static_assert(RK_N % RK_SPLIT == 0 && (RK_N / RK_SPLIT) % 4 == 0, "token slices of the reduction");

__device__ __forceinline__ uint32_t peer_smem(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_peer_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// grid (RK_SPLIT * token tiles, expert tiles), clusters of RK_SPLIT along x
__global__ void __launch_bounds__(RK_THREADS, 1)
    tc_router_split_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, int T, int E, int H,
                           float* __restrict__ logits, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RK_STAGES * RK_STAGE_BYTES);
  // bars: full[RK_STAGES], empty[RK_STAGES], tfull
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * RK_STAGES + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* part = reinterpret_cast<float*>(smem);  // [RK_N][RK_PART_PITCH] after the MMAs
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * RK_STAGES;
  const uint32_t tfull = empty0 + 8 * RK_STAGES;
  const uint32_t rank = cluster_rank();
  const int n0 = (blockIdx.x / RK_SPLIT) * RK_N, m0 = blockIdx.y * BM;
  const int nrows = min(RK_N, (T - n0 + 15) / 16 * 16);
  const int nkb_all = 3 * H / BK;
  const int kb0 = (int)rank * nkb_all / RK_SPLIT, kb1 = ((int)rank + 1) * nkb_all / RK_SPLIT;
  const int nkb = kb1 - kb0;  // may be 0 for a short K: the partial is then zero

  if (threadIdx.x == 0) {
    for (int s = 0; s < RK_STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(RK_N)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  bool failed = false;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------------ TMA producer
      uint32_t issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % RK_STAGES;
        if (!mbar_wait(empty0 + 8 * s, ((kb / RK_STAGES) & 1) ^ 1, abort_flag)) {
          failed = true;
          break;
        }
        const uint32_t a_dst = smem_u32(smem + s * RK_STAGE_BYTES);
        const uint32_t fb = full0 + 8 * s;
        const int k0 = (kb0 + kb) * BK;
        mbar_expect_tx(fb, RK_STAGE_BYTES);
        tma_2d(a_dst, &tmA, fb, k0, m0);
        tma_2d(a_dst + A_BYTES, &tmB, fb, k0 % H, n0);  // x, once for each part of Wr
        ++issued;
      }
      if (failed) *abort_flag = 1;
      // let every issued copy land before the CTA can move on
      const long long deadline = clock64() + TIMEOUT_CYCLES;
      for (int s = 0; s < RK_STAGES && (uint32_t)s < issued; ++s) {
        const uint32_t last = issued - 1 - ((issued - 1 - s) % RK_STAGES);
        mbar_drain(full0 + 8 * s, (last / RK_STAGES) & 1, deadline);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA issuer
      const uint64_t ad0 = sdesc(smem_u32(smem), 16, 1024);
      const uint64_t bd0 = sdesc(smem_u32(smem) + A_BYTES, 16, 1024);
      const uint32_t idesc = idesc_bf16(nrows, false, false);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % RK_STAGES;
        if (!mbar_wait(full0 + 8 * s, (kb / RK_STAGES) & 1, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint64_t so = (uint64_t)((s * RK_STAGE_BYTES) >> 4);
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks)
          umma_bf16(tmem_base, ad0 + so + ((ks * 32) >> 4), bd0 + so + ((ks * 32) >> 4), idesc,
                    (kb | ks) != 0 ? 1u : 0u);
        umma_commit(empty0 + 8 * s);
      }
      if (failed) *abort_flag = 1;
      umma_commit(tfull);  // after every MMA above (at once when there were none)
      // no MMA in flight when TMEM and the ring are reused
      mbar_drain(tfull, 0, clock64() + TIMEOUT_CYCLES);
    }
  } else {  // ---------------------------------------------------- epilogue warps 2..5
    const int q = warp & 3;  // TMEM lane quarter: experts m0 + 32 q + lane
    int ok = 1;
    if (lane == 0) {
      ok = mbar_wait(tfull, 0, abort_flag) ? 1 : 0;
      if (!ok) *abort_flag = 1;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      tc_fence_after();
      const int e = q * 32 + lane;
      for (int ch = 0; ch * 32 < nrows; ++ch) {
        float v[32];
        if (nkb > 0) {
          tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + ch * 32, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) part[(ch * 32 + j) * RK_PART_PITCH + e] = v[j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag_status(status, USAF_DEV_TIMEOUT);
  cluster_barrier();  // every CTA's partial (or its failure flag) is in its shared memory
  // a CTA that gave up left no partial: the cluster then writes none of the tile's logits
  uint32_t peer_failed = 0;
  for (uint32_t r = 0; r < RK_SPLIT; ++r)
    peer_failed |= ld_peer_u32(peer_smem(smem_u32((const void*)abort_flag), r));
  if (!peer_failed) {
    // this CTA's tokens of the tile, all experts of the tile, float4 at a time
    constexpr int TOK = RK_N / RK_SPLIT;
    const uint32_t base = smem_u32(part);
    const bool vec = (E & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
    for (int i = threadIdx.x; i < TOK * (BM / 4); i += RK_THREADS) {
      const int t = (int)rank * TOK + i / (BM / 4), e4 = (i % (BM / 4)) * 4;
      const int tok = n0 + t;
      if (tok >= T || t >= nrows) continue;
      const uint32_t off = (uint32_t)((t * RK_PART_PITCH + e4) * 4);
      float4 acc = ld_peer_f4(peer_smem(base + off, 0));
#pragma unroll
      for (int r = 1; r < RK_SPLIT; ++r) {
        const float4 w = ld_peer_f4(peer_smem(base + off, (uint32_t)r));
        acc.x += w.x;
        acc.y += w.y;
        acc.z += w.z;
        acc.w += w.w;
      }
      float* dst = logits + (int64_t)tok * E + m0 + e4;
      if (vec && m0 + e4 + 3 < E) {
        *reinterpret_cast<float4*>(dst) = acc;
      } else {
        const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
        for (int j = 0; j < 4 && m0 + e4 + j < E; ++j) dst[j] = a4[j];
      }
    }
  }
  cluster_barrier();  // no peer reads this CTA's shared memory any more
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(RK_N)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------- bounded-wait check
// The failure path of the kernels above, run on purpose and without any fault: one CTA takes
// tensor memory, waits on an mbarrier that nothing arrives on through the same bounded wait
// (limited to `limit` cycles instead of about two seconds), records the timeout, drains its MMA
// pipeline (nothing was issued, so the commit completes at once) and frees the tensor memory.
__global__ void __launch_bounds__(64, 1) diag_wait_kernel(long long limit, uint32_t* status) {
  __shared__ __align__(8) uint64_t bars[2];  // never-arriving barrier, drain
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t never = smem_u32(&bars[0]), drain = smem_u32(&bars[1]);
  if (threadIdx.x == 0) {
    mbar_init(never, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(32)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  if (warp == 0 && lane == 0) {
    if (!mbar_wait(never, 0, abort_flag, limit)) {
      *abort_flag = 1;
      flag_status(status, USAF_DEV_TIMEOUT);
    }
  } else if (warp == 1 && lane == 0) {
    umma_commit(drain);
    mbar_drain(drain, 0, clock64() + limit);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(32)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool map_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
            uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// gate_up_proj [E, 2I, H] viewed as (h, gate|up, i, e) so a 128-row box interleaves gate row i
// and up row i (rows 2i and 2i+1 of the tile).
bool map_gate_up_interleaved(CUtensorMap* m, const void* base, uint64_t E, uint64_t I,
                             uint64_t H) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {H, 2, I, E};
  cuuint64_t strides[3] = {I * H * 2, H * 2, 2 * I * H * 2};
  cuuint32_t box[4] = {64, 2, 64, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// feature-major token operand [rows = K features, cols = R_cap tokens], boxes of 64 x 64
bool map_tokens(CUtensorMap* m, const void* base, uint64_t features, uint64_t R_cap) {
  return map_2d(m, base, R_cap, features, 64, 64);
}

constexpr const char* VAR_NAME[5] = {"tc_gate_up_swiglu", "tc_down_combine", "tc_gvec_swiglu_bwd",
                                     "tc_dx", "tc_router_logits"};

// The CTA-pair kernel where the M tiles pair up (an even count of 128-row tiles); the
// single-CTA kernel otherwise.
template <int VAR>
usaf_status launch_pair(const CUtensorMap& a, const CUtensorMap& b, const Params& p,
                        cudaStream_t st) {
  USAF_TRACE(VAR_NAME[VAR], st);
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(tc_gemm_pair_kernel<VAR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pr::SMEM) != cudaSuccess)
      return USAF_ERR_CUDA;
    attr_done = true;
  }
  tc_gemm_pair_kernel<VAR><<<device_sm_count() / 2 * 2, NUM_THREADS, pr::SMEM, st>>>(a, b, p);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

template <int VAR>
usaf_status launch(const CUtensorMap& a, const CUtensorMap& b, const Params& p, cudaStream_t st) {
  if constexpr (!VarTraits<VAR>::router) {
    if (p.MT % 2 == 0) return launch_pair<VAR>(a, b, p, st);
  }
  USAF_TRACE(VAR_NAME[VAR], st);
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(tc_gemm_kernel<VAR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return USAF_ERR_CUDA;
    attr_done = true;
  }
  tc_gemm_kernel<VAR><<<device_sm_count(), NUM_THREADS, SMEM_BYTES, st>>>(a, b, p);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

Params base_params(const MoeArgs& a) {
  Params p{};
  p.off = a.rt.expert_offset;
  p.ptok = a.rt.perm_tok;
  p.pslot = a.rt.perm_slot;
  p.topk_w = a.rt.topk_w;
  p.plan = a.plan;
  p.wperm = a.wperm;
  p.E = (int)a.s.E;
  p.H = (int)a.s.H;
  p.I = (int)a.s.I;
  p.T = (int)a.s.T;
  p.R_cap = a.R_cap;
  p.status = a.status;
  return p;
}

}  // namespace

bool tc_shape_ok(const usaf_moe_shape& s) {
  return s.H % 64 == 0 && s.I % 64 == 0 && s.E <= MAX_E && s.H <= (1 << 20) &&
         s.I <= (1 << 20) && s.E * s.H < (int64_t(1) << 31) && s.E * 2 * s.I < (int64_t(1) << 31);
}

// Whether clusters of RK_SPLIT CTAs of the split-K router kernel fit on this device (checked once).
static bool router_split_ok() {
  static int ok = -1;
  if (ok < 0) {
    ok = 0;
    if (cudaFuncSetAttribute(tc_router_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             RK_SMEM_BYTES) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = RK_SPLIT;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(RK_SPLIT);
      cfg.blockDim = dim3(RK_THREADS);
      cfg.dynamicSmemBytes = RK_SMEM_BYTES;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, tc_router_split_kernel, &cfg) == cudaSuccess && n > 0)
        ok = 1;
    }
    cudaGetLastError();  // a refused query leaves no error behind
  }
  return ok == 1;
}

bool tc_token_map(CUtensorMap* m, const void* base, uint64_t features, uint64_t R_cap) {
  return map_tokens(m, base, features, R_cap);
}

usaf_status tc_router_logits(const usaf_moe_shape& s, const void* x, const float* wr,
                             void* wr3, float* logits, uint32_t* status, cudaStream_t st) {
  {
    USAF_TRACE("router_split", st);
    const dim3 grid((unsigned)ceil_div(s.H, 512), (unsigned)s.E);
    router_split_kernel<<<grid, 256, 0, st>>>(wr, (int)s.H, static_cast<__nv_bfloat16*>(wr3));
    USAF_CHECK_LAUNCH();
  }
  if (router_split_ok()) {
    // K split over clusters of RK_SPLIT CTAs, 256-token tiles
    USAF_TRACE("tc_router_logits", st);
    CUtensorMap ma, mb;
    if (!map_2d(&ma, wr3, 3 * s.H, s.E, 64, 128) || !map_2d(&mb, x, s.H, s.T, 64, RK_N))
      return USAF_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = RK_SPLIT;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(RK_SPLIT * ceil_div(s.T, RK_N)), (unsigned)ceil_div(s.E, BM));
    cfg.blockDim = dim3(RK_THREADS);
    cfg.dynamicSmemBytes = RK_SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, tc_router_split_kernel, ma, mb, (int)s.T, (int)s.E, (int)s.H,
                           logits, status) != cudaSuccess)
      return USAF_ERR_CUDA;
    USAF_CHECK_LAUNCH();
    return USAF_OK;
  }
  CUtensorMap ma, mb;
  if (!map_2d(&ma, wr3, 3 * s.H, s.E, 64, 128) || !map_2d(&mb, x, s.H, s.T, 64, ROUTER_BN))
    return USAF_ERR_CUDA;
  Params p{};
  p.E = (int)s.E;
  p.H = (int)s.H;
  p.I = (int)s.I;
  p.T = (int)s.T;
  p.MT = (int)ceil_div(s.E, BM);
  p.NT = (int)ceil_div(s.T, ROUTER_BN);
  p.acc_out = logits;
  p.status = status;
  return launch<V_ROUTER>(ma, mb, p, st);
}

usaf_status tc_fwd_gate_up(const MoeArgs& a, const void* xT, void* hT, void* waT,
                           cudaStream_t st) {
  CUtensorMap ma, mb;
  if (!map_gate_up_interleaved(&ma, a.w_gate_up, a.s.E, a.s.I, a.s.H) ||
      !map_tokens(&mb, xT, a.s.H, a.R_cap))
    return USAF_ERR_CUDA;
  Params p = base_params(a);
  p.MT = (int)(a.s.I / 64);
  p.h = static_cast<__nv_bfloat16*>(hT);
  p.wa = static_cast<__nv_bfloat16*>(waT);
  return launch<V_GATEUP>(ma, mb, p, st);
}

usaf_status tc_fwd_down(const MoeArgs& a, const void* waT, float* y_acc, cudaStream_t st) {
  CUtensorMap ma, mb;
  if (!map_2d(&ma, a.w_down, a.s.I, a.s.E * a.s.H, 64, 128) || !map_tokens(&mb, waT, a.s.I, a.R_cap))
    return USAF_ERR_CUDA;
  Params p = base_params(a);
  p.MT = (int)ceil_div(a.s.H, BM);
  p.acc_out = y_acc;
  return launch<V_DOWN>(ma, mb, p, st);
}

usaf_status tc_bwd_gvec(const MoeArgs& a, const void* dyT, const void* hT, void* dhT,
                        float* dw_part,
                        cudaStream_t st) {
  CUtensorMap ma, mb;
  if (!map_2d(&ma, a.w_down, a.s.I, a.s.E * a.s.H, 64, 64) || !map_tokens(&mb, dyT, a.s.H, a.R_cap))
    return USAF_ERR_CUDA;
  Params p = base_params(a);
  p.MT = (int)ceil_div(a.s.I, BM);
  p.hin = static_cast<const __nv_bfloat16*>(hT);
  p.dh = static_cast<__nv_bfloat16*>(dhT);
  p.dw_part = dw_part;
  p.n_slots = a.s.T * a.s.k;
  return launch<V_GVEC>(ma, mb, p, st);
}

usaf_status tc_bwd_dx(const MoeArgs& a, const void* dhT, float* dx_acc, const float* dl_perm,
                      cudaStream_t st) {
  CUtensorMap ma, mb;
  if (!map_2d(&ma, a.w_gate_up, a.s.H, a.s.E * 2 * a.s.I, 64, 64) ||
      !map_tokens(&mb, dhT, 2 * a.s.I, a.R_cap))
    return USAF_ERR_CUDA;
  Params p = base_params(a);
  p.MT = (int)ceil_div(a.s.H, BM);
  p.acc_out = dx_acc;
  p.dl_perm = dl_perm;
  p.w_router = a.w_router;
  return launch<V_DX>(ma, mb, p, st);
}

usaf_status diag_wait_launch(int64_t limit_cycles, uint32_t* status, cudaStream_t st) {
  USAF_TRACE("diag_bounded_wait", st);
  diag_wait_kernel<<<1, 64, 0, st>>>((long long)limit_cycles, status);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

usaf_status tc_wgrad_dense(const MoeArgs& a, const void* aT, int64_t a_rows, const void* bT,
                           int64_t b_rows, float* g, int accumulate, cudaStream_t st) {
  USAF_TRACE(accumulate ? "tc_wgrad_dense_add" : "tc_wgrad_dense", st);
  auto fn = encode_fn();
  if (!fn) return USAF_ERR_CUDA;
  CUtensorMap ma, mb, mo;
  if (!map_2d(&ma, aT, a.R_cap, a_rows, 64, 128) || !map_2d(&mb, bT, a.R_cap, b_rows, 64, 256))
    return USAF_ERR_CUDA;
  {
    // g as [E][a_rows][b_rows] fp32, stored in 32 x 32 boxes with 128-byte swizzle
    cuuint64_t dims[3] = {(cuuint64_t)b_rows, (cuuint64_t)a_rows, (cuuint64_t)a.s.E};
    cuuint64_t strides[2] = {(cuuint64_t)b_rows * 4, (cuuint64_t)(a_rows * b_rows * 4)};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (fn(&mo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, g, dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return USAF_ERR_CUDA;
  }
  WgParams p{};
  p.off = a.rt.expert_offset;
  p.E = (int)a.s.E;
  p.M = (int)a_rows;
  p.N = (int)b_rows;
  p.MT = (int)ceil_div(a_rows, 128);
  p.NT = (int)ceil_div(b_rows, 256);
  p.accumulate = accumulate;
  p.status = a.status;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(tc_wgrad_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             wg::SMEM) != cudaSuccess)
      return USAF_ERR_CUDA;
    attr_done = true;
  }
  tc_wgrad_kernel<false><<<device_sm_count(), NUM_THREADS, wg::SMEM, st>>>(ma, mb, mo, p);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

usaf_status tc_wgrad_gather(const MoeArgs& a, const void* aT, int64_t a_rows, const void* bT,
                            int64_t b_rows, const MaskedPlan& plan, int tensor, const int64_t* act,
                            float* g_act, int accumulate, cudaStream_t st) {
  USAF_TRACE(tensor == 0 ? "tc_wgrad_gather_gate_up" : "tc_wgrad_gather_down", st);
  CUtensorMap ma, mb;
  if (!map_2d(&ma, aT, a.R_cap, a_rows, 64, 128) || !map_2d(&mb, bT, a.R_cap, b_rows, 64, 256))
    return USAF_ERR_CUDA;
  WgParams p{};
  p.off = a.rt.expert_offset;
  p.E = (int)a.s.E;
  p.M = (int)a_rows;
  p.N = (int)b_rows;
  p.MT = (int)ceil_div(a_rows, 128);
  p.NT = (int)ceil_div(b_rows, 256);
  p.accumulate = accumulate;
  p.status = a.status;
  p.dlist = plan.dense_list;
  p.n_list = plan.n_dense;
  p.row_ptr = plan.row_ptr;
  p.rp_stride = plan.rp_stride;
  p.rp_off = tensor == 0 ? 0 : (int)(2 * a.s.I + 1);
  p.act = act;
  p.flat0 = tensor == 0 ? 0 : a.s.E * 2 * a.s.I * a.s.H;
  p.g_act = g_act;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(tc_wgrad_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             wg::SMEM) != cudaSuccess)
      return USAF_ERR_CUDA;
    attr_done = true;
  }
  // the output map is not used by the gather form; ma is passed in its place
  tc_wgrad_kernel<true><<<device_sm_count(), NUM_THREADS, wg::SMEM, st>>>(ma, mb, ma, p);
  USAF_CHECK_LAUNCH();
  return USAF_OK;
}

}  // namespace usaf
