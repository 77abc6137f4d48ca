// Fused attention backward on the tensor cores (tcgen05, TMEM, TMA): the
// gradients of L = <dO, O> for O = softmax(scale * Q K^T) V per head, given
// Q, K, V and dO, without the [s, s] matrices in memory:
//   P  = softmax_j(scale * Q K^T)      recomputed from the row statistics
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D),   D_i = sum_j P_ij dP_ij
//   dQ = scale * dS K,   dK = scale * dS^T Q
// Page "Twice the training speed on a BC-250 from tuned matrix kernels",
// section "What's left": a fused attention kernel in place of the batched
// products inside attention (the six products the library also runs
// unfused: S, O, dP, dV, dQ, dK) and the softmax between them.
//
// Three launches, each over 128-row tiles with one TMEM lane per row and
// every product of a block on the tensor cores:
//   STATS  (attn_stats_kernel) per query tile, over key blocks of 128:
//          S = Q K^T and dP = dO V^T; each row's log2-sum-exp (online, as in
//          the forward) and D_i (the P-weighted sum of dP, rescaled with the
//          running maximum);
//   DKDV   (attn_bwd2_kernel) per key tile, over query blocks of 64:
//          S^T = K Q^T and dP^T = V dO^T; P^T and dS^T written back over
//          them as 16-bit hi + lo parts; dV += P^T dO and dK += dS^T Q with
//          P^T, dS^T read from TMEM;
//   DQ     (attn_bwd2_kernel) per query tile, over key blocks of 64: S, dP,
//          then dQ += dS K.
// P (for dV) and dS (for dK and dQ) enter the products as v 2^sigma with a
// per-row exponent sigma kept online for each: a block whose largest |v|
// would reach 2^14 at the current exponent lowers it and rescales the row's
// accumulator by the power of two, so every 16-bit part stays below fp16's
// overflow and, for values above 2^-17 of the row's largest, clear of its
// subnormal range (a row whose probabilities are all tiny keeps its
// precision).  The powers of two come off in FP32 at the end.
#include "attn.h"
#include "attn_common.cuh"

namespace tg {
namespace {

using namespace attn;

constexpr float BTAU = 8.f, BCP = 7.f;
constexpr int NO_SIGMA = -1000;  // a row whose dS has been zero so far

enum Mode : int { DKDV = 1, DQ = 2 };

struct BwdArgs {
  int s, s_pad, nblk;
  float scale, scale_log2;
  float* stats;  // [2][heads][s_pad]: log2-sum-exp, D
  void* dA;      // DQ: dQ; DKDV: dK
  void* dB;      // DKDV: dV
  int out_kind;
  uint32_t idesc_s, idesc_o;
  unsigned long long timeout_ns;
  unsigned int* status;
};

// the exponent sigma with m 2^sigma < 2^14 for m > 0
__device__ __forceinline__ int sigma_for(float m) {
  int e;
  frexpf(m, &e);  // m = f 2^e, f in [0.5, 1): m < 2^e
  return max(-120, min(120, 14 - e));
}

// ---------------------------------------------------------------------------
// Row statistics.  Two CTAs per SM (256 TMEM columns each: S [0, 128) and
// dP [128, 256) of a key block); eight row warps, two per TMEM lane quadrant,
// each over half of a block's columns, exchanging a row's block maximum and
// final sums through shared memory.
constexpr int SSTAGES = 2;
constexpr uint32_t T_S = 0, T_P = 128;

struct StatsCfg {
  static constexpr int STAGE = 2 * TILE;  // the key block's K and V tiles
  static constexpr int BAR_BYTES = 128;
  static constexpr int XCH_BYTES = 2 * 4 * 2 * 32 * 8;
  static constexpr int SMEM = 1024 + 2 * TILE + SSTAGES * STAGE + BAR_BYTES + XCH_BYTES;
  static constexpr uint32_t TMEM_COLS = 256;
};

// Tensor maps: X0, X1 the CTA's own Q and dO tiles; Y0, Y1 the key block's
// K and V tiles.  All [heads][s][64], boxes of 128 rows.
template <bool BF16>
__global__ void __launch_bounds__(THREADS, 2)
    attn_stats_kernel(const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmX1,
                      const __grid_constant__ CUtensorMap tmY0, const __grid_constant__ CUtensorMap tmY1,
                      const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sX = smem;           // X0, X1
  uint8_t* sY = sX + 2 * TILE;  // stages: Y0, Y1
  uint64_t* bars = reinterpret_cast<uint64_t*>(sY + SSTAGES * StatsCfg::STAGE);
  uint64_t* x_full = bars;
  uint64_t* y_full = x_full + 1;
  uint64_t* y_empty = y_full + SSTAGES;
  uint64_t* s_full = y_empty + SSTAGES;
  uint64_t* p_full = s_full + 1;
  uint64_t* drain = p_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + StatsCfg::BAR_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.y, r0 = blockIdx.x * BT;
  const int nblk = a.nblk;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(x_full), 1);
    for (int i = 0; i < SSTAGES; ++i) {
      mbar_init(smem_u32(&y_full[i]), 1);
      mbar_init(smem_u32(&y_empty[i]), 1);
    }
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(p_full), ROW_WARPS);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX0);
    prefetch_tmap(&tmX1);
    prefetch_tmap(&tmY0);
    prefetch_tmap(&tmY1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), StatsCfg::TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long tmo = a.timeout_ns;
  pdl_wait();
  pdl_trigger();
  const size_t hs = static_cast<size_t>(head) * a.s_pad;
  float* lse_g = a.stats;
  float* dd_g = a.stats + static_cast<size_t>(gridDim.y) * a.s_pad;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(x_full), 2 * TILE);
      tma_load_3d(smem_u32(sX), &tmX0, smem_u32(x_full), 0, r0, head);
      tma_load_3d(smem_u32(sX + TILE), &tmX1, smem_u32(x_full), 0, r0, head);
      int issued[SSTAGES];
#pragma unroll
      for (int i = 0; i < SSTAGES; ++i) issued[i] = -1;
      for (int j = 0; j < nblk; ++j) {
        const int st = j % SSTAGES;
        const uint32_t ph = static_cast<uint32_t>((j / SSTAGES) & 1);
        if (!mbar_wait(smem_u32(&y_empty[st]), ph ^ 1u, tmo, abort_flag, a.status, 41)) break;
        const uint32_t fb = smem_u32(&y_full[st]);
        uint8_t* stage = sY + st * StatsCfg::STAGE;
        mbar_arrive_expect_tx(fb, StatsCfg::STAGE);
        tma_load_3d(smem_u32(stage), &tmY0, fb, 0, j * BT, head);
        tma_load_3d(smem_u32(stage + TILE), &tmY1, fb, 0, j * BT, head);
        issued[st] = static_cast<int>(ph);
      }
      mbar_wait(smem_u32(x_full), 0, 200000000ull, nullptr, a.status, 49);
#pragma unroll
      for (int i = 0; i < SSTAGES; ++i)
        if (issued[i] >= 0)
          mbar_wait(smem_u32(&y_full[i]), static_cast<uint32_t>(issued[i]), 200000000ull, nullptr, a.status, 49);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(smem_u32(x_full), 0, tmo, abort_flag, a.status, 42);
      tc_fence_after();
      const uint32_t x0 = smem_u32(sX), x1 = x0 + TILE;
      for (int j = 0; ok && j < nblk; ++j) {
        const int st = j % SSTAGES;
        const uint32_t ph = static_cast<uint32_t>((j / SSTAGES) & 1);
        if (!mbar_wait(smem_u32(&y_full[st]), ph, tmo, abort_flag, a.status, 43)) {
          ok = false;
          break;
        }
        // TMEM columns 0..255 are free again once the rows have read S and dP
        if (j > 0 && !mbar_wait(smem_u32(p_full), static_cast<uint32_t>((j - 1) & 1), tmo, abort_flag, a.status,
                                44)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t y0 = smem_u32(sY + st * StatsCfg::STAGE), y1 = y0 + TILE;
        // S = Q K^T, dP = dO V^T (all K-major, head dimension contiguous)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          umma_f16(tmem + T_S, sdesc_sw128(x0 + kk * 32, 16, 1024), sdesc_sw128(y0 + kk * 32, 16, 1024), a.idesc_s,
                   kk > 0 ? 1u : 0u);
          umma_f16(tmem + T_P, sdesc_sw128(x1 + kk * 32, 16, 1024), sdesc_sw128(y1 + kk * 32, 16, 1024), a.idesc_s,
                   kk > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(s_full));
        umma_commit(smem_u32(&y_empty[st]));
      }
      if (!ok) {
        umma_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, 200000000ull, nullptr, a.status, 50);
      }
    }
  } else {
    // ------------------------------------------------------------- the rows
    // After a failed wait the loop still runs to the end (every later wait
    // returns at once), so the two warps of a pair always meet at the same
    // named barriers; tensor memory is then garbage but never addressed out
    // of bounds, and nothing is stored.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;  // which 64 columns of each block
    const int row = q * 32 + lane;
    const int grow = r0 + row;  // this thread's query
    const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float sl = a.scale_log2;
    const bool neg = sl < 0.f;
    const float asl = fabsf(sl);
    float m_used = -INFINITY, l = 0.f, dsum = 0.f;
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      ok = mbar_wait(smem_u32(s_full), static_cast<uint32_t>(j & 1), tmo, abort_flag, a.status, 46) && ok;
      tc_fence_after();
      const int nvalid = min(BT, a.s - j * BT) - half * 64;  // this warp's columns inside the sequence
      const uint32_t cS = t_row + T_S + half * 64, cP = t_row + T_P + half * 64;
      float vm = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(cS + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (c * 32 + e < nvalid) vm = fmaxf(vm, neg ? -__uint_as_float(r[e]) : __uint_as_float(r[e]));
      }
      vm = fmaxf(vm, pair_exchange(xch, j & 1, q, half, lane, vm));
      const float mx = vm * asl;
      float rs = 1.f;
      if (j == 0 || mx > m_used + BTAU) {
        rs = ex2(m_used - mx);
        m_used = mx;
      }
      const float mc = m_used - BCP;
      float sum = 0.f, ds = 0.f;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32], g[32];
        tmem_ld_32x32b_x32(cS + c * 32, r);
        tmem_ld_32x32b_x32(cP + c * 32, g);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p = c * 32 + e < nvalid ? ex2(fmaf(__uint_as_float(r[e]), sl, -mc)) : 0.f;
          sum += p;
          ds = fmaf(p, __uint_as_float(g[e]), ds);
        }
      }
      l = l * rs + sum;
      dsum = dsum * rs + ds;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(p_full));
    }
    // ---- the row's results
    l += pair_exchange(xch, nblk & 1, q, half, lane, l);
    dsum += pair_exchange(xch, (nblk + 1) & 1, q, half, lane, dsum);
    if (ok && half == 0 && grow < a.s) {
      lse_g[hs + grow] = m_used - BCP + log2f(l);
      dd_g[hs + grow] = dsum / l;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, StatsCfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// dK, dV (DKDV) and dQ (DQ) over 64-wide inner blocks.  A CTA owns 128 rows
// (keys for DKDV, queries for DQ; one TMEM lane each) and walks the other
// side in blocks of BI = 64, so its tensor memory is 256 columns (S and dP
// 64 each, then the accumulators) and two CTAs share an SM: one CTA's row
// work runs while the other's products are on the tensor cores.  One row
// warp per TMEM lane quadrant owns whole rows, so a row's largest values
// need no exchange between warps.
constexpr int BI = 64;               // inner block: queries (DKDV) or keys (DQ)
constexpr int TILE_I = BI * D * 2;   // 8 KB: 64 rows of 128 bytes
constexpr int IVEC = BI * 4;         // one 64-entry FP32 vector
constexpr int ROW_WARPS2 = 4;
constexpr int THREADS2 = 64 + 32 * ROW_WARPS2;
constexpr int ISTAGES = 3;
constexpr uint32_t U_S = 0, U_P = 64, U_ACC = 128;

struct Bwd2Cfg {
  static constexpr int TILES = ISTAGES * 2 * TILE_I;  // Y0, Y1 per stage (1024-aligned)
  static constexpr int VECS = ISTAGES * 2 * IVEC;     // DKDV: the block's LSE and D per stage
  static constexpr int BAR_BYTES = 128;
  static constexpr int SMEM = 1024 + 2 * TILE + TILES + VECS + BAR_BYTES;
  static constexpr uint32_t TMEM_COLS = 256;
  static_assert(2 * SMEM <= 232448, "two CTAs per SM");
};

template <int MODE, bool BF16>
__global__ void __launch_bounds__(THREADS2, 2)
    attn_bwd2_kernel(const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmX1,
                     const __grid_constant__ CUtensorMap tmY0, const __grid_constant__ CUtensorMap tmY1,
                     const BwdArgs a) {
  static_assert(MODE == DKDV || MODE == DQ, "the row statistics run in attn_stats_kernel");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sX = smem;                          // X0, X1: this CTA's 128 rows
  uint8_t* sY = sX + 2 * TILE;                 // stages: Y0, Y1 (64 rows each)
  float* sV = reinterpret_cast<float*>(sY + Bwd2Cfg::TILES);  // stages: LSE, D (DKDV)
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sV) + Bwd2Cfg::VECS);
  uint64_t* x_full = bars;
  uint64_t* y_full = x_full + 1;
  uint64_t* y_empty = y_full + ISTAGES;
  uint64_t* s_full = y_empty + ISTAGES;
  uint64_t* p_full = s_full + 1;
  uint64_t* mma_done = p_full + 1;
  uint64_t* drain = mma_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert((2 * ISTAGES + 6) * 8 + 8 <= Bwd2Cfg::BAR_BYTES, "barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.y, r0 = blockIdx.x * BT;
  const int nsub = (a.s + BI - 1) / BI;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(x_full), 1);
    for (int i = 0; i < ISTAGES; ++i) {
      mbar_init(smem_u32(&y_full[i]), 1);
      mbar_init(smem_u32(&y_empty[i]), 1);
    }
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(p_full), ROW_WARPS2);
    mbar_init(smem_u32(mma_done), 1);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX0);
    prefetch_tmap(&tmX1);
    prefetch_tmap(&tmY0);
    prefetch_tmap(&tmY1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Bwd2Cfg::TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long tmo = a.timeout_ns;
  pdl_wait();
  pdl_trigger();
  const size_t hs = static_cast<size_t>(head) * a.s_pad;
  const float* lse_g = a.stats;
  const float* dd_g = a.stats + static_cast<size_t>(gridDim.y) * a.s_pad;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(x_full), 2 * TILE);
      tma_load_3d(smem_u32(sX), &tmX0, smem_u32(x_full), 0, r0, head);
      tma_load_3d(smem_u32(sX + TILE), &tmX1, smem_u32(x_full), 0, r0, head);
      int issued[ISTAGES];
#pragma unroll
      for (int i = 0; i < ISTAGES; ++i) issued[i] = -1;
      for (int j = 0; j < nsub; ++j) {
        const int st = j % ISTAGES;
        const uint32_t ph = static_cast<uint32_t>((j / ISTAGES) & 1);
        if (!mbar_wait(smem_u32(&y_empty[st]), ph ^ 1u, tmo, abort_flag, a.status, 61)) break;
        const uint32_t fb = smem_u32(&y_full[st]);
        uint8_t* ty = sY + st * 2 * TILE_I;
        mbar_arrive_expect_tx(fb, 2 * TILE_I + (MODE == DKDV ? 2 * IVEC : 0));
        tma_load_3d(smem_u32(ty), &tmY0, fb, 0, j * BI, head);
        tma_load_3d(smem_u32(ty + TILE_I), &tmY1, fb, 0, j * BI, head);
        if (MODE == DKDV) {
          float* tv = sV + st * 2 * BI;
          bulk_load(smem_u32(tv), lse_g + hs + j * BI, IVEC, fb);
          bulk_load(smem_u32(tv + BI), dd_g + hs + j * BI, IVEC, fb);
        }
        issued[st] = static_cast<int>(ph);
      }
      mbar_wait(smem_u32(x_full), 0, 200000000ull, nullptr, a.status, 69);
#pragma unroll
      for (int i = 0; i < ISTAGES; ++i)
        if (issued[i] >= 0)
          mbar_wait(smem_u32(&y_full[i]), static_cast<uint32_t>(issued[i]), 200000000ull, nullptr, a.status, 69);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(smem_u32(x_full), 0, tmo, abort_flag, a.status, 62);
      tc_fence_after();
      const uint32_t x0 = smem_u32(sX), x1 = x0 + TILE;
      for (int j = 0; ok && j < nsub; ++j) {
        const int st = j % ISTAGES;
        const uint32_t ph = static_cast<uint32_t>((j / ISTAGES) & 1);
        if (!mbar_wait(smem_u32(&y_full[st]), ph, tmo, abort_flag, a.status, 63)) {
          ok = false;
          break;
        }
        // columns [0, 128) are free again once the previous block's second
        // products have read them
        if (j > 0 &&
            !mbar_wait(smem_u32(mma_done), static_cast<uint32_t>((j - 1) & 1), tmo, abort_flag, a.status, 64)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t y0 = smem_u32(sY + st * 2 * TILE_I), y1 = y0 + TILE_I;
        // S = X0 Y0^T and dP = X1 Y1^T (K-major, head dimension contiguous), N = 64
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          umma_f16(tmem + U_S, sdesc_sw128(x0 + kk * 32, 16, 1024), sdesc_sw128(y0 + kk * 32, 16, 1024), a.idesc_s,
                   kk > 0 ? 1u : 0u);
          umma_f16(tmem + U_P, sdesc_sw128(x1 + kk * 32, 16, 1024), sdesc_sw128(y1 + kk * 32, 16, 1024), a.idesc_s,
                   kk > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(s_full));
        if (!mbar_wait(smem_u32(p_full), static_cast<uint32_t>(j & 1), tmo, abort_flag, a.status, 65)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // second products: A from TMEM (32 columns of a block as 16 hi pairs
        // then 16 lo pairs), B MN-major (the block's rows, 16 per step)
#pragma unroll
        for (int kk = 0; kk < BI / 16; ++kk) {
          const uint32_t pc = static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8);
          const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
          const uint64_t d0 = sdesc_sw128(y0 + kk * 2048, 8192, 1024);
          if (MODE == DKDV) {
            // dV += P^T dO (Y1), dK += dS^T Q (Y0)
            const uint64_t d1 = sdesc_sw128(y1 + kk * 2048, 8192, 1024);
            umma_f16_ta(tmem + U_ACC, tmem + U_S + pc, d1, a.idesc_o, acc);
            umma_f16_ta(tmem + U_ACC, tmem + U_S + pc + 16, d1, a.idesc_o, 1u);
            umma_f16_ta(tmem + U_ACC + 64, tmem + U_P + pc, d0, a.idesc_o, acc);
            umma_f16_ta(tmem + U_ACC + 64, tmem + U_P + pc + 16, d0, a.idesc_o, 1u);
          } else {
            // dQ += dS K (Y0)
            umma_f16_ta(tmem + U_ACC, tmem + U_P + pc, d0, a.idesc_o, acc);
            umma_f16_ta(tmem + U_ACC, tmem + U_P + pc + 16, d0, a.idesc_o, 1u);
          }
        }
        umma_commit(smem_u32(&y_empty[st]));
        umma_commit(smem_u32(mma_done));
      }
      if (!ok) {
        umma_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, 200000000ull, nullptr, a.status, 70);
      }
    }
  } else {
    // ------------------------------------------------------------- the rows
    // A failed wait makes every later one return at once; the loop runs to
    // its end and nothing is stored.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int grow = r0 + row;  // this thread's key (DKDV) or query (DQ)
    const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float sl = a.scale_log2;
    float lse = 0.f, dd = 0.f;
    if (MODE == DQ && grow < a.s) {
      lse = lse_g[hs + grow];
      dd = dd_g[hs + grow];
    }
    int sigma = NO_SIGMA;    // exponent of the row's dS
    int sigma_p = NO_SIGMA;  // DKDV: exponent of the row's P
    bool ok = true;
    for (int j = 0; j < nsub; ++j) {
      ok = mbar_wait(smem_u32(s_full), static_cast<uint32_t>(j & 1), tmo, abort_flag, a.status, 66) && ok;
      if (MODE == DKDV)  // the block's LSE and D in the stage: make the copies visible here
        ok = mbar_wait(smem_u32(&y_full[j % ISTAGES]), static_cast<uint32_t>((j / ISTAGES) & 1), tmo, abort_flag,
                       a.status, 68) && ok;
      tc_fence_after();
      const int nvalid = min(BI, a.s - j * BI);
      const float* slse = sV + (j % ISTAGES) * 2 * BI;
      const float* sdd = slse + BI;
      // pass A: P (DKDV: in FP32 back to its columns) and dS (kept in
      // registers), with the row's largest magnitudes
      float mp = 0.f, mds = 0.f;
      float dv[BI];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32], g[32];
        tmem_ld_32x32b_x32(t_row + U_S + c * 32, r);
        tmem_ld_32x32b_x32(t_row + U_P + c * 32, g);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = c * 32 + e;
          float p = 0.f, dsv = 0.f;
          if (col < nvalid) {
            const float lc = MODE == DQ ? lse : slse[col];
            const float dc = MODE == DQ ? dd : sdd[col];
            p = ex2(fmaf(__uint_as_float(r[e]), sl, -lc));
            dsv = p * (__uint_as_float(g[e]) - dc);
          }
          mp = fmaxf(mp, p);
          mds = fmaxf(mds, fabsf(dsv));
          r[e] = __float_as_uint(p);
          dv[col] = dsv;
        }
        if (MODE == DKDV) tmem_st_32x32b_x32(t_row + U_S + c * 32, r);
      }
      // the row's exponents: lowered when this block's largest value would
      // reach 2^14 at the current one, the accumulator rescaled with it
      float fs = 1.f, fp = 1.f;
      if (mds > 0.f && (sigma == NO_SIGMA || mds * pow2i(sigma) >= 16384.f)) {
        const int sn = sigma_for(mds);
        if (sigma != NO_SIGMA) fs = sn - sigma < -126 ? 0.f : pow2i(sn - sigma);
        sigma = sn;
      }
      if (MODE == DKDV && mp > 0.f && (sigma_p == NO_SIGMA || mp * pow2i(sigma_p) >= 16384.f)) {
        const int sn = sigma_for(mp);
        if (sigma_p != NO_SIGMA) fp = sn - sigma_p < -126 ? 0.f : pow2i(sn - sigma_p);
        sigma_p = sn;
      }
      // DKDV: dV [128, 192), dK [192, 256); DQ: dQ [128, 192)
      if (__any_sync(0xffffffffu, fs != 1.f)) {
        rescale32(t_row + U_ACC + (MODE == DKDV ? 64 : 0), fs);
        rescale32(t_row + U_ACC + (MODE == DKDV ? 64 : 0) + 32, fs);
      }
      if (MODE == DKDV && __any_sync(0xffffffffu, fp != 1.f)) {
        rescale32(t_row + U_ACC, fp);
        rescale32(t_row + U_ACC + 32, fp);
      }
      // pass B: v 2^sigma as hi + lo, written over the block's S and dP columns
      const float ss = sigma == NO_SIGMA ? 1.f : pow2i(sigma);
      const float sp = sigma_p == NO_SIGMA ? 1.f : pow2i(sigma_p);
      if (MODE == DKDV) tmem_st_wait();  // P's FP32 stores, read back below
#pragma unroll
      for (int c = 0; c < (MODE == DKDV ? 4 : 2); ++c) {
        const bool isp = MODE == DKDV && c >= 2;  // DKDV: dS chunks, then P chunks
        const uint32_t col = t_row + (isp ? U_S : U_P) + (c & 1) * 32;
        float v[32];
        if (isp) {
          uint32_t g[32];
          tmem_ld_32x32b_x32(col, g);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(g[e]) * sp;
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = dv[(c & 1) * 32 + e] * ss;
        }
        uint32_t w[32];
        split32<BF16>(v, w);
        tmem_st_32x32b_x32(col, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(p_full));
    }
    // ---- the row's results
    if (ok) ok = mbar_wait(smem_u32(mma_done), static_cast<uint32_t>((nsub - 1) & 1), tmo, abort_flag, a.status, 67);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const float ds_un = sigma == NO_SIGMA ? 0.f : a.scale * pow2i(-sigma);
      const float p_un = sigma_p == NO_SIGMA ? 0.f : pow2i(-sigma_p);
#pragma unroll 1
      for (int o = 0; o < (MODE == DKDV ? 2 : 1); ++o) {
        // DQ: dQ = scale 2^-sigma acc; DKDV: o = 0 dV = 2^-sigma_p acc, o = 1 dK as dQ
        const float f = (MODE == DKDV && o == 0) ? p_un : ds_un;
        void* out = (MODE == DKDV && o == 0) ? a.dB : a.dA;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + U_ACC + o * 64 + h * 32, r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]) * f;
          if (grow < a.s) store_row32(out, a.out_kind, (static_cast<size_t>(head) * a.s + grow) * D + h * 32, v);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Bwd2Cfg::TMEM_COLS);
  }
}

template <bool BF16>
cudaError_t launch_stats(const CUtensorMap& x0, const CUtensorMap& x1, const CUtensorMap& y0, const CUtensorMap& y1,
                         const BwdArgs& a, int heads, cudaStream_t stream) {
  auto kern = attn_stats_kernel<BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, StatsCfg::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const dim3 grid(static_cast<unsigned>(a.nblk), static_cast<unsigned>(heads));
  return launch_k(kern, grid, dim3(THREADS), StatsCfg::SMEM, stream, x0, x1, y0, y1, a);
}

template <int MODE, bool BF16>
cudaError_t launch_mode2(const CUtensorMap& x0, const CUtensorMap& x1, const CUtensorMap& y0, const CUtensorMap& y1,
                         const BwdArgs& a, int heads, cudaStream_t stream) {
  auto kern = attn_bwd2_kernel<MODE, BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Bwd2Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const dim3 grid(static_cast<unsigned>(a.nblk), static_cast<unsigned>(heads));
  return launch_k(kern, grid, dim3(THREADS2), Bwd2Cfg::SMEM, stream, x0, x1, y0, y1, a);
}

// tq, tk, tv, tdo: boxes of 128 rows (a CTA's own tile, and the statistics'
// key blocks); tq64 ... tdo64: boxes of 64 rows (the inner blocks of the
// dK/dV and dQ passes)
template <bool BF16>
cudaError_t launch_all(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tq64, const CUtensorMap& tk64, const CUtensorMap& tv64,
                       const CUtensorMap& tdo64, BwdArgs a, void* dQ, void* dK, void* dV, int heads,
                       cudaStream_t stream) {
  a.idesc_s = idesc_f16(BF16, false, false, 128, BT);  // S and dP over a 128-wide key block
  cudaError_t e = launch_stats<BF16>(tq, tdo, tk, tv, a, heads, stream);
  if (e != cudaSuccess) return e;
  a.idesc_s = idesc_f16(BF16, false, false, 128, BI);  // S and dP over a 64-wide inner block
  a.dA = dK;
  a.dB = dV;
  e = launch_mode2<DKDV, BF16>(tk, tv, tq64, tdo64, a, heads, stream);
  if (e != cudaSuccess) return e;
  a.dA = dQ;
  a.dB = nullptr;
  return launch_mode2<DQ, BF16>(tq, tdo, tk64, tv64, a, heads, stream);
}

}  // namespace

size_t attn_bwd_ws_bytes(int64_t heads, int64_t s) {
  const int64_t s_pad = (s + BT - 1) / BT * BT;
  return static_cast<size_t>(2) * heads * s_pad * 4;
}

cudaError_t attn_bwd_tc_launch(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK,
                               void* dV, int64_t heads, int64_t s, int64_t d, float scale, int in_kind,
                               int out_kind, void* ws, unsigned int* status, unsigned long long timeout_ns,
                               cudaStream_t stream) {
  if (heads == 0 || s == 0) return cudaSuccess;
  if (d != D) return cudaErrorInvalidValue;
  alignas(64) CUtensorMap tq, tk, tv, tdo, tq64, tk64, tv64, tdo64;
  const uint64_t pitch = D * 2;
  if (!encode_tmap_3d(&tq, Q, in_kind, D, s, heads, pitch, pitch * s, D, BT, 128) ||
      !encode_tmap_3d(&tk, K, in_kind, D, s, heads, pitch, pitch * s, D, BT, 128) ||
      !encode_tmap_3d(&tv, V, in_kind, D, s, heads, pitch, pitch * s, D, BT, 128) ||
      !encode_tmap_3d(&tdo, dO, in_kind, D, s, heads, pitch, pitch * s, D, BT, 128) ||
      !encode_tmap_3d(&tq64, Q, in_kind, D, s, heads, pitch, pitch * s, D, BI, 128) ||
      !encode_tmap_3d(&tk64, K, in_kind, D, s, heads, pitch, pitch * s, D, BI, 128) ||
      !encode_tmap_3d(&tv64, V, in_kind, D, s, heads, pitch, pitch * s, D, BI, 128) ||
      !encode_tmap_3d(&tdo64, dO, in_kind, D, s, heads, pitch, pitch * s, D, BI, 128))
    return cudaErrorInvalidValue;
  BwdArgs a{};
  a.s = static_cast<int>(s);
  a.nblk = static_cast<int>((s + BT - 1) / BT);
  a.s_pad = a.nblk * BT;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.stats = static_cast<float*>(ws);
  a.out_kind = out_kind;
  const bool bf = in_kind == EK_BF16;
  a.idesc_o = idesc_f16(bf, false, true, 128, D);
  a.timeout_ns = timeout_ns;
  a.status = status;
  return bf ? launch_all<true>(tq, tk, tv, tdo, tq64, tk64, tv64, tdo64, a, dQ, dK, dV, static_cast<int>(heads), stream)
            : launch_all<false>(tq, tk, tv, tdo, tq64, tk64, tv64, tdo64, a, dQ, dK, dV, static_cast<int>(heads),
                                stream);
}

}  // namespace tg
