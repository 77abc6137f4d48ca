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
// Two launches of one kernel template, each over 128-row tiles with one TMEM
// lane per row, walking the other side in blocks of 64 with every product of
// a block on the tensor cores:
//   QSIDE  per query tile, two sweeps over the key blocks.  Sweep 1: S = Q K^T
//          and dP = dO V^T; each row's log2-sum-exp (online, as in the
//          forward) and D_i (the P-weighted sum of dP, rescaled with the
//          running maximum), kept for sweep 2 and written to the workspace
//          for the key side.  Sweep 2: S, dP again, then dQ += dS K;
//   KSIDE  per key tile, over query blocks: S^T = K Q^T and dP^T = V dO^T;
//          P^T and dS^T written back over them as 16-bit hi + lo parts;
//          dV += P^T dO and dK += dS^T Q with P^T, dS^T read from TMEM.
// A CTA's tensor memory is 256 columns (S and dP 64 each, then the
// accumulators), so two CTAs share an SM and one CTA's row work runs while
// the other's products are on the tensor cores.  One row warp per TMEM lane
// quadrant owns whole rows, so a row's largest values need no exchange
// between warps.
// P (for dV) and dS (for dK and dQ) enter the products as v 2^sigma with a
// per-row exponent sigma kept online for each: a block whose largest |v|
// would reach 2^14 at the current exponent lowers it and rescales the row's
// accumulator by the power of two, so every 16-bit part stays below fp16's
// overflow and, for values above 2^-17 of the row's largest, clear of its
// subnormal range (a row whose probabilities are all tiny keeps its
// precision).  The powers of two come off in FP32 at the end.
#include "attn.h"
#include "attn_common.cuh"
#include "smem_attr.h"

namespace tg {
namespace {

using namespace attn;

constexpr float BTAU = 8.f, BCP = 7.f;
constexpr int NO_SIGMA = -1000;  // a row whose dS has been zero so far

enum Mode : int { KSIDE = 1, QSIDE = 2 };

struct BwdArgs {
  int s, s_pad, nblk;
  float scale, scale_log2;
  float* stats;  // [2][heads][s_pad]: log2-sum-exp, D
  void* dA;      // QSIDE: dQ; KSIDE: dK
  void* dB;      // KSIDE: dV
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

constexpr int BI = 64;               // inner block: queries (KSIDE) or keys (QSIDE)
constexpr int TILE_I = BI * D * 2;   // 8 KB: 64 rows of 128 bytes
constexpr int IVEC = BI * 4;         // one 64-entry FP32 vector
constexpr int ROW_WARPS2 = 4;
constexpr int THREADS2 = 64 + 32 * ROW_WARPS2;
constexpr int ISTAGES = 3;
constexpr uint32_t U_S = 0, U_P = 64, U_ACC = 128;

struct Bwd2Cfg {
  static constexpr int TILES = ISTAGES * 2 * TILE_I;  // Y0, Y1 per stage (1024-aligned)
  static constexpr int VECS = ISTAGES * 2 * IVEC;     // KSIDE: the block's LSE and D per stage
  static constexpr int BAR_BYTES = 128;
  static constexpr int SMEM = 1024 + 2 * TILE + TILES + VECS + BAR_BYTES;
  static constexpr uint32_t TMEM_COLS = 256;
  static_assert(2 * SMEM <= 232448, "two CTAs per SM");
};

// Tensor maps: X0, X1 the CTA's own 128-row tiles (QSIDE: Q and dO; KSIDE:
// K and V), boxes of 128 rows; Y0, Y1 the inner blocks (QSIDE: K and V;
// KSIDE: Q and dO), boxes of 64 rows.  All [heads][s][64].
template <int MODE, bool BF16>
__global__ void __launch_bounds__(THREADS2, 2)
    attn_bwd2_kernel(const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmX1,
                     const __grid_constant__ CUtensorMap tmY0, const __grid_constant__ CUtensorMap tmY1,
                     const BwdArgs a) {
  constexpr bool QS = MODE == QSIDE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sX = smem;                          // X0, X1: this CTA's 128 rows
  uint8_t* sY = sX + 2 * TILE;                 // stages: Y0, Y1 (64 rows each)
  float* sV = reinterpret_cast<float*>(sY + Bwd2Cfg::TILES);  // stages: LSE, D (KSIDE)
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
  // iterations: QSIDE sweeps the key blocks twice (statistics, then dQ);
  // iteration j works on block j % nsub
  const int nit = QS ? 2 * nsub : nsub;

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
  float* lse_g = a.stats;
  float* dd_g = a.stats + static_cast<size_t>(gridDim.y) * a.s_pad;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(x_full), 2 * TILE);
      tma_load_3d(smem_u32(sX), &tmX0, smem_u32(x_full), 0, r0, head);
      tma_load_3d(smem_u32(sX + TILE), &tmX1, smem_u32(x_full), 0, r0, head);
      int issued[ISTAGES];
#pragma unroll
      for (int i = 0; i < ISTAGES; ++i) issued[i] = -1;
      for (int j = 0; j < nit; ++j) {
        const int st = j % ISTAGES, jb = j % nsub;
        const uint32_t ph = static_cast<uint32_t>((j / ISTAGES) & 1);
        if (!mbar_wait(smem_u32(&y_empty[st]), ph ^ 1u, tmo, abort_flag, a.status, 61)) break;
        const uint32_t fb = smem_u32(&y_full[st]);
        uint8_t* ty = sY + st * 2 * TILE_I;
        mbar_arrive_expect_tx(fb, 2 * TILE_I + (QS ? 0 : 2 * IVEC));
        tma_load_3d(smem_u32(ty), &tmY0, fb, 0, jb * BI, head);
        tma_load_3d(smem_u32(ty + TILE_I), &tmY1, fb, 0, jb * BI, head);
        if (!QS) {
          float* tv = sV + st * 2 * BI;
          bulk_load(smem_u32(tv), lse_g + hs + jb * BI, IVEC, fb);
          bulk_load(smem_u32(tv + BI), dd_g + hs + jb * BI, IVEC, fb);
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
      for (int j = 0; ok && j < nit; ++j) {
        const int st = j % ISTAGES;
        const uint32_t ph = static_cast<uint32_t>((j / ISTAGES) & 1);
        const bool stats = QS && j < nsub;  // QSIDE sweep 1: no second products
        if (!mbar_wait(smem_u32(&y_full[st]), ph, tmo, abort_flag, a.status, 63)) {
          ok = false;
          break;
        }
        // columns [0, 128) are free again once the previous iteration is done
        // with them: the rows have read S and dP (a statistics iteration) or
        // the second products have read P and dS
        if (j > 0) {
          const bool prev_stats = QS && j - 1 < nsub;
          const bool w = prev_stats
                             ? mbar_wait(smem_u32(p_full), static_cast<uint32_t>((j - 1) & 1), tmo, abort_flag,
                                         a.status, 64)
                             : mbar_wait(smem_u32(mma_done), static_cast<uint32_t>((j - 1 - (QS ? nsub : 0)) & 1),
                                         tmo, abort_flag, a.status, 64);
          if (!w) {
            ok = false;
            break;
          }
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
        if (stats) {
          umma_commit(smem_u32(&y_empty[st]));
          continue;
        }
        if (!mbar_wait(smem_u32(p_full), static_cast<uint32_t>(j & 1), tmo, abort_flag, a.status, 65)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // second products: A from TMEM (32 columns of a block as 16 hi pairs
        // then 16 lo pairs), B MN-major (the block's rows, 16 per step)
        const bool first = j == (QS ? nsub : 0);
#pragma unroll
        for (int kk = 0; kk < BI / 16; ++kk) {
          const uint32_t pc = static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8);
          const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
          const uint64_t d0 = sdesc_sw128(y0 + kk * 2048, 8192, 1024);
          if (!QS) {
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
    const int grow = r0 + row;  // this thread's query (QSIDE) or key (KSIDE)
    const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float sl = a.scale_log2;
    const bool neg = sl < 0.f;  // then the largest logit is at the smallest score
    const float asl = fabsf(sl);
    float lse = 0.f, dd = 0.f;                      // QSIDE: the row's statistics, from sweep 1
    float m_used = -INFINITY, l = 0.f, dsum = 0.f;  // QSIDE sweep 1: running state
    int sigma = NO_SIGMA;    // exponent of the row's dS
    int sigma_p = NO_SIGMA;  // KSIDE: exponent of the row's P
    bool ok = true;
    for (int j = 0; j < nit; ++j) {
      const int jb = j % nsub;
      ok = mbar_wait(smem_u32(s_full), static_cast<uint32_t>(j & 1), tmo, abort_flag, a.status, 66) && ok;
      if (!QS)  // the block's LSE and D in the stage: make the copies visible here
        ok = mbar_wait(smem_u32(&y_full[j % ISTAGES]), static_cast<uint32_t>((j / ISTAGES) & 1), tmo, abort_flag,
                       a.status, 68) && ok;
      tc_fence_after();
      const int nvalid = min(BI, a.s - jb * BI);
      if (QS && j < nsub) {
        // ---- sweep 1: the row's running maximum, sum of P and sum of P dP
        uint32_t r[64];
        tmem_ld_32x32b_x32(t_row + U_S, r);
        tmem_ld_32x32b_x32(t_row + U_S + 32, r + 32);
        tmem_ld_wait();
        float vm = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e < nvalid) vm = fmaxf(vm, neg ? -__uint_as_float(r[e]) : __uint_as_float(r[e]));
        const float mx = vm * asl;
        float rs = 1.f;
        if (j == 0 || mx > m_used + BTAU) {
          rs = ex2(m_used - mx);  // 0 on the first block
          m_used = mx;
        }
        const float mc = m_used - BCP;
        float sum = 0.f, ds = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t g[32];
          tmem_ld_32x32b_x32(t_row + U_P + c * 32, g);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float p = c * 32 + e < nvalid ? ex2(fmaf(__uint_as_float(r[c * 32 + e]), sl, -mc)) : 0.f;
            sum += p;
            ds = fmaf(p, __uint_as_float(g[e]), ds);
          }
        }
        l = l * rs + sum;
        dsum = dsum * rs + ds;
        if (j == nsub - 1) {  // the row's statistics: kept for sweep 2, and for the key side
          lse = m_used - BCP + log2f(l);
          dd = dsum / l;
          if (ok && grow < a.s) {
            lse_g[hs + grow] = lse;
            dd_g[hs + grow] = dd;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(p_full));
        continue;
      }
      const float* slse = sV + (j % ISTAGES) * 2 * BI;
      const float* sdd = slse + BI;
      // pass A: P (KSIDE: in FP32 back to its columns) and dS (kept in
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
            const float lc = QS ? lse : slse[col];
            const float dc = QS ? dd : sdd[col];
            p = ex2(fmaf(__uint_as_float(r[e]), sl, -lc));
            dsv = p * (__uint_as_float(g[e]) - dc);
          }
          mp = fmaxf(mp, p);
          mds = fmaxf(mds, fabsf(dsv));
          r[e] = __float_as_uint(p);
          dv[col] = dsv;
        }
        if (!QS) tmem_st_32x32b_x32(t_row + U_S + c * 32, r);
      }
      // the row's exponents: lowered when this block's largest value would
      // reach 2^14 at the current one, the accumulator rescaled with it
      float fs = 1.f, fp = 1.f;
      if (mds > 0.f && (sigma == NO_SIGMA || mds * pow2i(sigma) >= 16384.f)) {
        const int sn = sigma_for(mds);
        if (sigma != NO_SIGMA) fs = sn - sigma < -126 ? 0.f : pow2i(sn - sigma);
        sigma = sn;
      }
      if (!QS && mp > 0.f && (sigma_p == NO_SIGMA || mp * pow2i(sigma_p) >= 16384.f)) {
        const int sn = sigma_for(mp);
        if (sigma_p != NO_SIGMA) fp = sn - sigma_p < -126 ? 0.f : pow2i(sn - sigma_p);
        sigma_p = sn;
      }
      // KSIDE: dV [128, 192), dK [192, 256); QSIDE: dQ [128, 192)
      if (__any_sync(0xffffffffu, fs != 1.f)) {
        rescale32(t_row + U_ACC + (QS ? 0 : 64), fs);
        rescale32(t_row + U_ACC + (QS ? 0 : 64) + 32, fs);
      }
      if (!QS && __any_sync(0xffffffffu, fp != 1.f)) {
        rescale32(t_row + U_ACC, fp);
        rescale32(t_row + U_ACC + 32, fp);
      }
      // pass B: v 2^sigma as hi + lo, written over the block's S and dP columns
      const float ss = sigma == NO_SIGMA ? 1.f : pow2i(sigma);
      const float sp = sigma_p == NO_SIGMA ? 1.f : pow2i(sigma_p);
      if (!QS) tmem_st_wait();  // P's FP32 stores, read back below
#pragma unroll
      for (int c = 0; c < (QS ? 2 : 4); ++c) {
        const bool isp = !QS && c >= 2;  // KSIDE: dS chunks, then P chunks
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
      for (int o = 0; o < (QS ? 1 : 2); ++o) {
        // QSIDE: dQ = scale 2^-sigma acc; KSIDE: o = 0 dV = 2^-sigma_p acc, o = 1 dK as dQ
        const float f = (!QS && o == 0) ? p_un : ds_un;
        void* out = (!QS && o == 0) ? a.dB : a.dA;
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

template <int MODE, bool BF16>
cudaError_t launch_mode2(const CUtensorMap& x0, const CUtensorMap& x1, const CUtensorMap& y0, const CUtensorMap& y1,
                         const BwdArgs& a, int heads, cudaStream_t stream) {
  auto kern = attn_bwd2_kernel<MODE, BF16>;
  const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), Bwd2Cfg::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.nblk), static_cast<unsigned>(heads));
  return launch_k(kern, grid, dim3(THREADS2), Bwd2Cfg::SMEM, stream, x0, x1, y0, y1, a);
}

// tq, tk, tv, tdo: boxes of 128 rows (a CTA's own tile); tq64 ... tdo64:
// boxes of 64 rows (the inner blocks)
template <bool BF16>
cudaError_t launch_all(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tq64, const CUtensorMap& tk64, const CUtensorMap& tv64,
                       const CUtensorMap& tdo64, BwdArgs a, void* dQ, void* dK, void* dV, int heads,
                       cudaStream_t stream) {
  a.idesc_s = idesc_f16(BF16, false, false, 128, BI);  // S and dP over a 64-wide inner block
  // the query side first: its first sweep writes the row statistics the key side reads
  a.dA = dQ;
  a.dB = nullptr;
  cudaError_t e = launch_mode2<QSIDE, BF16>(tq, tdo, tk64, tv64, a, heads, stream);
  if (e != cudaSuccess) return e;
  a.dA = dK;
  a.dB = dV;
  return launch_mode2<KSIDE, BF16>(tk, tv, tq64, tdo64, a, heads, stream);
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
