// lora.cu -- rank-16 LoRA products as HBM-streaming kernels.
//
// Page "Twice the training speed on a BC-250 from tuned matrix kernels",
// section "Tuning the kernels": the rank-16 LoRA matrices are among the
// products a training step runs.  Each of them reads or writes one [T, d]
// tensor and touches only small [*, 16] factors otherwise, so they are bound
// by HBM bandwidth, not by the tensor cores.  The arithmetic (about 16 flop
// per streamed byte) still needs the tensor pipe: FP32 FFMA on the CUDA cores
// cannot keep up with HBM at that intensity, so it runs on warp-level
// mma.sync (m16n8k16, FP32 accumulate).
//
// Streaming.  The kernels that read a [T, d] tensor are warp-specialised:
// one producer warp moves tiles into a ring of shared-memory stages with TMA
// (cp.async.bulk.tensor, swizzled) and eight consumer warps read fragments
// from the stages with ldmatrix.  A CTA keeps up to ~150 KB of loads in flight
// without holding them in registers, and every streamed byte crosses HBM once.
//   row-down   OUT[t, r] = sum_k IN[t, k] S(r, k)      (H = X A^T, dH = dY B)
//              CTA = R consecutive rows (R <= 32: about one CTA per SM), all
//              of K; a warp owns one 64-column chunk of each stage.
//   col-red    P[j, r] = sum_t IN[t, j] Hm[t, r]        (dB = dY^T H, dA^T = X^T dH)
//              the (128-column block, 128-token step) space is cut into
//              contiguous ranges of equal length on the fewest CTAs that keep
//              the largest share (every CTA streams about the same number of
//              bytes, and few CTAs share a column block); a column block cut
//              by range boundaries gets one FP32 partial per CTA, and the last
//              CTA to publish one adds them in CTA order.  The tiles are read
//              transposed by ldmatrix.trans, so there is no transposition
//              pass.  Optionally fused with the row-up of the same tile
//              (dX = dH A): the dH tile in the stage also feeds the
//              [128 x 128] dX tile, written straight from registers.
//   row-up     OUT[t, j] = sum_r Hm[t, r] S2(j, r)      (Y = H B^T)
//              writes a [T, d] tensor from the small factors, all from
//              registers (16-byte stores).
// FP32 operands (the gradient dH, FP32 LoRA factors) enter the 16-bit MMA as
// hi + lo parts, hi = rn(x) and lo = rn((x - hi) 2^11): the lo part is stored
// scaled by 2^11, its products go to their own FP32 sums and those are scaled
// back by 2^-11 at the end (exact: powers of two).  Both parts are
// multiplied, so x keeps about 16 (bf16) or 22 (fp16) significant bits; the
// scaling keeps fp16's lo part out of its subnormal range (without it, a lo
// part below 2^-14 would keep only the bits above 2^-24, a fixed absolute
// precision that fails the relative bound for small gradients or factors).
//
// Every result is a fixed-order sum: a warp adds its chunks in K order, the
// warps' partial tiles are added in warp order, the CTAs' partials of a column
// block in CTA order.  Every wait on an mbarrier is bounded (it gives up after
// the configured limit, raises the device status word and lets the CTA unwind).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdio.h>
#include <stdlib.h>

#include "ptx.cuh"
#include "smem_attr.h"
#include "tg_internal.h"

namespace tg {

constexpr int LR = 16;                    // the rank these kernels are written for
constexpr float LO_SCALE = 2048.f;        // lo parts are stored times 2^11 ...
constexpr float LO_UNSCALE = 1.f / 2048.f;  // ... and their products' sums scaled back
constexpr int LCW = 8;                    // consumer warps of a TMA-fed role
constexpr int LGROUP = (LCW + 1) * 32;    // one role: consumers + one producer warp
constexpr int LGROUP_UP = (2 * LCW + 1) * 32;  // col-red + row-up warps + one producer warp
constexpr int LMAX_STAGES = 8;
constexpr int CR_RS = 128;                // tokens per col-red step
constexpr int RD_RED_BYTES = LCW * 32 * 17 * 4;  // row-down cross-warp partials
constexpr int BAR_BYTES = 2 * LMAX_STAGES * 8 + 64;  // mbarriers + flags
constexpr int SMEM_LIMIT = 232448;
// gradient passes: row-down chunks per stage and smem budget, col-red stages,
// pass-2 CTAs per SM
constexpr int G1_RD_CH = 8, G1_RD_BUDGET = 156 * 1024, G1_CR_STAGES = 2, G2_CR_STAGES = 4, G2_CTAS_PER_SM = 1;

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// Address of 16-byte chunk `chunk` of row `row` in a tile written by TMA.
// 128-byte rows with the 128-byte swizzle (tile base 1024-byte aligned): the
// chunk index is XORed with row % 8.
__device__ __forceinline__ uint32_t sw128(uint32_t base, int row, int chunk) {
  return base + static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// 32-byte rows with the 32-byte swizzle (tile base 256-byte aligned): the
// chunk index (0 or 1) is XORed with bit 2 of the row.
__device__ __forceinline__ uint32_t sw32(uint32_t base, int row, int chunk) {
  return base + static_cast<uint32_t>(row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4));
}
// the consumer warps of one role (named barrier `id`, 256 threads)
__device__ __forceinline__ void group_bar(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(LCW * 32) : "memory");
}

__device__ __forceinline__ uint2 ld8(const void* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }

template <bool BF16>
__device__ __forceinline__ float round16(float x) {
  return BF16 ? __bfloat162float(__float2bfloat16_rn(x)) : __half2float(__float2half_rn(x));
}
template <bool BF16>
__device__ __forceinline__ uint16_t bits16(float x) {
  if (BF16) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
  } else {
    __half h = __float2half_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
  }
}

__device__ __forceinline__ void store_out(void* out, int kind, size_t i, float v) {
  if (kind == EK_F32)
    static_cast<float*>(out)[i] = v;
  else if (kind == EK_BF16)
    static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  else
    static_cast<__half*>(out)[i] = __float2half_rn(v);
}

// 8 consecutive outputs of one row (16-byte aligned start)
__device__ __forceinline__ void store8(void* out, int kind, size_t i, const float* v) {
  if (kind == EK_F32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + i);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else if (kind == EK_BF16) {
    uint4 w = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                         pack_bf16x2(v[6], v[7]));
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + i) = w;
  } else {
    uint4 w = make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                         pack_f16x2(v[6], v[7]));
    *reinterpret_cast<uint4*>(static_cast<__half*>(out) + i) = w;
  }
}

// the bits of the 8 consecutive outputs at i: two 16-byte words for FP32,
// one (w[0]) for the 16-bit kinds
__device__ __forceinline__ void load8_raw(const void* out, int kind, size_t i, uint4* w) {
  if (kind == EK_F32) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(out) + i);
    w[0] = p[0];
    w[1] = p[1];
  } else {
    w[0] = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(out) + i);
  }
}

// 16 bytes global -> shared without a register round trip (completion per
// thread: cp_async_wait_all)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// all but the most recent commit group are complete
__device__ __forceinline__ void cp_async_wait_group1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// those 8 outputs as FP32 (exact: every 16-bit value is one)
__device__ __forceinline__ void raw8_to_float(int kind, const uint4* w, float* v) {
  if (kind == EK_F32) {
    const uint32_t u[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __uint_as_float(u[k]);
  } else {
    const uint32_t u[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (kind == EK_BF16) {
        v[2 * k] = __uint_as_float(u[k] << 16);
        v[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
      } else {
        v[2 * k] = __half2float(__ushort_as_half(static_cast<unsigned short>(u[k] & 0xFFFFu)));
        v[2 * k + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(u[k] >> 16)));
      }
    }
  }
}

// Producer epilogue after an aborted wait: let every copy already issued
// land before the CTA unwinds (bounded, without the abort short-cut).
__device__ __forceinline__ void drain_issued(const uint64_t* full, const int* issued, int stages,
                                             unsigned int* status) {
  for (int s = 0; s < stages; ++s)
    if (issued[s] >= 0)
      mbar_wait(smem_u32(&full[s]), static_cast<uint32_t>(issued[s]), 200000000ull, nullptr, status, 0x2F);
}

// Per-CTA event timestamps of a role, only in -DTG_TRACE builds.
#ifdef TG_TRACE
#define LORA_EVENT(tr, ev)                                                \
  do {                                                                    \
    if (tr) (tr)[blockIdx.x * 16 + (ev)] = globaltimer_ns();             \
  } while (0)
#else
#define LORA_EVENT(tr, ev) \
  do {                     \
  } while (0)
#endif

// The barrier block of a role: full[LMAX_STAGES], empty[LMAX_STAGES], flags.
struct RoleBars {
  uint64_t* full;
  uint64_t* empty;
  volatile int* flags;  // [0] abort, [1] shared decision, [2] last-contributor, [3] last CTA of a column block
  __device__ RoleBars(uint8_t* p)
      : full(reinterpret_cast<uint64_t*>(p)),
        empty(reinterpret_cast<uint64_t*>(p) + LMAX_STAGES),
        flags(reinterpret_cast<volatile int*>(p + 2 * LMAX_STAGES * 8)) {}
  __device__ void init(int stages, int consumer_warps = LCW) const {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), static_cast<uint32_t>(consumer_warps));
    }
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
  }
};

// ===================================================================
// Role 1: row-down.  OUT[t, r] = sum_k IN[t, k] S(r, k), r < 16.
// A stage holds CH 64-column chunks of the CTA's R rows and of S, loaded by
// one 3-D TMA box each: IN viewed as [K/64 chunks][T rows][64], box
// {64, R, CH}; S viewed as [K/64][16][64] (S_KN = false: S stored [16][K],
// the LoRA A) or [K/64][64][16] (S_KN = true: S stored [K][16], the LoRA B).
// Only whole chunks are viewed that way; a last partial chunk (K % 64 != 0)
// has a stage of its own, loaded through plain 2-D maps whose box reads
// zeros past K.  Chunks of a 3-D box past the last whole chunk read as zeros.
// Shared memory per stage: IN [CH][R rows][128 B] (128-byte swizzle, counted
// in 128-byte rows from the stage base), S [CH][2 KB]; then the cross-warp
// partials [8][32][17] f32 and the barrier block.
// ===================================================================
struct RdArgs {
  int T, K, R, CH, stages;
  int sparts;  // factor parts per chunk: 1, or 2 (hi and lo 16-bit parts of an FP32 factor)
  int nfull;  // whole 64-column chunks
  int nst3;   // stages of whole chunks (3-D boxes)
  int tail;   // 1: one more stage with the partial chunk
  int xs;     // bytes of a stage's IN part
  void* out;     // [T][16]
  int out_kind;
  uint16_t* hi;  // optional hi/lo split of the FP32 result, [T][16] 16-bit each
  uint16_t* lo;
  unsigned long long timeout_ns;
  unsigned int* status;
  unsigned long long* trace;
};

__host__ __device__ inline int rd_r16(int R) { return (R + 15) & ~15; }
// IN part of a stage: the rows a consumer may address (the last chunk's row
// groups run R16 - R rows past its box), rounded to the 1024-byte swizzle atom
__host__ __device__ inline int rd_xs(int R, int CH) { return ((CH * R + rd_r16(R) - R) * 128 + 1023) & ~1023; }
__host__ __device__ inline int rd_ring_bytes(int R, int CH, int stages, int sparts) {
  return stages * (rd_xs(R, CH) + CH * 2048 * sparts);
}
// the role's share of shared memory (1024-byte multiple)
__host__ __device__ inline int rd_region_bytes(int R, int CH, int stages, int sparts) {
  return (rd_ring_bytes(R, CH, stages, sparts) + RD_RED_BYTES + BAR_BYTES + 1023) & ~1023;
}
// 16-byte chunk `chunk` of 128-byte row `seg` counted from a 1024-aligned base
__device__ __forceinline__ uint32_t sw128s(uint32_t base, int seg, int chunk) {
  return base + static_cast<uint32_t>(seg * 128 + ((chunk ^ (seg & 7)) << 4));
}

struct RdMaps {
  CUtensorMap x, s, x3, s3;  // 2-D (partial chunk) and 3-D (whole chunks) views
  CUtensorMap slo, s3lo;     // the same views of the factor's lo part (sparts = 2)
};

__device__ __forceinline__ RoleBars rd_bars(const RdArgs& a, uint8_t* smem) {
  return RoleBars(smem + rd_ring_bytes(a.R, a.CH, a.stages, a.sparts) + RD_RED_BYTES);
}

__device__ __forceinline__ void rowdown_init(const RdArgs& a, const RdMaps* m, uint8_t* smem, int tid) {
  if (tid == 0) rd_bars(a, smem).init(a.stages);
  if (tid == LCW * 32) {
    if (a.nst3 > 0) {
      prefetch_tmap(&m->x3);
      prefetch_tmap(&m->s3);
      if (a.sparts == 2) prefetch_tmap(&m->s3lo);
    }
    if (a.tail) {
      prefetch_tmap(&m->x);
      prefetch_tmap(&m->s);
      if (a.sparts == 2) prefetch_tmap(&m->slo);
    }
  }
}

// SLO: the factor is an FP32 one given as hi + lo 16-bit parts (sparts = 2):
// each stage also holds the lo chunks, after the hi ones, and every MMA with
// the factor is issued for both parts into the same FP32 accumulators.
template <bool BF16, bool S_KN, bool SLO = false>
__device__ void rowdown_run(int tile, const RdMaps* mp, const RdArgs& a, uint8_t* smem, int tid, int bar_id) {
  const int R16 = rd_r16(a.R);
  const int stage_bytes = a.xs + a.CH * 2048 * (SLO ? 2 : 1);
  const uint32_t sbase = smem_u32(smem);
  float* red = reinterpret_cast<float*>(smem + rd_ring_bytes(a.R, a.CH, a.stages, SLO ? 2 : 1));
  const RoleBars rb = rd_bars(a, smem);
  volatile int* abort_flag = rb.flags;
  const int warp = tid >> 5, lane = tid & 31;
  const int nst = a.nst3 + a.tail;
  const int row0 = tile * a.R;

  if (warp == LCW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    LORA_EVENT(a.trace, 0);
    int issued[LMAX_STAGES];
    for (int s = 0; s < LMAX_STAGES; ++s) issued[s] = -1;
    for (int s = 0; s < nst; ++s) {
      const int slot = s % a.stages;
      const uint32_t ph = static_cast<uint32_t>((s / a.stages) & 1);
      if (!mbar_wait(smem_u32(&rb.empty[slot]), ph ^ 1u, a.timeout_ns, abort_flag, a.status, 0x21)) {
        drain_issued(rb.full, issued, a.stages, a.status);
        return;
      }
      const uint32_t fb = smem_u32(&rb.full[slot]);
      const uint32_t xd = sbase + static_cast<uint32_t>(slot * stage_bytes);
      const uint32_t sd = xd + static_cast<uint32_t>(a.xs);
      const uint32_t sdl = sd + static_cast<uint32_t>(a.CH * 2048);  // SLO: the lo chunks
      if (s < a.nst3) {
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(a.CH * (a.R * 128 + 2048 * (SLO ? 2 : 1))));
        tma_load_3d(xd, &mp->x3, fb, 0, row0, s * a.CH);
        tma_load_3d(sd, &mp->s3, fb, 0, 0, s * a.CH);
        if (SLO) tma_load_3d(sdl, &mp->s3lo, fb, 0, 0, s * a.CH);
      } else {  // the partial last chunk
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(a.R * 128 + 2048 * (SLO ? 2 : 1)));
        tma_load_3d(xd, &mp->x, fb, a.nfull * 64, row0, 0);
        if (S_KN) {
          tma_load_3d(sd, &mp->s, fb, 0, a.nfull * 64, 0);
          if (SLO) tma_load_3d(sdl, &mp->slo, fb, 0, a.nfull * 64, 0);
        } else {
          tma_load_3d(sd, &mp->s, fb, a.nfull * 64, 0, 0);
          if (SLO) tma_load_3d(sdl, &mp->slo, fb, a.nfull * 64, 0, 0);
        }
      }
      issued[slot] = static_cast<int>(ph);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int m = lane >> 3, i = lane & 7, g = lane >> 2, c = lane & 3;
  const int cw = warp % a.CH;                     // chunk of each stage this warp takes
  const int rgs = LCW / a.CH, rg0 = warp / a.CH;  // row groups rg with rg % rgs == rg0
  const int nrg = R16 / 16;
  float acc[2][2][4], accl[SLO ? 2 : 1][2][4];  // SLO: the factor's lo-part products apart
#pragma unroll
  for (int rg = 0; rg < 2; ++rg)
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[rg][nb][q] = accl[SLO ? rg : 0][nb][q] = 0.f;
  for (int s = 0; s < nst; ++s) {
    const int slot = s % a.stages;
    const uint32_t ph = static_cast<uint32_t>((s / a.stages) & 1);
    if (!mbar_wait(smem_u32(&rb.full[slot]), ph, a.timeout_ns, abort_flag, a.status, 0x22)) break;
    if (tid == 0 && s == 0) LORA_EVENT(a.trace, 2);
    if (tid == 0 && s == nst - 1) LORA_EVENT(a.trace, 3);
    if (s < a.nst3 || cw == 0) {
      const uint32_t xb = sbase + static_cast<uint32_t>(slot * stage_bytes);
      const uint32_t sb = xb + static_cast<uint32_t>(a.xs + cw * 2048);
      const uint32_t sbl = sb + static_cast<uint32_t>(a.CH * 2048);  // SLO: this chunk's lo part
      const int seg0 = cw * a.R;  // first 128-byte row of this chunk in the stage
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // b[0..1]: n-block 0 (r 0-7), b[2..3]: n-block 1 (r 8-15)
        uint32_t b[4], bl[4];
        if (S_KN)
          ldsm_x4_t(sw32(sb, kk * 16 + (m & 1) * 8 + i, m >> 1), b);
        else
          ldsm_x4(sw128(sb, (m >> 1) * 8 + i, 2 * kk + (m & 1)), b);
        if (SLO) {
          if (S_KN)
            ldsm_x4_t(sw32(sbl, kk * 16 + (m & 1) * 8 + i, m >> 1), bl);
          else
            ldsm_x4(sw128(sbl, (m >> 1) * 8 + i, 2 * kk + (m & 1)), bl);
        }
#pragma unroll
        for (int rg = 0; rg < 2; ++rg) {
          if (rg < nrg && rg % rgs == rg0) {
            uint32_t af[4];
            ldsm_x4(sw128s(xb, seg0 + rg * 16 + (m & 1) * 8 + i, 2 * kk + (m >> 1)), af);
            mma_16816<BF16>(acc[rg][0], af, b);
            mma_16816<BF16>(acc[rg][1], af, b + 2);
            if (SLO) {  // the factor's lo part (stored times 2^11): its own sums
              mma_16816<BF16>(accl[rg][0], af, bl);
              mma_16816<BF16>(accl[rg][1], af, bl + 2);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&rb.empty[slot]));
  }
  if (SLO) {  // the lo products' sums, scaled back
#pragma unroll
    for (int rg = 0; rg < 2; ++rg)
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[rg][nb][q] += accl[SLO ? rg : 0][nb][q] * LO_UNSCALE;
  }
  // this warp's partial tile -> red[warp]; rows rg*16 + g (+8), columns nb*8 + 2c (+1)
  float* rw = red + warp * (32 * 17);
#pragma unroll
  for (int rg = 0; rg < 2; ++rg)
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      const int r0 = rg * 16 + g, col = nb * 8 + 2 * c;
      rw[r0 * 17 + col] = acc[rg][nb][0];
      rw[r0 * 17 + col + 1] = acc[rg][nb][1];
      rw[(r0 + 8) * 17 + col] = acc[rg][nb][2];
      rw[(r0 + 8) * 17 + col + 1] = acc[rg][nb][3];
    }
  group_bar(bar_id);
  if (*abort_flag) return;  // no barrier follows: a divergent decision is harmless
  for (int o = tid; o < R16 * LR; o += LCW * 32) {
    const int row = o >> 4, col = o & 15;
    float v = red[row * 17 + col];
#pragma unroll
    for (int w = 1; w < LCW; ++w) v += red[w * (32 * 17) + row * 17 + col];
    const int t = row0 + row;
    if (row < a.R && t < a.T) {
      const size_t e = static_cast<size_t>(t) * LR + col;
      store_out(a.out, a.out_kind, e, v);
      if (a.hi != nullptr) {
        const float h = round16<BF16>(v);
        a.hi[e] = bits16<BF16>(h);
        a.lo[e] = bits16<BF16>((v - h) * LO_SCALE);
      }
    }
  }
  if (tid == 0) LORA_EVENT(a.trace, 4);
}

// ===================================================================
// Role 2: column reduction over tokens, optionally fused with a row-up.
//   P[j, r] = sum_t IN[t, j] Hm[t, r]           (Hm 16-bit, or hi + lo parts)
//   UP:  OUT[t, j] = sum_r Hm[t, r] S2[r, j]    (S2 = the LoRA A, [16][J])
// Work: steps p = jb * nsteps + s over 128-column blocks jb and 128-token
// steps s; CTA c takes steps [c*N/G, (c+1)*N/G).  A stage holds the IN tile
// [128 tokens][128 columns] (two boxes {64, 128}, 128-byte swizzle), the Hm
// tile(s) [128][16] (box {16, 128}, 32-byte swizzle) and, with UP, the S2
// tile [16][128 columns] (two boxes {64, 16}).
// Column reduction: consumer warp w owns the 16-column M-tile w of the block
// over all 128 tokens of a step; MMA with M = column, K = token;
// ldmatrix.trans of the [token][column] tile gives the A fragments and of the
// [token][r] tile the B fragments.  When the CTA's range leaves a column
// block (or ends) each warp stores its partial to P[c][k] (k-th block of the
// range); a separate pass adds the partials of a block in CTA order.
// Row-up (UP): a second group of 8 warps reads the Hm and S2 tiles of the
// same stages; warp w computes tokens 16w..16w+15 of a step x 128 columns
// (M = token, N = column, K = r) and stores them straight from registers:
// the N index is permuted within each 32-column group (n-slot g of N-tile t
// is column 8*(g/2) + 2t + g%2), so each thread ends with 8 consecutive
// columns of its two rows, one 16-byte store each.
// ===================================================================
constexpr int CR_CB = 128;  // columns per block

struct CrArgs {
  int T, J, nj, nsteps, stages, G;
  long long N;   // nj * nsteps
  int max_segs;  // partial slots per CTA
  float* P;      // [G][max_segs][128][16]
  void* out;     // UP: the row-up output [T][J]
  int out_kind;
  int add;       // UP: out += scale * the row-up (one rounding) instead of out = the row-up (the kernel's
                 // ADD instance)
  int s2parts;   // UP: parts of the S2 tile, 1, or 2 (hi and lo 16-bit parts of an FP32 factor)
  float scale;   // also multiplies the ordered sums of the partials (1: unchanged bits)
  unsigned long long timeout_ns;
  unsigned int* status;
  unsigned long long* trace;
  unsigned int* cnt;  // pass 2: arrival counters, one per column block (the last CTA of a block adds its
                      // partials); pass 1 clears cnt_n of them for it
  int cnt_n;
};

// What pass 2 of the gradient finishes besides its own column reduction:
// dB from pass 1's partials (complete when pass 2 starts) and dA from its own.
struct FinArgs {
  CrArgs crb;  // pass 1's column reduction
  void* dB;    // [d_out][16]
  void* dA;    // [16][d_in]
  int kind;    // element kind of dA and dB
};

__host__ __device__ inline long long cr_start(long long c, const CrArgs& a) { return c * a.N / a.G; }

// v = old + scale * v, with old the bits read from the output
__device__ __forceinline__ void add8(const CrArgs& a, const uint4* old, float* v) {
  float o[8];
  raw8_to_float(a.out_kind, old, o);
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = fmaf(a.scale, v[k], o[k]);
}
// the CTA whose range holds step p
__host__ __device__ inline int cr_cta_of(long long p, const CrArgs& a) {
  int c = static_cast<int>(p * a.G / a.N);
  while (c + 1 < a.G && cr_start(c + 1, a) <= p) ++c;
  while (c > 0 && cr_start(c, a) > p) --c;
  return c;
}

__host__ __device__ inline int cr_stage_bytes(int nh, bool up, bool s2lo = false) {
  return 32768 + nh * 4096 + (up ? 4096 : 0) + (up && s2lo ? 4096 : 0);
}
__host__ __device__ inline int cr_region_bytes(int stages, int nh, bool up, bool s2lo = false) {
  return (stages * cr_stage_bytes(nh, up, s2lo) + BAR_BYTES + 1023) & ~1023;
}

struct CrMaps {
  CUtensorMap in, h, hlo, s2, s2lo;
};

__device__ __forceinline__ RoleBars cr_bars(const CrArgs& a, int nh, bool up, uint8_t* smem) {
  return RoleBars(smem + a.stages * cr_stage_bytes(nh, up, a.s2parts == 2));
}

// Finish of a column reduction: out element (j, r) = sum over the CTAs that
// worked on column block j / 128, in CTA order, of their partials, times
// a.scale (exact for scale 1).  One call takes 8 consecutive elements
// e0..e0+7 of the block (one output column j, ranks 0..7 or 8..15): two
// 16-byte loads per contributor, the loads of CB contributors in flight
// together.
//   transposed = 0: out is [J][16] (dB);  1: out is [16][J] (dA)
__device__ __forceinline__ void cr_finish(const CrArgs& a, void* out, int kind, int transposed, int jb, int e0) {
  const int c0 = cr_cta_of(static_cast<long long>(jb) * a.nsteps, a);
  const int c1 = cr_cta_of(static_cast<long long>(jb + 1) * a.nsteps - 1, a);
  const int k0 = jb - static_cast<int>(cr_start(c0, a) / a.nsteps);  // slot of c0; every later one uses slot 0
  constexpr int CB = 8;  // contributors whose loads are in flight together
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int cb = c0; cb <= c1; cb += CB) {
    float4 x[CB][2];
#pragma unroll
    for (int q = 0; q < CB; ++q) {
      const int cc = cb + q;
      if (cc <= c1) {
        const float* src = a.P + (static_cast<size_t>(cc) * a.max_segs + (cc == c0 ? k0 : 0)) * (CR_CB * LR) + e0;
        x[q][0] = __ldcg(reinterpret_cast<const float4*>(src));
        x[q][1] = __ldcg(reinterpret_cast<const float4*>(src) + 1);
      } else {
        x[q][0] = x[q][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int q = 0; q < CB; ++q) {
      v[0] += x[q][0].x;
      v[1] += x[q][0].y;
      v[2] += x[q][0].z;
      v[3] += x[q][0].w;
      v[4] += x[q][1].x;
      v[5] += x[q][1].y;
      v[6] += x[q][1].z;
      v[7] += x[q][1].w;
    }
  }
  const int j = jb * CR_CB + (e0 >> 4), r0 = e0 & 15;
  if (j >= a.J) return;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    store_out(out, kind, transposed ? static_cast<size_t>(r0 + k) * a.J + j : static_cast<size_t>(j) * LR + r0 + k,
              v[k] * a.scale);
}

template <bool HILO, bool UP>
__device__ __forceinline__ void colred_init(const CrArgs& a, const CrMaps* m, uint8_t* smem, int tid) {
  if (tid == 0) cr_bars(a, HILO ? 2 : 1, UP, smem).init(a.stages, UP ? 2 * LCW : LCW);
  if (tid == (UP ? 2 * LCW : LCW) * 32) {
    prefetch_tmap(&m->in);
    prefetch_tmap(&m->h);
    if (HILO) prefetch_tmap(&m->hlo);
    if (UP) prefetch_tmap(&m->s2);
    if (UP && a.s2parts == 2) prefetch_tmap(&m->s2lo);
  }
}

// ADD staging of the old outputs a row-up warp rewrites in a step, double
// buffered (the copies of step s + 1 fly during step s): per warp and buffer
// [4 column groups q][2 rows][W words][32 lanes] 16-byte chunks (W = 2 for
// FP32 outputs, else 1); lane-major so that a warp's accesses are conflict-free
__host__ __device__ inline int ru_old_buf(int out_kind) { return 8 * (out_kind == EK_F32 ? 2 : 1) * 512; }
__host__ __device__ inline int ru_old_bytes(int out_kind) { return LCW * 2 * ru_old_buf(out_kind); }

// SLO (with UP): S2 is an FP32 factor given as hi + lo 16-bit parts; the lo
// tile follows the hi one in each stage and the row-up adds its products too.
//
// FIN (pass 2 of the gradient): the consumers first add up their share of
// dB from pass 1's partials; at the end of its part of a column block each
// CTA counts itself in, and the last of the block's CTAs adds the block's
// partials (in CTA order, as every other column reduction) into dA.  No CTA
// waits for another: the last one to arrive does the sum.
template <bool BF16, bool HILO, bool UP, bool ADD = false, bool SLO = false, bool FIN = false>
__device__ void colred_run(const CrMaps* mp, const CrArgs& a, uint8_t* smem, int tid,
                           const FinArgs* fin = nullptr) {
  constexpr int NH = HILO ? 2 : 1;
  constexpr int SB = 32768 + NH * 4096 + (UP ? 4096 : 0) + (UP && SLO ? 4096 : 0);
  constexpr int HOFF = 32768, S2OFF = 32768 + NH * 4096;
  const int cta = blockIdx.x;
  if (cta >= a.G) return;
  const long long p0 = cr_start(cta, a), p1 = cr_start(cta + 1, a);
  const int nst = static_cast<int>(p1 - p0);
  const uint32_t sbase = smem_u32(smem);
  const RoleBars rb = cr_bars(a, NH, UP, smem);
  volatile int* abort_flag = rb.flags;
  const int warp = tid >> 5, lane = tid & 31;

  if (warp == (UP ? 2 * LCW : LCW)) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    LORA_EVENT(a.trace, 0);
    int issued[LMAX_STAGES];
    for (int s = 0; s < LMAX_STAGES; ++s) issued[s] = -1;
    for (int s = 0; s < nst; ++s) {
      const long long p = p0 + s;
      const int jb = static_cast<int>(p / a.nsteps), t0 = static_cast<int>(p % a.nsteps) * CR_RS;
      const int slot = s % a.stages;
      const uint32_t ph = static_cast<uint32_t>((s / a.stages) & 1);
      if (!mbar_wait(smem_u32(&rb.empty[slot]), ph ^ 1u, a.timeout_ns, abort_flag, a.status, 0x23)) {
        drain_issued(rb.full, issued, a.stages, a.status);
        return;
      }
      const uint32_t fb = smem_u32(&rb.full[slot]);
      const uint32_t dst = sbase + static_cast<uint32_t>(slot * SB);
      mbar_arrive_expect_tx(fb, static_cast<uint32_t>(SB));
      tma_load_3d(dst, &mp->in, fb, jb * CR_CB, t0, 0);
      tma_load_3d(dst + 16384, &mp->in, fb, jb * CR_CB + 64, t0, 0);
      tma_load_3d(dst + HOFF, &mp->h, fb, 0, t0, 0);
      if (HILO) tma_load_3d(dst + HOFF + 4096, &mp->hlo, fb, 0, t0, 0);
      if (UP) {
        tma_load_3d(dst + S2OFF, &mp->s2, fb, jb * CR_CB, 0, 0);
        tma_load_3d(dst + S2OFF + 2048, &mp->s2, fb, jb * CR_CB + 64, 0, 0);
      }
      if (UP && SLO) {
        tma_load_3d(dst + S2OFF + 4096, &mp->s2lo, fb, jb * CR_CB, 0, 0);
        tma_load_3d(dst + S2OFF + 6144, &mp->s2lo, fb, jb * CR_CB + 64, 0, 0);
      }
      issued[slot] = static_cast<int>(ph);
    }
    return;
  }

  const int m = lane >> 3, i = lane & 7, g = lane >> 2, c = lane & 3;
  if (UP && warp >= LCW) {
    // ---------------------------------------------- row-up warps (UP only)
    // warp LCW + w computes tokens 16w..16w+15 of every step x 128 columns
    const int w = warp - LCW;
    uint32_t bup[4][4][2];  // B fragments of the column block (4 groups of 32 columns x 4 N-tiles)
    bool uok = true;
    const int ow = a.out_kind == EK_F32 ? 2 : 1, esz = a.out_kind == EK_F32 ? 4 : 2;  // ADD staging words, bytes
    const uint32_t obase0 = sbase + static_cast<uint32_t>(cr_region_bytes(a.stages, NH, UP, SLO) +
                                                          w * 2 * ru_old_buf(a.out_kind));
    // ADD: copy the old outputs of step sp into staging buffer sp & 1 (one commit group)
    auto stage_old = [&](int sp) {
      const long long pp = p0 + sp;
      const int jbp = static_cast<int>(pp / a.nsteps);
      const int ra = static_cast<int>(pp % a.nsteps) * CR_RS + w * 16 + g;
      const uint32_t ob = obase0 + static_cast<uint32_t>((sp & 1) * ru_old_buf(a.out_kind));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int jq = jbp * CR_CB + 32 * q + 8 * c;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = ra + 8 * h;
          if (jq < a.J && row < a.T) {
            const char* src = static_cast<const char*>(a.out) + (static_cast<size_t>(row) * a.J + jq) * esz;
            for (int wd = 0; wd < ow; ++wd) cp_async16(ob + ((q * 2 + h) * ow + wd) * 512 + lane * 16, src + 16 * wd);
          }
        }
      }
      cp_async_commit();
    };
    if (ADD && nst > 0) stage_old(0);
    for (int s = 0; s < nst; ++s) {
      const long long p = p0 + s;
      const int jb = static_cast<int>(p / a.nsteps), t0 = static_cast<int>(p % a.nsteps) * CR_RS;
      const int slot = s % a.stages;
      const uint32_t ph = static_cast<uint32_t>((s / a.stages) & 1);
      // ADD: the next step's old outputs start moving (an empty group at the end)
      if (ADD) {
        if (uok && s + 1 < nst)
          stage_old(s + 1);
        else
          cp_async_commit();
      }
      if (uok && !mbar_wait(smem_u32(&rb.full[slot]), ph, a.timeout_ns, abort_flag, a.status, 0x25)) uok = false;
      const uint32_t st = sbase + static_cast<uint32_t>(slot * SB);
      uint32_t ah[4] = {0u, 0u, 0u, 0u}, al[4] = {0u, 0u, 0u, 0u};
      if (uok) {
        if (s == 0 || p % a.nsteps == 0) {
          // b0 = rows r 2c,2c+1 and b1 = rows 2c+8,2c+9 of the S2 tile at
          // column 32q + 8(g/2) + 2t + g%2 (S2 tiles: 64 columns each)
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int col = 32 * (q & 1) + 8 * (g >> 1) + 2 * t + (g & 1);
              const uint32_t s2b = st + S2OFF + (q >> 1) * 2048;
              uint32_t v[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int r = (u >> 1) * 8 + 2 * c + (u & 1);
                uint16_t x;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(x) : "r"(sw128(s2b, r, col >> 3) + (col & 7) * 2));
                v[u] = x;
              }
              bup[q][t][0] = v[0] | (v[1] << 16);
              bup[q][t][1] = v[2] | (v[3] << 16);
            }
        }
        ldsm_x4(sw32(st + HOFF, w * 16 + (m & 1) * 8 + i, m >> 1), ah);
        if (HILO) ldsm_x4(sw32(st + HOFF + 4096, w * 16 + (m & 1) * 8 + i, m >> 1), al);
      }
      if (!SLO || !uok) {  // SLO reads the stage's lo tile below: it frees the stage after that
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&rb.empty[slot]));  // the stage is no longer read
      }
      if (!uok) continue;
      const int ra = t0 + w * 16 + g, rb2 = ra + 8;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float d[4][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          // the lo parts (of Hm, and of an FP32 S2) are stored times 2^11: their
          // products have their own sum, scaled back before it joins d
          float dl[4] = {0.f, 0.f, 0.f, 0.f};
          d[t][0] = d[t][1] = d[t][2] = d[t][3] = 0.f;
          mma_16816<BF16>(d[t], ah, bup[q][t]);
          if (HILO) mma_16816<BF16>(dl, al, bup[q][t]);
          if (SLO) {
            // the lo fragment, read from this stage as bup was (the lo part times
            // the lo part of Hm is below FP32 resolution and is left out)
            const int col = 32 * (q & 1) + 8 * (g >> 1) + 2 * t + (g & 1);
            const uint32_t s2l = st + S2OFF + 4096 + (q >> 1) * 2048;
            uint32_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int r = (u >> 1) * 8 + 2 * c + (u & 1);
              uint16_t x;
              asm volatile("ld.shared.u16 %0, [%1];" : "=h"(x) : "r"(sw128(s2l, r, col >> 3) + (col & 7) * 2));
              v[u] = x;
            }
            const uint32_t bl[2] = {v[0] | (v[1] << 16), v[2] | (v[3] << 16)};
            mma_16816<BF16>(dl, ah, bl);
          }
          if (HILO || SLO) {
#pragma unroll
            for (int e = 0; e < 4; ++e) d[t][e] += dl[e] * LO_UNSCALE;
          }
        }
        const int j = jb * CR_CB + 32 * q + 8 * c;  // this thread's 8 consecutive columns
        if (ADD && q == 0) cp_async_wait_group1();  // this step's staged old outputs have landed
        if (j < a.J) {
          float v[8];
          uint4 oa[2], ob[2];  // add: the old outputs, from the staging
          if (ADD) {
            const uint32_t obs = obase0 + static_cast<uint32_t>((s & 1) * ru_old_buf(a.out_kind));
#pragma unroll
            for (int wd = 0; wd < 2; ++wd)
              if (wd < ow) {
                oa[wd] = ld_shared_v4(obs + ((q * 2) * ow + wd) * 512 + lane * 16);
                ob[wd] = ld_shared_v4(obs + ((q * 2 + 1) * ow + wd) * 512 + lane * 16);
              }
          }
          if (ra < a.T) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              v[2 * t] = d[t][0];
              v[2 * t + 1] = d[t][1];
            }
            if (ADD) add8(a, oa, v);
            store8(a.out, a.out_kind, static_cast<size_t>(ra) * a.J + j, v);
          }
          if (rb2 < a.T) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              v[2 * t] = d[t][2];
              v[2 * t + 1] = d[t][3];
            }
            if (ADD) add8(a, ob, v);
            store8(a.out, a.out_kind, static_cast<size_t>(rb2) * a.J + j, v);
          }
        }
      }
      if (SLO) {  // the lo tile has been read
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&rb.empty[slot]));
      }
    }
    if (ADD) cp_async_wait_all();  // no copy outlives the kernel (a step given up after a failed wait)
    if (w == 0 && lane == 0) LORA_EVENT(a.trace, 9);
    return;
  }

  // ------------------------------------------------------ col-red consumers
  if (FIN) {
    // this CTA's share of dB (pass 1's partials are complete and visible),
    // eight elements of a column block per task, dealt out across the CTAs
    // (task i to CTA i % G) so that no CTA starts its own steps late
    const int per = CR_CB * LR / 8, total = fin->crb.nj * per;
    for (int i = tid * a.G + cta; i < total; i += a.G * LCW * 32)
      cr_finish(fin->crb, fin->dB, fin->kind, 0, i / per, (i - (i / per) * per) * 8);
    if (tid == 0) LORA_EVENT(a.trace, 6);
  }
  // warp w: columns 16w..16w+15 of the block = chunks 2(w%4), 2(w%4)+1 of IN tile w/4
  float acc[2][4], accl[2][4];  // hi and lo products: two independent chains
#pragma unroll
  for (int nb = 0; nb < 2; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nb][e] = accl[nb][e] = 0.f;
  int seg = 0;
  bool ok = true;
  for (int s = 0; s < nst; ++s) {
    const long long p = p0 + s;
    const int slot = s % a.stages;
    const uint32_t ph = static_cast<uint32_t>((s / a.stages) & 1);
    if (ok && !mbar_wait(smem_u32(&rb.full[slot]), ph, a.timeout_ns, abort_flag, a.status, 0x24)) ok = false;
    if (tid == 0 && s == 0) LORA_EVENT(a.trace, 2);
    if (tid == 0 && s == nst - 1) LORA_EVENT(a.trace, 3);
    const uint32_t st = sbase + static_cast<uint32_t>(slot * SB);
    const uint32_t inb = st + (warp >> 2) * 16384;
    if (ok) {
#pragma unroll
      for (int ks = 0; ks < CR_RS / 16; ++ks) {
        uint32_t af[4], bf[4];
        ldsm_x4_t(sw128(inb, ks * 16 + (m >> 1) * 8 + i, (warp & 3) * 2 + (m & 1)), af);
        ldsm_x4_t(sw32(st + HOFF, ks * 16 + (m & 1) * 8 + i, m >> 1), bf);
        mma_16816<BF16>(acc[0], af, bf);
        mma_16816<BF16>(acc[1], af, bf + 2);
        if (HILO) {
          ldsm_x4_t(sw32(st + HOFF + 4096, ks * 16 + (m & 1) * 8 + i, m >> 1), bf);
          mma_16816<BF16>(accl[0], af, bf);
          mma_16816<BF16>(accl[1], af, bf + 2);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&rb.empty[slot]));
    // end of this CTA's part of a column block: this warp's 16 columns of the partial
    if ((p + 1) % a.nsteps == 0 || s == nst - 1) {
      if (ok) {
        float* dst = a.P + (static_cast<size_t>(cta) * a.max_segs + seg) * CR_CB * LR;
        const int jl = warp * 16 + g;
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          const int r = nb * 8 + 2 * c;
          // the lo parts were stored times 2^11: their sums scaled back
          *reinterpret_cast<float2*>(dst + jl * LR + r) =
              make_float2(acc[nb][0] + accl[nb][0] * LO_UNSCALE, acc[nb][1] + accl[nb][1] * LO_UNSCALE);
          *reinterpret_cast<float2*>(dst + (jl + 8) * LR + r) =
              make_float2(acc[nb][2] + accl[nb][2] * LO_UNSCALE, acc[nb][3] + accl[nb][3] * LO_UNSCALE);
        }
      }
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nb][e] = accl[nb][e] = 0.f;
      ++seg;
      if (FIN) {
        const int jb = static_cast<int>(p / a.nsteps);
        __threadfence();  // this thread's partial, visible device-wide before the CTA counts itself in
        group_bar(1);     // every consumer warp has stored its columns of the partial
        if (tid == 0) {
          int last = 0;
          if (ok) {
            const int c0 = cr_cta_of(static_cast<long long>(jb) * a.nsteps, a);
            const int c1 = cr_cta_of(static_cast<long long>(jb + 1) * a.nsteps - 1, a);
            last = atomicAdd(&a.cnt[jb], 1u) == static_cast<unsigned int>(c1 - c0);
          }
          rb.flags[3] = last;
        }
        group_bar(1);
        if (rb.flags[3]) {
          __threadfence();  // the other CTAs' partials, seen after their arrivals
          static_assert(CR_CB * LR == LCW * 32 * 8, "eight elements of a column block per consumer thread");
          if (tid == 0) LORA_EVENT(a.trace, 7);
          cr_finish(a, fin->dA, fin->kind, 1, jb, tid * 8);
          if (tid == 0) a.cnt[jb] = 0u;  // ready for the next call (pass 1 clears them too)
          if (tid == 0) LORA_EVENT(a.trace, 8);
        }
      }
    }
  }
  if (tid == 0) LORA_EVENT(a.trace, 4);
}

// ===================================================================
// Role 3: row-up.  OUT[t, j] = sum_r Hm[t, r] S2(j, r), S2 = the LoRA B [J][16].
// A warp owns 32 output columns of a 256-column CTA slab and walks 16-row
// blocks blk = cta_t, cta_t + n_t, ...; the Hm fragments of RU_PRE blocks are
// loaded before the first of them is used.  Output columns are permuted
// across the four n-blocks so that each thread ends with 8 consecutive
// columns of its two rows (one 16-byte store per row).  K = 16 is permuted
// too: MMA slots 2c,2c+1 <- r 4c,4c+1 and slots 2c+8,2c+9 <- r 4c+2,4c+3, so
// 8 bytes of Hm feed a fragment.
// ===================================================================
constexpr int RU_PRE = 4;

struct RuArgs {
  const uint16_t* H;
  const uint16_t* S2;
  const float* S2f;      // SLO: the factor in FP32, split into 16-bit hi + lo fragments in registers
  void* out;
  int out_kind;
  int T, J, n_t;
  int add;      // out += scale * H S2^T (one rounding, in FP32) instead of out = H S2^T
  float scale;
};

// out[i .. i+8) = v, or (ADD) out = old + scale * v with old the bits read
// earlier from the same place
template <bool ADD>
__device__ __forceinline__ void put8(const RuArgs& a, size_t i, float* v, const uint4* old) {
  if (ADD) {
    float o[8];
    raw8_to_float(a.out_kind, old, o);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = fmaf(a.scale, v[k], o[k]);
  }
  store8(a.out, a.out_kind, i, v);
}

// ADD: the old outputs of the RU_PRE blocks are read together with their Hm
// fragments, so that every thread has all of its reads in flight at once
// instead of one 16-byte read ahead of each store.
template <bool BF16, bool ADD, bool SLO = false>
__device__ void rowup_role(int cta_j, int cta_t, const RuArgs& a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int J = a.J, T = a.T;
  const int j0 = cta_j * 256 + warp * 32;
  if (j0 >= J) return;
  // B fragments for the 4 n-blocks: column of n-slot g in block jb
  uint32_t bfr[4][2], bfl[SLO ? 4 : 1][2];
#pragma unroll
  for (int jb = 0; jb < 4; ++jb) {
    const int col = j0 + 8 * (g >> 1) + 2 * jb + (g & 1);
    if (SLO) {  // r = 4c .. 4c+3 of the FP32 factor: hi = RNE(w), lo = RNE(w - hi), packed in pairs
      const float4 w = col < J ? *reinterpret_cast<const float4*>(a.S2f + static_cast<size_t>(col) * LR + 4 * c)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      const float wv[4] = {w.x, w.y, w.z, w.w};
      uint32_t hb[4], lb[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float h = round16<BF16>(wv[e]);
        hb[e] = bits16<BF16>(h);
        lb[e] = bits16<BF16>((wv[e] - h) * LO_SCALE);
      }
      bfr[jb][0] = hb[0] | (hb[1] << 16);
      bfr[jb][1] = hb[2] | (hb[3] << 16);
      bfl[SLO ? jb : 0][0] = lb[0] | (lb[1] << 16);
      bfl[SLO ? jb : 0][1] = lb[2] | (lb[3] << 16);
    } else {
      const uint2 v = col < J ? ld8(a.S2 + static_cast<size_t>(col) * LR + 4 * c) : make_uint2(0u, 0u);
      bfr[jb][0] = v.x;
      bfr[jb][1] = v.y;
    }
  }
  const bool colv = j0 + 8 * c < J;  // this thread's 8 output columns exist (J % 8 == 0)
  const int nblk = (T + 15) / 16;
  for (int blk0 = cta_t; blk0 < nblk; blk0 += RU_PRE * a.n_t) {
    uint2 ha[RU_PRE], hb[RU_PRE];
    uint4 oa[ADD ? RU_PRE : 1][2], ob[ADD ? RU_PRE : 1][2];
#pragma unroll
    for (int u = 0; u < RU_PRE; ++u) {
      const int ra = (blk0 + u * a.n_t) * 16 + g, rb = ra + 8;
      const uint2 z = make_uint2(0u, 0u);
      ha[u] = ra < T ? ld8(a.H + static_cast<size_t>(ra) * LR + 4 * c) : z;
      hb[u] = rb < T ? ld8(a.H + static_cast<size_t>(rb) * LR + 4 * c) : z;
      if (ADD && colv) {
        if (ra < T) load8_raw(a.out, a.out_kind, static_cast<size_t>(ra) * J + j0 + 8 * c, oa[u]);
        if (rb < T) load8_raw(a.out, a.out_kind, static_cast<size_t>(rb) * J + j0 + 8 * c, ob[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < RU_PRE; ++u) {
      const int blk = blk0 + u * a.n_t;
      if (blk >= nblk) break;  // warp-uniform: the MMAs below need the whole warp
      const int ra = blk * 16 + g, rb = ra + 8;
      float acc[4][4];
#pragma unroll
      for (int jb = 0; jb < 4; ++jb) acc[jb][0] = acc[jb][1] = acc[jb][2] = acc[jb][3] = 0.f;
      const uint32_t ah[4] = {ha[u].x, hb[u].x, ha[u].y, hb[u].y};
#pragma unroll
      for (int jb = 0; jb < 4; ++jb) {
        mma_16816<BF16>(acc[jb], ah, bfr[jb]);
        if (SLO) {  // the factor's lo part (stored times 2^11): its own sum, scaled back
          float l[4] = {0.f, 0.f, 0.f, 0.f};
          mma_16816<BF16>(l, ah, bfl[SLO ? jb : 0]);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[jb][e] += l[e] * LO_UNSCALE;
        }
      }
      // thread (g, c): rows ra / rb, columns j0 + 8c + 2*jb + {0,1}
      if (colv) {
        float v[8];
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
          v[2 * jb] = acc[jb][0];
          v[2 * jb + 1] = acc[jb][1];
        }
        if (ra < T) put8<ADD>(a, static_cast<size_t>(ra) * J + j0 + 8 * c, v, oa[ADD ? u : 0]);
        if (rb < T) {
#pragma unroll
          for (int jb = 0; jb < 4; ++jb) {
            v[2 * jb] = acc[jb][2];
            v[2 * jb + 1] = acc[jb][3];
          }
          put8<ADD>(a, static_cast<size_t>(rb) * J + j0 + 8 * c, v, ob[ADD ? u : 0]);
        }
      }
    }
  }
}

// ===================================================================
// kernels
// ===================================================================
__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

// H = X A^T
template <bool BF16, bool SLO>
__global__ void __launch_bounds__(LGROUP, 1) lora_down_kernel(const __grid_constant__ RdMaps maps, const RdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  if (threadIdx.x == 0) LORA_EVENT(a.trace, 5);
  rowdown_init(a, &maps, smem, threadIdx.x);
  fence_mbar_init();
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  rowdown_run<BF16, false, SLO>(blockIdx.x, &maps, a, smem, threadIdx.x, 1);
}

// Y = H B^T
template <bool BF16, bool ADD, bool SLO>
__global__ void __launch_bounds__(256) lora_up_kernel(const RuArgs a) {
  pdl_wait();
  pdl_trigger();
  rowup_role<BF16, ADD, SLO>(blockIdx.x, blockIdx.y, a);
}

// Pass 1 over dY, two roles per CTA (threads 0..287 and 288..575):
// row-down dH = dY B (FP32, and its hi/lo parts) for the CTA's rows, and the
// column reduction dB = dY^T H over the CTA's share of (column block, step)
// space (partials only).
template <bool BF16, bool SLO>
__global__ void __launch_bounds__(2 * LGROUP, 1)
    lora_grad1_kernel(const __grid_constant__ RdMaps rmaps, const __grid_constant__ CrMaps cmaps, const RdArgs rd,
                      const CrArgs cr, int rd_region) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  uint8_t* smem_cr = smem + rd_region;
  const int tid = threadIdx.x;
  if (tid == 0) LORA_EVENT(rd.trace, 5);
  if (tid < LGROUP)
    rowdown_init(rd, &rmaps, smem, tid);
  else
    colred_init<false, false>(cr, &cmaps, smem_cr, tid - LGROUP);
  fence_mbar_init();
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  // pass 2's arrival counters start at zero (whatever an earlier call left)
  if (blockIdx.x == 0)
    for (int i = tid; i < cr.cnt_n; i += blockDim.x) cr.cnt[i] = 0u;
  if (tid < LGROUP) {
    if (static_cast<int>(blockIdx.x) * rd.R < rd.T) rowdown_run<BF16, true, SLO>(blockIdx.x, &rmaps, rd, smem, tid, 1);
  } else {
    colred_run<BF16, false, false>(&cmaps, cr, smem_cr, tid - LGROUP);
  }
}

// Pass 2 over X: each step reads an X tile with its dH hi/lo tiles and the
// matching columns of A; one warp group accumulates dA^T = X^T dH (partials,
// then dA by the last CTA of each column block; first, dB from pass 1's
// partials), the other writes the dX = dH A tile.
template <bool BF16, bool ADD, bool SLO>
__global__ void __launch_bounds__(LGROUP_UP, 1)
    lora_grad2_kernel(const __grid_constant__ CrMaps cmaps, const CrArgs cr, const __grid_constant__ FinArgs fin) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  const int tid = threadIdx.x;
  if (tid == 0) LORA_EVENT(cr.trace, 5);
  colred_init<true, true>(cr, &cmaps, smem, tid);
  fence_mbar_init();
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  colred_run<BF16, true, true, ADD, SLO, true>(&cmaps, cr, smem, tid, &fin);
}

// ===================================================================
// host side
// ===================================================================
static int clampi(int64_t v, int lo, int hi) { return static_cast<int>(v < lo ? lo : (v > hi ? hi : v)); }

// Raise a kernel's dynamic shared-memory limit (once per device and kernel).
static cudaError_t allow_smem(const void* kern) { return raise_smem_limit(kern, SMEM_LIMIT); }

static unsigned long long* trace_ptr(int which) {
#ifdef TG_TRACE
  if (const char* e = getenv("TG_TRACE_ADDR"))
    return reinterpret_cast<unsigned long long*>(strtoull(e, nullptr, 0)) + static_cast<size_t>(which) * 8192 * 16;
#endif
  (void)which;
  return nullptr;
}

// Row-down plan: R rows per CTA (about one CTA per SM, at most 32 rows),
// CH 64-column chunks per stage, as many stages as fit in smem_budget.
static RdArgs rd_plan(int64_t T, int64_t K, int sms, int CH, int smem_budget, int sparts = 1) {
  RdArgs r{};
  r.sparts = sparts;
  r.T = static_cast<int>(T);
  r.K = static_cast<int>(K);
  r.R = clampi((T + sms - 1) / sms, 1, 32);
  r.nfull = static_cast<int>(K / 64);
  r.CH = clampi(CH, 1, r.nfull > 0 ? r.nfull : 1);
  while (LCW % r.CH) --r.CH;  // CH divides the 8 consumer warps
  r.nst3 = (r.nfull + r.CH - 1) / r.CH;
  r.tail = K % 64 != 0 ? 1 : 0;
  r.xs = rd_xs(r.R, r.CH);
  const int per_stage = r.xs + r.CH * 2048 * sparts;
  r.stages = clampi((smem_budget - RD_RED_BYTES - BAR_BYTES - 1023) / per_stage, 1, LMAX_STAGES);
  if (r.stages > r.nst3 + r.tail) r.stages = r.nst3 + r.tail;
  return r;
}

// 2-D maps (the partial last chunk) and 3-D chunked views (whole chunks) of
// the streamed tensor IN [T][K] and of the factor S (and of its lo part Slo,
// when the factor is an FP32 one split into two 16-bit parts)
static bool rd_factor_maps(CUtensorMap* s2d, CUtensorMap* s3d, const void* S, int kind, const RdArgs& r, bool s_kn) {
  const uint64_t K = r.K;
  if (s_kn) {
    if (!encode_tmap_3d(s2d, S, kind, LR, K, 1, LR * 2, LR * K * 2, LR, 64, 32)) return false;
  } else {
    if (!encode_tmap_3d(s2d, S, kind, K, LR, 1, K * 2, K * LR * 2, 64, LR, 128)) return false;
  }
  if (r.nfull == 0) {  // no whole chunk: the 3-D view is never used
    *s3d = *s2d;
    return true;
  }
  const uint64_t nf = r.nfull;
  if (s_kn) {  // S [K][16] as [chunk][64 k][16]
    const uint64_t d[3] = {LR, 64, nf}, st[2] = {LR * 2, 64 * LR * 2};
    const uint32_t b[3] = {LR, 64, static_cast<uint32_t>(r.CH)};
    return encode_tmap_nd(s3d, S, kind, 3, d, st, b, 32);
  }
  // S [16][K] as [chunk][16][64]
  const uint64_t d[3] = {64, LR, nf}, st[2] = {K * 2, 128};
  const uint32_t b[3] = {64, LR, static_cast<uint32_t>(r.CH)};
  return encode_tmap_nd(s3d, S, kind, 3, d, st, b, 128);
}

static bool rd_maps(RdMaps* m, const void* in, const void* S, const void* Slo, int kind, const RdArgs& r, bool s_kn) {
  const uint64_t T = r.T, K = r.K;
  if (!encode_tmap_3d(&m->x, in, kind, K, T, 1, K * 2, K * T * 2, 64, r.R, 128)) return false;
  if (!rd_factor_maps(&m->s, &m->s3, S, kind, r, s_kn)) return false;
  if (Slo) {
    if (!rd_factor_maps(&m->slo, &m->s3lo, Slo, kind, r, s_kn)) return false;
  } else {
    m->slo = m->s;
    m->s3lo = m->s3;
  }
  if (r.nfull == 0) {  // no whole chunk: the 3-D view is never used
    m->x3 = m->x;
    return true;
  }
  // IN as [chunk][row][64]
  const uint64_t d[3] = {64, T, static_cast<uint64_t>(r.nfull)}, st[2] = {K * 2, 128};
  const uint32_t b[3] = {64, static_cast<uint32_t>(r.R), static_cast<uint32_t>(r.CH)};
  return encode_tmap_nd(&m->x3, in, kind, 3, d, st, b, 128);
}

// Column-reduction plan over (at most) G CTAs.
static CrArgs cr_plan(int64_t T, int64_t J, int G, int stages) {
  CrArgs c{};
  c.T = static_cast<int>(T);
  c.J = static_cast<int>(J);
  c.nj = static_cast<int>((J + CR_CB - 1) / CR_CB);
  c.nsteps = static_cast<int>((T + CR_RS - 1) / CR_RS);
  c.N = static_cast<long long>(c.nj) * c.nsteps;
  // the fewest CTAs with the same largest share as G of them: ranges of equal
  // length, so fewer CTAs share a column block (their partials are summed)
  const long long per = (c.N > 0 && G > 0) ? (c.N + G - 1) / G : 1;
  c.G = static_cast<int>((c.N + per - 1) / per);
  c.stages = stages;
  c.scale = 1.f;
  c.max_segs = 1;
  for (int cc = 0; cc < c.G; ++cc) {
    const long long s0 = cr_start(cc, c), s1 = cr_start(cc + 1, c);
    const int segs = static_cast<int>((s1 - 1) / c.nsteps - s0 / c.nsteps + 1);
    if (segs > c.max_segs) c.max_segs = segs;
  }
  return c;
}

static bool cr_maps(CrMaps* m, const void* in, const void* H, const void* Hlo, const void* S2, int kind, int64_t T,
                    int64_t J, const void* S2lo = nullptr) {
  if (!encode_tmap_3d(&m->in, in, kind, J, T, 1, J * 2, J * T * 2, 64, CR_RS, 128)) return false;
  if (!encode_tmap_3d(&m->h, H, kind, LR, T, 1, LR * 2, LR * T * 2, LR, CR_RS, 32)) return false;
  m->hlo = m->h;
  m->s2 = m->h;
  m->s2lo = m->h;
  if (Hlo && !encode_tmap_3d(&m->hlo, Hlo, kind, LR, T, 1, LR * 2, LR * T * 2, LR, CR_RS, 32)) return false;
  if (S2 && !encode_tmap_3d(&m->s2, S2, kind, J, LR, 1, J * 2, J * LR * 2, 64, LR, 128)) return false;
  if (S2lo && !encode_tmap_3d(&m->s2lo, S2lo, kind, J, LR, 1, J * 2, J * LR * 2, 64, LR, 128)) return false;
  return true;
}

size_t lora_down_ws_bytes(int64_t, int64_t, int64_t, int) { return 0; }

// ---- FP32 factors: each is split once per call into 16-bit hi and lo parts
// (hi = RNE(w), lo = RNE(w - hi), so hi + lo is w to within 2^-18 of |w| in
// bf16), which the streaming kernels multiply in turn into the same FP32 sums.

// one or two factors in one launch: element i < n1 of w1 -> (hi1, hi1 + n1),
// element n1 + i of the index space -> element i of w2 -> (hi2, hi2 + n2)
template <bool BF16>
__global__ void __launch_bounds__(256)
    lora_split_kernel(const float* w1, uint16_t* hi1, int64_t n1, const float* w2, uint16_t* hi2, int64_t n2) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n1 + n2;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool first = i < n1;
    const int64_t k = first ? i : i - n1, n = first ? n1 : n2;
    uint16_t* hi = first ? hi1 : hi2;
    const float v = (first ? w1 : w2)[k];
    const float h = round16<BF16>(v);
    hi[k] = bits16<BF16>(h);
    hi[n + k] = bits16<BF16>((v - h) * LO_SCALE);
  }
}

// bytes of the hi and lo parts of an FP32 factor of n elements (256-byte multiple)
static size_t parts_bytes(int64_t n) { return (static_cast<size_t>(n) * 4 + 255) / 256 * 256; }

// parts of w1 [n1] at hi1 (hi, then lo) and, if n2 > 0, of w2 [n2] at hi2
static cudaError_t split_factors(const float* w1, uint16_t* hi1, int64_t n1, const float* w2, uint16_t* hi2, int64_t n2,
                                 int in_kind, cudaStream_t st) {
  const int64_t n = n1 + n2;
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  return launch_k(in_kind == EK_BF16 ? lora_split_kernel<true> : lora_split_kernel<false>, dim3(blocks), dim3(256), 0,
                  st, w1, hi1, n1, w2, hi2, n2);
}

size_t lora_w32_ws_bytes(int op, int64_t T, int64_t d_in, int64_t d_out, int sms) {
  if (op == 0) return parts_bytes(LR * d_in);   // down: A
  if (op == 1) return 0;                         // up: B is split in registers
  return lora_grad_ws_bytes(T, d_in, d_out, LR, sms) + parts_bytes(LR * d_in) + parts_bytes(LR * d_out);
}

cudaError_t lora_down_launch(const LoraArgs& a) {
  if (a.T == 0) return cudaSuccess;
  const int sp = a.w32 ? 2 : 1;
  RdArgs rd = rd_plan(a.T, a.d_in, a.num_sms, 8, 212 * 1024, sp);
  rd.out = a.out;
  rd.out_kind = a.out_kind;
  rd.hi = rd.lo = nullptr;
  rd.timeout_ns = a.timeout_ns;
  rd.status = a.status;
  rd.trace = trace_ptr(0);
  const void* S = a.A;
  const void* Slo = nullptr;
  if (a.w32) {  // A is FP32: its hi and lo parts in the workspace
    uint16_t* hi = reinterpret_cast<uint16_t*>(a.ws);
    cudaError_t e =
        split_factors(static_cast<const float*>(a.A), hi, LR * a.d_in, nullptr, nullptr, 0, a.in_kind, a.stream);
    if (e != cudaSuccess) return e;
    S = hi;
    Slo = hi + LR * a.d_in;
  }
  alignas(64) RdMaps maps;
  if (!rd_maps(&maps, a.X, S, Slo, a.in_kind, rd, false)) return cudaErrorInvalidValue;
  const bool bf = a.in_kind == EK_BF16;
  auto kern = a.w32 ? (bf ? lora_down_kernel<true, true> : lora_down_kernel<false, true>)
                    : (bf ? lora_down_kernel<true, false> : lora_down_kernel<false, false>);
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>((a.T + rd.R - 1) / rd.R);
  return launch_k(kern, dim3(grid), dim3(LGROUP), rd_region_bytes(rd.R, rd.CH, rd.stages, sp) + 1024, a.stream,
                  maps, rd);
}

// Row-block CTAs per 256-column slab: at most `ctas` CTAs in all (rounded
// down, so that the grid is one wave of resident CTAs, with no straggler
// CTAs left for a second one)
static int rowup_nt(int64_t T, int64_t J, int ctas) {
  const int64_t nj = (J + 255) / 256, nblk = (T + 15) / 16;
  return clampi(ctas / nj, 1, static_cast<int>(nblk));
}

cudaError_t lora_up_launch(const LoraArgs& a) {
  const int nj = static_cast<int>((a.d_out + 255) / 256);
  if (nj == 0 || a.T == 0) return cudaSuccess;
  RuArgs ru{};
  ru.H = static_cast<const uint16_t*>(a.H);
  ru.S2 = static_cast<const uint16_t*>(a.B);
  if (a.w32) ru.S2f = static_cast<const float*>(a.B);  // split into hi + lo in the kernel
  ru.out = a.out;
  ru.out_kind = a.out_kind;
  ru.T = static_cast<int>(a.T);
  ru.J = static_cast<int>(a.d_out);
  // one wave: 4 CTAs per SM fit the plain kernel's registers, 3 the FP32-factor one's, 2 the adding one's
  ru.n_t = rowup_nt(a.T, a.d_out, (a.add ? 2 : a.w32 ? 3 : 4) * a.num_sms);
  ru.add = a.add;
  ru.scale = a.scale;
  const bool bf = a.in_kind == EK_BF16;
  auto k = a.w32 ? (bf ? lora_up_kernel<true, false, true> : lora_up_kernel<false, false, true>)
           : a.add ? (bf ? lora_up_kernel<true, true, false> : lora_up_kernel<false, true, false>)
                   : (bf ? lora_up_kernel<true, false, false> : lora_up_kernel<false, false, false>);
  return launch_k(k, dim3(nj, ru.n_t), dim3(256), 0, a.stream, ru);
}

// ---- gradient: plans and workspace

struct GradPlan {
  RdArgs rd;   // pass 1 row-down
  CrArgs crb;  // pass 1 column reduction (dB)
  CrArgs cra;  // pass 2 column reduction + row-up (dA, dX)
  int g1;
  size_t dh, hi, lo, pb, pa, cnt, total;  // workspace layout
};
static size_t up256(size_t v) { return (v + 255) / 256 * 256; }

static GradPlan grad_plan(int64_t T, int64_t d_in, int64_t d_out, int sms, int out_kind, int sparts = 1) {
  GradPlan g;
  g.rd = rd_plan(T, d_out, sms, G1_RD_CH, G1_RD_BUDGET, sparts);
  g.g1 = static_cast<int>((T + g.rd.R - 1) / g.rd.R);
  g.crb = cr_plan(T, d_out, g.g1, G1_CR_STAGES);
  g.cra = cr_plan(T, d_in, G2_CTAS_PER_SM * sms, G2_CR_STAGES);
  g.cra.out_kind = out_kind;
  g.dh = 0;
  g.hi = g.dh + up256(static_cast<size_t>(T) * LR * 4);
  g.lo = g.hi + up256(static_cast<size_t>(T) * LR * 2);
  g.pb = g.lo + up256(static_cast<size_t>(T) * LR * 2);
  g.pa = g.pb + up256(static_cast<size_t>(g.crb.G) * g.crb.max_segs * CR_CB * LR * 4);
  g.cnt = g.pa + up256(static_cast<size_t>(g.cra.G) * g.cra.max_segs * CR_CB * LR * 4);
  g.total = g.cnt + up256(static_cast<size_t>(g.cra.nj) * 4);
  return g;
}

size_t lora_grad_ws_bytes(int64_t T, int64_t d_in, int64_t d_out, int64_t, int sms) {
  // the partial layout does not depend on the output type
  return grad_plan(T, d_in, d_out, sms, EK_F32).total;
}

// a.out = dA, a.out2 = dB, a.out3 = dX, a.out4 = optional dH (FP32)
cudaError_t lora_grad_launch(const LoraArgs& a) {
  const int sp = a.w32 ? 2 : 1;
  GradPlan gp = grad_plan(a.T, a.d_in, a.d_out, a.num_sms, a.out_kind, sp);
  char* base = reinterpret_cast<char*>(a.ws);
  float* dH = a.out4 ? static_cast<float*>(a.out4) : reinterpret_cast<float*>(base + gp.dh);
  uint16_t* hi = reinterpret_cast<uint16_t*>(base + gp.hi);
  uint16_t* lo = reinterpret_cast<uint16_t*>(base + gp.lo);
  const bool bf = a.in_kind == EK_BF16;
  const int kind = a.in_kind;
  // factors: 16-bit as given, or (FP32) their hi and lo parts after the plan's workspace
  const void* Ahi = a.A;
  const void* Bhi = a.B;
  const void* Alo = nullptr;
  const void* Blo = nullptr;
  if (a.w32) {
    uint16_t* pa = reinterpret_cast<uint16_t*>(base + gp.total);
    uint16_t* pb = reinterpret_cast<uint16_t*>(base + gp.total + parts_bytes(LR * a.d_in));
    cudaError_t e = split_factors(static_cast<const float*>(a.A), pa, LR * a.d_in, static_cast<const float*>(a.B), pb,
                                  a.d_out * LR, kind, a.stream);
    if (e != cudaSuccess) return e;
    Ahi = pa;
    Alo = pa + LR * a.d_in;
    Bhi = pb;
    Blo = pb + a.d_out * LR;
  }

  // ---- pass 1: dH (row-down over dY with B) and dB partials (col-red over dY with H)
  RdArgs& rd = gp.rd;
  rd.out = dH;
  rd.out_kind = EK_F32;
  rd.hi = hi;
  rd.lo = lo;
  rd.timeout_ns = a.timeout_ns;
  rd.status = a.status;
  rd.trace = trace_ptr(0);
  CrArgs& crb = gp.crb;
  crb.P = reinterpret_cast<float*>(base + gp.pb);
  crb.cnt = reinterpret_cast<unsigned int*>(base + gp.cnt);  // cleared by pass 1 for pass 2
  crb.cnt_n = gp.cra.nj;
  crb.scale = a.add ? a.scale : 1.f;
  crb.timeout_ns = a.timeout_ns;
  crb.status = a.status;
  crb.trace = trace_ptr(1);
  alignas(64) RdMaps rmaps;
  alignas(64) CrMaps cmaps1;
  if (!rd_maps(&rmaps, a.dY, Bhi, Blo, kind, rd, true)) return cudaErrorInvalidValue;
  if (!cr_maps(&cmaps1, a.dY, a.H, nullptr, nullptr, kind, a.T, a.d_out)) return cudaErrorInvalidValue;
  // the two roles share the SM's shared memory: fewer row-down stages if they do not fit
  while (rd.stages > 1 &&
         1024 + rd_region_bytes(rd.R, rd.CH, rd.stages, sp) + cr_region_bytes(crb.stages, 1, false) > SMEM_LIMIT)
    --rd.stages;
  const int rd_region = rd_region_bytes(rd.R, rd.CH, rd.stages, sp);
  const int smem1 = 1024 + rd_region + cr_region_bytes(crb.stages, 1, false);
  auto k1 = a.w32 ? (bf ? lora_grad1_kernel<true, true> : lora_grad1_kernel<false, true>)
                  : (bf ? lora_grad1_kernel<true, false> : lora_grad1_kernel<false, false>);
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(k1));
  if (e != cudaSuccess) return e;
  e = launch_k(k1, dim3(gp.g1), dim3(2 * LGROUP), smem1, a.stream, rmaps, cmaps1, rd, crb, rd_region);
  if (e != cudaSuccess) return e;

  // ---- pass 2: dA partials (col-red over X with dH hi/lo) and dX (row-up of the same tiles)
  CrArgs& cra = gp.cra;
  cra.P = reinterpret_cast<float*>(base + gp.pa);
  cra.cnt = reinterpret_cast<unsigned int*>(base + gp.cnt);
  cra.out = a.out3;  // dX
  cra.add = a.add;   // dX += scale * dH A
  cra.scale = a.add ? a.scale : 1.f;
  cra.timeout_ns = a.timeout_ns;
  cra.status = a.status;
  cra.trace = trace_ptr(2);
  alignas(64) CrMaps cmaps2;
  cra.s2parts = sp;
  if (!cr_maps(&cmaps2, a.X, hi, lo, Ahi, kind, a.T, a.d_in, Alo)) return cudaErrorInvalidValue;
  auto k2 = a.w32 ? (bf ? lora_grad2_kernel<true, false, true> : lora_grad2_kernel<false, false, true>)
            : a.add ? (bf ? lora_grad2_kernel<true, true, false> : lora_grad2_kernel<false, true, false>)
                    : (bf ? lora_grad2_kernel<true, false, false> : lora_grad2_kernel<false, false, false>);
  e = allow_smem(reinterpret_cast<const void*>(k2));
  if (e != cudaSuccess) return e;
  // the adding instance stages the old dX of two steps: one operand stage
  // fewer for 16-bit dX, two for FP32
  if (a.add) cra.stages = G2_CR_STAGES - (a.out_kind == EK_F32 ? 2 : 1);
  const int smem2 =
      1024 + cr_region_bytes(cra.stages, 2, true, a.w32 != 0) + (a.add ? ru_old_bytes(a.out_kind) : 0);
  // and the sums of the partials: dB (pass 1's) and dA (its own), FP32 for
  // FP32 factors (the gradients of FP32 weights), else the output type
  FinArgs fin{};
  fin.crb = crb;
  fin.dB = a.out2;
  fin.dA = a.out;
  fin.kind = a.w32 ? static_cast<int>(EK_F32) : a.out_kind;
  return launch_k(k2, dim3(cra.G), dim3(LGROUP_UP), smem2, a.stream, cmaps2, cra, fin);
}

}  // namespace tg
