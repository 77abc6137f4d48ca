// attn_common.cuh -- pieces shared by the fused attention kernels (forward
// attn_tc.cu, backward attn_bwd_tc.cu): the tensor-memory A-operand MMA, a
// bulk copy, the base-2 exponential, the hi + lo 16-bit split, the rescale
// of accumulator columns, and (forward) the exchange of per-row values
// between the two warps that share a TMEM lane quadrant.
//
// Every tcgen05.ld / tcgen05.st is a warp-collective (.sync.aligned)
// instruction: the row code around them keeps whole warps together and
// makes per-row decisions with per-lane values, never with a branch around
// the tensor-memory access.
#pragma once
#include "ptx.cuh"

namespace tg {
namespace attn {

constexpr int D = 64;             // head dimension
constexpr int BT = 128;           // rows per tile; keys (or queries) per block
constexpr int TILE = BT * D * 2;  // 16 KB: 128 rows of 128 bytes
constexpr int ROW_WARPS = 8;      // two warps per TMEM lane quadrant, each half of a block's columns
constexpr int THREADS = 64 + 32 * ROW_WARPS;  // warp 0 TMA, warp 1 MMA, warps 2..9 rows

// D[tmem] (+)= A[tmem] * B[smem]: the A operand (M = 128 rows x K = 16) is 8
// TMEM columns of packed 16-bit pairs, row i in lane i.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// global -> shared bulk copy completing on an mbarrier (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// 2^x by the SFU instruction (results below 2^-126 flush to zero; relative
// error about 2^-22, far inside the products' 1e-5 bound)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^e for an integer e in [-126, 127], exactly
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

// Two FP32 values as hi = RNE16(v), lo = RNE16(v - hi), packed pairwise.
template <bool BF16>
__device__ __forceinline__ void split2(float v0, float v1, uint32_t* hi, uint32_t* lo) {
  if constexpr (BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 f = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - f.x, v1 - f.y);
    *hi = *reinterpret_cast<const uint32_t*>(&h);
    *lo = *reinterpret_cast<const uint32_t*>(&l);
  } else {
    const __half2 h = __floats2half2_rn(v0, v1);
    const float2 f = __half22float2(h);
    const __half2 l = __floats2half2_rn(v0 - f.x, v1 - f.y);
    *hi = *reinterpret_cast<const uint32_t*>(&h);
    *lo = *reinterpret_cast<const uint32_t*>(&l);
  }
}

// 32 FP32 values of a row as one TMEM chunk of the A operand: hi pairs in
// the chunk's first 16 columns, lo pairs in its last 16
template <bool BF16>
__device__ __forceinline__ void split32(const float* v, uint32_t* w) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) split2<BF16>(v[e], v[e + 1], &w[e / 2], &w[16 + e / 2]);
}

// The two row warps of TMEM lane quadrant q (half 0 and half 1) exchange one
// value per row: each writes its own, both wait on the pair's named barrier
// (ids 1..4), each reads the other's.  buf: [2 slots][4 quadrants][2 halves][32].
__device__ __forceinline__ float pair_exchange(float* buf, int slot, int q, int half, int lane, float v) {
  buf[((slot * 4 + q) * 2 + half) * 32 + lane] = v;
  asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory");
  return buf[((slot * 4 + q) * 2 + (half ^ 1)) * 32 + lane];
}

__device__ __forceinline__ void store_row32(void* out, int out_kind, size_t base, const float* v) {
  if (out_kind == EK_F32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + base);
#pragma unroll
    for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + base);
    const bool bf = out_kind == EK_BF16;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float* f = v + 8 * e;
      dst[e] = bf ? make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                               pack_bf16x2(f[6], f[7]))
                  : make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                               pack_f16x2(f[6], f[7]));
    }
  }
}

// Multiply 32 TMEM columns of this warp's rows by a per-row factor (1 for
// rows that keep their scale).  Warp-collective: call with the whole warp.
__device__ __forceinline__ void rescale32(uint32_t taddr, float f) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
  tmem_st_32x32b_x32(taddr, r);
}

}  // namespace attn
}  // namespace tg
