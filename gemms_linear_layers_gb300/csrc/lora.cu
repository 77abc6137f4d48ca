// lora.cu -- rank-16 LoRA products as HBM-streaming kernels.
//
// Page "Twice the training speed on a BC-250 from tuned matrix kernels",
// section "Tuning the kernels": the rank-16 LoRA matrices are among the
// products a training step runs.  Every one of them reads or writes one
// [T, d] tensor and touches only small [*, 16] factors otherwise, so they are
// bound by HBM bandwidth, not by the tensor cores.  Each kernel streams its
// big operand exactly once with 16-byte vector loads or stores and keeps the
// rank-16 side in registers; the arithmetic runs on warp-level mma.sync
// (m16n8k16, FP32 accumulate) because FP32 FFMA alone cannot keep up with
// ~16 flop per byte at HBM speed.
//
// Register layouts.  mma.sync m16n8k16 splits a warp's lane into g = lane/4
// and c = lane%4.  A reduction index may be permuted freely as long as both
// operands use the same permutation, and an output index may be permuted as
// long as the store undoes it; the kernels use this to feed fragments
// straight from 16-byte loads:
//   * a thread that loads 8 consecutive k values of a row feeds two MMAs:
//     values 0-3 go to MMA 0 (slots 2c,2c+1 <- k 0,1; slots 2c+8,2c+9 <- k 2,3)
//     and values 4-7 to MMA 1;
//   * for reductions over tokens, movmatrix.trans turns row-major register
//     tiles into the (pairs along tokens) layout the fragments need.
// FP32 operands (the gradient dH) are split into hi + lo 16-bit parts and
// both parts are multiplied, so dH keeps ~16 significant bits instead of 8.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "tg_internal.h"

namespace tg {

constexpr int LR = 16;  // the rank these kernels are written for
constexpr int LTHREADS = 256;

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ uint2 ld8(const void* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
__device__ __forceinline__ float4 ld16f(const void* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ uint32_t movtrans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}
template <bool BF16>
__device__ __forceinline__ float round16(float x) {
  return BF16 ? __bfloat162float(__float2bfloat16_rn(x)) : __half2float(__float2half_rn(x));
}
// x = hi + lo + O(2^-16 |x|): both parts as packed pairs
template <bool BF16>
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const float h0 = round16<BF16>(x0), h1 = round16<BF16>(x1);
  hi = pack16x2<BF16>(h0, h1);
  lo = pack16x2<BF16>(x0 - h0, x1 - h1);
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

// ===================================================================
// Role 1: row-down.  OUT[t, r] = sum_k IN[t, k] * S[r, k]   (r < 16)
//   IN [T, K] 16-bit (the streamed tensor), S [16, K] 16-bit row-major.
// CTA = 16 rows; its 8 warps take 64-wide K chunks round-robin, two chunks
// per iteration (16 x 16-byte loads in flight per thread); the 8 partial
// 16x16 tiles are added in warp order through shared memory.
// ===================================================================
struct RdFrag {
  uint4 xa[2], xb[2], s0[2], s1[2];
};

// loads of one 64-wide K chunk (zeros past K or past T)
__device__ __forceinline__ void rowdown_load(RdFrag& f, const uint16_t* pa, const uint16_t* pb, const uint16_t* S,
                                             int K, int k0, bool va, bool vb, int g, int c) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int k = k0 + 32 * h + 8 * c;
    const bool kv = k < K;
    const uint4 z = make_uint4(0, 0, 0, 0);
    f.xa[h] = (kv && va) ? ld_stream16(pa + k) : z;
    f.xb[h] = (kv && vb) ? ld_stream16(pb + k) : z;
    f.s0[h] = kv ? ld16(S + static_cast<size_t>(g) * K + k) : z;
    f.s1[h] = kv ? ld16(S + static_cast<size_t>(8 + g) * K + k) : z;
  }
}

template <bool BF16>
__device__ __forceinline__ void rowdown_mma(const RdFrag& f, float (&acc)[2][4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    {
      const uint32_t a[4] = {f.xa[h].x, f.xb[h].x, f.xa[h].y, f.xb[h].y};
      const uint32_t b0[2] = {f.s0[h].x, f.s0[h].y}, b1[2] = {f.s1[h].x, f.s1[h].y};
      mma_16816<BF16>(acc[0], a, b0);
      mma_16816<BF16>(acc[1], a, b1);
    }
    {
      const uint32_t a[4] = {f.xa[h].z, f.xb[h].z, f.xa[h].w, f.xb[h].w};
      const uint32_t b0[2] = {f.s0[h].z, f.s0[h].w}, b1[2] = {f.s1[h].z, f.s1[h].w};
      mma_16816<BF16>(acc[0], a, b0);
      mma_16816<BF16>(acc[1], a, b1);
    }
  }
}

template <bool BF16>
__device__ void rowdown_role(int cta, const uint16_t* __restrict__ IN, const uint16_t* __restrict__ S,
                             void* __restrict__ OUT, int out_kind, int T, int K, float* red /* [8][16][17] */) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int t0 = cta * 16;
  const int ra = t0 + g, rb = t0 + g + 8;
  const bool va = ra < T, vb = rb < T;
  const uint16_t* pa = IN + static_cast<size_t>(va ? ra : 0) * K;
  const uint16_t* pb = IN + static_cast<size_t>(vb ? rb : 0) * K;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  const int nch = (K + 63) / 64;
  // two chunks per iteration: all 16 loads are issued before the MMAs
  for (int ch = warp; ch < nch; ch += 16) {
    RdFrag f0, f1;
    rowdown_load(f0, pa, pb, S, K, ch * 64, va, vb, g, c);
    rowdown_load(f1, pa, pb, S, K, (ch + 8) * 64, va, vb, g, c);  // zeros when past K
    rowdown_mma<BF16>(f0, acc);
    rowdown_mma<BF16>(f1, acc);
  }
  // acc[nb]: rows g / g+8, columns 8*nb + 2c, +1
  float* rw = red + warp * (16 * 17);
#pragma unroll
  for (int nb = 0; nb < 2; ++nb) {
    rw[g * 17 + 8 * nb + 2 * c] = acc[nb][0];
    rw[g * 17 + 8 * nb + 2 * c + 1] = acc[nb][1];
    rw[(g + 8) * 17 + 8 * nb + 2 * c] = acc[nb][2];
    rw[(g + 8) * 17 + 8 * nb + 2 * c + 1] = acc[nb][3];
  }
  __syncthreads();
  {
    const int o = threadIdx.x;  // 256 threads: one output each
    const int rr = o >> 4, cc = o & 15;
    float s = red[rr * 17 + cc];
#pragma unroll
    for (int w = 1; w < 8; ++w) s += red[w * (16 * 17) + rr * 17 + cc];
    if (t0 + rr < T) store_out(OUT, out_kind, static_cast<size_t>(t0 + rr) * LR + cc, s);
  }
}

// ===================================================================
// Role 2: row-up.  OUT[t, j] = sum_r Hm[t, r] * S2[j, r]
//   Hm [T, 16] 16-bit, or FP32 (HF32: split into hi + lo), S2 [J, 16] 16-bit.
// A warp owns 32 output columns of a 256-column CTA slab and walks 16-row
// blocks.  Output columns are permuted across the four n-blocks so that each
// thread ends with 8 consecutive columns of its two rows: one 16-byte store
// per row.  K = 16 is permuted too: slots 2c,2c+1 <- r 4c,4c+1 and slots
// 2c+8,2c+9 <- r 4c+2,4c+3, so 8 bytes of Hm and of S2 feed a fragment.
// ===================================================================
template <bool BF16, bool HF32>
__device__ void rowup_role(int cta_j, int cta_t, int n_t, const void* __restrict__ Hm,
                           const uint16_t* __restrict__ S2, void* __restrict__ OUT, int out_kind, int T, int J) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int j0 = cta_j * 256 + warp * 32;
  if (j0 >= J) return;
  // B fragments for the 4 n-blocks: column of n-slot g in block jb
  uint32_t bfr[4][2];
#pragma unroll
  for (int jb = 0; jb < 4; ++jb) {
    const int col = j0 + 8 * (g >> 1) + 2 * jb + (g & 1);
    const uint2 v = col < J ? ld8(S2 + static_cast<size_t>(col) * LR + 4 * c) : make_uint2(0, 0);
    bfr[jb][0] = v.x;
    bfr[jb][1] = v.y;
  }
  const bool colv = j0 + 8 * c < J;  // this thread's 8 output columns exist (J % 8 == 0)
  const int nblk = (T + 15) / 16;
  for (int blk = cta_t; blk < nblk; blk += n_t) {
    const int ra = blk * 16 + g, rb = ra + 8;
    const bool va = ra < T, vb = rb < T;
    float acc[4][4];
#pragma unroll
    for (int jb = 0; jb < 4; ++jb) acc[jb][0] = acc[jb][1] = acc[jb][2] = acc[jb][3] = 0.f;
    if (HF32) {
      const float* H = static_cast<const float*>(Hm);
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 ha = va ? ld16f(H + static_cast<size_t>(ra) * LR + 4 * c) : z;
      const float4 hb = vb ? ld16f(H + static_cast<size_t>(rb) * LR + 4 * c) : z;
      uint32_t ah[4], al[4];
      split2<BF16>(ha.x, ha.y, ah[0], al[0]);
      split2<BF16>(hb.x, hb.y, ah[1], al[1]);
      split2<BF16>(ha.z, ha.w, ah[2], al[2]);
      split2<BF16>(hb.z, hb.w, ah[3], al[3]);
#pragma unroll
      for (int jb = 0; jb < 4; ++jb) {
        mma_16816<BF16>(acc[jb], ah, bfr[jb]);
        mma_16816<BF16>(acc[jb], al, bfr[jb]);
      }
    } else {
      const uint16_t* H = static_cast<const uint16_t*>(Hm);
      const uint2 z = make_uint2(0, 0);
      const uint2 ha = va ? ld8(H + static_cast<size_t>(ra) * LR + 4 * c) : z;
      const uint2 hb = vb ? ld8(H + static_cast<size_t>(rb) * LR + 4 * c) : z;
      const uint32_t a[4] = {ha.x, hb.x, ha.y, hb.y};
#pragma unroll
      for (int jb = 0; jb < 4; ++jb) mma_16816<BF16>(acc[jb], a, bfr[jb]);
    }
    // thread (g, c): rows ra / rb, columns j0 + 8c + 2*jb + {0,1}
    if (colv) {
      float v[8];
      if (va) {
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
          v[2 * jb] = acc[jb][0];
          v[2 * jb + 1] = acc[jb][1];
        }
        store8(OUT, out_kind, static_cast<size_t>(ra) * J + j0 + 8 * c, v);
      }
      if (vb) {
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
          v[2 * jb] = acc[jb][2];
          v[2 * jb + 1] = acc[jb][3];
        }
        store8(OUT, out_kind, static_cast<size_t>(rb) * J + j0 + 8 * c, v);
      }
    }
  }
}

// ===================================================================
// Role 3: column reduction over tokens.
//   P[part, j, r] = sum_{t in part} IN[t, j] * Hm[t, r]
// IN [T, J] 16-bit (streamed), Hm [T, 16] 16-bit or FP32 (hi + lo).
// A warp owns 32 columns and a row range; per 16-row step each thread loads
// 8 columns of rows g and g+8 (16 bytes each).  movmatrix.trans turns word w
// of those loads into (token pairs 2c,2c+1 ; column jcol(g, w)) -- the A
// fragment of an MMA whose M index is the column (M slot g <- word 2p,
// slot g+8 <- word 2p+1) and whose K index is the token.  The Hm rows are
// transposed the same way into B fragments (n slot g <- r = 4(g>>1)+2v+(g&1)).
// CTA = 8 warps = 2 column groups x 4 row sub-ranges; the 4 sub-range
// partials are added in order through shared memory.
// ===================================================================
template <bool BF16, bool HF32>
__device__ __forceinline__ void colred_step(const uint16_t* IN, const void* Hm, int T, int J, int t0, int j0,
                                            int g, int c, float (&acc)[2][2][4], float (&accl)[2][2][4]) {
  const int ra = t0 + g, rb = t0 + g + 8;
  const bool va = ra < T, vb = rb < T;
  const int jc = j0 + 8 * c;
  const bool jv = jc < J;
  const uint4 z4 = make_uint4(0, 0, 0, 0);
  const uint4 xa = (va && jv) ? ld_stream16(IN + static_cast<size_t>(ra) * J + jc) : z4;
  const uint4 xb = (vb && jv) ? ld_stream16(IN + static_cast<size_t>(rb) * J + jc) : z4;
  // A fragments: [p][reg]
  uint32_t a[2][4];
  a[0][0] = movtrans(xa.x);
  a[0][1] = movtrans(xa.y);
  a[0][2] = movtrans(xb.x);
  a[0][3] = movtrans(xb.y);
  a[1][0] = movtrans(xa.z);
  a[1][1] = movtrans(xa.w);
  a[1][2] = movtrans(xb.z);
  a[1][3] = movtrans(xb.w);
  // B fragments: [v][reg]
  uint32_t b[2][2], bl[2][2];
  if (HF32) {
    const float* H = static_cast<const float*>(Hm);
    const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 ha = va ? ld16f(H + static_cast<size_t>(ra) * LR + 4 * c) : zf;
    const float4 hb = vb ? ld16f(H + static_cast<size_t>(rb) * LR + 4 * c) : zf;
    uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
    split2<BF16>(ha.x, ha.y, h0, l0);  // row g,   r 4c, 4c+1
    split2<BF16>(ha.z, ha.w, h1, l1);  // row g,   r 4c+2, 4c+3
    split2<BF16>(hb.x, hb.y, h2, l2);  // row g+8, r 4c, 4c+1
    split2<BF16>(hb.z, hb.w, h3, l3);  // row g+8, r 4c+2, 4c+3
    b[0][0] = movtrans(h0);
    b[1][0] = movtrans(h1);
    b[0][1] = movtrans(h2);
    b[1][1] = movtrans(h3);
    bl[0][0] = movtrans(l0);
    bl[1][0] = movtrans(l1);
    bl[0][1] = movtrans(l2);
    bl[1][1] = movtrans(l3);
  } else {
    const uint16_t* H = static_cast<const uint16_t*>(Hm);
    const uint2 z2 = make_uint2(0, 0);
    const uint2 ha = va ? ld8(H + static_cast<size_t>(ra) * LR + 4 * c) : z2;
    const uint2 hb = vb ? ld8(H + static_cast<size_t>(rb) * LR + 4 * c) : z2;
    b[0][0] = movtrans(ha.x);
    b[1][0] = movtrans(ha.y);
    b[0][1] = movtrans(hb.x);
    b[1][1] = movtrans(hb.y);
  }
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      mma_16816<BF16>(acc[p][v], a[p], b[v]);
      if (HF32) mma_16816<BF16>(accl[p][v], a[p], bl[v]);
    }
}

template <bool BF16, bool HF32>
__device__ void colred_role(int cta_j, int part, int parts, const uint16_t* __restrict__ IN,
                            const void* __restrict__ Hm, float* __restrict__ P, int T, int J,
                            float* red /* [4][64][17] */) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int cg = warp & 1;   // column group within the CTA
  const int sub = warp >> 1; // row sub-range
  const int j0 = cta_j * 64 + cg * 32;
  // rows of this part, split into 4 sub-ranges of whole 16-row steps
  const int nsteps = (T + 15) / 16;
  const int s_begin = static_cast<int>((static_cast<int64_t>(nsteps) * part) / parts);
  const int s_end = static_cast<int>((static_cast<int64_t>(nsteps) * (part + 1)) / parts);
  const int per = (s_end - s_begin + 3) / 4;
  const int my_b = s_begin + sub * per;
  const int my_e = min(s_end, my_b + per);
  float acc[2][2][4], accl[2][2][4];
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int v = 0; v < 2; ++v)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[p][v][q] = accl[p][v][q] = 0.f;
  int s = my_b;
  for (; s + 1 < my_e; s += 2) {
    colred_step<BF16, HF32>(IN, Hm, T, J, s * 16, j0, g, c, acc, accl);
    colred_step<BF16, HF32>(IN, Hm, T, J, (s + 1) * 16, j0, g, c, acc, accl);
  }
  if (s < my_e) colred_step<BF16, HF32>(IN, Hm, T, J, s * 16, j0, g, c, acc, accl);
  // acc[p][v]: rows (M slots) g / g+8 -> columns jcol(g, 2p) / jcol(g, 2p+1);
  // columns (N slots) 2c, 2c+1 -> r = 4c + 2v, 4c + 2v + 1
  float* rs = red + sub * (64 * 17);
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int jl0 = cg * 32 + 8 * (g >> 1) + 2 * (2 * p) + (g & 1);
      const int jl1 = cg * 32 + 8 * (g >> 1) + 2 * (2 * p + 1) + (g & 1);
      const int r0 = 4 * c + 2 * v;
      rs[jl0 * 17 + r0] = acc[p][v][0] + accl[p][v][0];
      rs[jl0 * 17 + r0 + 1] = acc[p][v][1] + accl[p][v][1];
      rs[jl1 * 17 + r0] = acc[p][v][2] + accl[p][v][2];
      rs[jl1 * 17 + r0 + 1] = acc[p][v][3] + accl[p][v][3];
    }
  __syncthreads();
  for (int o = threadIdx.x; o < 64 * LR; o += LTHREADS) {
    const int jl = o >> 4, r = o & 15;
    float sum = red[jl * 17 + r];
#pragma unroll
    for (int w = 1; w < 4; ++w) sum += red[w * (64 * 17) + jl * 17 + r];
    const int j = cta_j * 64 + jl;
    if (j < J) P[(static_cast<size_t>(part) * J + j) * LR + r] = sum;
  }
}

// ===================================================================
// kernels
// ===================================================================
template <bool BF16>
__global__ void __launch_bounds__(LTHREADS) lora_down_kernel(const uint16_t* X, const uint16_t* A, void* H,
                                                             int out_kind, int T, int d_in) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8 * 16 * 17];
  rowdown_role<BF16>(blockIdx.x, X, A, H, out_kind, T, d_in, red);
}

template <bool BF16>
__global__ void __launch_bounds__(LTHREADS) lora_up_kernel(const uint16_t* H, const uint16_t* B, void* Y,
                                                           int out_kind, int T, int d_out, int n_t) {
  pdl_wait();
  pdl_trigger();
  rowup_role<BF16, false>(blockIdx.x, blockIdx.y, n_t, H, B, Y, out_kind, T, d_out);
}

// prep: Bt[r][o] = B[o][r], At[i][r] = A[r][i]
__global__ void lora_prep_kernel(const uint16_t* A, const uint16_t* B, uint16_t* At, uint16_t* Bt, int d_in,
                                 int d_out) {
  pdl_wait();
  pdl_trigger();
  const int64_t nA = static_cast<int64_t>(d_in) * LR, nB = static_cast<int64_t>(d_out) * LR;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < nA + nB;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (e < nA) {
      const int64_t i = e / LR, r = e % LR;
      At[e] = A[r * d_in + i];
    } else {
      const int64_t f = e - nA, r = f / d_out, o = f % d_out;
      Bt[f] = B[o * LR + r];
    }
  }
}

// pass 1 over dY: row-down CTAs compute dH = dY B (FP32), column CTAs
// compute partial dB over token parts
template <bool BF16>
__global__ void __launch_bounds__(LTHREADS) lora_grad1_kernel(const uint16_t* dY, const uint16_t* Bt,
                                                              const uint16_t* H, float* dH, float* Pb, int T,
                                                              int d_out, int n_rowdown, int nj_b, int parts_b) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[4 * 64 * 17];
  const int b = blockIdx.x;
  if (b < n_rowdown) {
    rowdown_role<BF16>(b, dY, Bt, dH, EK_F32, T, d_out, red);
  } else {
    const int q = b - n_rowdown;
    colred_role<BF16, false>(q % nj_b, q / nj_b, parts_b, dY, H, Pb, T, d_out, red);
  }
}

// pass 2: column CTAs compute partial dA^T over token parts from X and the
// FP32 dH; row-up CTAs write dX = dH A
template <bool BF16>
__global__ void __launch_bounds__(LTHREADS) lora_grad2_kernel(const uint16_t* X, const float* dH,
                                                              const uint16_t* At, void* dX, int out_kind,
                                                              float* Pa, int T, int d_in, int n_colred, int nj_a,
                                                              int parts_a, int nj_x, int n_tx) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[4 * 64 * 17];
  const int b = blockIdx.x;
  if (b < n_colred) {
    colred_role<BF16, true>(b % nj_a, b / nj_a, parts_a, X, dH, Pa, T, d_in, red);
  } else {
    const int q = b - n_colred;
    rowup_role<BF16, true>(q % nj_x, q / nj_x, n_tx, dH, At, dX, out_kind, T, d_in);
  }
}

// pass 3: dB[o][r] = sum_parts Pb ; dA[r][i] = sum_parts Pa[.][i][r] (parts in order)
__global__ void lora_grad3_kernel(const float* Pb, const float* Pa, void* dB, void* dA, int out_kind, int d_out,
                                  int d_in, int parts_b, int parts_a) {
  pdl_wait();
  pdl_trigger();
  const int64_t nB = static_cast<int64_t>(d_out) * LR, nA = static_cast<int64_t>(d_in) * LR;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < nB + nA;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (e < nB) {
      float s = Pb[e];
      for (int p = 1; p < parts_b; ++p) s += Pb[static_cast<int64_t>(p) * nB + e];
      store_out(dB, out_kind, e, s);
    } else {
      const int64_t f = e - nB;  // f = r * d_in + i  (dA layout)
      const int64_t r = f / d_in, i = f % d_in;
      const int64_t src = i * LR + r;
      float s = Pa[src];
      for (int p = 1; p < parts_a; ++p) s += Pa[static_cast<int64_t>(p) * nA + src];
      store_out(dA, out_kind, f, s);
    }
  }
}

// ===================================================================
// host launchers
// ===================================================================
static int clampi(int64_t v, int lo, int hi) { return static_cast<int>(v < lo ? lo : (v > hi ? hi : v)); }

static int rowup_nt(int64_t T, int64_t J, int sms) {
  const int64_t nj = (J + 255) / 256, nblk = (T + 15) / 16;
  return clampi((4LL * sms + nj - 1) / nj, 1, static_cast<int>(nblk));
}
static int colred_parts(int64_t T, int64_t J, int sms) {
  const int64_t nj = (J + 63) / 64, nsteps = (T + 15) / 16;
  return clampi((2LL * sms + nj - 1) / nj, 1, static_cast<int>(nsteps < 64 ? nsteps : 64));
}

size_t lora_down_ws_bytes(int64_t, int64_t, int64_t, int) { return 0; }

cudaError_t lora_down_launch(const LoraArgs& a) {
  const int grid = static_cast<int>((a.T + 15) / 16);
  if (grid == 0) return cudaSuccess;
  return launch_k(a.in_kind == EK_BF16 ? lora_down_kernel<true> : lora_down_kernel<false>, dim3(grid),
                  dim3(LTHREADS), 0, a.stream, static_cast<const uint16_t*>(a.X), static_cast<const uint16_t*>(a.A),
                  a.out, a.out_kind, static_cast<int>(a.T), static_cast<int>(a.d_in));
}

cudaError_t lora_up_launch(const LoraArgs& a) {
  const int nj = static_cast<int>((a.d_out + 255) / 256);
  const int nt = rowup_nt(a.T, a.d_out, a.num_sms);
  if (nj == 0 || a.T == 0) return cudaSuccess;
  dim3 grid(nj, nt);
  return launch_k(a.in_kind == EK_BF16 ? lora_up_kernel<true> : lora_up_kernel<false>, grid, dim3(LTHREADS), 0,
                  a.stream, static_cast<const uint16_t*>(a.H), static_cast<const uint16_t*>(a.B), a.out, a.out_kind,
                  static_cast<int>(a.T), static_cast<int>(a.d_out), nt);
}

// workspace: [At d_in*16 x 2B][Bt d_out*16 x 2B][dH T*16 x 4B][Pb][Pa], 256-byte aligned pieces
struct GradWs {
  size_t at, bt, dh, pb, pa, total;
  int parts_a, parts_b;
};
static size_t up256(size_t v) { return (v + 255) / 256 * 256; }
static GradWs grad_ws(int64_t T, int64_t d_in, int64_t d_out, int sms) {
  GradWs w;
  w.parts_b = colred_parts(T, d_out, sms);
  w.parts_a = colred_parts(T, d_in, sms);
  w.at = 0;
  w.bt = w.at + up256(static_cast<size_t>(d_in) * LR * 2);
  w.dh = w.bt + up256(static_cast<size_t>(d_out) * LR * 2);
  w.pb = w.dh + up256(static_cast<size_t>(T) * LR * 4);
  w.pa = w.pb + up256(static_cast<size_t>(w.parts_b) * d_out * LR * 4);
  w.total = w.pa + up256(static_cast<size_t>(w.parts_a) * d_in * LR * 4);
  return w;
}

size_t lora_grad_ws_bytes(int64_t T, int64_t d_in, int64_t d_out, int64_t, int sms) {
  return grad_ws(T, d_in, d_out, sms).total;
}

// a.out = dA, a.out2 = dB, a.out3 = dX, a.out4 = optional dH (FP32)
cudaError_t lora_grad_launch(const LoraArgs& a) {
  const GradWs w = grad_ws(a.T, a.d_in, a.d_out, a.num_sms);
  char* base = reinterpret_cast<char*>(a.ws);
  uint16_t* At = reinterpret_cast<uint16_t*>(base + w.at);
  uint16_t* Bt = reinterpret_cast<uint16_t*>(base + w.bt);
  float* dH = a.out4 ? static_cast<float*>(a.out4) : reinterpret_cast<float*>(base + w.dh);
  float* Pb = reinterpret_cast<float*>(base + w.pb);
  float* Pa = reinterpret_cast<float*>(base + w.pa);
  const int T = static_cast<int>(a.T), d_in = static_cast<int>(a.d_in), d_out = static_cast<int>(a.d_out);
  const bool bf = a.in_kind == EK_BF16;
  const uint16_t* X = static_cast<const uint16_t*>(a.X);
  const uint16_t* A = static_cast<const uint16_t*>(a.A);
  const uint16_t* B = static_cast<const uint16_t*>(a.B);
  const uint16_t* H = static_cast<const uint16_t*>(a.H);
  const uint16_t* dY = static_cast<const uint16_t*>(a.dY);

  const int prep_blocks = clampi((static_cast<int64_t>(d_in + d_out) * LR + 255) / 256, 1, 4 * a.num_sms);
  cudaError_t e = launch_k(lora_prep_kernel, dim3(prep_blocks), dim3(256), 0, a.stream, A, B, At, Bt, d_in, d_out);
  if (e != cudaSuccess) return e;

  const int n_rowdown = (T + 15) / 16;
  const int nj_b = (d_out + 63) / 64;
  const int g1 = n_rowdown + nj_b * w.parts_b;
  e = launch_k(bf ? lora_grad1_kernel<true> : lora_grad1_kernel<false>, dim3(g1), dim3(LTHREADS), 0, a.stream, dY,
               static_cast<const uint16_t*>(Bt), H, dH, Pb, T, d_out, n_rowdown, nj_b, w.parts_b);
  if (e != cudaSuccess) return e;

  const int nj_a = (d_in + 63) / 64;
  const int n_colred = nj_a * w.parts_a;
  const int nj_x = (d_in + 255) / 256;
  const int n_tx = rowup_nt(T, d_in, a.num_sms);
  const int g2 = n_colred + nj_x * n_tx;
  e = launch_k(bf ? lora_grad2_kernel<true> : lora_grad2_kernel<false>, dim3(g2), dim3(LTHREADS), 0, a.stream, X,
               static_cast<const float*>(dH), static_cast<const uint16_t*>(At), a.out3, a.out_kind, Pa, T, d_in,
               n_colred, nj_a, w.parts_a, nj_x, n_tx);
  if (e != cudaSuccess) return e;

  const int g3 = clampi((static_cast<int64_t>(d_in + d_out) * LR + 255) / 256, 1, 4 * a.num_sms);
  return launch_k(lora_grad3_kernel, dim3(g3), dim3(256), 0, a.stream, static_cast<const float*>(Pb),
                  static_cast<const float*>(Pa), a.out2, a.out, a.out_kind, d_out, d_in, w.parts_b, w.parts_a);
}

}  // namespace tg
