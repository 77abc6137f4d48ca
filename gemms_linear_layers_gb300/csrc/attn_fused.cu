// Fused attention forward: O = softmax(scale * Q K^T) V per head, without
// writing the [s, s] score or probability matrices.
//
// Page "Twice the training speed on a BC-250 from tuned matrix kernels",
// section "What got in the way" / the closing notes: the batched products
// inside attention, with the softmax between them, are the part a fused
// attention kernel would take over.  The two products are the ones the library
// also runs unfused (S = Q K^T, O = P V); here they run back to back on chip
// with the softmax of each row kept online (running maximum m and sum l, the
// partial output rescaled by exp(m_old - m_new) whenever m grows).
//
// Kernel: 4 warps per CTA, 16 query rows per warp (64 per CTA), keys in blocks
// of 64 through a double-buffered shared-memory ring filled with cp.async.
// Both products run on mma.sync m16n8k16 with FP32 accumulation: the score
// accumulator of one key block is, unchanged, the A operand of the P V product
// (two 8-key tiles form one 16-key step).  P is split into 16-bit hi and lo
// parts and both are multiplied by V, so P is carried to within 2^-18 of its
// FP32 value.  Exponentials are base 2 on scores prescaled by scale * log2(e).
#include "attn.h"
#include "ptx.cuh"

namespace tg {
namespace {

constexpr int AD = 64;            // head dimension
constexpr int ABQ = 64;           // query rows per CTA
constexpr int ABK = 64;           // keys per block
constexpr int AROW = AD + 8;      // padded shared-memory row (16-bit elements): 144 bytes
constexpr int ATHREADS = 128;

struct AttnArgs {
  const uint16_t* Q;
  const uint16_t* K;
  const uint16_t* V;
  void* O;
  int out_kind;
  int s;
  float scale_log2;  // scale * log2(e)
};

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// 16 bytes global -> shared; src_bytes = 0 fills zeros (rows past the end)
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// rows [r0, r0 + 64) of a [s][64] 16-bit matrix into a padded tile
__device__ __forceinline__ void load_tile(uint32_t tile, const uint16_t* src, int r0, int s, int tid) {
#pragma unroll
  for (int u = 0; u < (ABK * AD * 2 / 16) / ATHREADS; ++u) {  // 4 chunks of 16 bytes per thread
    const int q = tid + u * ATHREADS, row = q >> 3, ch = q & 7;
    const int r = r0 + row;
    const bool ok = r < s;
    cp16(tile + static_cast<uint32_t>(row * AROW * 2 + ch * 16), src + static_cast<size_t>(ok ? r : 0) * AD + ch * 8,
         ok ? 16 : 0);
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}
template <bool BF16>
__device__ __forceinline__ float rnd16(float x) {
  return BF16 ? __bfloat162float(__float2bfloat16_rn(x)) : __half2float(__float2half_rn(x));
}

template <bool BF16>
__global__ void __launch_bounds__(ATHREADS, 1) attn_fwd_kernel(const AttnArgs a) {
  __shared__ __align__(128) uint16_t Qs[ABQ * AROW];
  __shared__ __align__(128) uint16_t Ks[2][ABK * AROW];
  __shared__ __align__(128) uint16_t Vs[2][ABK * AROW];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int head = blockIdx.y, q0 = blockIdx.x * ABQ;
  const size_t hoff = static_cast<size_t>(head) * a.s * AD;
  const uint16_t* Q = a.Q + hoff;
  const uint16_t* K = a.K + hoff;
  const uint16_t* V = a.V + hoff;
  const uint32_t qs = smem_u32(Qs), ks0 = smem_u32(Ks[0]), vs0 = smem_u32(Vs[0]);
  constexpr uint32_t TILE = ABK * AROW * 2;
  const int nblk = (a.s + ABK - 1) / ABK;

  load_tile(qs, Q, q0, a.s, tid);
  load_tile(ks0, K, 0, a.s, tid);
  load_tile(vs0, V, 0, a.s, tid);
  cp_commit();

  float o[8][4];  // 16 rows x 64 columns of the output: d-tile j, (g, 2c..2c+1) and (g+8, ...)
#pragma unroll
  for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows g and g+8
  uint32_t qf[4][4];                                        // Q fragments, 4 steps of 16 columns

  for (int b = 0; b < nblk; ++b) {
    if (b + 1 < nblk) {  // the next block's K and V start moving
      load_tile(ks0 + ((b + 1) & 1) * TILE, K, (b + 1) * ABK, a.s, tid);
      load_tile(vs0 + ((b + 1) & 1) * TILE, V, (b + 1) * ABK, a.s, tid);
    }
    cp_commit();
    cp_wait<1>();  // every group but the newest: Q (first time) and this block's K, V
    __syncthreads();
    if (b == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        ldsm4(qs + static_cast<uint32_t>(((warp * 16 + (lane & 15)) * AROW + kk * 16 + (lane >> 4) * 8) * 2), qf[kk]);
    }
    const uint32_t ks = ks0 + (b & 1) * TILE, vs = vs0 + (b & 1) * TILE;

    // S = Q K^T for this warp's 16 rows x 64 keys
    float sc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {  // key tiles 2jp, 2jp+1
        uint32_t kb[4];
        const int key = jp * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm4(ks + static_cast<uint32_t>((key * AROW + kk * 16 + ((lane >> 3) & 1) * 8) * 2), kb);
        mma_16816<BF16>(sc[2 * jp], qf[kk], kb);
        mma_16816<BF16>(sc[2 * jp + 1], qf[kk], kb + 2);
      }
    }
    // online softmax over the block's valid keys
    const int kbase = b * ABK;
    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool ok = kbase + 8 * j + 2 * c + e < a.s;
        sc[j][e] = ok ? sc[j][e] * a.scale_log2 : -INFINITY;
        sc[j][2 + e] = ok ? sc[j][2 + e] * a.scale_log2 : -INFINITY;
        bm0 = fmaxf(bm0, sc[j][e]);
        bm1 = fmaxf(bm1, sc[j][2 + e]);
      }
    }
#pragma unroll
    for (int x = 1; x <= 2; x <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
    }
    const float n0 = fmaxf(m0, bm0), n1 = fmaxf(m1, bm1);  // finite: every block has a valid key
    const float r0 = exp2f(m0 - n0), r1 = exp2f(m1 - n1);  // 0 on the first block
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[j][e] = exp2f(sc[j][e] - n0);
        sc[j][2 + e] = exp2f(sc[j][2 + e] - n1);
        s0 += sc[j][e];
        s1 += sc[j][2 + e];
      }
    }
#pragma unroll
    for (int x = 1; x <= 2; x <<= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, x);
      s1 += __shfl_xor_sync(0xffffffffu, s1, x);
    }
    l0 = l0 * r0 + s0;
    l1 = l1 * r1 + s1;
    m0 = n0;
    m1 = n1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j][0] *= r0;
      o[j][1] *= r0;
      o[j][2] *= r1;
      o[j][3] *= r1;
    }
    // O += P V: P's 16-key steps are the score tiles (2kk, 2kk+1), as hi + lo 16-bit parts
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t ph[4], pl[4];
      const float* t0 = sc[2 * kk];
      const float* t1 = sc[2 * kk + 1];
      const float v[8] = {t0[0], t0[1], t0[2], t0[3], t1[0], t1[1], t1[2], t1[3]};
      float h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = rnd16<BF16>(v[e]);
      ph[0] = pack2<BF16>(h[0], h[1]);  // row g, keys 2c, 2c+1
      ph[1] = pack2<BF16>(h[2], h[3]);  // row g+8
      ph[2] = pack2<BF16>(h[4], h[5]);  // row g, keys 8 + 2c, ...
      ph[3] = pack2<BF16>(h[6], h[7]);  // row g+8
      pl[0] = pack2<BF16>(v[0] - h[0], v[1] - h[1]);
      pl[1] = pack2<BF16>(v[2] - h[2], v[3] - h[3]);
      pl[2] = pack2<BF16>(v[4] - h[4], v[5] - h[5]);
      pl[3] = pack2<BF16>(v[6] - h[6], v[7] - h[7]);
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {  // d tiles 2jp, 2jp+1
        uint32_t vb[4];
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm4_t(vs + static_cast<uint32_t>((key * AROW + jp * 16 + (lane >> 4) * 8) * 2), vb);
        mma_16816<BF16>(o[2 * jp], ph, vb);
        mma_16816<BF16>(o[2 * jp], pl, vb);
        mma_16816<BF16>(o[2 * jp + 1], ph, vb + 2);
        mma_16816<BF16>(o[2 * jp + 1], pl, vb + 2);
      }
    }
    __syncthreads();  // this block's K and V tiles may be refilled
  }
  cp_wait<0>();

  // O / l, rows q0 + 16 warp + g (+8), columns 8j + 2c (+1)
  const float i0 = 1.f / l0, i1 = 1.f / l1;
  const int ra = q0 + warp * 16 + g, rb = ra + 8;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int col = 8 * j + 2 * c;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = h ? rb : ra;
      if (row >= a.s) continue;
      const float x = o[j][2 * h] * (h ? i1 : i0), y = o[j][2 * h + 1] * (h ? i1 : i0);
      const size_t e = hoff + static_cast<size_t>(row) * AD + col;
      if (a.out_kind == EK_F32) {
        *reinterpret_cast<float2*>(static_cast<float*>(a.O) + e) = make_float2(x, y);
      } else {
        *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.O) + e) =
            a.out_kind == EK_BF16 ? pack_bf16x2(x, y) : pack_f16x2(x, y);
      }
    }
  }
}

}  // namespace

cudaError_t attn_fwd_launch(const void* Q, const void* K, const void* V, void* O, int64_t heads, int64_t s, int64_t d,
                            float scale, int in_kind, int out_kind, cudaStream_t stream) {
  if (heads == 0 || s == 0) return cudaSuccess;
  if (d != AD) return cudaErrorInvalidValue;
  AttnArgs a{};
  a.Q = static_cast<const uint16_t*>(Q);
  a.K = static_cast<const uint16_t*>(K);
  a.V = static_cast<const uint16_t*>(V);
  a.O = O;
  a.out_kind = out_kind;
  a.s = static_cast<int>(s);
  a.scale_log2 = scale * 1.4426950408889634f;
  const dim3 grid(static_cast<unsigned>((s + ABQ - 1) / ABQ), static_cast<unsigned>(heads));
  if (in_kind == EK_BF16)
    attn_fwd_kernel<true><<<grid, ATHREADS, 0, stream>>>(a);
  else
    attn_fwd_kernel<false><<<grid, ATHREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace tg
