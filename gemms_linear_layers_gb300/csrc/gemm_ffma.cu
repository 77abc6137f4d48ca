// FP32-input products of a linear layer on the CUDA cores (FFMA).
//
// Page "Twice the training speed on a BC-250 from tuned matrix kernels",
// section "Where the time went": the forward pass, the input gradient and the
// weight gradient of every linear layer, each in its own layout; the page
// times the FP32 versions of these products as well (its FP32 numbers are the
// baseline the 16-bit kernels are compared with).  Here the operands are FP32
// and every product a*b is fused into its FP32 sum (one rounding per step,
// k ascending within a split), so the result is the FP32 evaluation of the
// exact definition; the tensor cores' TF32 path would round the operands to
// 10-bit mantissas and is not used.
//
// Kernel: 128 x 128 output tile per CTA of 256 threads, each thread 8 x 8
// outputs (two 4-row and two 4-column groups 64 apart, so that a warp's
// shared-memory reads are broadcasts or contiguous); K in steps of 16 through
// two shared-memory buffers, the next step's operands held in registers while
// the current one is multiplied.  Operand tiles are stored [k][m] and [k][n]:
// a K-major operand (rows with K contiguous) is transposed on the way in, an
// MN-major one is copied as it is.  Long reductions over few tiles are split
// along K into FP32 partials that the ordered split-K reduction adds up
// (bitwise reproducible).
//
// The same products also run on the tensor cores (api.cu chooses when the
// operand pitches allow TMA): split3_kernel below cuts each FP32 operand into
// three bf16 parts, and the layer-product kernels form the six part products
// a_i b_j with i + j <= 2 in FP32 sums.
#include <cuda_bf16.h>

#include "tg_internal.h"

namespace tg {
namespace {

constexpr int FM = 128, FN = 128, FK = 16, FT = 256;
constexpr int FROW = FM + 4;  // padded row of a [k][128] tile (float4 aligned)

struct FfmaArgs {
  const float* A;
  const float* B;
  float* C;  // the output, or the split partials [split][M][N]
  int64_t M, N, K, lda, ldb;
  int64_t kps;       // K per split (a multiple of FK)
  int vec_a, vec_b;  // 16-byte loads along the operand's contiguous dimension are aligned
  int vec_c;         // 16-byte stores of C are aligned
  int accumulate;    // C += the product (unsplit launches only)
};

// 8 consecutive elements of one row of a row-major [rows][ld] array starting
// at column c, zero outside [0, rows) x [0, cols)
__device__ __forceinline__ void load_run8(const float* p, int64_t rows, int64_t cols, int64_t ld, int64_t r,
                                          int64_t c, bool vec, float* v) {
  if (r < rows && c + 8 <= cols && vec) {
    const float4* q = reinterpret_cast<const float4*>(p + r * ld + c);
    const float4 x = __ldg(q), y = __ldg(q + 1);
    v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w, v[4] = y.x, v[5] = y.y, v[6] = y.z, v[7] = y.w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = (r < rows && c + e < cols) ? __ldg(p + r * ld + c + e) : 0.f;
  }
}

// A(i, k): K-major (A[i][k], NT and NN) or MN-major (A[k][i], TN).
// B(k, j): K-major (B[j][k], NT) or MN-major (B[k][j], NN and TN).
template <int LAYOUT>
__global__ void __launch_bounds__(FT, 2) ffma_gemm_kernel(const FfmaArgs g) {
  constexpr bool A_KMAJ = LAYOUT != LAYOUT_TN;
  constexpr bool B_KMAJ = LAYOUT == LAYOUT_NT;
  __shared__ __align__(16) float As[2][FK][FROW];
  __shared__ __align__(16) float Bs[2][FK][FROW];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * FM, n0 = static_cast<int64_t>(blockIdx.x) * FN;
  const int64_t kbeg = static_cast<int64_t>(blockIdx.z) * g.kps;
  const int64_t kend = kbeg + g.kps < g.K ? kbeg + g.kps : g.K;

  // this thread's share of a K step: 8 elements of A and 8 of B
  float ra[8], rb[8];
  auto load = [&](int64_t k0) {
    if (A_KMAJ)  // row m0 + tid/2 of A, columns k0 + 8 (tid&1) ..
      load_run8(g.A, g.M, kend, g.lda, m0 + (tid >> 1), k0 + (tid & 1) * 8, g.vec_a, ra);
    else  // row k0 + tid/16 of A^T, columns m0 + 8 (tid&15) ..
      load_run8(g.A, kend, g.M, g.lda, k0 + (tid >> 4), m0 + (tid & 15) * 8, g.vec_a, ra);
    if (B_KMAJ)
      load_run8(g.B, g.N, kend, g.ldb, n0 + (tid >> 1), k0 + (tid & 1) * 8, g.vec_b, rb);
    else
      load_run8(g.B, kend, g.N, g.ldb, k0 + (tid >> 4), n0 + (tid & 15) * 8, g.vec_b, rb);
  };
  auto store = [&](int buf) {
    if (A_KMAJ) {
#pragma unroll
      for (int e = 0; e < 8; ++e) As[buf][(tid & 1) * 8 + e][tid >> 1] = ra[e];
    } else {
      float4* d = reinterpret_cast<float4*>(&As[buf][tid >> 4][(tid & 15) * 8]);
      d[0] = make_float4(ra[0], ra[1], ra[2], ra[3]);
      d[1] = make_float4(ra[4], ra[5], ra[6], ra[7]);
    }
    if (B_KMAJ) {
#pragma unroll
      for (int e = 0; e < 8; ++e) Bs[buf][(tid & 1) * 8 + e][tid >> 1] = rb[e];
    } else {
      float4* d = reinterpret_cast<float4*>(&Bs[buf][tid >> 4][(tid & 15) * 8]);
      d[0] = make_float4(rb[0], rb[1], rb[2], rb[3]);
      d[1] = make_float4(rb[4], rb[5], rb[6], rb[7]);
    }
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  int buf = 0;
  if (kbeg < kend) {
    load(kbeg);
    store(0);
  }
  __syncthreads();
  for (int64_t k0 = kbeg; k0 < kend; k0 += FK) {
    const bool more = k0 + FK < kend;
    if (more) load(k0 + FK);  // in flight while this step is multiplied
#pragma unroll
    for (int k = 0; k < FK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) store(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }

  // rows m0 + 4 ty + i (+64 for i >= 4), columns n0 + 4 tx + j (+64 for j >= 4)
  float* C = g.C + static_cast<int64_t>(blockIdx.z) * g.M * g.N;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = m0 + ty * 4 + (i & 3) + (i >> 2) * 64;
    if (r >= g.M) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t c = n0 + tx * 4 + h * 64;
      float* p = C + r * g.N + c;
      float v[4] = {acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]};
      if (c + 4 <= g.N && g.vec_c) {
        if (g.accumulate) {
          const float4 o = *reinterpret_cast<const float4*>(p);
          v[0] += o.x, v[1] += o.y, v[2] += o.z, v[3] += o.w;
        }
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c + e < g.N) p[e] = g.accumulate ? p[e] + v[e] : v[e];
      }
    }
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int ffma_splits(int64_t M, int64_t N, int64_t K, int sms) {
  const int64_t tiles = ((M + FM - 1) / FM) * ((N + FN - 1) / FN);
  const int64_t slots = 2 * static_cast<int64_t>(sms);  // two CTAs per SM
  if (tiles >= slots || K < 2 * 512) return 1;
  int64_t s = slots / tiles;
  if (s > 16) s = 16;
  if (s > K / 512) s = K / 512;  // at least 512 products per split
  if (s < 2) return 1;
  const int64_t kps = ((K + s - 1) / s + FK - 1) / FK * FK;
  return static_cast<int>((K + kps - 1) / kps);
}

size_t ffma_ws_bytes(int64_t M, int64_t N, int64_t K, int sms) {
  const int s = ffma_splits(M, N, K, sms);
  return s > 1 ? static_cast<size_t>(s) * M * N * sizeof(float) : 0;
}

cudaError_t ffma_gemm_launch(const FfmaGemm& g) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  FfmaArgs a{};
  a.A = g.A;
  a.B = g.B;
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.lda = g.lda;
  a.ldb = g.ldb;
  const int s = g.splits > 1 ? g.splits : 1;
  a.kps = s > 1 ? ((g.K + s - 1) / s + FK - 1) / FK * FK : g.K;
  a.C = s > 1 ? g.ws : g.C;
  a.vec_a = al16(g.A) && g.lda % 4 == 0;
  a.vec_b = al16(g.B) && g.ldb % 4 == 0;
  a.vec_c = al16(a.C) && g.N % 4 == 0;
  a.accumulate = s > 1 ? 0 : g.accumulate;
  const dim3 grid(static_cast<unsigned>((g.N + FN - 1) / FN), static_cast<unsigned>((g.M + FM - 1) / FM),
                  static_cast<unsigned>(s));
  if (g.layout == LAYOUT_NT)
    ffma_gemm_kernel<LAYOUT_NT><<<grid, FT, 0, g.stream>>>(a);
  else if (g.layout == LAYOUT_NN)
    ffma_gemm_kernel<LAYOUT_NN><<<grid, FT, 0, g.stream>>>(a);
  else
    ffma_gemm_kernel<LAYOUT_TN><<<grid, FT, 0, g.stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || s == 1) return e;
  return splitk_reduce_launch(g.ws, g.C, EK_F32, 1, s, g.M * g.N, g.stream, g.accumulate);
}

// ---------------------------------------------------------------------------
// FP32 operands on the tensor cores: each operand split into three bf16 parts
// (8 significant bits each; FP32 has 24) so that the 16-bit MMA, which
// multiplies exactly and adds in FP32, can form the six part products that
// carry the product to within 2^-24 of its magnitude.
namespace {
// the three parts of one value: v - p0 and its remainder are exact in FP32
// (each part takes the leading 8 bits of what is left, rounded to nearest)
__device__ __forceinline__ void split3_one(float v, uint16_t* p) {
  const __nv_bfloat16 p0 = __float2bfloat16_rn(v);
  const float r1 = isfinite(v) ? v - __bfloat162float(p0) : 0.f;
  const __nv_bfloat16 p1 = __float2bfloat16_rn(r1);
  const __nv_bfloat16 p2 = __float2bfloat16_rn(r1 - __bfloat162float(p1));
  p[0] = __bfloat16_as_ushort(p0);
  p[1] = __bfloat16_as_ushort(p1);
  p[2] = __bfloat16_as_ushort(p2);
}

// vec4: four values per step (16-byte loads, 8-byte stores of each part)
template <bool VEC4>
__global__ void split3_kernel(const float* __restrict__ src, int64_t n, int64_t pstride, uint16_t* __restrict__ dst) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // src may be the previous kernel's output
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (VEC4) {
    for (int64_t q = i0; q < n / 4; q += stride) {
      const float4 v = reinterpret_cast<const float4*>(src)[q];
      uint16_t a[3], b[3], c[3], d[3];
      split3_one(v.x, a);
      split3_one(v.y, b);
      split3_one(v.z, c);
      split3_one(v.w, d);
#pragma unroll
      for (int p = 0; p < 3; ++p)
        *reinterpret_cast<uint2*>(dst + p * pstride + 4 * q) =
            make_uint2(a[p] | (static_cast<uint32_t>(b[p]) << 16), c[p] | (static_cast<uint32_t>(d[p]) << 16));
    }
  } else {
    for (int64_t i = i0; i < n; i += stride) {
      uint16_t a[3];
      split3_one(src[i], a);
      dst[i] = a[0];
      dst[pstride + i] = a[1];
      dst[2 * pstride + i] = a[2];
    }
  }
}
}  // namespace

cudaError_t split3_launch(const float* src, int64_t n, int64_t pstride, uint16_t* dst, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  // whole float4 groups when the source and every part start 16 / 8 bytes aligned
  const bool vec = n % 4 == 0 && pstride % 4 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dst) % 8 == 0;
  const int64_t work = vec ? n / 4 : n;
  int64_t blocks = (work + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  return vec ? launch_k(split3_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, src, n, pstride,
                        dst)
             : launch_k(split3_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, src, n,
                        pstride, dst);
}

}  // namespace tg
