// lora_block.cu -- a rank-r LoRA branch staged as one 64-deep K block that
// the tensor-core layer product appends to its own reduction, so the branch
// is added to the base layer's output inside the product's FP32 accumulator
// (one rounding, no second pass over the output):
//   forward:         Y  = X W^T  + scale H  B^T      A2 = H'  [T][64], B2 = B'  [d_out][64]
//   input gradient:  dX = dY W   + scale dH A        A2 = dH' [T][64], B2 = A'  [64][d_in]
// Page "Twice the training speed on a BC-250 from tuned matrix kernels",
// section "What's left": fusing the small element-wise operations, here the
// addition of the LoRA branch into the base layer's output.
//
// The scale is applied in FP32 to the activation side and carried to the
// 16-bit MMA as two parts, hi = RNE16(scale h) and lo = RNE16(scale h - hi),
// in columns [0, r) and [r, 2r) of A2; the factor is repeated in the same
// two column (or row) ranges of B2, and the rest of the block is zero.  So
// the block contributes hi B + lo B = scale h B to within 2^-17 |scale h B|
// (bf16), below the products' 1e-5 bound.
#include "ptx.cuh"

namespace tg {
namespace {

struct BlockPrep {
  const void* H;  // [T][r]: 16-bit (in_kind) or FP32 (h_f32)
  const void* F;  // forward: B [N][r]; input gradient: A [r][N] (16-bit)
  uint16_t* A2;   // [T][64]
  uint16_t* B2;   // forward [N][64]; input gradient [64][N]
  long long T, N;
  int r, bf16, h_f32, dgrad;
  float scale;
};

__device__ __forceinline__ float to_f32(uint16_t v, int bf16) {
  return bf16 ? __bfloat162float(__ushort_as_bfloat16(v)) : __half2float(__ushort_as_half(v));
}
__device__ __forceinline__ uint16_t to_16(float x, int bf16) {
  return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
}

// one 8-element (16-byte) group of A2 or B2 per step
__global__ void lora_block_prep_kernel(const BlockPrep p) {
  pdl_wait();  // H may be the previous kernel's output
  pdl_trigger();
  const long long ga = p.T * 8, gb = p.N * 8;  // 8 groups per 64-column row; B2 of the dgrad: 64 rows of N / 8
  const long long nb8 = p.N / 8;
  for (long long gi = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; gi < ga + gb;
       gi += static_cast<long long>(gridDim.x) * blockDim.x) {
    uint16_t v[8];
    uint16_t* dst;
    if (gi < ga) {  // A2 row t, columns c0 .. c0 + 7: hi / lo parts of scale h
      const long long t = gi >> 3;
      const int c0 = static_cast<int>(gi & 7) * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = c0 + e;
        uint16_t out = 0;
        if (c < 2 * p.r) {
          const long long el = t * p.r + (c < p.r ? c : c - p.r);
          const float h =
              p.h_f32 ? static_cast<const float*>(p.H)[el] : to_f32(static_cast<const uint16_t*>(p.H)[el], p.bf16);
          const float x = p.scale * h;
          const uint16_t hi = to_16(x, p.bf16);
          out = c < p.r ? hi : to_16(x - to_f32(hi, p.bf16), p.bf16);
        }
        v[e] = out;
      }
      dst = p.A2 + gi * 8;
    } else if (!p.dgrad) {  // B' [N][64]: B[n][k] in columns k and r + k
      const long long j = gi - ga, n = j >> 3;
      const int c0 = static_cast<int>(j & 7) * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = c0 + e;
        v[e] = c < 2 * p.r ? static_cast<const uint16_t*>(p.F)[n * p.r + (c < p.r ? c : c - p.r)] : uint16_t(0);
      }
      dst = p.B2 + j * 8;
    } else {  // A' [64][N]: A[k][n] in rows k and r + k
      const long long j = gi - ga, k = j / nb8, n0 = (j - k * nb8) * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        v[e] = k < 2 * p.r ? static_cast<const uint16_t*>(p.F)[(k < p.r ? k : k - p.r) * p.N + n0 + e] : uint16_t(0);
      dst = p.B2 + j * 8;
    }
    *reinterpret_cast<uint4*>(dst) = make_uint4(v[0] | (static_cast<uint32_t>(v[1]) << 16),
                                                v[2] | (static_cast<uint32_t>(v[3]) << 16),
                                                v[4] | (static_cast<uint32_t>(v[5]) << 16),
                                                v[6] | (static_cast<uint32_t>(v[7]) << 16));
  }
}

}  // namespace

size_t lora_block_ws_bytes(int64_t T, int64_t N) {
  const size_t a = static_cast<size_t>(T) * 128;
  return ((a + 255) / 256) * 256 + static_cast<size_t>(N) * 128;
}

cudaError_t lora_block_prep_launch(const void* H, int h_f32, const void* F, int64_t T, int64_t N, int64_t r, float scale,
                                   int in_kind, int dgrad, void* ws, const void** A2, const void** B2, int sms,
                                   cudaStream_t stream) {
  BlockPrep p{};
  p.H = H;
  p.F = F;
  p.A2 = static_cast<uint16_t*>(ws);
  p.B2 = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + ((static_cast<size_t>(T) * 128 + 255) / 256) * 256);
  p.T = T;
  p.N = N;
  p.r = static_cast<int>(r);
  p.bf16 = in_kind == EK_BF16 ? 1 : 0;
  p.h_f32 = h_f32;
  p.dgrad = dgrad;
  p.scale = scale;
  *A2 = p.A2;
  *B2 = p.B2;
  // the input gradient's A' is 64 rows of N: N is a multiple of 8 on the tensor-core path
  if (dgrad && N % 8 != 0) return cudaErrorInvalidValue;
  const long long total = (T + N) * 8;  // 16-byte groups
  long long blocks = (total + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  if (blocks < 1) blocks = 1;
  return launch_k(lora_block_prep_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, p);
}

}  // namespace tg
