// gemm_simt.cu -- CUDA-core kernels beside the tensor-core path:
//  * the ordered reduction of FP32 split-K partials (deterministic: split
//    order fixed, no atomics), with the final cast to the output type;
//  * a plain strided GEMM for shapes the tensor-core path cannot address
//    (a row pitch that is not a multiple of 16 bytes, an unaligned base
//    pointer, an FP32 operand).  It is a GPU path, not a CPU fallback:
//    FP32 accumulation, k ascending for every output element.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "tg_internal.h"

namespace tg {

__device__ __forceinline__ float load_as_float(const void* p, int kind, int64_t i) {
  if (kind == EK_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  if (kind == EK_F16) return __half2float(static_cast<const __half*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

__device__ __forceinline__ void store_from_float(void* p, int kind, int64_t i, float v) {
  if (kind == EK_BF16)
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else if (kind == EK_F16)
    static_cast<__half*>(p)[i] = __float2half_rn(v);
  else
    static_cast<float*>(p)[i] = v;
}

// ------------------------------------------------------------- tail split
// C tile dp_tiles + t = sum over s ascending of partial slot t * splits + s
// (each a dense [bm][bn] FP32 tile); rows past M and columns past N skipped.
// One thread per 4 adjacent columns: its loads of every split are issued
// together (unrolled), so the reduction costs a few L2 round trips rather than
// one per split.  bn and N are multiples of 4, so 4 columns are all inside or
// all past N.
__global__ void tail_reduce_kernel(const float* __restrict__ P, void* __restrict__ C, int out_kind, TailGeo g,
                                   int accumulate) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  int b, m0, n0;
  tile_origin(g.dp_tiles + t, g.m_tiles, g.n_tiles, g.raster_n, g.bn, &b, &m0, &n0, g.bm);
  const int per4 = g.bm * g.bn / 4;
  const float4* tile = reinterpret_cast<const float4*>(P) + static_cast<size_t>(t) * g.splits * per4;
  for (int e4 = blockIdx.x * blockDim.x + threadIdx.x; e4 < per4; e4 += gridDim.x * blockDim.x) {
    const int r = (4 * e4) / g.bn, col = 4 * e4 - r * g.bn;
    const int64_t m = m0 + r, n = n0 + col;
    if (m >= g.M || n >= g.N) continue;
    const float4* src = tile + e4;
    float4 v = src[0];
#pragma unroll 8
    for (int s = 1; s < g.splits; ++s) {
      const float4 w = src[static_cast<size_t>(s) * per4];
      v.x += w.x;
      v.y += w.y;
      v.z += w.z;
      v.w += w.w;
    }
    const int64_t o = (b * g.M + m) * g.N + n;
    if (out_kind == EK_F32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(C) + o);
      if (accumulate) {  // C += the sum of the pieces
        const float4 c0 = *dst;
        v.x = c0.x + v.x;
        v.y = c0.y + v.y;
        v.z = c0.z + v.z;
        v.w = c0.w + v.w;
      }
      *dst = v;
    } else if (out_kind == EK_BF16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(C) + o) = pk;
    } else {
      __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__half*>(C) + o) = pk;
    }
  }
}

cudaError_t tail_reduce_launch(const float* P, void* C, int out_kind, const TailGeo& t, cudaStream_t stream,
                               int accumulate) {
  if (t.tail_tiles == 0) return cudaSuccess;
  const int per4 = t.bm * t.bn / 4;
  return launch_k(tail_reduce_kernel, dim3((per4 + 255) / 256, t.tail_tiles), dim3(256), 0, stream, P, C, out_kind,
                  t, accumulate);
}

// ---------------------------------------------------------------- split-K
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, void* __restrict__ C, int out_kind,
                                     int64_t batch, int64_t splits, int64_t MN, int accumulate) {
  pdl_wait();
  pdl_trigger();
  const int64_t n4 = MN / 4;  // MN is a multiple of 4 on the tensor-core path
  const int64_t total = batch * n4;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < total;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = v / n4;
    const int64_t i4 = v - b * n4;
    const float4* src = reinterpret_cast<const float4*>(ws) + (b * splits) * n4 + i4;
    float4 s = src[0];
#pragma unroll 8
    for (int64_t k = 1; k < splits; ++k) {
      const float4 t = src[k * n4];
      s.x += t.x;
      s.y += t.y;
      s.z += t.z;
      s.w += t.w;
    }
    const int64_t o = b * MN + i4 * 4;
    if (out_kind == EK_F32) {
      float4* dst = reinterpret_cast<float4*>(C) + o / 4;
      if (accumulate) {  // C += the sum of the splits
        const float4 c0 = *dst;
        s.x = c0.x + s.x;
        s.y = c0.y + s.y;
        s.z = c0.z + s.z;
        s.w = c0.w + s.w;
      }
      *dst = s;
    } else if (out_kind == EK_BF16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y), hi = __floats2bfloat162_rn(s.z, s.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(C)[o / 4] = pk;
    } else {
      __half2 lo = __floats2half2_rn(s.x, s.y), hi = __floats2half2_rn(s.z, s.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(C)[o / 4] = pk;
    }
  }
}

cudaError_t splitk_reduce_launch(const float* ws, void* C, int out_kind, int64_t batch, int64_t splits,
                                 int64_t MN, cudaStream_t stream, int accumulate) {
  const int64_t total = batch * (MN / 4);
  if (total <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_k(splitk_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, ws, C, out_kind,
                  batch, splits, MN, accumulate);
}

// ---------------------------------------------------------------- strided
constexpr int ST = 16;  // 16 x 16 outputs per block, K staged 16 at a time

__global__ void simt_gemm_kernel(SimtGemm g) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[ST][ST + 1];
  __shared__ float Bs[ST][ST + 1];
  const int64_t b = blockIdx.z;
  const int64_t i = static_cast<int64_t>(blockIdx.y) * ST + threadIdx.y;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * ST + threadIdx.x;
  float acc = 0.f;
  for (int64_t k0 = 0; k0 < g.K; k0 += ST) {
    const int64_t ka = k0 + threadIdx.x;  // A tile: row threadIdx.y, column k
    const int64_t ia = static_cast<int64_t>(blockIdx.y) * ST + threadIdx.y;
    As[threadIdx.y][threadIdx.x] =
        (ia < g.M && ka < g.K) ? load_as_float(g.A, g.a_kind, b * g.a_bs + ia * g.a_rs + ka * g.a_cs) : 0.f;
    const int64_t kb = k0 + threadIdx.y;  // B tile: row k, column threadIdx.x
    const int64_t jb = static_cast<int64_t>(blockIdx.x) * ST + threadIdx.x;
    Bs[threadIdx.y][threadIdx.x] =
        (kb < g.K && jb < g.N) ? load_as_float(g.B, g.b_kind, b * g.b_bs + kb * g.b_rs + jb * g.b_cs) : 0.f;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < ST; ++kk) acc = fmaf(As[threadIdx.y][kk], Bs[kk][threadIdx.x], acc);
    __syncthreads();
  }
  if (i < g.M && j < g.N) {
    const int64_t o = (b * g.M + i) * g.N + j;
    if (g.accumulate)
      acc = fmaf(g.scale, acc, load_as_float(g.C, g.out_kind, o));  // C += scale * the product
    else
      acc *= g.scale;  // C = scale * the product (exact for scale 1)
    store_from_float(g.C, g.out_kind, o, acc);
  }
}

cudaError_t simt_gemm_launch(const SimtGemm& g) {
  if (g.M <= 0 || g.N <= 0 || g.batch <= 0) return cudaSuccess;
  dim3 block(ST, ST);
  dim3 grid(static_cast<unsigned>((g.N + ST - 1) / ST), static_cast<unsigned>((g.M + ST - 1) / ST),
            static_cast<unsigned>(g.batch));
  if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidConfiguration;
  return launch_k(simt_gemm_kernel, grid, block, 0, g.stream, g);
}

}  // namespace tg
