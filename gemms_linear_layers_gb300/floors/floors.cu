// floors.cu -- stand-alone measurements of what this GPU allows, the floors
// the library's kernels are compared with (not linked into libtg.so):
//   1. the cost of an empty kernel launched back to back;
//   2. streaming a [T, K] bf16 matrix from HBM with TMA boxes shaped like the
//      LoRA row-down kernel's ({64, R, 8}, 4 stages), with no arithmetic;
//   3. the same bytes with plain 16-byte loads;
//   4. the rate of one 128 x N x 16 tcgen05.mma (one CTA per SM, operands
//      resident in shared memory) for N = 64 .. 256, K- and MN-major.
// Buffers are rotated beyond twice the L2 so every launch reads HBM.  Every
// wait is bounded; a wait that times out sets a flag that is reported.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <vector>

#include "ptx.cuh"

using namespace tg;

#define CK(x)                                                                       \
  do {                                                                              \
    cudaError_t e_ = (x);                                                           \
    if (e_ != cudaSuccess) {                                                        \
      printf("CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
      exit(1);                                                                      \
    }                                                                               \
  } while (0)

__global__ void k_empty(unsigned* out) {
  if (threadIdx.x == 12345) out[0] = 1;
}

// ---------------------------------------------------------------- streaming
struct StreamArgs {
  int T, R, CH, NS, nchunks, stage_bytes;
  unsigned* status;
};

__global__ void __launch_bounds__(64, 1) k_tma_stream(const __grid_constant__ CUtensorMap tm, StreamArgs p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + p.NS * p.stage_bytes);
  uint64_t* empty = full + 16;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int r0 = blockIdx.x * p.R;
  if (r0 >= p.T) return;
  const int nst = (p.nchunks + p.CH - 1) / p.CH;
  if (threadIdx.x == 0) {  // producer
    for (int s = 0; s < nst; ++s) {
      const int slot = s % p.NS;
      const uint32_t ph = (s / p.NS) & 1;
      if (!mbar_wait(smem_u32(&empty[slot]), ph ^ 1u, 2000000000ull, nullptr, p.status, 1)) return;
      const uint32_t fb = smem_u32(&full[slot]);
      mbar_arrive_expect_tx(fb, 64 * 2 * p.R * p.CH);
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(ring + slot * p.stage_bytes)),
          "l"(reinterpret_cast<uint64_t>(&tm)), "r"(fb), "r"(0), "r"(r0), "r"(s * p.CH)
          : "memory");
    }
  } else if (threadIdx.x == 32) {  // consumer: releases each stage as it lands
    for (int s = 0; s < nst; ++s) {
      const int slot = s % p.NS;
      const uint32_t ph = (s / p.NS) & 1;
      if (!mbar_wait(smem_u32(&full[slot]), ph, 2000000000ull, nullptr, p.status, 2)) return;
      mbar_arrive(smem_u32(&empty[slot]));
    }
  }
}

template <int UNR>
__global__ void k_ldg_stream(const uint4* __restrict__ src, long long n16, unsigned* out) {
  unsigned acc = 0;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (UNR - 1) * stride < n16; i += UNR * stride) {
    uint4 v[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < UNR; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = __ldcs(src + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x12345678u) out[0] = acc;
}

// ------------------------------------------------------------- tensor pipe
template <int N, bool AMN, bool BMN>
__global__ void __launch_bounds__(128, 1) k_mma(long long* out, int iters, unsigned* status) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = sm;          // 128 x 64 bf16, 16 KB
  uint8_t* sB = sm + 16384;  // N x 64 bf16
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  for (int i = threadIdx.x; i < (16384 + N * 128) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(&tslot), 256);
    tmem_relinquish();
    tc_fence_before();
  }
  fence_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tslot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_f16(true, AMN, BMN, 128, N);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    const long long t0 = clock64();
    uint32_t ph = 0;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_f16(tbase, AMN ? sdesc_sw128(a0 + kk * 2048, 8192, 1024) : sdesc_sw128(a0 + kk * 32, 16, 1024),
                 BMN ? sdesc_sw128(b0 + kk * 2048, 8192, 1024) : sdesc_sw128(b0 + kk * 32, 16, 1024), idesc, 1u);
      if ((it & 15) == 15) {
        umma_commit(smem_u32(&bar));
        mbar_wait(smem_u32(&bar), ph, 2000000000ull, nullptr, status, 3);
        ph ^= 1u;
      }
    }
    umma_commit(smem_u32(&bar));
    mbar_wait(smem_u32(&bar), ph, 2000000000ull, nullptr, status, 4);
    out[blockIdx.x] = clock64() - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tbase, 256);
  }
}

typedef CUresult (*EncFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                          const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                          CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <typename F>
static float per_launch_us(F launch, int n) {
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  float best = 1e30f;
  for (int rep = 0; rep < 5; ++rep) {
    CK(cudaEventRecord(e0));
    for (int i = 0; i < n; ++i) launch(i);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    CK(cudaGetLastError());
    float ms;
    CK(cudaEventElapsedTime(&ms, e0, e1));
    if (ms / n < best) best = ms / n;
  }
  return best * 1e3f;
}

template <int N, bool AMN, bool BMN>
static void mma_rate(long long* d_out, unsigned* st, int sms) {
  const int iters = 2048;
  auto k = k_mma<N, AMN, BMN>;
  const int smem = 1024 + 16384 + N * 128;
  CK(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  for (int rep = 0; rep < 2; ++rep) k<<<sms, 128, smem>>>(d_out, iters, st);
  CK(cudaDeviceSynchronize());
  std::vector<long long> h(sms);
  CK(cudaMemcpy(h.data(), d_out, sms * 8, cudaMemcpyDeviceToHost));
  double cyc = 0;
  for (long long v : h) cyc += static_cast<double>(v);
  cyc /= sms;
  printf("| 128 x %3d x 16, A %s-major, B %s-major | %.1f | %.0f |\n", N, AMN ? "MN" : "K", BMN ? "MN" : "K",
         cyc / (iters * 4.0), 2.0 * 128 * N * 64 * iters / cyc);
}

int main() {
  int sms;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  int l2;
  CK(cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, 0));
  EncFn enc;
  cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&enc), 12000,
                                      cudaEnableDefault, &q));
  unsigned* st;
  CK(cudaMalloc(&st, 4));
  CK(cudaMemset(st, 0, 4));
  unsigned* out;
  CK(cudaMalloc(&out, 4));

  printf("## launch floor\n\nempty kernel (%d x 256), back to back: %.2f us\n\n", sms,
         per_launch_us([&](int) { k_empty<<<sms, 256>>>(out); }, 200));

  printf("## streaming floors (T = 4096 rows, back-to-back launches, buffers rotated beyond 2 x L2)\n\n");
  printf("| pattern | MB | us per launch | GB/s |\n|---|---:|---:|---:|\n");
  CK(cudaFuncSetAttribute(k_tma_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448));
  const int T = 4096;
  for (int K : {2304, 5760}) {
    const long long bytes = static_cast<long long>(T) * K * 2;
    const int nb = static_cast<int>(2LL * l2 / bytes) + 2;
    std::vector<char*> bufs(nb);
    for (auto& b : bufs) {
      CK(cudaMalloc(&b, bytes));
      CK(cudaMemset(b, 1, bytes));
    }
    // TMA boxes {64, R, 8} over [K/64][T][64], 4 stages: the row-down pattern
    const int R = (T + sms - 1) / sms, CH = 8, NS = 4;
    const int stage = (64 * 2 * R * CH + 1023) & ~1023;
    std::vector<CUtensorMap> tms(nb);
    for (int i = 0; i < nb; ++i) {
      cuuint64_t d[3] = {64, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(K / 64)};
      cuuint64_t s[2] = {static_cast<cuuint64_t>(K) * 2, 128};
      cuuint32_t b[3] = {64, static_cast<cuuint32_t>(R), static_cast<cuuint32_t>(CH)}, e[3] = {1, 1, 1};
      if (enc(&tms[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, bufs[i], d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
          CUDA_SUCCESS) {
        printf("tensor map encode failed\n");
        return 1;
      }
    }
    StreamArgs pa{T, R, CH, NS, K / 64, stage, st};
    const int smem = NS * stage + 1024 + 256;
    float us = per_launch_us([&](int i) { k_tma_stream<<<sms, 64, smem>>>(tms[i % nb], pa); }, 4 * nb);
    printf("| TMA boxes {64, %d, 8}, 4 stages | %.1f | %.2f | %.0f |\n", R, bytes / 1e6, us, bytes / us / 1e3);
    us = per_launch_us(
        [&](int i) { k_ldg_stream<4><<<sms * 8, 256>>>(reinterpret_cast<const uint4*>(bufs[i % nb]), bytes / 16, out); },
        4 * nb);
    printf("| 16-byte loads, 8 x 256 threads per SM | %.1f | %.2f | %.0f |\n", bytes / 1e6, us, bytes / us / 1e3);
    for (auto& b : bufs) CK(cudaFree(b));
  }

  printf("\n## tensor pipe: one 128 x N x 16 tcgen05.mma, one CTA per SM\n\n");
  printf("| MMA | cycles | flop/clk/SM |\n|---|---:|---:|\n");
  long long* d_cyc;
  CK(cudaMalloc(&d_cyc, sms * 8));
  mma_rate<64, false, false>(d_cyc, st, sms);
  mma_rate<128, false, false>(d_cyc, st, sms);
  mma_rate<144, false, false>(d_cyc, st, sms);
  mma_rate<192, false, false>(d_cyc, st, sms);
  mma_rate<256, false, false>(d_cyc, st, sms);
  mma_rate<256, true, true>(d_cyc, st, sms);
  unsigned hs;
  CK(cudaMemcpy(&hs, st, 4, cudaMemcpyDeviceToHost));
  printf("\nbounded waits: %s\n", hs ? "a wait timed out (numbers invalid)" : "none timed out");
  return hs ? 2 : 0;
}
