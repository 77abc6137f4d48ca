// gemm_tc_cs.cuh -- split-K inside a thread-block cluster for the tcgen05 GEMM.
//
// Same products and arithmetic as gemm_tc.cuh (page "Twice the training
// speed on a BC-250 from tuned matrix kernels", sections "Where the time
// went" and "Tuning the kernels": 16-bit inputs, FP32 accumulation).  For
// the products of small layers, a 128 x BN output tile is cut along K into
// S ranges computed by the S CTAs of one cluster (one SM each), and the S
// FP32 partial tiles are added on chip:
//   - CTA rank r of the cluster accumulates K blocks [r kps, (r+1) kps) in
//     its tensor memory (one accumulator, one tile per cluster);
//   - its epilogue warps copy the accumulator to a padded [128][BN + 4]
//     FP32 buffer in its own shared memory (the operand ring, idle by then);
//   - after a cluster barrier, CTA r adds rows [128 r / S, 128 (r+1) / S) of
//     all S buffers, in rank order, reading them through distributed shared
//     memory, and writes them to the output with coalesced stores;
//   - a second cluster barrier keeps every buffer alive until all reads end.
// (Measured: pushing the slices with bulk copies into a receive area first
// was slower than these direct loads.)
// No partial tile goes through global memory and no second kernel runs; the
// sum is in a fixed order (bitwise deterministic).  Every mbarrier wait is
// bounded; every CTA reaches both cluster barriers, on abort too.
#pragma once
#include "gemm_tc.cuh"

namespace tg {

template <int BN>
struct TcsCfg {
  static constexpr int B_CHUNKS = (BN + 63) / 64;
  static constexpr int B_STAGE = B_CHUNKS * 64 * TC_BK * 2;  // MN-major chunks; a K-major B uses BN x 128 B of it
  static constexpr int B_BYTES_K = BN * TC_BK * 2;
  static constexpr int STAGE = TC_A_STAGE + B_STAGE;
  static constexpr int RED_STRIDE = BN + 4;  // floats per buffer row (16-byte pad: 4-way store conflicts at most)
  static constexpr int RED_BYTES = TC_BM * RED_STRIDE * 4;
  static constexpr int BAR_BYTES = 256;
  static constexpr int RING_BUDGET = 232448 - 1024 - BAR_BYTES;
  static constexpr int STAGES = RING_BUDGET / STAGE > 8 ? 8 : RING_BUDGET / STAGE;
  static constexpr int RING = STAGES * STAGE;
  static constexpr int SMEM = 1024 + (RING > RED_BYTES ? RING : RED_BYTES) + BAR_BYTES;
  static constexpr int TMEM_COLS = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);
  static_assert(BN == 64 || BN == 128 || BN == 192 || BN == 256, "tile width");
  static_assert(SMEM <= 232448 && STAGES >= 4, "shared memory budget");
  static_assert(2 * STAGES + 2 <= BAR_BYTES / 8 - 2, "barrier area");
};

struct CsArgs {
  int m_tiles, n_tiles;
  int kb_total;  // K blocks of 64
  int kps;       // K blocks per cluster rank
  int raster_n;
  uint32_t idesc;
  int out_f16;  // 16-bit output type: 1 = fp16, 0 = bf16
  int a_chunked, b_chunked;
  void* C;  // [batch][M][N], row-major
  long long M, N;
  int accumulate;  // FP32 output: C += the product
  unsigned long long timeout_ns;
  unsigned int* status;
  unsigned long long* trace;  // event timestamps per CTA (only in -DTG_TRACE builds)
};

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

template <bool A_MN, bool B_MN, int BN, bool OUT16>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_cs_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const CsArgs args) {
  using Cfg = TcsCfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * TC_A_STAGE;
  const int rank = static_cast<int>(cluster_ctarank());
  const int nsplit = static_cast<int>(cluster_nctarank());
  float* red = reinterpret_cast<float*>(smem);  // the ring, once every MMA has read it
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (Cfg::RING > Cfg::RED_BYTES ? Cfg::RING : Cfg::RED_BYTES));
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // this cluster's tile and this CTA's K range
  int b, m0, n0;
  tile_origin(static_cast<int>(blockIdx.x) / nsplit, args.m_tiles, args.n_tiles, args.raster_n, BN, &b, &m0, &n0);
  const int kb0 = rank * args.kps;
  const int kb1 = min(args.kb_total, kb0 + args.kps);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(tfull), 1);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const unsigned long long tmo = args.timeout_ns;
  if (threadIdx.x == 0) TG_EVENT(15);  // before the wait for the previous kernel
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) TG_EVENT(0);

  bool have_acc = true;  // this CTA's partial tile is valid (no wait ran out)
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued[S];
#pragma unroll
      for (int s = 0; s < S; ++s) issued[s] = -1;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, tmo, abort_flag, args.status, 1)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&full[stage]);
        mbar_arrive_expect_tx(fb, TC_A_STAGE + (B_MN ? Cfg::B_STAGE : Cfg::B_BYTES_K));
        const uint32_t a_dst = smem_u32(sA + stage * TC_A_STAGE);
        const uint32_t b_dst = smem_u32(sB + stage * Cfg::B_STAGE);
        const int k0 = kb * TC_BK;
        if (A_MN) {
          if (args.a_chunked) {
            tma_load_4d(a_dst, &tmA, fb, 0, k0, m0 / 64, b);
          } else {
            tma_load_3d(a_dst, &tmA, fb, m0, k0, b);
            tma_load_3d(a_dst + 8192, &tmA, fb, m0 + 64, k0, b);
          }
        } else {
          tma_load_3d(a_dst, &tmA, fb, k0, m0, b);
        }
        if (B_MN) {
          if (args.b_chunked) {
            tma_load_4d(b_dst, &tmB, fb, 0, k0, n0 / 64, b);
          } else {
#pragma unroll
            for (int j = 0; j < Cfg::B_CHUNKS; ++j) tma_load_3d(b_dst + j * 8192, &tmB, fb, n0 + 64 * j, k0, b);
          }
        } else {
          tma_load_3d(b_dst, &tmB, fb, k0, n0, b);
        }
        issued[stage] = static_cast<int>(phase);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
#pragma unroll
        for (int s = 0; s < S; ++s)
          if (issued[s] >= 0)
            mbar_wait(smem_u32(&full[s]), static_cast<uint32_t>(issued[s]), 200000000ull, nullptr, args.status, 9);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(smem_u32(&full[stage]), phase, tmo, abort_flag, args.status, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(sA + stage * TC_A_STAGE);
        const uint32_t b_base = smem_u32(sB + stage * Cfg::B_STAGE);
#pragma unroll
        for (int kk = 0; kk < TC_BK / 16; ++kk) {
          const uint64_t ad = A_MN ? sdesc_sw128(a_base + kk * 2048, 8192, 1024) : sdesc_sw128(a_base + kk * 32, 16, 1024);
          const uint64_t bd = B_MN ? sdesc_sw128(b_base + kk * 2048, 8192, 1024) : sdesc_sw128(b_base + kk * 32, 16, 1024);
          umma_f16(tmem_base, ad, bd, args.idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&empty[stage]));
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        umma_commit(smem_u32(tfull));
      } else {
        umma_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, 200000000ull, nullptr, args.status, 10);
      }
    }
  } else {
    // ------------------------------------- epilogue: accumulator -> buffer
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    if (mbar_wait(smem_u32(tfull), 0, tmo, abort_flag, args.status, 4)) {
      if (warp == 2 && lane == 0) TG_EVENT(1);
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      float* dst = red + static_cast<size_t>(q * 32 + lane) * Cfg::RED_STRIDE;
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + ch * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(dst + ch * 32 + 4 * j) = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
      }
      if (warp == 2 && lane == 0) TG_EVENT(2);
    } else {
      have_acc = false;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
  // every CTA's buffer is written (and visible cluster-wide) past this point
  cluster_sync_all();
  if (threadIdx.x == 0) TG_EVENT(3);

  // ------------------------------------------ reduction of this CTA's rows
  if (!*abort_flag && have_acc) {
    constexpr int G = BN / 4;  // float4 groups per row
    const int r0 = rank * TC_BM / nsplit, r1 = (rank + 1) * TC_BM / nsplit;
    const int groups = (r1 - r0) * G;
    // two groups per thread and round: up to 16 remote loads in flight
    for (int base = threadIdx.x; base < groups; base += 2 * blockDim.x) {
      float4 w[2][8];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = base + u * blockDim.x;
        if (idx >= groups) break;
        const int row = r0 + idx / G, g = idx - (idx / G) * G;
        const uint32_t local = smem_u32(red + static_cast<size_t>(row) * Cfg::RED_STRIDE + 4 * g);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          if (s < nsplit) w[u][s] = ld_dsmem_f4(mapa_shared(local, static_cast<uint32_t>(s)));
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = base + u * blockDim.x;
        if (idx >= groups) break;
        const int row = r0 + idx / G, g = idx - (idx / G) * G;
        const long long m = static_cast<long long>(m0) + row, n = static_cast<long long>(n0) + 4 * g;
        if (m >= args.M || n >= args.N) continue;
        float4 v = w[u][0];  // the sum in rank order
#pragma unroll
        for (int s = 1; s < 8; ++s)
          if (s < nsplit) {
            v.x += w[u][s].x;
            v.y += w[u][s].y;
            v.z += w[u][s].z;
            v.w += w[u][s].w;
          }
        const long long o = (static_cast<long long>(b) * args.M + m) * args.N + n;
        if (OUT16) {
          uint2 pk;
          if (args.out_f16) {
            pk.x = pack_f16x2(v.x, v.y);
            pk.y = pack_f16x2(v.z, v.w);
          } else {
            pk.x = pack_bf16x2(v.x, v.y);
            pk.y = pack_bf16x2(v.z, v.w);
          }
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(args.C) + o) = pk;
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(args.C) + o);
          if (args.accumulate) {
            const float4 c0 = *dst;  // this thread alone writes these four elements
            v.x = c0.x + v.x;
            v.y = c0.y + v.y;
            v.z = c0.z + v.z;
            v.w = c0.w + v.w;
          }
          *dst = v;
        }
      }
    }
  }
  if (threadIdx.x == 0) TG_EVENT(5);
  // no CTA leaves while another may still read its buffer
  cluster_sync_all();
  if (threadIdx.x == 0) TG_EVENT(6);
}

}  // namespace tg
