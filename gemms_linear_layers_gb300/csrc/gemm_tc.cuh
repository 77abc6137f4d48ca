// gemm_tc.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// The three products of a linear layer in a training step (page "Twice the
// training speed on a BC-250 from tuned matrix kernels", section "Where the
// time went") differ only in which operand index is contiguous in memory, so
// one kernel template covers them, specialised on the major-ness of A and B:
//   forward   Y  = X W^T   : A = X  K-major,    B = W  K-major
//   dgrad     dX = dY W    : A = dY K-major,    B = W  MN-major
//   wgrad     dW = dY^T X  : A = dY MN-major,   B = X  MN-major
// 16-bit inputs, FP32 accumulation in tensor memory (section "Tuning the
// kernels": bf16 and fp16 with FP32 accumulation).
//
// CTA = 6 warps, one CTA per SM, persistent over output tiles of 128 x BN:
//   warp 0      TMA producer: 64-deep K blocks of A and B into a STAGES-deep
//               shared-memory ring (128-byte swizzle), full/empty mbarriers
//   warp 1      allocates tensor memory; one lane issues tcgen05.mma
//               (M=128, N=BN, K=16 per instruction) into one of two TMEM
//               accumulators, and tcgen05.commit frees smem stages
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quadrant, cast (RNE)
//               to the output type, swizzled staging tile, TMA store; the
//               accumulator is handed back as soon as it has been read, so
//               the next tile's MMAs overlap this tile's stores.
// Split-K: a unit is (tile, K range); partial sums go to an FP32 workspace
// and a separate kernel adds them in split order (deterministic).
// Tail split: when the tiles are not a whole number of waves, the tiles of
// the last, partial wave are split along K (tail_splits ways) while every
// other tile runs whole; the split pieces leave as FP32 partial tiles and
// a small kernel adds them in split order.
// Stream-K: the (tile x K block) iteration space is cut into gridDim.x equal
// contiguous ranges, one per CTA.  A tile cut by a range boundary is finished
// by the CTA holding its first K block (the owner): every later CTA that
// worked on the tile writes its FP32 partial tile to the workspace and
// publishes it with a flag; the owner waits for those flags, adds the
// partials to its accumulator in CTA order, clears their flags and writes the
// tile.  A flag holds a per-launch value, and is zero between launches.  Waits only
// ever point to higher-numbered CTAs, which produce their partial first
// thing, and all CTAs of the persistent grid are resident, so the waits end.
#pragma once
#include "ptx.cuh"

namespace tg {

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;  // 128 bytes of 16-bit values: one swizzle row
constexpr int TC_THREADS = 192;
constexpr int TC_EPI_WARPS = 4;
constexpr int TC_A_STAGE = TC_BM * TC_BK * 2;  // 16 KB
constexpr int TC_EPI_BUF = 32 * 128;           // 32 rows x 128 bytes

template <int BN, bool DEEP = false>
struct TcCfg {
  // B tile: BN rows of 128 bytes (K-major) or ceil(BN/64) 64-column chunks
  // of 8 KB (MN-major; a width that is not a multiple of 64 loads a full last
  // chunk and the MMA reads only its first columns)
  static constexpr int B_CHUNKS = (BN + 63) / 64;
  static constexpr int B_STAGE = B_CHUNKS * 64 * TC_BK * 2;
  static constexpr int B_BYTES_K = BN * TC_BK * 2;
  static constexpr int B_BYTES_MN = B_STAGE;
  // DEEP (widths 144 and 192 only): each epilogue warp keeps one staging
  // buffer instead of two, which makes room for a fifth operand stage (more
  // loads in flight); it pays when a CTA streams many K blocks, so that the
  // slower epilogue hides behind the next unit's MMAs.
  static_assert(!DEEP || BN == 192 || BN == 144, "deep ring only for 144 and 192");
  static constexpr int EPI_BUFS = DEEP ? 1 : 2;
  static constexpr int STAGES = DEEP ? 5 : (BN > 128) ? 4 : (BN == 128) ? 6 : 8;
  static constexpr int ACC_STRIDE = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);
  static constexpr int TMEM_COLS = 2 * ACC_STRIDE;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 + STAGES * (TC_A_STAGE + B_STAGE) +
                              TC_EPI_WARPS * EPI_BUFS * TC_EPI_BUF + BAR_BYTES;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(BN % 16 == 0 && BN >= 64 && BN <= 256, "tile width");
  static_assert(2 * STAGES + 5 <= BAR_BYTES / 8 - 2, "barrier area");
};

struct TcArgs {
  int m_tiles, n_tiles;
  int kb_total;  // K blocks of 64
  int kps;       // K blocks per split
  int splits;
  int units;     // batch * m_tiles * n_tiles * splits
  uint32_t idesc;
  int out_f16;   // 16-bit output type: 1 = fp16, 0 = bf16
  int raster_n;  // 1: consecutive units walk along N (they share the A tile)
  int a_chunked, b_chunked;  // MN-major operand loaded by one 4-D box ([batch][chunk][k][64]) per stage
  int dp_tiles;     // tail split: tiles run whole (the first dp_tiles in raster order)
  int tail_splits;  // > 1: each later tile is split into this many K ranges of tail_kps blocks
  int tail_kps;
  int sk;        // 1: stream-K schedule over batch * m_tiles * n_tiles * kb_total iterations
  long long sk_iters;
  float* sk_part;                // [gridDim.x][128][BN] FP32 partial tiles
  unsigned long long* sk_flags;  // [gridDim.x][4] publication flags, one per 32-row quadrant, 128 B apart
  unsigned long long sk_epoch;   // this launch's flag value
  unsigned long long timeout_ns;
  unsigned int* status;
  unsigned long long* trace;  // event timestamps per CTA (only in -DTG_TRACE builds)
  int accumulate;             // FP32 output: the tile writer adds its tile into C (C += A B)
  int kb_lora;                // >= 0: K block kb_lora comes from tmA2 / tmB2 at K offset 0 (a LoRA
                              // branch appended to the reduction); -1: none
  int split3;                 // 1: FP32 operands as three 16-bit parts each (the maps' batch index is
                              // the part); the reduction runs over 6 segments of kbs K blocks
  int kbs;
};

// FP32 operands split into three bf16 parts a = a0 + a1 + a2 (exactly, for
// normal values): a b is the sum of the six part products a_i b_j with
// i + j <= 2 (the three left out are below 2^-24 |a b|).  Segment s of the
// reduction multiplies part PA(s) of A by part PB(s) of B, the largest terms
// first: (0,0) (0,1) (1,0) (0,2) (1,1) (2,0).
__device__ __forceinline__ void split3_block(int kb, int kbs, int* k0, int* za, int* zb) {
  const int seg = kb / kbs;
  *k0 = (kb - seg * kbs) * TC_BK;
  *za = (0x210100 >> (4 * seg)) & 0xF;
  *zb = (0x012010 >> (4 * seg)) & 0xF;
}

#ifdef TG_TRACE
#define TG_EVENT(ev)                                                                    \
  do {                                                                                  \
    if (args.trace) args.trace[blockIdx.x * 16 + (ev)] = globaltimer_ns();             \
  } while (0)
#else
#define TG_EVENT(ev) \
  do {               \
  } while (0)
#endif

struct Unit {
  int b, m0, n0, split, kb0, kb1;
  int owner;   // this CTA writes the tile (stream-K: it holds the tile's first K block)
  int c_last;  // stream-K owner: last CTA holding a piece of the tile (> blockIdx.x: wait for partials)
  int part;    // tail split: this unit writes FP32 partial slot pz instead of the output
  int pz;
};

template <int BN>
__device__ __forceinline__ void tile_coords(int t, const TcArgs& a, Unit& c) {
  tile_origin(t, a.m_tiles, a.n_tiles, a.raster_n, BN, &c.b, &c.m0, &c.n0);
}

__device__ __forceinline__ long long sk_start(long long cta, const TcArgs& a) {
  return cta * a.sk_iters / gridDim.x;
}

// the CTA whose stream-K range holds iteration p
__device__ __forceinline__ int sk_cta_of(long long p, const TcArgs& a) {
  int c = static_cast<int>(p * gridDim.x / a.sk_iters);
  while (c + 1 < static_cast<int>(gridDim.x) && sk_start(c + 1, a) <= p) ++c;
  while (c > 0 && sk_start(c, a) > p) --c;
  return c;
}

// The sequence of units one CTA works on; every role walks the same one.
struct WorkIter {
  long long pos, end;  // stream-K range, or (unit index, -) for the split schedule
};

__device__ __forceinline__ WorkIter work_begin(const TcArgs& a) {
  WorkIter it;
  if (a.sk) {
    it.pos = sk_start(blockIdx.x, a);
    it.end = sk_start(blockIdx.x + 1, a);
  } else {
    it.pos = blockIdx.x;
    it.end = a.units;
  }
  return it;
}

template <int BN>
__device__ __forceinline__ bool work_next(const TcArgs& a, WorkIter& it, Unit& c) {
  if (it.pos >= it.end) return false;
  if (!a.sk) {
    const int u = static_cast<int>(it.pos);
    c.owner = 1;
    c.c_last = -1;
    if (a.tail_splits > 1 && u >= a.dp_tiles) {
      const int v = u - a.dp_tiles;
      tile_coords<BN>(a.dp_tiles + v / a.tail_splits, a, c);
      c.split = v % a.tail_splits;
      c.kb0 = c.split * a.tail_kps;
      c.kb1 = min(a.kb_total, c.kb0 + a.tail_kps);
      c.part = 1;
      c.pz = v;
    } else {
      c.split = u % a.splits;
      tile_coords<BN>(u / a.splits, a, c);
      c.kb0 = c.split * a.kps;
      c.kb1 = min(a.kb_total, c.kb0 + a.kps);
      c.part = 0;
      c.pz = 0;
    }
    it.pos += gridDim.x;
    return true;
  }
  const long long kb = a.kb_total;
  const int t = static_cast<int>(it.pos / kb);
  const long long kt0 = static_cast<long long>(t) * kb;
  const long long seg_end = min(it.end, kt0 + kb);
  tile_coords<BN>(t, a, c);
  c.split = 0;
  c.kb0 = static_cast<int>(it.pos - kt0);
  c.kb1 = static_cast<int>(seg_end - kt0);
  c.owner = it.pos == kt0;
  c.c_last = (c.owner && seg_end < kt0 + kb) ? sk_cta_of(kt0 + kb - 1, a) : -1;
  c.part = 0;
  c.pz = 0;
  it.pos = seg_end;
  return true;
}

// float4 index in the partial-tile area of (CTA, 32-row quadrant q, 32-column
// block, 4-column group j, lane): lanes innermost, so warp accesses coalesce
template <int BN>
__device__ __forceinline__ size_t sk_part_index(int cta, int q, int blk, int j, int lane) {
  return ((((static_cast<size_t>(cta) * 4 + q) * (BN / 32) + blk) * 8 + j) * 32) + lane;
}

// flag of (CTA, 32-row quadrant), one per 128-byte line
__device__ __forceinline__ int sk_flag_index(int cta, int q) { return (cta * 4 + q) * 16; }

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}
// ---- stream-K epilogue steps, shared by the single-CTA and CTA-pair kernels.
// The CTAs holding later pieces of a tile are first, first + step, ..., last
// (step 2 for pairs: the same rank in each later pair).

// Owner: wait until those CTAs have published their partial of this warp's
// 32 rows (quadrant q), then stage their sum, in CTA order, in tensor memory
// at t_pre (the idle accumulator).  False when a wait ran out.
template <int BN>
__device__ __forceinline__ bool sk_gather_parts(const TcArgs& args, int first, int last, int step, int q, int lane,
                                                uint32_t t_pre, volatile int* abort_flag) {
  // one lane polls, with back-off: flags sit on their own 128-byte lines
  // and a storm of polls would crowd the L2 slices the TMA loads need
  int ok = 1;
  if (lane == 0) {
    for (int cc = first; cc <= last && ok; cc += step) {
      const unsigned long long* fl = args.sk_flags + sk_flag_index(cc, q);
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_u64(fl) != args.sk_epoch) {
        __nanosleep(128);
        if (*abort_flag || globaltimer_ns() - t0 > args.timeout_ns) {
          if (!*abort_flag) {
            *abort_flag = 1;
            atomicOr(args.status, TG_DEVSTAT_TIMEOUT | 5u);
          }
          ok = 0;
          break;
        }
      }
    }
  }
  const bool have = __shfl_sync(0xffffffffu, ok, 0) != 0;
  __syncwarp();  // lane 0's acquire orders the other lanes' reads below
  if (!have) return false;
  // G 32-column blocks per round: their loads are all in flight together, so
  // the gather costs BN / (32 G) L2 round trips instead of BN / 32 (it runs
  // after the last piece is published, on the tile's critical path); more
  // than two blocks per round spill registers
  constexpr int NB = BN / 32;
  constexpr int G = NB % 2 == 0 ? 2 : 1;
#pragma unroll 1
  for (int b0 = 0; b0 < NB; b0 += G) {
    uint32_t sp[G * 32];
    for (int cc = first; cc <= last; cc += step) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float* src = args.sk_part + 4 * sk_part_index<BN>(cc, q, b0 + g, 0, lane);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 v = ld_cg_f4(src + 4 * 32 * j);
          uint32_t* d = sp + 32 * g + 4 * j;
          if (cc == first) {
            d[0] = __float_as_uint(v.x);
            d[1] = __float_as_uint(v.y);
            d[2] = __float_as_uint(v.z);
            d[3] = __float_as_uint(v.w);
          } else {
            d[0] = __float_as_uint(__uint_as_float(d[0]) + v.x);
            d[1] = __float_as_uint(__uint_as_float(d[1]) + v.y);
            d[2] = __float_as_uint(__uint_as_float(d[2]) + v.z);
            d[3] = __float_as_uint(__uint_as_float(d[3]) + v.w);
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) tmem_st_32x32b_x32(t_pre + (b0 + g) * 32, sp + 32 * g);
  }
  tmem_st_wait();
  return true;
}

// Contributor: this warp's 32 rows of the accumulator at t_row to partial
// slot `cta`, calling release() once the accumulator has been read (it hands
// the accumulator back), then publish the slot's quadrant flag.  Private
// layout: for each 32-column block and each 4-column group, the 32 lanes'
// float4s are adjacent, so every warp store writes 512 contiguous bytes.
template <int BN, typename Release>
__device__ __forceinline__ void sk_put_part(const TcArgs& args, int cta, int q, int lane, uint32_t t_row,
                                            Release release) {
#pragma unroll 1
  for (int ch = 0; ch < BN / 32; ++ch) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + ch * 32, r);
    tmem_ld_wait();
    if (ch == BN / 32 - 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release();
    }
    float4* dst = reinterpret_cast<float4*>(args.sk_part) + sk_part_index<BN>(cta, q, ch, 0, lane);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      dst[j * 32] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
  }
  // each warp publishes its own 32 rows: no barrier between the epilogue warps
  __threadfence();
  __syncwarp();
  if (lane == 0) st_release_u64(args.sk_flags + sk_flag_index(cta, q), args.sk_epoch);
}

// Owner, after its tile is written: clear the flags it consumed, so flags
// are zero between launches (a replayed CUDA graph reuses the same value)
__device__ __forceinline__ void sk_clear_flags(const TcArgs& args, int first, int last, int step, int q, int lane) {
  __syncwarp();
  if (lane == 0)
    for (int cc = first; cc <= last; cc += step) st_release_u64(args.sk_flags + sk_flag_index(cc, q), 0ull);
}

template <bool A_MN, bool B_MN, int BN, bool OUT16, bool DEEP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2,
                   const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB2, const TcArgs args) {
  using Cfg = TcCfg<BN, DEEP>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * TC_A_STAGE;
  uint8_t* sE = sB + S * Cfg::B_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + TC_EPI_WARPS * Cfg::EPI_BUFS * TC_EPI_BUF);
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), TC_EPI_WARPS);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    if (BN % 64 != 0) prefetch_tmap(&tmC2);
    if (args.tail_splits > 1) prefetch_tmap(&tmP);
    if (args.kb_lora >= 0) {
      prefetch_tmap(&tmA2);
      prefetch_tmap(&tmB2);
    }
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
  // the prologue above overlapped the previous kernel; global memory from here
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) TG_EVENT(0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued[S];
#pragma unroll
      for (int s = 0; s < S; ++s) issued[s] = -1;
      bool ok = true;
      WorkIter it = work_begin(args);
      Unit c;
      while (ok && work_next<BN>(args, it, c)) {
        for (int kb = c.kb0; kb < c.kb1; ++kb) {
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, tmo, abort_flag, args.status, 1)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, TC_A_STAGE + (B_MN ? Cfg::B_BYTES_MN : Cfg::B_BYTES_K));
          const uint32_t a_dst = smem_u32(sA + stage * TC_A_STAGE);
          const uint32_t b_dst = smem_u32(sB + stage * Cfg::B_STAGE);
          // the appended LoRA block: the same boxes from the second pair of maps
          const bool lx = kb == args.kb_lora;
          const CUtensorMap* mA = lx ? &tmA2 : &tmA;
          const CUtensorMap* mB = lx ? &tmB2 : &tmB;
          int k0 = lx ? 0 : kb * TC_BK, za = c.b, zb = c.b;
          if (args.split3) split3_block(kb, args.kbs, &k0, &za, &zb);
          if (A_MN) {
            if (args.a_chunked) {  // one box: 2 chunks of 64 columns x 64 k-rows
              tma_load_4d(a_dst, mA, fb, 0, k0, c.m0 / 64, za);
            } else {
              tma_load_3d(a_dst, mA, fb, c.m0, k0, za);
              tma_load_3d(a_dst + 8192, mA, fb, c.m0 + 64, k0, za);
            }
          } else {
            tma_load_3d(a_dst, mA, fb, k0, c.m0, za);
          }
          if (B_MN) {
            if (args.b_chunked) {
              tma_load_4d(b_dst, mB, fb, 0, k0, c.n0 / 64, zb);
            } else {
#pragma unroll
              for (int j = 0; j < Cfg::B_CHUNKS; ++j)
                tma_load_3d(b_dst + j * 8192, mB, fb, c.n0 + 64 * j, k0, zb);
            }
          } else {
            tma_load_3d(b_dst, mB, fb, k0, c.n0, zb);
          }
          issued[stage] = static_cast<int>(phase);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (it.pos == it.end || c.kb1 - c.kb0 >= 0) TG_EVENT(c.owner ? 9 : 1);
      }
      TG_EVENT(8);
      if (!ok) {
        // let every copy already issued land before the CTA unwinds
#pragma unroll
        for (int s = 0; s < S; ++s)
          if (issued[s] >= 0)
            mbar_wait(smem_u32(&full[s]), static_cast<uint32_t>(issued[s]), 200000000ull, nullptr,
                      args.status, 9);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      WorkIter it = work_begin(args);
      Unit c;
      while (ok && work_next<BN>(args, it, c)) {
        if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, tmo, abort_flag, args.status, 2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::ACC_STRIDE);
        for (int kb = c.kb0; kb < c.kb1; ++kb) {
          if (!mbar_wait(smem_u32(&full[stage]), phase, tmo, abort_flag, args.status, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * TC_A_STAGE);
          const uint32_t b_base = smem_u32(sB + stage * Cfg::B_STAGE);
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(a_base + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b_base + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(b_base + kk * 32, 16, 1024);
            umma_f16(d_tmem, ad, bd, args.idesc, (kb > c.kb0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&empty[stage]));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[acc]));
        TG_EVENT(c.owner ? 10 : 2);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        // every MMA issued so far must finish before tensor memory is freed
        umma_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, 200000000ull, nullptr, args.status, 10);
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int ew = warp - 2;  // staging buffers owned by this warp
    const int q = warp & 3;   // TMEM lane quadrant this warp may access
    uint8_t* ebuf = sE + ew * Cfg::EPI_BUFS * TC_EPI_BUF;
    constexpr int CW = OUT16 ? 64 : 32;  // columns per 128-byte staging row
    constexpr int NCH = BN / CW;
    constexpr int TW = BN % CW;  // a last, narrower chunk (16 columns) for BN = 144
    int acc = 0;
    uint32_t acc_phase = 0;
    int nstore = 0;
    WorkIter it = work_begin(args);
    Unit c;
    while (work_next<BN>(args, it, c)) {
      // A stream-K owner whose tile later CTAs finish: this is the CTA's
      // last unit, so the other accumulator is idle.  While this unit's MMAs
      // run, wait for the later pieces of this warp's 32 rows and stage their
      // sum (in CTA order) there, so the fix-up below reads tensor memory.
      const bool fixup = c.owner && c.c_last > static_cast<int>(blockIdx.x);
      bool have_parts = true;
      const uint32_t t_pre = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>((acc ^ 1) * Cfg::ACC_STRIDE);
      if (BN % 64 == 0 && fixup) {
        if (warp == 2 && lane == 0) TG_EVENT(4);
        have_parts = sk_gather_parts<BN>(args, blockIdx.x + 1, c.c_last, 1, q, lane, t_pre, abort_flag);
        if (warp == 2 && lane == 0) TG_EVENT(5);
      }
      if (!mbar_wait(smem_u32(&tfull[acc]), acc_phase, tmo, abort_flag, args.status, 4)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::ACC_STRIDE);
      const int row = q * 32 + lane;  // row of the tile this thread holds
      if (!c.owner) {
        // ---- stream-K contributor: FP32 partial tile to this CTA's slot, then publish
        sk_put_part<BN>(args, blockIdx.x, q, lane, t_row, [&] { mbar_arrive(smem_u32(&tempty[acc])); });
        if (warp == 2 && lane == 0) TG_EVENT(3);
      } else if (BN % 64 == 0 && c.part) {
        // ---- tail split piece: FP32 partial tile [128][BN] to slot pz
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + ch * 32, r);
          tmem_ld_wait();
          if (ch == BN / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
          }
          uint8_t* buf = ebuf + (nstore % Cfg::EPI_BUFS) * TC_EPI_BUF;
          // the staging buffer's previous store must have read it
          if (lane == 0 && nstore >= Cfg::EPI_BUFS) bulk_wait_read<Cfg::EPI_BUFS - 1>();
          __syncwarp();
          uint8_t* rowp = buf + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmP, smem_u32(buf), ch * 32, q * 32, c.pz);
            bulk_commit();
          }
          ++nstore;
        }
      } else {
        // ---- tile writer (a stream-K owner adds the later pieces staged above)
        const int zc = c.b * args.splits + c.split;
#pragma unroll 1
        for (int ch = 0; ch < NCH; ++ch) {
          uint32_t r[CW];
          tmem_ld_32x32b_x32(t_row + ch * CW, r);
          if (OUT16) tmem_ld_32x32b_x32(t_row + ch * CW + 32, r + 32);
          tmem_ld_wait();
          if (ch == NCH - 1 && TW == 0) {
            // accumulator fully read: hand it back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
          }
          if (BN % 64 == 0 && fixup && have_parts) {
            // add the later CTAs' pieces (their sum, staged in the idle accumulator)
#pragma unroll
            for (int sub = 0; sub < CW / 32; ++sub) {
              uint32_t sp[32];
              tmem_ld_32x32b_x32(t_pre + ch * CW + sub * 32, sp);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j)
                r[32 * sub + j] = __float_as_uint(__uint_as_float(r[32 * sub + j]) + __uint_as_float(sp[j]));
            }
          }
          uint8_t* buf = ebuf + (nstore % Cfg::EPI_BUFS) * TC_EPI_BUF;
          // the staging buffer's previous store must have read it
          if (lane == 0 && nstore >= Cfg::EPI_BUFS) bulk_wait_read<Cfg::EPI_BUFS - 1>();
          __syncwarp();
          uint8_t* rowp = buf + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint4 v;
            if (OUT16) {
              const uint32_t* f = r + 8 * j;
              if (args.out_f16) {
                v.x = pack_f16x2(__uint_as_float(f[0]), __uint_as_float(f[1]));
                v.y = pack_f16x2(__uint_as_float(f[2]), __uint_as_float(f[3]));
                v.z = pack_f16x2(__uint_as_float(f[4]), __uint_as_float(f[5]));
                v.w = pack_f16x2(__uint_as_float(f[6]), __uint_as_float(f[7]));
              } else {
                v.x = pack_bf16x2(__uint_as_float(f[0]), __uint_as_float(f[1]));
                v.y = pack_bf16x2(__uint_as_float(f[2]), __uint_as_float(f[3]));
                v.z = pack_bf16x2(__uint_as_float(f[4]), __uint_as_float(f[5]));
                v.w = pack_bf16x2(__uint_as_float(f[6]), __uint_as_float(f[7]));
              }
            } else {
              v = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            }
            // 128-byte swizzle: 16-byte chunk j of row `lane` sits at chunk j ^ (lane % 8)
            *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) = v;
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (!OUT16 && args.accumulate)
              tma_reduce_add_3d(&tmC, smem_u32(buf), c.n0 + ch * CW, c.m0 + q * 32, zc);
            else
              tma_store_3d(&tmC, smem_u32(buf), c.n0 + ch * CW, c.m0 + q * 32, zc);
            bulk_commit();
          }
          ++nstore;
        }
        if constexpr (TW != 0) {
          // the last TW columns: staged as dense rows of TW elements (no
          // swizzle) and stored through a map whose box is TW wide
          static_assert(TW == 16, "tail width");
          uint32_t r[16];
          tmem_ld_32x32b_x16(t_row + NCH * CW, r);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
          uint8_t* buf = ebuf + (nstore % Cfg::EPI_BUFS) * TC_EPI_BUF;
          // the staging buffer's previous store must have read it
          if (lane == 0 && nstore >= Cfg::EPI_BUFS) bulk_wait_read<Cfg::EPI_BUFS - 1>();
          __syncwarp();
          if (OUT16) {
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              w[j] = args.out_f16 ? pack_f16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]))
                                  : pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            uint4* rowp = reinterpret_cast<uint4*>(buf + lane * 32);
            rowp[0] = make_uint4(w[0], w[1], w[2], w[3]);
            rowp[1] = make_uint4(w[4], w[5], w[6], w[7]);
          } else {
            uint4* rowp = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
            for (int j = 0; j < 4; ++j) rowp[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (!OUT16 && args.accumulate)
              tma_reduce_add_3d(&tmC2, smem_u32(buf), c.n0 + NCH * CW, c.m0 + q * 32, zc);
            else
              tma_store_3d(&tmC2, smem_u32(buf), c.n0 + NCH * CW, c.m0 + q * 32, zc);
            bulk_commit();
          }
          ++nstore;
        }
        if (fixup && have_parts) sk_clear_flags(args, blockIdx.x + 1, c.c_last, 1, q, lane);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_all();
    if (warp == 2 && lane == 0) TG_EVENT(6);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace tg
