// gemm_tc2.cuh -- the CTA-pair variant of the persistent tcgen05 GEMM.
//
// Same products and arithmetic as gemm_tc.cuh (page "Twice the training
// speed on a BC-250 from tuned matrix kernels", sections "Where the time
// went" and "Tuning the kernels": 16-bit inputs, FP32 accumulation), with
// output tiles of 256 x BN computed by a cluster of two CTAs on two SMs:
//   - each CTA loads its own 128 rows of A and its own half of B (BN/2 rows
//     of a K-major B, BN/2 columns of an MN-major one) into a ring at the
//     same shared-memory offsets in both CTAs;
//   - the even CTA (rank 0) issues tcgen05.mma.cta_group::2 with M = 256,
//     which reads both CTAs' operand halves and accumulates each CTA's 128
//     rows in that CTA's tensor memory;
//   - its commits arrive on the "stage free" and "accumulator full" barriers
//     of both CTAs (multicast); both CTAs' loads complete on rank 0's "stage
//     full" barrier, which rank 0 arms with the pair's byte count;
//   - each CTA's epilogue stores its 128 rows and arrives on rank 0's
//     "accumulator free" barrier.
// Per SM this halves the B bytes each K block moves from L2 (an SM streams
// 16 KB of A and BN/2 x 128 bytes of B per 128 x BN x 64 of MMA work, where
// the single-CTA kernel moves all BN rows of B), and the freed shared
// memory holds a deeper ring (6 stages at BN = 192/256, 8 at 128).
// Schedules as in the single-CTA kernel: data-parallel over (tile, split)
// units with FP32 split partials; the tail split (whole tiles for the full
// waves, the last wave's tiles cut along K into FP32 partials that a second
// kernel adds); stream-K over pairs.  Every wait is bounded; an
// aborting CTA waits at the final cluster barrier, so neither CTA of a pair
// leaves while the other may still touch its shared or tensor memory.
#pragma once
#include "gemm_tc.cuh"

namespace tg {

constexpr int TC2_BM = 256;

template <int BN, bool B_MN>
struct Tc2Cfg {
  static constexpr int BH = BN / 2;  // B rows (K-major) or columns (MN-major) held by one CTA
  static constexpr int B_CHUNKS = (BH + 63) / 64;
  static constexpr int B_BYTES = B_MN ? B_CHUNKS * 64 * TC_BK * 2 : BH * TC_BK * 2;
  static constexpr int STAGE = TC_A_STAGE + B_BYTES;
  static constexpr int EPI_BYTES = TC_EPI_WARPS * 2 * TC_EPI_BUF;
  static constexpr int BAR_BYTES = 256;
  static constexpr int RING_BUDGET = 232448 - 1024 - EPI_BYTES - BAR_BYTES;
  static constexpr int STAGES = RING_BUDGET / STAGE > 8 ? 8 : RING_BUDGET / STAGE;
  static constexpr int ACC_STRIDE = BN <= 128 ? 128 : 256;
  static constexpr int TMEM_COLS = 2 * ACC_STRIDE;
  static constexpr int SMEM = 1024 + STAGES * STAGE + EPI_BYTES + BAR_BYTES;
  static_assert(BN == 128 || BN == 192 || BN == 256, "pair tile width");
  static_assert(B_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(SMEM <= 232448 && STAGES >= 4, "shared memory budget");
  static_assert(2 * STAGES + 5 <= BAR_BYTES / 8 - 2, "barrier area");
};

struct Unit2 {
  int b, m0, n0, zc, kb0, kb1;
  int owner;   // this pair writes the tile (stream-K: it holds the tile's first K block)
  int c_last;  // stream-K owner: last pair holding a piece of the tile (> this pair: gather partials)
  int part;    // tail split: this unit writes FP32 partial slot pz instead of the output
  int pz;
};

// The sequence of units one pair works on (both CTAs and every role walk
// the same one): (tile, split) units dealt round-robin to the pairs, or, for
// stream-K, an equal contiguous range of the (tile x K block) iterations.
struct PairIter {
  long long pos, end;
};

__device__ __forceinline__ int pair_count() { return static_cast<int>(gridDim.x >> 1); }
__device__ __forceinline__ int pair_index() { return static_cast<int>(blockIdx.x >> 1); }

__device__ __forceinline__ long long pair_sk_start(long long p, const TcArgs& a) {
  return p * a.sk_iters / pair_count();
}

// the pair whose stream-K range holds iteration i
__device__ __forceinline__ int pair_sk_of(long long i, const TcArgs& a) {
  const int np = pair_count();
  int p = static_cast<int>(i * np / a.sk_iters);
  while (p + 1 < np && pair_sk_start(p + 1, a) <= i) ++p;
  while (p > 0 && pair_sk_start(p, a) > i) --p;
  return p;
}

__device__ __forceinline__ PairIter pair_begin(const TcArgs& a) {
  PairIter it;
  if (a.sk) {
    it.pos = pair_sk_start(pair_index(), a);
    it.end = pair_sk_start(pair_index() + 1, a);
  } else {
    it.pos = pair_index();
    it.end = a.units;
  }
  return it;
}

__device__ __forceinline__ void pair_tile(int t, const TcArgs& a, int bn, Unit2& c) {
  const int tiles = a.m_tiles * a.n_tiles;
  c.b = t / tiles;
  const int r = t - c.b * tiles;
  if (a.raster_n) {
    c.n0 = (r % a.n_tiles) * bn;
    c.m0 = (r / a.n_tiles) * TC2_BM;
  } else {
    c.m0 = (r % a.m_tiles) * TC2_BM;
    c.n0 = (r / a.m_tiles) * bn;
  }
}

__device__ __forceinline__ bool pair_next(const TcArgs& a, int bn, PairIter& it, Unit2& c) {
  if (it.pos >= it.end) return false;
  if (!a.sk) {
    const int u = static_cast<int>(it.pos);
    c.owner = 1;
    c.c_last = -1;
    if (a.tail_splits > 1 && u >= a.dp_tiles) {
      // tail split: a K range of one of the tiles past the last whole wave
      const int v = u - a.dp_tiles;
      pair_tile(a.dp_tiles + v / a.tail_splits, a, bn, c);
      c.zc = c.b;
      c.kb0 = (v % a.tail_splits) * a.tail_kps;
      c.kb1 = min(a.kb_total, c.kb0 + a.tail_kps);
      c.part = 1;
      c.pz = v;
    } else {
      const int split = u % a.splits;
      pair_tile(u / a.splits, a, bn, c);
      c.zc = c.b * a.splits + split;
      c.kb0 = split * a.kps;
      c.kb1 = min(a.kb_total, c.kb0 + a.kps);
      c.part = 0;
      c.pz = 0;
    }
    it.pos += pair_count();
    return true;
  }
  const long long kb = a.kb_total;
  const int t = static_cast<int>(it.pos / kb);
  const long long kt0 = static_cast<long long>(t) * kb;
  const long long seg_end = min(it.end, kt0 + kb);
  pair_tile(t, a, bn, c);
  c.zc = c.b;
  c.kb0 = static_cast<int>(it.pos - kt0);
  c.kb1 = static_cast<int>(seg_end - kt0);
  c.owner = it.pos == kt0;
  c.c_last = (c.owner && seg_end < kt0 + kb) ? pair_sk_of(kt0 + kb - 1, a) : -1;
  c.part = 0;
  c.pz = 0;
  it.pos = seg_end;
  return true;
}

#ifdef TG_TRACE
// time spent in a wait, summed per role; written to trace slot `slot`
#define TG_WAIT_BEGIN(v) const uint64_t v##_t0 = globaltimer_ns()
#define TG_WAIT_END(acc, v) acc += globaltimer_ns() - v##_t0
#define TG_WAIT_STORE(slot, acc) \
  do {                           \
    if (args.trace) args.trace[blockIdx.x * 16 + (slot)] = (acc); \
  } while (0)
#else
#define TG_WAIT_BEGIN(v) \
  do {                   \
  } while (0)
#define TG_WAIT_END(acc, v) \
  do {                      \
  } while (0)
#define TG_WAIT_STORE(slot, acc) \
  do {                           \
  } while (0)
#endif

template <bool A_MN, bool B_MN, int BN, bool OUT16>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
                    const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                    const TcArgs args) {
  using Cfg = Tc2Cfg<BN, B_MN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * TC_A_STAGE;
  uint8_t* sE = sB + S * Cfg::B_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + Cfg::EPI_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);   // rank 0's producer arms it; both CTAs' bytes complete it
      mbar_init(smem_u32(&empty[s]), 1);  // one multicast commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), 2 * TC_EPI_WARPS);  // the epilogue warps of both CTAs
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    if (args.tail_splits > 1) prefetch_tmap(&tmP);
    if (args.kb_lora >= 0) {
      prefetch_tmap(&tmA2);
      prefetch_tmap(&tmB2);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  __syncthreads();
  // both CTAs' barriers are initialised before either CTA signals the other's
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const unsigned long long tmo = args.timeout_ns;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) TG_EVENT(0);

  if (warp == 0) {
    // ------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued[S];
#pragma unroll
      for (int s = 0; s < S; ++s) issued[s] = -1;
      bool ok = true;
      unsigned long long w_empty = 0;
      (void)w_empty;
      PairIter it = pair_begin(args);
      Unit2 c;
      const int a_row = static_cast<int>(rank) * TC_BM;    // this CTA's rows of the pair tile
      const int b_off = static_cast<int>(rank) * Cfg::BH;  // this CTA's half of B
      while (ok && pair_next(args, BN, it, c)) {
        for (int kb = c.kb0; kb < c.kb1; ++kb) {
          TG_WAIT_BEGIN(we);
          if (!mbar_wait<true>(smem_u32(&empty[stage]), phase ^ 1u, tmo, abort_flag, args.status, 1)) {
            ok = false;
            break;
          }
          TG_WAIT_END(w_empty, we);
          const uint32_t fb_local = smem_u32(&full[stage]);
          if (rank == 0) mbar_arrive_expect_tx(fb_local, 2 * Cfg::STAGE);
          const uint32_t fb = mapa_shared(fb_local, 0);
          const uint32_t a_dst = smem_u32(sA + stage * TC_A_STAGE);
          const uint32_t b_dst = smem_u32(sB + stage * Cfg::B_BYTES);
          // the appended LoRA block: the same boxes from the second pair of maps
          const bool lx = kb == args.kb_lora;
          const CUtensorMap* mA = lx ? &tmA2 : &tmA;
          const CUtensorMap* mB = lx ? &tmB2 : &tmB;
          int k0 = lx ? 0 : kb * TC_BK, za = c.b, zb = c.b;
          if (args.split3) split3_block(kb, args.kbs, &k0, &za, &zb);
          const int m = c.m0 + a_row;
          if (A_MN) {
            if (args.a_chunked) {
              tma_load_4d_pair(a_dst, mA, fb, 0, k0, m / 64, za);
            } else {
              tma_load_3d_pair(a_dst, mA, fb, m, k0, za);
              tma_load_3d_pair(a_dst + 8192, mA, fb, m + 64, k0, za);
            }
          } else {
            tma_load_3d_pair(a_dst, mA, fb, k0, m, za);
          }
          const int n = c.n0 + b_off;
          if (B_MN) {
            if (args.b_chunked) {
              tma_load_4d_pair(b_dst, mB, fb, 0, k0, n / 64, zb);
            } else {
#pragma unroll
              for (int j = 0; j < Cfg::B_CHUNKS; ++j) tma_load_3d_pair(b_dst + j * 8192, mB, fb, n + 64 * j, k0, zb);
            }
          } else {
            tma_load_3d_pair(b_dst, mB, fb, k0, n, zb);
          }
          if (issued[stage] < 0 && stage == 0) TG_EVENT(1);
          issued[stage] = static_cast<int>(phase);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      TG_EVENT(8);
      TG_WAIT_STORE(10, w_empty);
      if (ok) {
        // the last commits of rank 0's MMAs arrive on these barriers: see
        // them all before this CTA can leave
#pragma unroll
        for (int s = 0; s < S; ++s)
          if (issued[s] >= 0 &&
              !mbar_wait<true>(smem_u32(&empty[s]), static_cast<uint32_t>(issued[s]), tmo, abort_flag, args.status, 11))
            break;
      } else if (rank == 0) {
        // copies already issued complete on this CTA's barriers: let them land
#pragma unroll
        for (int s = 0; s < S; ++s)
          if (issued[s] >= 0)
            mbar_wait<true>(smem_u32(&full[s]), static_cast<uint32_t>(issued[s]), 200000000ull, nullptr, args.status,
                            9);
      } else {
        // the peer's copies complete on rank 0's barriers, which this CTA
        // cannot wait on: give copies issued just before the abort time to land
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer (rank 0 only)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      unsigned long long w_tempty = 0, w_full = 0;
      (void)w_tempty;
      (void)w_full;
      PairIter it = pair_begin(args);
      Unit2 c;
      while (ok && pair_next(args, BN, it, c)) {
        TG_WAIT_BEGIN(wt);
        if (!mbar_wait<true>(smem_u32(&tempty[acc]), acc_phase ^ 1u, tmo, abort_flag, args.status, 2)) {
          ok = false;
          break;
        }
        TG_WAIT_END(w_tempty, wt);
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::ACC_STRIDE);
        for (int kb = c.kb0; kb < c.kb1; ++kb) {
          TG_WAIT_BEGIN(wf);
          if (!mbar_wait<true>(smem_u32(&full[stage]), phase, tmo, abort_flag, args.status, 3)) {
            ok = false;
            break;
          }
          TG_WAIT_END(w_full, wf);
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * TC_A_STAGE);
          const uint32_t b_base = smem_u32(sB + stage * Cfg::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(a_base + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b_base + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(b_base + kk * 32, 16, 1024);
            umma_f16_pair(d_tmem, ad, bd, args.idesc, (kb > c.kb0 || kk > 0) ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&empty[stage]), 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&tfull[acc]), 0x3);
        TG_EVENT(7);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      TG_WAIT_STORE(11, w_tempty);
      TG_WAIT_STORE(12, w_full);
      // every MMA issued must finish before either CTA frees tensor memory
      umma_commit_pair(smem_u32(drain), 0x1);
      mbar_wait<true>(smem_u32(drain), 0, ok ? tmo : 200000000ull, nullptr, args.status, 10);
    }
  } else {
    // ------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - 2;
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    uint8_t* ebuf = sE + ew * 2 * TC_EPI_BUF;
    constexpr int CW = OUT16 ? 64 : 32;  // columns per 128-byte staging row
    constexpr int NCH = BN / CW;
    static_assert(BN % CW == 0, "pair tile width and output width");
    const uint32_t tempty_cl = mapa_shared(smem_u32(&tempty[0]), 0);
    const int pair = pair_index();
    unsigned long long w_tfull = 0, w_ld = 0, w_bw = 0, w_pack = 0, w_fs = 0, w_chunks = 0, w_unit = 0;
    (void)w_chunks;
    (void)w_unit;
    (void)w_pack;
    (void)w_fs;
    (void)w_tfull;
    (void)w_ld;
    (void)w_bw;
    int acc = 0;
    uint32_t acc_phase = 0;
    int nstore = 0;
    PairIter it = pair_begin(args);
    Unit2 c;
    while (pair_next(args, BN, it, c)) {
      // A stream-K owner whose tile later pairs finish: this is the pair's
      // last unit, so the other accumulator is idle.  While this unit's MMAs
      // run, gather the later pieces of this warp's 32 rows (from the CTA of
      // the same rank in each later pair) and stage their sum there.
      const bool fixup = c.owner && c.c_last > pair;
      const int first = 2 * (pair + 1) + static_cast<int>(rank);
      const int last = 2 * c.c_last + static_cast<int>(rank);
      bool have_parts = true;
      const uint32_t t_pre = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>((acc ^ 1) * Cfg::ACC_STRIDE);
      if (fixup) {
        if (warp == 2 && lane == 0) TG_EVENT(4);
        have_parts = sk_gather_parts<BN>(args, first, last, 2, q, lane, t_pre, abort_flag);
        if (warp == 2 && lane == 0) TG_EVENT(5);
      }
      TG_WAIT_BEGIN(wtf);
      if (!mbar_wait<true>(smem_u32(&tfull[acc]), acc_phase, tmo, abort_flag, args.status, 4)) break;
      TG_WAIT_END(w_tfull, wtf);
      TG_WAIT_BEGIN(wu);
      if (warp == 2 && lane == 0) TG_EVENT(9);
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::ACC_STRIDE);
      if (!c.owner) {
        // stream-K contributor: FP32 partial of this CTA's 128 rows to its slot
        const uint32_t te = tempty_cl + static_cast<uint32_t>(acc * 8);
        sk_put_part<BN>(args, blockIdx.x, q, lane, t_row, [&] { mbar_arrive_cluster(te); });
        if (warp == 2 && lane == 0) TG_EVENT(3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
        continue;
      }
      if (c.part) {
        // tail split piece: this CTA's 128 rows of FP32 partial slot pz
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + ch * 32, r);
          tmem_ld_wait();
          if (ch == BN / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_cl + static_cast<uint32_t>(acc * 8));
          }
          uint8_t* buf = ebuf + (nstore & 1) * TC_EPI_BUF;
          if (lane == 0 && nstore >= 2) bulk_wait_read<1>();
          __syncwarp();
          uint8_t* rowp = buf + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmP, smem_u32(buf), ch * 32, static_cast<int>(rank) * TC_BM + q * 32, c.pz);
            bulk_commit();
          }
          ++nstore;
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
        continue;
      }
      const int row0 = c.m0 + static_cast<int>(rank) * TC_BM + q * 32;
      TG_WAIT_BEGIN(wc);
#pragma unroll 1
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t r[CW];
        TG_WAIT_BEGIN(wl);
        tmem_ld_32x32b_x32(t_row + ch * CW, r);
        if (OUT16) tmem_ld_32x32b_x32(t_row + ch * CW + 32, r + 32);
        tmem_ld_wait();
        TG_WAIT_END(w_ld, wl);
        if (ch == NCH - 1) {
          // accumulator read: hand it back to rank 0's MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty_cl + static_cast<uint32_t>(acc * 8));
        }
        if (fixup && have_parts) {
          // add the later pairs' pieces (their sum, staged in the idle accumulator)
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
        uint8_t* buf = ebuf + (nstore & 1) * TC_EPI_BUF;
        TG_WAIT_BEGIN(wb);
        if (lane == 0 && nstore >= 2) bulk_wait_read<1>();
        __syncwarp();
        TG_WAIT_END(w_bw, wb);
        uint8_t* rowp = buf + lane * 128;
        TG_WAIT_BEGIN(wp);
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
        TG_WAIT_END(w_pack, wp);
        TG_WAIT_BEGIN(wfs);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (!OUT16 && args.accumulate)
            tma_reduce_add_3d(&tmC, smem_u32(buf), c.n0 + ch * CW, row0, c.zc);
          else
            tma_store_3d(&tmC, smem_u32(buf), c.n0 + ch * CW, row0, c.zc);
          bulk_commit();
        }
        TG_WAIT_END(w_fs, wfs);
        ++nstore;
      }
      TG_WAIT_END(w_chunks, wc);
      if (fixup && have_parts) sk_clear_flags(args, first, last, 2, q, lane);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      TG_WAIT_END(w_unit, wu);
    }
    if (lane == 0) bulk_wait_all();
    if (warp == 2 && lane == 0) TG_EVENT(6);
    if (warp == 2 && lane == 0) TG_WAIT_STORE(13, w_tfull);
    if (warp == 2 && lane == 0) TG_WAIT_STORE(14, w_ld);
    if (warp == 2 && lane == 0) TG_WAIT_STORE(15, w_bw);
    if (warp == 2 && lane == 0) TG_WAIT_STORE(3, w_pack);
    if (warp == 2 && lane == 0) TG_WAIT_STORE(4, w_fs);
    if (warp == 2 && lane == 0) TG_WAIT_STORE(5, w_chunks);
    if (warp == 2 && lane == 0) TG_WAIT_STORE(1, w_unit);
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA leaves (or frees tensor memory) while the other may still
  // read its shared memory, write its tensor memory or arrive on its barriers
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace tg
