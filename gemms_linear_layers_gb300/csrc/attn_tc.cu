// Fused attention forward on the tensor cores (tcgen05, TMEM, TMA):
//   O[h] = softmax(scale * Q[h] K[h]^T) V[h]   per head, softmax over keys,
// without writing the [s, s] score or probability matrices.
//
// Page "Twice the training speed on a BC-250 from tuned matrix kernels",
// section "What's left": the batched products inside attention, with the
// softmax between them, are what a fused attention kernel would take over.
// The two products are the ones the library also runs unfused (S = Q K^T,
// O = P V); here they run back to back on chip with each row's softmax kept
// online (running maximum m and sum l).
//
// One CTA computes 128 query rows of one head (one TMEM lane per row), two
// CTAs per SM so that one CTA's softmax overlaps the other's MMAs.  Per
// block of 128 keys:
//   warp 0      TMA: the Q tile once, then K and V blocks [128 keys][64] into
//               a two-stage ring (128-byte swizzle)
//   warp 1      tcgen05.mma: S = Q K^T into TMEM (M = 128, N = 128 keys),
//               then O += P V with P read from TMEM (M = 128, N = 64)
//   warps 2..9  softmax, two warps per TMEM lane quadrant, each over half of
//               the block's keys: its rows of S from TMEM, the block maximum
//               (combined with the partner warp's), and P = 2^(x - m + C)
//               written back over S as 16-bit hi + lo parts (hi = RNE(p),
//               lo = RNE(p - hi)), so P enters the second product to within
//               2^-17 of its FP32 value (bf16; 2^-22 for fp16); at the end
//               O / l goes to memory.
// The running maximum is refreshed only when a block's maximum exceeds it by
// more than TAU (in log2 units): P then stays below 2^(TAU + C), and O and l
// are rescaled only on those blocks (exact: the softmax is invariant to the
// shift).  C = 7 keeps P's lo parts clear of the fp16 subnormal range for
// every weight above 2^-10 of the row's largest (the scale cancels in O / l).
#include "attn.h"
#include "attn_common.cuh"
#include "smem_attr.h"

namespace tg {
namespace {

using namespace attn;

constexpr int FSTAGES = 2;  // K/V ring depth
constexpr int FBAR_BYTES = 128;
constexpr int FXCH_BYTES = 2 * 4 * 2 * 32 * 4;  // pair-exchange buffer (2 slots)
constexpr int FSMEM = 1024 + TILE + FSTAGES * 2 * TILE + FBAR_BYTES + FXCH_BYTES;
constexpr uint32_t FTMEM_COLS = 256;  // S/P [0, 128), O [128, 192)
constexpr uint32_t T_S = 0, T_O = 128;
constexpr float TAU = 8.f;
constexpr float CP = 7.f;

struct FwdArgs {
  int s, nblk;
  float scale_log2;  // scale * log2(e)
  void* O;
  int out_kind;
  uint32_t idesc_qk, idesc_pv;
  unsigned long long timeout_ns;
  unsigned int* status;
};

template <bool BF16>
__global__ void __launch_bounds__(THREADS, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + TILE;
  uint8_t* sV = sK + FSTAGES * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + FSTAGES * TILE);
  uint64_t* q_full = bars;
  uint64_t* kv_full = q_full + 1;
  uint64_t* kv_empty = kv_full + FSTAGES;
  uint64_t* s_full = kv_empty + FSTAGES;
  uint64_t* p_full = s_full + 1;
  uint64_t* pv_done = p_full + 1;
  uint64_t* drain = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + FBAR_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.y, q0 = blockIdx.x * BT;
  const int nblk = a.nblk;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int i = 0; i < FSTAGES; ++i) {
      mbar_init(smem_u32(&kv_full[i]), 1);
      mbar_init(smem_u32(&kv_empty[i]), 1);
    }
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(p_full), ROW_WARPS);
    mbar_init(smem_u32(pv_done), 1);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), FTMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long tmo = a.timeout_ns;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(q_full), TILE);
      tma_load_3d(smem_u32(sQ), &tmQ, smem_u32(q_full), 0, q0, head);
      int issued[FSTAGES];
#pragma unroll
      for (int i = 0; i < FSTAGES; ++i) issued[i] = -1;
      for (int j = 0; j < nblk; ++j) {
        const int st = j % FSTAGES;
        const uint32_t ph = static_cast<uint32_t>((j / FSTAGES) & 1);
        if (!mbar_wait(smem_u32(&kv_empty[st]), ph ^ 1u, tmo, abort_flag, a.status, 21)) break;
        const uint32_t fb = smem_u32(&kv_full[st]);
        mbar_arrive_expect_tx(fb, 2 * TILE);
        tma_load_3d(smem_u32(sK + st * TILE), &tmK, fb, 0, j * BT, head);
        tma_load_3d(smem_u32(sV + st * TILE), &tmV, fb, 0, j * BT, head);
        issued[st] = static_cast<int>(ph);
      }
      // every copy issued must land before the CTA may exit
      mbar_wait(smem_u32(q_full), 0, 200000000ull, nullptr, a.status, 29);
#pragma unroll
      for (int i = 0; i < FSTAGES; ++i)
        if (issued[i] >= 0)
          mbar_wait(smem_u32(&kv_full[i]), static_cast<uint32_t>(issued[i]), 200000000ull, nullptr, a.status, 29);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(smem_u32(q_full), 0, tmo, abort_flag, a.status, 22);
      tc_fence_after();
      const uint32_t qa = smem_u32(sQ);
      for (int j = 0; ok && j < nblk; ++j) {
        const int st = j % FSTAGES;
        const uint32_t ph = static_cast<uint32_t>((j / FSTAGES) & 1);
        if (!mbar_wait(smem_u32(&kv_full[st]), ph, tmo, abort_flag, a.status, 23)) {
          ok = false;
          break;
        }
        // the previous block's P V must have read P before S overwrites it
        if (j > 0 && !mbar_wait(smem_u32(pv_done), static_cast<uint32_t>((j - 1) & 1), tmo, abort_flag, a.status, 24)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ka = smem_u32(sK + st * TILE), va = smem_u32(sV + st * TILE);
        // S = Q K^T: both operands K-major (head dimension contiguous)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_f16(tmem + T_S, sdesc_sw128(qa + kk * 32, 16, 1024), sdesc_sw128(ka + kk * 32, 16, 1024), a.idesc_qk,
                   kk > 0 ? 1u : 0u);
        umma_commit(smem_u32(s_full));
        if (!mbar_wait(smem_u32(p_full), static_cast<uint32_t>(j & 1), tmo, abort_flag, a.status, 25)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // O += P_hi V + P_lo V: P from TMEM (keys 32c..32c+31 sit in columns
        // 32c..32c+15 as hi pairs, 32c+16..32c+31 as lo pairs), V MN-major
        // (one 64-column chunk, 16 key rows per step)
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk) {
          const uint32_t pc = T_S + static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8);
          const uint64_t vd = sdesc_sw128(va + kk * 2048, 8192, 1024);
          umma_f16_ta(tmem + T_O, tmem + pc, vd, a.idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          umma_f16_ta(tmem + T_O, tmem + pc + 16, vd, a.idesc_pv, 1u);
        }
        umma_commit(smem_u32(&kv_empty[st]));
        umma_commit(smem_u32(pv_done));
      }
      if (!ok) {
        // every MMA issued so far must finish before tensor memory is freed
        umma_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, 200000000ull, nullptr, a.status, 30);
      }
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int q = warp & 3;            // TMEM lane quadrant of this warp
    const int half = (warp - 2) >> 2;  // which 64 keys of each block (and 32 columns of O)
    const int row = q * 32 + lane;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float sl = a.scale_log2;
    const bool neg = sl < 0.f;  // then the largest logit is at the smallest score
    const float asl = fabsf(sl);
    float m_used = -INFINITY, l = 0.f;
    // After a failed wait the loop still runs to the end (every later wait
    // returns at once), so the two warps of a pair always meet at the same
    // named barriers; tensor memory is then read and written as garbage
    // but never out of bounds, and nothing is stored.
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      ok = mbar_wait(smem_u32(s_full), static_cast<uint32_t>(j & 1), tmo, abort_flag, a.status, 26) && ok;
      tc_fence_after();
      const int kvalid = min(BT, a.s - j * BT) - half * 64;  // keys of this warp's half inside the sequence
      // pass 1: the largest (or smallest, for a negative scale) score of the row's half block
      float vm = -INFINITY;
      {
        uint32_t r[64];  // both 32-column chunks in flight together
        tmem_ld_32x32b_x32(t_row + T_S + half * 64, r);
        tmem_ld_32x32b_x32(t_row + T_S + half * 64 + 32, r + 32);
        tmem_ld_wait();
        if (kvalid >= 64) {
#pragma unroll
          for (int e = 0; e < 64; ++e) vm = fmaxf(vm, neg ? -__uint_as_float(r[e]) : __uint_as_float(r[e]));
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e < kvalid) vm = fmaxf(vm, neg ? -__uint_as_float(r[e]) : __uint_as_float(r[e]));
        }
      }
      vm = fmaxf(vm, pair_exchange(xch, j & 1, q, half, lane, vm));
      const float mx = vm * asl;  // the block's largest logit (log2 units)
      float rescale = 1.f;
      const bool refresh = j == 0 || mx > m_used + TAU;
      if (refresh) {
        rescale = ex2(m_used - mx);  // 0 on the first block
        m_used = mx;
      }
      const float mc = m_used - CP;
      // pass 2: P = 2^(x - m + C) as hi + lo 16-bit pairs over the same columns
      float sum = 0.f;
      uint32_t r[64];  // both chunks in flight together again
      tmem_ld_32x32b_x32(t_row + T_S + half * 64, r);
      tmem_ld_32x32b_x32(t_row + T_S + half * 64 + 32, r + 32);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float p[32];
        if (kvalid >= 64) {
#pragma unroll
          for (int e = 0; e < 32; ++e) p[e] = ex2(fmaf(__uint_as_float(r[c * 32 + e]), sl, -mc));
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            p[e] = c * 32 + e < kvalid ? ex2(fmaf(__uint_as_float(r[c * 32 + e]), sl, -mc)) : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) sum += p[e];
        uint32_t w[32];
        split32<BF16>(p, w);
        tmem_st_32x32b_x32(t_row + T_S + half * 64 + c * 32, w);
      }
      l = l * rescale + sum;
      // O (this warp's 32 columns) scaled to a refreshed maximum; every earlier
      // P V has completed, since this block's S was committed after them
      if (__any_sync(0xffffffffu, refresh && j > 0)) rescale32(t_row + T_O + half * 32, rescale);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(p_full));
    }
    // ---- epilogue: O / l to memory, row q0 + row of this head, this warp's 32 columns
    if (ok) ok = mbar_wait(smem_u32(pv_done), static_cast<uint32_t>((nblk - 1) & 1), tmo, abort_flag, a.status, 27);
    l += pair_exchange(xch, nblk & 1, q, half, lane, l);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const float inv = 1.f / l;
      const int grow = q0 + row;
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + T_O + half * 32, r);
      tmem_ld_wait();
      float v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]) * inv;
      if (grow < a.s) store_row32(a.O, a.out_kind, (static_cast<size_t>(head) * a.s + grow) * D + half * 32, v);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, FTMEM_COLS);
  }
}

}  // namespace

cudaError_t attn_fwd_tc_launch(const void* Q, const void* K, const void* V, void* O, int64_t heads, int64_t s,
                               int64_t d, float scale, int in_kind, int out_kind, unsigned int* status,
                               unsigned long long timeout_ns, cudaStream_t stream) {
  if (heads == 0 || s == 0) return cudaSuccess;
  if (d != D) return cudaErrorInvalidValue;
  alignas(64) CUtensorMap tmQ, tmK, tmV;
  const uint64_t pitch = D * 2;
  if (!encode_tmap_3d(&tmQ, Q, in_kind, D, s, heads, pitch, pitch * s, D, BT, 128) ||
      !encode_tmap_3d(&tmK, K, in_kind, D, s, heads, pitch, pitch * s, D, BT, 128) ||
      !encode_tmap_3d(&tmV, V, in_kind, D, s, heads, pitch, pitch * s, D, BT, 128))
    return cudaErrorInvalidValue;
  FwdArgs a{};
  a.s = static_cast<int>(s);
  a.nblk = static_cast<int>((s + BT - 1) / BT);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.O = O;
  a.out_kind = out_kind;
  const bool bf = in_kind == EK_BF16;
  a.idesc_qk = idesc_f16(bf, false, false, 128, BT);
  a.idesc_pv = idesc_f16(bf, false, true, 128, D);
  a.timeout_ns = timeout_ns;
  a.status = status;
  auto kern = bf ? attn_fwd_tc_kernel<true> : attn_fwd_tc_kernel<false>;
  const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), FSMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((s + BT - 1) / BT), static_cast<unsigned>(heads));
  return launch_k(kern, grid, dim3(THREADS), FSMEM, stream, tmQ, tmK, tmV, a);
}

}  // namespace tg
