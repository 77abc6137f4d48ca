// gemm_tc_launch.cuh -- host side of one tensor-core GEMM launch: tensor maps,
// kernel selection by tile width and output width, dynamic shared memory.
// Included once per layout family (gemm_tc_nt.cu, _nn.cu, _tn.cu) so the
// three families compile in parallel.
#pragma once
#include <cuda.h>
#include <stdlib.h>

#include "gemm_tc.cuh"
#include "gemm_tc2.cuh"
#include "gemm_tc_cs.cuh"
#include "tg_internal.h"

namespace tg {

// Tensor maps of the LoRA block appended to the reduction (same boxes as the
// main operands' maps, K = 64): A2 [M][64] K-major; B2 [N][64] K-major or
// [64][N] MN-major (chunked like the main B when that is chunked).  Without a
// LoRA block the main maps are copied (never read).
static bool lora_maps(const TcGemm& g, bool b_mn, bool b4, uint32_t b_box_rows, int b_chunks, const CUtensorMap& tmA,
                      const CUtensorMap& tmB, CUtensorMap* tmA2, CUtensorMap* tmB2) {
  if (g.lora_A2 == nullptr) {
    *tmA2 = tmA;
    *tmB2 = tmB;
    return true;
  }
  const uint64_t M = g.M, N = g.N;
  if (!encode_tmap_3d(tmA2, g.lora_A2, g.in_kind, 64, M, 1, 128, M * 128, 64, TC_BM, 128)) return false;
  if (b4) {
    const uint64_t d[4] = {64, 64, N / 64, 1}, st[3] = {N * 2, 128, 64 * N * 2};
    const uint32_t b[4] = {64, 64, static_cast<uint32_t>(b_chunks), 1};
    return encode_tmap_nd(tmB2, g.lora_B2, g.in_kind, 4, d, st, b, 128);
  }
  if (b_mn) return encode_tmap_3d(tmB2, g.lora_B2, g.in_kind, N, 64, 1, N * 2, 64 * N * 2, 64, 64, 128);
  return encode_tmap_3d(tmB2, g.lora_B2, g.in_kind, 64, N, 1, 128, N * 128, 64, b_box_rows, 128);
}

template <bool A_MN, bool B_MN, int BN, bool OUT16, bool DEEP = false>
static cudaError_t tc_launch_one(const TcGemm& g) {
  using Cfg = TcCfg<BN, DEEP>;
  auto kern = tc_gemm_kernel<A_MN, B_MN, BN, OUT16, DEEP>;
  // the attribute is per function and per device: set it once per device, so
  // later calls (including calls under stream capture) make no such call
  static bool attr_set[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }

  alignas(64) CUtensorMap tmA, tmB, tmC, tmC2, tmP;
  const uint64_t M = g.M, N = g.N, K = g.K, nb = g.batch;
  const uint64_t nbm = g.split3 ? 3 : nb;  // the operand maps' batch: the three parts of a split
  bool ok;
  // An MN-major operand whose width is a multiple of 64 is viewed as
  // [batch][width/64 chunks][K][64], so one box loads all of a stage's chunks
  // in the layout the MMA reads (chunks 8 KB apart).  Otherwise one 2-D box
  // per chunk (boxes past the width read zeros).
  const bool a4 = A_MN && M % 64 == 0 && chunked_mn_enabled();
  const bool b4 = B_MN && N % 64 == 0 && BN % 64 == 0 && chunked_mn_enabled();
  if (a4) {
    const uint64_t d[4] = {64, K, M / 64, nbm}, st[3] = {static_cast<uint64_t>(g.lda) * 2, 128,
                                                      static_cast<uint64_t>(g.a_bstride) * 2};
    const uint32_t b[4] = {64, 64, TC_BM / 64, 1};
    ok = encode_tmap_nd(&tmA, g.A, g.in_kind, 4, d, st, b, 128);
  } else if (A_MN) {  // stored [batch][K][M]
    ok = encode_tmap_3d(&tmA, g.A, g.in_kind, M, K, nbm, g.lda * 2, g.a_bstride * 2, 64, 64, 128);
  } else {  // stored [batch][M][K]
    ok = encode_tmap_3d(&tmA, g.A, g.in_kind, K, M, nbm, g.lda * 2, g.a_bstride * 2, 64, TC_BM, 128);
  }
  if (!ok) return cudaErrorInvalidValue;
  if (b4) {
    const uint64_t d[4] = {64, K, N / 64, nbm}, st[3] = {static_cast<uint64_t>(g.ldb) * 2, 128,
                                                      static_cast<uint64_t>(g.b_bstride) * 2};
    const uint32_t b[4] = {64, 64, static_cast<uint32_t>(Cfg::B_CHUNKS), 1};
    ok = encode_tmap_nd(&tmB, g.B, g.in_kind, 4, d, st, b, 128);
  } else if (B_MN) {  // stored [batch][K][N]
    ok = encode_tmap_3d(&tmB, g.B, g.in_kind, N, K, nbm, g.ldb * 2, g.b_bstride * 2, 64, 64, 128);
  } else {  // stored [batch][N][K]
    ok = encode_tmap_3d(&tmB, g.B, g.in_kind, K, N, nbm, g.ldb * 2, g.b_bstride * 2, 64, BN, 128);
  }
  if (!ok) return cudaErrorInvalidValue;
  alignas(64) CUtensorMap tmA2, tmB2;
  if (!lora_maps(g, B_MN, b4, BN, Cfg::B_CHUNKS, tmA, tmB, &tmA2, &tmB2)) return cudaErrorInvalidValue;

  // output (or FP32 split partials): [batch * splits][M][N], dense
  const bool split_parts = !g.sk && g.splits > 1;
  const int ck = split_parts ? EK_F32 : g.out_kind;
  const uint64_t esz = elem_bytes(ck);
  void* cptr = split_parts ? g.ws : g.C;
  ok = encode_tmap_3d(&tmC, cptr, ck, N, M, nb * (split_parts ? g.splits : 1), N * esz, M * N * esz,
                      OUT16 ? 64 : 32, 32, 128);
  if (!ok) return cudaErrorInvalidValue;
  // the 16-column tail of a tile width that is not a multiple of 64 / 32
  tmC2 = tmC;
  if (BN % (OUT16 ? 64 : 32) != 0) {
    ok = encode_tmap_3d(&tmC2, cptr, ck, N, M, nb * (split_parts ? g.splits : 1), N * esz, M * N * esz, 16, 32, 0);
    if (!ok) return cudaErrorInvalidValue;
  }

  TcArgs a;
  a.m_tiles = static_cast<int>((M + TC_BM - 1) / TC_BM);
  a.n_tiles = static_cast<int>((N + BN - 1) / BN);
  a.kbs = static_cast<int>((K + TC_BK - 1) / TC_BK);
  a.split3 = g.split3 ? 1 : 0;
  a.kb_total = g.split3 ? 6 * a.kbs : a.kbs;
  a.kb_lora = -1;
  if (g.lora_A2 != nullptr) {  // one more K block, after the product's own
    a.kb_lora = a.kb_total;
    a.kb_total += 1;
  }
  a.splits = g.sk ? 1 : g.splits;
  a.kps = (a.kb_total + a.splits - 1) / a.splits;
  a.units = static_cast<int>(nb) * a.m_tiles * a.n_tiles * a.splits;
  a.idesc = idesc_f16(g.in_kind == EK_BF16, A_MN, B_MN, TC_BM, BN);
  a.out_f16 = g.out_kind == EK_F16 ? 1 : 0;
  a.raster_n = g.raster_n;
  a.sk = g.sk;
  a.a_chunked = a4 ? 1 : 0;
  a.b_chunked = b4 ? 1 : 0;
  // tail split (never with stream-K or split partials)
  const TailGeo tg = tail_geo(M, N, static_cast<uint64_t>(a.kb_total) * TC_BK, nb, BN, g.grid,
                              (g.sk || g.splits > 1 || g.lora_A2) ? 1 : g.tail_splits, g.raster_n);
  a.dp_tiles = tg.dp_tiles;
  a.tail_splits = tg.splits;
  a.tail_kps = tg.kps;
  tmP = tmC;
  if (tg.tail_tiles > 0) {
    a.units = tg.dp_tiles + tg.tail_tiles * tg.splits;
    ok = encode_tmap_3d(&tmP, g.ws, EK_F32, BN, 128, static_cast<uint64_t>(tg.tail_tiles) * tg.splits, BN * 4,
                        128 * BN * 4, 32, 32, 128);
    if (!ok) return cudaErrorInvalidValue;
  }
  a.sk_iters = static_cast<long long>(a.units) * a.kb_total;
  a.sk_part = nullptr;
  a.sk_flags = nullptr;
  a.sk_epoch = g.sk_epoch;
  a.timeout_ns = g.timeout_ns;
  a.status = g.status;
  a.trace = nullptr;
#ifdef TG_TRACE
  if (const char* e = getenv("TG_TRACE_ADDR")) a.trace = reinterpret_cast<unsigned long long*>(strtoull(e, nullptr, 0));
#endif
  a.accumulate = g.accumulate && !split_parts ? 1 : 0;  // split partials: the reduction adds into C
  int grid = g.grid < a.units ? g.grid : a.units;
  if (g.sk) {
    // every CTA gets at least one iteration; the workspace holds grid slots
    grid = a.sk_iters < g.grid ? static_cast<int>(a.sk_iters) : g.grid;
    a.sk_part = static_cast<float*>(g.ws);
    a.sk_flags = reinterpret_cast<unsigned long long*>(static_cast<char*>(g.ws) +
                                                       static_cast<size_t>(grid) * TC_BM * BN * 4);
  }
  cudaError_t e2 =
      launch_k(kern, dim3(grid), dim3(TC_THREADS), Cfg::SMEM, g.stream, tmA, tmB, tmC, tmC2, tmP, tmA2, tmB2, a);
  if (e2 != cudaSuccess || tg.tail_tiles == 0) return e2;
  return tail_reduce_launch(static_cast<const float*>(g.ws), g.C, g.out_kind, tg, g.stream, g.accumulate);
}

// CTA-pair kernel: clusters of two CTAs, one per SM, persistent over
// 256 x BN tiles (x splits, or stream-K ranges).  The grid is the number of
// pairs that fit on the device at once (at most half the SMs), times two:
// stream-K needs every pair resident.
template <bool A_MN, bool B_MN, int BN, bool OUT16>
static cudaError_t tc2_launch_one(const TcGemm& g) {
  using Cfg = Tc2Cfg<BN, B_MN>;
  auto kern = tc2_gemm_kernel<A_MN, B_MN, BN, OUT16>;
  static bool attr_set[128] = {};
  static int max_pairs[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = g.stream;
  cfg.attrs = attr;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    int n = 0;
    cfg.gridDim = dim3(2 * (g.grid / 2 > 0 ? g.grid / 2 : 1));
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    max_pairs[dev] = n;
    attr_set[dev] = true;
  }

  alignas(64) CUtensorMap tmA, tmB, tmC, tmP;
  const uint64_t M = g.M, N = g.N, K = g.K, nb = g.batch;
  const uint64_t nbm = g.split3 ? 3 : nb;  // the operand maps' batch: the three parts of a split
  bool ok;
  const bool a4 = A_MN && M % 64 == 0 && chunked_mn_enabled();
  const bool b4 = B_MN && N % 64 == 0 && Cfg::BH % 64 == 0 && chunked_mn_enabled();
  if (a4) {
    const uint64_t d[4] = {64, K, M / 64, nbm}, st[3] = {static_cast<uint64_t>(g.lda) * 2, 128,
                                                      static_cast<uint64_t>(g.a_bstride) * 2};
    const uint32_t b[4] = {64, 64, TC_BM / 64, 1};
    ok = encode_tmap_nd(&tmA, g.A, g.in_kind, 4, d, st, b, 128);
  } else if (A_MN) {
    ok = encode_tmap_3d(&tmA, g.A, g.in_kind, M, K, nbm, g.lda * 2, g.a_bstride * 2, 64, 64, 128);
  } else {
    ok = encode_tmap_3d(&tmA, g.A, g.in_kind, K, M, nbm, g.lda * 2, g.a_bstride * 2, 64, TC_BM, 128);
  }
  if (!ok) return cudaErrorInvalidValue;
  if (b4) {
    const uint64_t d[4] = {64, K, N / 64, nbm}, st[3] = {static_cast<uint64_t>(g.ldb) * 2, 128,
                                                      static_cast<uint64_t>(g.b_bstride) * 2};
    const uint32_t b[4] = {64, 64, static_cast<uint32_t>(Cfg::B_CHUNKS), 1};
    ok = encode_tmap_nd(&tmB, g.B, g.in_kind, 4, d, st, b, 128);
  } else if (B_MN) {
    ok = encode_tmap_3d(&tmB, g.B, g.in_kind, N, K, nbm, g.ldb * 2, g.b_bstride * 2, 64, 64, 128);
  } else {
    ok = encode_tmap_3d(&tmB, g.B, g.in_kind, K, N, nbm, g.ldb * 2, g.b_bstride * 2, 64, Cfg::BH, 128);
  }
  if (!ok) return cudaErrorInvalidValue;
  alignas(64) CUtensorMap tmA2, tmB2;
  if (!lora_maps(g, B_MN, b4, Cfg::BH, Cfg::B_CHUNKS, tmA, tmB, &tmA2, &tmB2)) return cudaErrorInvalidValue;
  const bool split_parts = !g.sk && g.splits > 1;
  const int ck = split_parts ? EK_F32 : g.out_kind;
  const uint64_t esz = elem_bytes(ck);
  void* cptr = split_parts ? g.ws : g.C;
  ok = encode_tmap_3d(&tmC, cptr, ck, N, M, nb * (split_parts ? g.splits : 1), N * esz, M * N * esz,
                      OUT16 ? 64 : 32, 32, 128);
  if (!ok) return cudaErrorInvalidValue;

  TcArgs a = {};
  a.m_tiles = static_cast<int>((M + TC2_BM - 1) / TC2_BM);
  a.n_tiles = static_cast<int>((N + BN - 1) / BN);
  a.kbs = static_cast<int>((K + TC_BK - 1) / TC_BK);
  a.split3 = g.split3 ? 1 : 0;
  a.kb_total = g.split3 ? 6 * a.kbs : a.kbs;
  a.kb_lora = -1;
  if (g.lora_A2 != nullptr) {  // one more K block, after the product's own
    a.kb_lora = a.kb_total;
    a.kb_total += 1;
  }
  a.splits = g.sk ? 1 : g.splits;
  a.kps = (a.kb_total + a.splits - 1) / a.splits;
  a.units = static_cast<int>(nb) * a.m_tiles * a.n_tiles * a.splits;
  a.idesc = idesc_f16(g.in_kind == EK_BF16, A_MN, B_MN, TC2_BM, BN);
  a.out_f16 = g.out_kind == EK_F16 ? 1 : 0;
  a.raster_n = g.raster_n;
  a.a_chunked = a4 ? 1 : 0;
  a.b_chunked = b4 ? 1 : 0;
  // tail split (never with stream-K or split partials); the geometry is that
  // of a full wave of grid / 2 pairs, whatever number of pairs runs
  const TailGeo tg = tail_geo(M, N, static_cast<uint64_t>(a.kb_total) * TC_BK, nb, BN, g.grid / 2,
                              (g.sk || g.splits > 1 || g.lora_A2) ? 1 : g.tail_splits, g.raster_n, TC2_BM);
  a.dp_tiles = tg.dp_tiles;
  a.tail_splits = tg.splits;
  a.tail_kps = tg.kps;
  tmP = tmC;
  if (tg.tail_tiles > 0) {
    a.units = tg.dp_tiles + tg.tail_tiles * tg.splits;
    ok = encode_tmap_3d(&tmP, g.ws, EK_F32, BN, TC2_BM, static_cast<uint64_t>(tg.tail_tiles) * tg.splits, BN * 4,
                        TC2_BM * BN * 4, 32, 32, 128);
    if (!ok) return cudaErrorInvalidValue;
  }
  a.timeout_ns = g.timeout_ns;
  a.status = g.status;
  a.accumulate = g.accumulate && !split_parts ? 1 : 0;  // split partials: the reduction adds into C
  a.sk = g.sk;
  a.sk_iters = static_cast<long long>(a.units) * a.kb_total;
  a.sk_epoch = g.sk_epoch;
#ifdef TG_TRACE
  if (const char* e = getenv("TG_TRACE_ADDR")) a.trace = reinterpret_cast<unsigned long long*>(strtoull(e, nullptr, 0));
#endif
  int pairs = g.grid / 2;
  if (pairs > max_pairs[dev]) pairs = max_pairs[dev];
  const long long work = g.sk ? a.sk_iters : a.units;  // every pair gets at least one unit / iteration
  if (pairs > work) pairs = static_cast<int>(work);
  if (pairs < 1) pairs = 1;
  if (g.sk) {
    // stream-K slots: one FP32 partial tile per CTA, then the flags
    a.sk_part = static_cast<float*>(g.ws);
    a.sk_flags = reinterpret_cast<unsigned long long*>(static_cast<char*>(g.ws) +
                                                       static_cast<size_t>(2 * pairs) * TC_BM * BN * 4);
  }
  cfg.gridDim = dim3(2 * pairs);
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  cudaError_t e2 = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, tmP, tmA2, tmB2, a);
  if (e2 != cudaSuccess || tg.tail_tiles == 0) return e2;
  return tail_reduce_launch(static_cast<const float*>(g.ws), g.C, g.out_kind, tg, g.stream, g.accumulate);
}

template <bool A_MN, bool B_MN>
static cudaError_t tc2_launch_layout(const TcGemm& g) {
  const bool out16 = (g.sk || g.splits == 1) && g.out_kind != EK_F32;
  switch (g.bn) {
    case 128: return out16 ? tc2_launch_one<A_MN, B_MN, 128, true>(g) : tc2_launch_one<A_MN, B_MN, 128, false>(g);
    case 192: return out16 ? tc2_launch_one<A_MN, B_MN, 192, true>(g) : tc2_launch_one<A_MN, B_MN, 192, false>(g);
    case 256: return out16 ? tc2_launch_one<A_MN, B_MN, 256, true>(g) : tc2_launch_one<A_MN, B_MN, 256, false>(g);
    default: return cudaErrorInvalidValue;
  }
}

// Cluster split-K: one 128 x BN tile per cluster of csplit CTAs, every CTA
// one K range; the grid is tiles x csplit (no persistence, no workspace).
template <bool A_MN, bool B_MN, int BN, bool OUT16>
static cudaError_t tcs_launch_one(const TcGemm& g) {
  using Cfg = TcsCfg<BN>;
  auto kern = tc_cs_gemm_kernel<A_MN, B_MN, BN, OUT16>;
  static bool attr_set[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  alignas(64) CUtensorMap tmA, tmB;
  const uint64_t M = g.M, N = g.N, K = g.K, nb = g.batch;
  bool ok;
  const bool a4 = A_MN && M % 64 == 0 && chunked_mn_enabled();
  const bool b4 = B_MN && N % 64 == 0 && BN % 64 == 0 && chunked_mn_enabled();
  if (a4) {
    const uint64_t d[4] = {64, K, M / 64, nb}, st[3] = {static_cast<uint64_t>(g.lda) * 2, 128,
                                                      static_cast<uint64_t>(g.a_bstride) * 2};
    const uint32_t b[4] = {64, 64, TC_BM / 64, 1};
    ok = encode_tmap_nd(&tmA, g.A, g.in_kind, 4, d, st, b, 128);
  } else if (A_MN) {
    ok = encode_tmap_3d(&tmA, g.A, g.in_kind, M, K, nb, g.lda * 2, g.a_bstride * 2, 64, 64, 128);
  } else {
    ok = encode_tmap_3d(&tmA, g.A, g.in_kind, K, M, nb, g.lda * 2, g.a_bstride * 2, 64, TC_BM, 128);
  }
  if (!ok) return cudaErrorInvalidValue;
  if (b4) {
    const uint64_t d[4] = {64, K, N / 64, nb}, st[3] = {static_cast<uint64_t>(g.ldb) * 2, 128,
                                                      static_cast<uint64_t>(g.b_bstride) * 2};
    const uint32_t b[4] = {64, 64, static_cast<uint32_t>(Cfg::B_CHUNKS), 1};
    ok = encode_tmap_nd(&tmB, g.B, g.in_kind, 4, d, st, b, 128);
  } else if (B_MN) {
    ok = encode_tmap_3d(&tmB, g.B, g.in_kind, N, K, nb, g.ldb * 2, g.b_bstride * 2, 64, 64, 128);
  } else {
    ok = encode_tmap_3d(&tmB, g.B, g.in_kind, K, N, nb, g.ldb * 2, g.b_bstride * 2, 64, BN, 128);
  }
  if (!ok) return cudaErrorInvalidValue;

  CsArgs a = {};
  a.m_tiles = static_cast<int>((M + TC_BM - 1) / TC_BM);
  a.n_tiles = static_cast<int>((N + BN - 1) / BN);
  a.kb_total = static_cast<int>((K + TC_BK - 1) / TC_BK);
  // every rank gets a non-empty K range
  a.kps = (a.kb_total + g.csplit - 1) / g.csplit;
  const int ranks = (a.kb_total + a.kps - 1) / a.kps;
  a.raster_n = g.raster_n;
  a.idesc = idesc_f16(g.in_kind == EK_BF16, A_MN, B_MN, TC_BM, BN);
  a.out_f16 = g.out_kind == EK_F16 ? 1 : 0;
  a.a_chunked = a4 ? 1 : 0;
  a.b_chunked = b4 ? 1 : 0;
  a.C = g.C;
  a.M = static_cast<long long>(M);
  a.N = static_cast<long long>(N);
  a.accumulate = g.accumulate;
  a.timeout_ns = g.timeout_ns;
  a.status = g.status;
  a.trace = nullptr;
#ifdef TG_TRACE
  if (const char* e = getenv("TG_TRACE_ADDR")) a.trace = reinterpret_cast<unsigned long long*>(strtoull(e, nullptr, 0));
#endif
  const long long tiles = static_cast<long long>(nb) * a.m_tiles * a.n_tiles;
  if (tiles * ranks > 0x7fffffffLL) return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(ranks);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * ranks));
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = g.stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, a);
}

template <bool A_MN, bool B_MN>
static cudaError_t tcs_launch_layout(const TcGemm& g) {
  const bool out16 = g.out_kind != EK_F32;
  switch (g.bn) {
    case 64: return out16 ? tcs_launch_one<A_MN, B_MN, 64, true>(g) : tcs_launch_one<A_MN, B_MN, 64, false>(g);
    case 128: return out16 ? tcs_launch_one<A_MN, B_MN, 128, true>(g) : tcs_launch_one<A_MN, B_MN, 128, false>(g);
    case 192: return out16 ? tcs_launch_one<A_MN, B_MN, 192, true>(g) : tcs_launch_one<A_MN, B_MN, 192, false>(g);
    case 256: return out16 ? tcs_launch_one<A_MN, B_MN, 256, true>(g) : tcs_launch_one<A_MN, B_MN, 256, false>(g);
    default: return cudaErrorInvalidValue;
  }
}

template <bool A_MN, bool B_MN>
static cudaError_t tc_launch_layout(const TcGemm& g) {
  if (g.csplit > 1) return tcs_launch_layout<A_MN, B_MN>(g);
  if (g.pair) return tc2_launch_layout<A_MN, B_MN>(g);
  // split partials are FP32; so is an FP32 output
  const bool out16 = (g.sk || g.splits == 1) && g.out_kind != EK_F32;
  switch (g.bn) {
    case 64: return out16 ? tc_launch_one<A_MN, B_MN, 64, true>(g) : tc_launch_one<A_MN, B_MN, 64, false>(g);
    case 128: return out16 ? tc_launch_one<A_MN, B_MN, 128, true>(g) : tc_launch_one<A_MN, B_MN, 128, false>(g);
    case 144:
      if (g.deep) return out16 ? tc_launch_one<A_MN, B_MN, 144, true, true>(g) : tc_launch_one<A_MN, B_MN, 144, false, true>(g);
      return out16 ? tc_launch_one<A_MN, B_MN, 144, true>(g) : tc_launch_one<A_MN, B_MN, 144, false>(g);
    case 192:
      if (g.deep) return out16 ? tc_launch_one<A_MN, B_MN, 192, true, true>(g) : tc_launch_one<A_MN, B_MN, 192, false, true>(g);
      return out16 ? tc_launch_one<A_MN, B_MN, 192, true>(g) : tc_launch_one<A_MN, B_MN, 192, false>(g);
    case 256: return out16 ? tc_launch_one<A_MN, B_MN, 256, true>(g) : tc_launch_one<A_MN, B_MN, 256, false>(g);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tg
