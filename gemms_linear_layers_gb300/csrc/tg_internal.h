// tg_internal.h -- declarations shared between the translation units of
// libtg.so (never installed; the public interface is include/tg.h).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <utility>

// device status word: bit 31 = a bounded wait timed out; low bits = site id
#define TG_DEVSTAT_TIMEOUT 0x80000000u
#define TG_DEVSTAT_SITE_MASK 0x0000FFFFu

namespace tg {

// Programmatic dependent launch on (default) or off ($TG_PDL=0).
bool pdl_enabled();
// MN-major GEMM operands loaded as one chunked 4-D box per stage (default) or
// one 2-D box per 64-column chunk ($TG_CHUNKED_MN=0).
bool chunked_mn_enabled();

// Sets the calling thread's tg_last_call() text (and logs it under TG_LOG).
void note_last_call(const std::string& s);

// Launch with programmatic stream serialization, so the kernel's prologue
// overlaps the previous kernel's tail (the kernel calls pdl_wait() before it
// touches global memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

enum ElemKind : int { EK_BF16 = 0, EK_F16 = 1, EK_F32 = 2 };

inline int elem_bytes(int ek) { return ek == EK_F32 ? 4 : 2; }

// Operand layouts of the three kernel families.  "K-major": the reduction
// index is contiguous; "MN-major": the row (A) or column (B) index is.
enum Layout : int {
  LAYOUT_NT = 0,  // A K-major, B K-major   (forward)
  LAYOUT_NN = 1,  // A K-major, B MN-major  (input gradient)
  LAYOUT_TN = 2,  // A MN-major, B MN-major (weight gradient)
};

// One tensor-core GEMM launch: C[b] (MxN) = sum_k A[b](m,k) B[b](k,n).
//   A K-major : stored [batch][M][K] with row pitch lda;   MN-major: [batch][K][M]
//   B K-major : stored [batch][N][K] with row pitch ldb;   MN-major: [batch][K][N]
//   C         : stored [batch][M][N], dense
struct TcGemm {
  int layout;
  const void* A;
  const void* B;
  void* C;
  int in_kind;   // EK_BF16 / EK_F16
  int out_kind;  // EK_BF16 / EK_F16 / EK_F32
  int64_t batch, M, N, K;
  int64_t lda, ldb;           // row pitches in elements
  int64_t a_bstride, b_bstride;  // batch strides in elements
  int bn;                     // tile width: 64, 128, 144, 192 or 256
  int splits;                 // >1: FP32 partials to ws, then an ordered reduction
  int raster_n;               // 1: walk output tiles along N first (A tiles reused)
  int sk;                     // 1: stream-K schedule (ws holds per-CTA partial tiles + flags)
  unsigned long long sk_epoch;  // flag value unique to this launch
  int tail_splits;            // >1: tiles past the last whole wave are split along K (ws: partial tiles)
  int deep;                   // 1: widths 144/192 with a fifth operand stage (one epilogue buffer)
  int pair;                   // 1: CTA-pair kernel, 256 x bn tiles (bn 128, 192 or 256)
  int csplit;                 // > 1: split-K across the CTAs of a cluster, added on chip (bn 64..256)
  int accumulate;             // FP32 C only: C += the product (gradient accumulation)
  // a LoRA branch appended to the reduction as one more 64-deep K block:
  // A2 [M][64] (K-major) and B2 laid out as B with K = 64 ([N][64] K-major,
  // [64][N] MN-major); both nullptr when absent
  const void* lora_A2;
  const void* lora_B2;
  // 1: A and B are FP32 operands given as three bf16 parts each, stored
  // [3][...] with the parts a_bstride / b_bstride elements apart (batch 1);
  // the reduction runs over the six part products (gemm_tc.cuh, split3_block)
  int split3;
  void* ws;
  int grid;                   // persistent CTAs
  cudaStream_t stream;
  unsigned int* status;
  unsigned long long timeout_ns;
};

// Workspace of a stream-K launch: one FP32 partial tile and four flags per
// CTA, each flag on its own 128-byte line.
inline size_t sk_ws_bytes(int grid, int bn) {
  return static_cast<size_t>(grid) * (128 * static_cast<size_t>(bn) * 4 + 4 * 128);
}

// Tail split: the tiles past the last whole wave of `grid` CTAs are each cut
// into `splits` K ranges whose FP32 partial tiles ([128][bn] each) are added
// by tail_reduce_kernel in split order.
struct TailGeo {
  int dp_tiles, tail_tiles, splits, kps;
  int m_tiles, n_tiles, raster_n, bn;
  int bm;  // tile height: 128 (single CTA) or 256 (CTA pair)
  int64_t M, N;
};
// grid: CTAs (single CTA) or pairs (bm = 256) of one wave
inline TailGeo tail_geo(int64_t M, int64_t N, int64_t K, int64_t batch, int bn, int grid, int want_splits,
                        int raster_n, int bm = 128) {
  TailGeo t{};
  t.bm = bm;
  t.m_tiles = static_cast<int>((M + bm - 1) / bm);
  t.n_tiles = static_cast<int>((N + bn - 1) / bn);
  t.raster_n = raster_n;
  t.bn = bn;
  t.M = M;
  t.N = N;
  const int tiles = static_cast<int>(batch) * t.m_tiles * t.n_tiles;
  const int kb = static_cast<int>((K + 63) / 64);
  t.dp_tiles = grid > 0 ? (tiles / grid) * grid : tiles;
  t.tail_tiles = tiles - t.dp_tiles;
  if (t.dp_tiles == 0 || t.tail_tiles == 0 || want_splits < 2 || bn % 64 != 0) {
    t.dp_tiles = tiles;
    t.tail_tiles = 0;
    t.splits = 1;
    t.kps = kb;
    return t;
  }
  t.kps = (kb + want_splits - 1) / want_splits;
  t.splits = (kb + t.kps - 1) / t.kps;
  if (t.splits < 2) {
    t.dp_tiles = tiles;
    t.tail_tiles = 0;
    t.splits = 1;
    t.kps = kb;
  }
  return t;
}
inline size_t tail_ws_bytes(const TailGeo& t) {
  return static_cast<size_t>(t.tail_tiles) * t.splits * t.bm * static_cast<size_t>(t.bn) * 4;
}
// Origin of output tile t (batch-major, then raster order within the batch)
// for tiles bm rows high.
__host__ __device__ inline void tile_origin(int t, int m_tiles, int n_tiles, int raster_n, int bn, int* b, int* m0,
                                            int* n0, int bm = 128) {
  const int tiles = m_tiles * n_tiles;
  *b = t / tiles;
  const int r = t - *b * tiles;
  if (raster_n) {  // consecutive units walk along N: they share the A tile
    *n0 = (r % n_tiles) * bn;
    *m0 = (r / n_tiles) * bm;
  } else {  // consecutive units walk down M: they share the B tile
    *m0 = (r % m_tiles) * bm;
    *n0 = (r / m_tiles) * bn;
  }
}
// accumulate (FP32 C only): C += the sum instead of C = the sum
cudaError_t tail_reduce_launch(const float* P, void* C, int out_kind, const TailGeo& t, cudaStream_t stream,
                               int accumulate);

// per-layout launchers (gemm_tc_{nt,nn,tn}.cu)
cudaError_t tc_gemm_launch_nt(const TcGemm& g);
cudaError_t tc_gemm_launch_nn(const TcGemm& g);
cudaError_t tc_gemm_launch_tn(const TcGemm& g);

// FP32 split partials ws[b*splits + s][M][N] -> C[b][M][N], s ascending
// (accumulate, FP32 C only: C += the sum)
cudaError_t splitk_reduce_launch(const float* ws, void* C, int out_kind, int64_t batch,
                                 int64_t splits, int64_t MN, cudaStream_t stream, int accumulate);

// Plain strided GEMM on CUDA cores for shapes the tensor-core path cannot take
// (row pitches that are not 16-byte multiples, unaligned pointers, FP32 operands).
//   C[b][i][j] = sum_k A[b*a_bs + i*a_rs + k*a_cs] * B[b*b_bs + k*b_rs + j*b_cs]
struct SimtGemm {
  const void* A;
  const void* B;
  void* C;
  int a_kind, b_kind, out_kind;
  int64_t batch, M, N, K;
  int64_t a_bs, a_rs, a_cs, b_bs, b_rs, b_cs;
  int accumulate;  // C += scale * the product (FP32 arithmetic, one rounding to C's type)
  float scale;     // without accumulate: C = scale * the product
  cudaStream_t stream;
};
cudaError_t simt_gemm_launch(const SimtGemm& g);

// FP32-input layer product on the CUDA cores (gemm_ffma.cu), batch 1, dense
// row-major operands in the layouts above; C FP32 with row pitch N.
struct FfmaGemm {
  int layout;
  const float* A;
  const float* B;
  float* C;
  int64_t M, N, K, lda, ldb;
  int splits;      // > 1: FP32 partials in ws[split][M][N], added in split order afterwards
  float* ws;
  int accumulate;  // C += the product
  cudaStream_t stream;
};
int ffma_splits(int64_t M, int64_t N, int64_t K, int sms);
size_t ffma_ws_bytes(int64_t M, int64_t N, int64_t K, int sms);
cudaError_t ffma_gemm_launch(const FfmaGemm& g);

// Tensor-map encoding through the driver entry point (tmap.cpp).
bool encode_tmap_3d(void* tmap_out, const void* base, int elem_kind, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                    uint32_t box1, int swizzle_bytes);
bool encode_tmap_nd(void* tmap_out, const void* base, int elem_kind, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes);

// FP32 [n] -> three bf16 parts at dst, dst + pstride and dst + 2 pstride, with
// v = p0 + p1 + p2 exactly for normal v (gemm_ffma.cu); non-finite v keeps
// only p0.
cudaError_t split3_launch(const float* src, int64_t n, int64_t pstride, uint16_t* dst, cudaStream_t stream);

// rank-r LoRA streaming kernels (lora.cu)
struct LoraArgs {
  const void* X;   // [T, d_in]
  const void* A;   // [r, d_in]
  const void* B;   // [d_out, r]
  const void* H;   // [T, r]
  const void* dY;  // [T, d_out]
  void* out;       // op-dependent output
  void* out2;
  void* out3;
  void* out4;
  float* ws;
  int64_t T, d_in, d_out, r;
  int in_kind, out_kind;
  int num_sms;
  cudaStream_t stream;
  unsigned int* status;          // device status word (bounded waits report here)
  unsigned long long timeout_ns; // limit of every wait on an mbarrier
  int add;                       // up projection: out += scale * H B^T; gradient: dX += scale * dH A,
                                 // dA and dB scaled
  float scale;
  int w32;                       // A and B are FP32 (split into 16-bit hi + lo parts in ws); dA, dB FP32
};
size_t lora_down_ws_bytes(int64_t T, int64_t d_in, int64_t r, int num_sms);
cudaError_t lora_down_launch(const LoraArgs& a);
cudaError_t lora_up_launch(const LoraArgs& a);
size_t lora_grad_ws_bytes(int64_t T, int64_t d_in, int64_t d_out, int64_t r, int num_sms);
cudaError_t lora_grad_launch(const LoraArgs& a);
// workspace of the FP32-factor calls (op 0 down, 1 up, 2 gradient): the
// factors' hi/lo parts, after the gradient's own workspace
size_t lora_w32_ws_bytes(int op, int64_t T, int64_t d_in, int64_t d_out, int sms);

// A rank-r LoRA branch (r <= 32) staged as the 64-deep K block a layer product
// appends to its reduction (lora_block.cu): A2 = [hi(scale h) | lo(scale h) | 0]
// [T][64] from H [T][r] (16-bit, or FP32 when h_f32), B2 from F: forward
// F = B [N][r] -> [N][64]; input gradient (dgrad) F = A [r][N] -> [64][N].
// ws holds lora_block_ws_bytes(T, N) bytes; *A2, *B2 receive the two arrays.
size_t lora_block_ws_bytes(int64_t T, int64_t N);
cudaError_t lora_block_prep_launch(const void* H, int h_f32, const void* F, int64_t T, int64_t N, int64_t r, float scale,
                                   int in_kind, int dgrad, void* ws, const void** A2, const void** B2, int sms,
                                   cudaStream_t stream);

// wait-timeout probe kernel (api.cu)
cudaError_t wait_probe_launch(unsigned long long timeout_ns, unsigned int* status,
                              cudaStream_t stream);

}  // namespace tg
