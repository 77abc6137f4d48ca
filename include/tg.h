/*
 * tg.h -- training products of linear layers on GB300 (sm_103a): C ABI of libtg.so.
 *
 * What the library computes comes from the page "Twice the training speed on a
 * BC-250 from tuned matrix kernels":
 *   - section "Where the time went": every linear layer of a training step runs
 *     three matrix products -- the forward pass, the gradient for its input and
 *     the gradient for its weight -- each in a different memory layout;
 *   - section "Tuning the kernels": bf16 and fp16 inputs with FP32 accumulation,
 *     for every layer of a decoder at 1,024-4,096 tokens, the rank-16 LoRA
 *     matrices and the batched products inside attention;
 *   - section "Checking the results are right": all three layouts and the
 *     batched attention products are checked against a float64 CPU product.
 *
 * Conventions shared by every entry point
 *   - Tensors are row-major and dense (no stride arguments).  Names follow the
 *     page: X[T, d_in] activations, W[d_out, d_in] weight, dY[T, d_out] output
 *     gradient, T tokens.
 *   - Pointers are DEVICE pointers owned by the caller; the library keeps no
 *     reference after the call returns and allocates no device memory for a
 *     call.  Scratch space, when a call needs it, is the caller's `ws`
 *     (tg_workspace_size gives the size; `ws` may be NULL when that is 0).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous: TG_OK means the work was enqueued.  A device-side failure
 *     (a bounded wait that timed out) is reported by tg_stream_status.
 *   - Outputs are overwritten (no alpha/beta).  `in` is TG_BF16 or TG_F16;
 *     `out` is TG_F32 or the input type.  16-bit outputs are the FP32 result
 *     rounded to nearest even.  The layer products (tg_gemm_fwd, _dgrad,
 *     _wgrad and their _noalloc / _accumulate forms) also take in = TG_F32
 *     with out = TG_F32: FP32 operands, held to the same bound.  When every
 *     row pitch is a multiple of 8 elements (the output's of 4) they run on
 *     the tensor cores: each operand is cut into three bf16 parts that carry
 *     it exactly (staged in `ws`), and the product sums the six part products
 *     a_i b_j with i + j <= 2 in FP32; otherwise every product is fused into
 *     its FP32 sum on the CUDA cores (FFMA; also for every FP32 product when
 *     the environment sets TG_FP32_PATH=ffma).  No TF32 rounding either way.
 *   - Sizes: a negative size is TG_ERR_INVALID_ARG; an empty output (a zero
 *     row or column count) is TG_OK with nothing done; an empty reduction
 *     writes zeros.  Every size must be below 2^31.
 *   - Pointers: each must be aligned to its element size (else
 *     TG_ERR_MISALIGNED).  Base addresses aligned to 16 bytes with row pitches
 *     that are multiples of 16 bytes take the tensor-core path; anything else
 *     takes a slower CUDA-core GPU path with identical semantics.
 *   - Errors are return codes; nothing aborts, exits or throws across the ABI.
 *   - Calls on different streams may run concurrently if they do not share a
 *     workspace or an output.  One exception: a layer product whose tile-table
 *     entry selects the stream-K schedule (token "sk", see tg_load_table)
 *     needs every CTA of its launch resident at once, because CTAs wait for
 *     partial tiles of later CTAs of the same launch; run it with the GPU to
 *     itself (nothing else in flight on other streams), or a wait may run out
 *     and tg_stream_status report TG_ERR_DEVICE_TIMEOUT.  Only a table entry
 *     selects stream-K; the shipped table has none and the library never
 *     picks it by itself.
 */
#ifndef TG_H
#define TG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { TG_BF16 = 0, TG_F16 = 1, TG_F32 = 2 } tg_dtype;

typedef enum {
  TG_OK = 0,
  TG_ERR_INVALID_ARG = 1,         /* NULL pointer with a non-empty tensor, bad size, bad enum */
  TG_ERR_UNSUPPORTED_DTYPE = 2,   /* input not bf16/fp16 (or FP32 for a layer product), or output
                                     neither FP32 nor the input type */
  TG_ERR_MISALIGNED = 3,          /* pointer not aligned to its element size */
  TG_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below tg_workspace_size() for the call */
  TG_ERR_CUDA = 5,                /* a CUDA runtime call failed (launch, attribute, device query) */
  TG_ERR_DEVICE_TIMEOUT = 6,      /* a kernel's bounded wait ran out (tg_stream_status) */
  TG_ERR_TABLE = 7,               /* a tile table could not be read or parsed */
  TG_ERR_UNSUPPORTED_DEVICE = 8   /* the current device is not sm_103 */
} tg_status;

/* The six batched products inside attention (no mask, no softmax, no scale).
 * Tensors are [batch, rows, cols]; batch = heads, s = sequence, d = head dim. */
typedef enum {
  TG_ATTN_QK = 0,    /* S  = Q  K^T : A=Q [b,s,d],  B=K [b,s,d]  -> C [b,s,s] */
  TG_ATTN_PV = 1,    /* O  = P  V   : A=P [b,s,s],  B=V [b,s,d]  -> C [b,s,d] */
  TG_ATTN_DO_VT = 2, /* dP = dO V^T : A=dO [b,s,d], B=V [b,s,d]  -> C [b,s,s] */
  TG_ATTN_PT_DO = 3, /* dV = P^T dO : A=P [b,s,s],  B=dO [b,s,d] -> C [b,s,d] */
  TG_ATTN_DS_K = 4,  /* dQ = dS K   : A=dS [b,s,s], B=K [b,s,d]  -> C [b,s,d] */
  TG_ATTN_DST_Q = 5  /* dK = dS^T Q : A=dS [b,s,s], B=Q [b,s,d]  -> C [b,s,d] */
} tg_attn_op;

/* Operation ids for tg_workspace_size. */
typedef enum {
  TG_OP_GEMM_FWD = 0,   /* d0=T, d1=d_out, d2=d_in */
  TG_OP_GEMM_DGRAD = 1, /* d0=T, d1=d_out, d2=d_in */
  TG_OP_GEMM_WGRAD = 2, /* d0=T, d1=d_out, d2=d_in */
  TG_OP_LORA_DOWN = 3,  /* d0=T, d1=d_in, d2=r */
  TG_OP_LORA_UP = 4,    /* d0=T, d1=d_out, d2=r */
  TG_OP_LORA_GRAD = 5,  /* d0=T, d1=d_in, d2=d_out, d3=r */
  TG_OP_BMM_ATTN = 6,   /* d0=tg_attn_op, d1=batch, d2=s, d3=d */
  TG_OP_LORA_DOWN_F32W = 7,  /* d0=T, d1=d_in, d2=r */
  TG_OP_LORA_UP_F32W = 8,    /* d0=T, d1=d_out, d2=r */
  TG_OP_LORA_GRAD_F32W = 9,  /* d0=T, d1=d_in, d2=d_out, d3=r */
  TG_OP_ATTN_BWD = 10,       /* d0=heads, d1=s, d2=d */
  TG_OP_GEMM_FWD_LORA = 11,  /* d0=T, d1=d_out, d2=d_in, d3=r */
  TG_OP_GEMM_DGRAD_LORA = 12 /* d0=T, d1=d_out, d2=d_in, d3=r */
} tg_op;

/* Forward product of a linear layer ("Where the time went"):
 *   Y[T, d_out] = X[T, d_in] . W[d_out, d_in]^T
 * Both operands have the reduction index (d_in) contiguous. */
tg_status tg_gemm_fwd(const void* X, const void* W, void* Y, int64_t T, int64_t d_out, int64_t d_in,
                      tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream);

/* Input-gradient product ("Where the time went"):
 *   dX[T, d_in] = dY[T, d_out] . W[d_out, d_in]
 * The reduction index (d_out) is contiguous in dY but strided in W. */
tg_status tg_gemm_dgrad(const void* dY, const void* W, void* dX, int64_t T, int64_t d_out,
                        int64_t d_in, tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes,
                        void* stream);

/* Forward product with a rank-r LoRA branch added inside it (section "What's
 * left": fusing the small element-wise operations):
 *   Y[T, d_out] = X[T, d_in] . W[d_out, d_in]^T + scale . H[T, r] . B[d_out, r]^T
 * X, W, H, B have type `in` (bf16 or fp16); Y has type `out` (FP32 or `in`)
 * and is overwritten with one rounding of the FP32 sum.  On the tensor-core
 * path (the alignment rules of the layer products, r <= 32) one small launch
 * stages the branch as a 64-deep K block -- scale . H as 16-bit hi + lo
 * parts beside two copies of B -- that the product appends to its own
 * reduction, so Y is written once and never read (the product runs whole
 * tiles: no K split); otherwise both products are added in an FP32 buffer on
 * the CUDA cores and rounded once.  scale must be finite; r = 0 is
 * tg_gemm_fwd.  Workspace: tg_workspace_size(TG_OP_GEMM_FWD_LORA, T, d_out,
 * d_in, r, in, out) bytes (the larger of the two paths' needs). */
tg_status tg_gemm_fwd_lora(const void* X, const void* W, const void* H, const void* B, void* Y, int64_t T,
                           int64_t d_out, int64_t d_in, int64_t r, float scale, tg_dtype in, tg_dtype out, void* ws,
                           size_t ws_bytes, void* stream);

/* Input-gradient product with the LoRA branch's part added inside it, for
 * Y = X W^T + scale . (X A^T) B^T:
 *   dX[T, d_in] = dY[T, d_out] . W[d_out, d_in] + scale . dH[T, r] . A[r, d_in]
 * with dH = dY . B in FP32 (tg_lora_grad's optional output).  dY, W, A have
 * type `in`; dX has type `out`, overwritten with one rounding.  The same two
 * paths and rules as tg_gemm_fwd_lora (scale . dH staged as hi + lo parts
 * beside two copies of A).  Workspace: tg_workspace_size(
 * TG_OP_GEMM_DGRAD_LORA, T, d_out, d_in, r, in, out). */
tg_status tg_gemm_dgrad_lora(const void* dY, const void* W, const float* dH, const void* A, void* dX, int64_t T,
                             int64_t d_out, int64_t d_in, int64_t r, float scale, tg_dtype in, tg_dtype out, void* ws,
                             size_t ws_bytes, void* stream);

/* Weight-gradient product ("Where the time went"), reduced over tokens:
 *   dW[d_out, d_in] = dY[T, d_out]^T . X[T, d_in]
 * The reduction index (T) is strided in both operands.  Long reductions are
 * split across the GPU with FP32 partials in `ws` and summed in a fixed order,
 * so results are bitwise reproducible run to run. */
tg_status tg_gemm_wgrad(const void* dY, const void* X, void* dW, int64_t T, int64_t d_out,
                        int64_t d_in, tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes,
                        void* stream);

/* Weight-gradient product for callers that cannot allocate device memory.
 * (The page has no counterpart; this is an interface for such callers.)
 * Some callers may not call cudaMalloc or lend a workspace: code inside a host
 * framework that owns all device memory through its own pool, or a process
 * held to a fixed memory budget set at start-up.  This computes exactly what
 * tg_gemm_wgrad computes, with the same kernels and arguments, minus the
 * workspace: the split-K scratch is a 32 MiB array inside the library that
 * every device loading the library holds until the process exits.
 *   - Nothing is allocated: no cudaMalloc/cudaFree, no library allocator.
 *   - A shape whose plan needs more than 32 MiB of scratch (see
 *     tg_workspace_size(TG_OP_GEMM_WGRAD, ...)) is rejected with
 *     TG_ERR_WORKSPACE_TOO_SMALL and a message in tg_last_call(); nothing runs.
 *   - All calls share the one array.  Calls that may overlap on the GPU (on
 *     different streams, or on one stream with no ordering between them)
 *     race on it and can corrupt each other's results; order them.
 *   - The first call on a device looks up the array's device address (a CUDA
 *     runtime query, done once per device with that device current); make
 *     that first call before any stream capture begins. */
tg_status tg_gemm_wgrad_noalloc(const void* dY, const void* X, void* dW, int64_t T, int64_t d_out,
                                int64_t d_in, tg_dtype in, tg_dtype out, void* stream);

/* Weight gradient added into an FP32 gradient buffer (gradient accumulation
 * over micro-batches, a "main grad" kept in FP32 beside 16-bit weights):
 *   dW[d_out, d_in] += dY[T, d_out]^T . X[T, d_in]          (dW FP32)
 * Same products, plans and kernels as tg_gemm_wgrad with out = TG_F32 (and
 * the same workspace, tg_workspace_size(TG_OP_GEMM_WGRAD, ..., TG_F32));
 * every element of dW receives exactly one FP32 addition of its FP32
 * product, so repeated calls are bitwise reproducible.  T = 0 leaves dW
 * unchanged.  16-bit dW is not offered: a rounded product added to a
 * rounded sum would round twice. */
tg_status tg_gemm_wgrad_accumulate(const void* dY, const void* X, float* dW, int64_t T, int64_t d_out,
                                   int64_t d_in, tg_dtype in, void* ws, size_t ws_bytes, void* stream);

/* Rank-r LoRA down projection ("Tuning the kernels": the rank-16 LoRA matrices):
 *   H[T, r] = X[T, d_in] . A[r, d_in]^T
 * r = 16 takes the streaming kernel (X read once); other ranks are supported
 * on the general path. */
tg_status tg_lora_down(const void* X, const void* A, void* H, int64_t T, int64_t d_in, int64_t r,
                       tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream);

/* Rank-r LoRA up projection:
 *   Y[T, d_out] = H[T, r] . B[d_out, r]^T        (overwrites Y; no alpha/r scale) */
tg_status tg_lora_up(const void* H, const void* B, void* Y, int64_t T, int64_t d_out, int64_t r,
                     tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream);

/* The LoRA branch added into the base layer's output with its scale (the
 * usual alpha / r), one rounding to Y's type:
 *   Y[T, d_out] += scale . H[T, r] . B[d_out, r]^T
 * Same kernels as tg_lora_up (r = 16: the streaming kernel, which reads Y's
 * 8-element groups, adds in FP32 and writes them back; other ranks: the
 * CUDA-core path).  scale must be finite (TG_ERR_INVALID_ARG otherwise);
 * r = 0 leaves Y unchanged.  Workspace as tg_lora_up. */
tg_status tg_lora_up_add(const void* H, const void* B, void* Y, int64_t T, int64_t d_out, int64_t r, float scale,
                         tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream);

/* Gradients of the LoRA branch Y = (X A^T) B^T given dY:
 *   dH[T, r]     = dY . B          (kept in FP32; written to dH_f32 when non-NULL;
 *                                    enters the products below as 16-bit hi + lo
 *                                    parts, lo stored times 2^11, as for the FP32
 *                                    factors of tg_lora_grad_f32w)
 *   dB[d_out, r] = dY^T . H
 *   dA[r, d_in]  = dH^T . X        (uses the FP32 dH)
 *   dX[T, d_in]  = dH . A          (uses the FP32 dH)
 * X, A, B, H, dY have type `in`; dA, dB, dX have type `out`; dH_f32 is float.
 * The sums over tokens are FP32 partials added in a fixed order, so results
 * are bitwise reproducible; `ws` may hold anything on entry (the call clears
 * the counters it keeps there). */
tg_status tg_lora_grad(const void* X, const void* A, const void* B, const void* H, const void* dY,
                       void* dA, void* dB, void* dX, float* dH_f32, int64_t T, int64_t d_in,
                       int64_t d_out, int64_t r, tg_dtype in, tg_dtype out, void* ws,
                       size_t ws_bytes, void* stream);

/* Gradients of a LoRA branch added into its base layer with a scale (the
 * usual alpha / r), Y = X W^T + scale . (X A^T) B^T, given dY: the LoRA part
 * of the layer's input gradient is added into dX, which holds the base
 * layer's dgrad (dY . W) on entry.
 *   dH[T, r]      = dY . B               (FP32, unscaled as in tg_lora_grad;
 *                                          written to dH_f32 when non-NULL)
 *   dB[d_out, r]  = scale . dY^T . H     (overwritten)
 *   dA[r, d_in]   = scale . dH^T . X     (overwritten)
 *   dX[T, d_in]  += scale . dH . A       (read and rewritten, one rounding)
 * The scale multiplies the FP32 sums before the one rounding to `out`, so
 * scale = 1 with dX = 0 gives tg_lora_grad's bits.  Same kernels, workspace
 * and arguments as tg_lora_grad; scale must be finite (TG_ERR_INVALID_ARG
 * otherwise).  r = 0 leaves dX unchanged. */
tg_status tg_lora_grad_add(const void* X, const void* A, const void* B, const void* H, const void* dY,
                           void* dA, void* dB, void* dX, float* dH_f32, int64_t T, int64_t d_in,
                           int64_t d_out, int64_t r, float scale, tg_dtype in, tg_dtype out, void* ws,
                           size_t ws_bytes, void* stream);

/* The LoRA products with FP32 factors, as an optimizer keeps the LoRA
 * weights, and 16-bit activations ("Tuning the kernels": the rank-16 LoRA
 * matrices; the FP32 LoRA weights otherwise cost a conversion of every
 * activation to FP32 or of the weights to 16 bits per call):
 *   tg_lora_down_f32w:  H[T, r]      = X[T, d_in] . A[r, d_in]^T
 *   tg_lora_up_f32w:    Y[T, d_out]  = H[T, r] . B[d_out, r]^T
 *   tg_lora_grad_f32w:  dH = dY . B (FP32, optional out), dB = dY^T . H,
 *                       dA = dH^T . X, dX = dH . A;  dA and dB FP32
 * X, H, dY have type `in` (bf16 or fp16); A, B are FP32 and are not rounded
 * to `in`: r = 16 splits each factor into 16-bit parts hi = RNE(w) and
 * lo = RNE((w - hi) 2^11) (in `ws` by one small launch, or in registers for
 * the up product, whose B must then be 16-byte aligned) and the streaming
 * kernels multiply both parts, the lo products in FP32 sums of their own that
 * are scaled back by 2^-11, so the parts stand for w to within 2^-17 |w|
 * (bf16) or 2^-22 |w| (fp16, for |w| >= 2^-14; below that, to within 2^-36
 * absolutely, so fp16 factors below about 1.5e-6 in magnitude lose the 1e-5
 * relative bound); other ranks run on the CUDA cores with the FP32 factors
 * as they are.  H, Y, dX have type `out`.  Workspace:
 * tg_workspace_size(TG_OP_LORA_*_F32W, ...); arguments and errors otherwise
 * as tg_lora_down / _up / _grad. */
tg_status tg_lora_down_f32w(const void* X, const float* A, void* H, int64_t T, int64_t d_in, int64_t r,
                            tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream);
tg_status tg_lora_up_f32w(const void* H, const float* B, void* Y, int64_t T, int64_t d_out, int64_t r,
                          tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream);
tg_status tg_lora_grad_f32w(const void* X, const float* A, const float* B, const void* H, const void* dY,
                            float* dA, float* dB, void* dX, float* dH_f32, int64_t T, int64_t d_in,
                            int64_t d_out, int64_t r, tg_dtype in, tg_dtype out, void* ws,
                            size_t ws_bytes, void* stream);

/* Fused attention forward (the fused kernel that would replace the two
 * batched products and the softmax between them):
 *   O[h] = softmax(scale . Q[h] K[h]^T) V[h]     per head h, softmax over keys
 * Q, K, V, O are [heads, s, d] contiguous; d must be 64; every pointer
 * 16-byte aligned (TG_ERR_MISALIGNED otherwise); scale finite (the usual
 * 1/sqrt(d)).  No mask.  The [s, s] scores never reach memory: each row's
 * softmax is kept online in FP32 over key blocks, and the probabilities enter
 * the second product as 16-bit hi + lo parts (to within 2^-17 of FP32), on
 * the tensor cores (tcgen05, with S, P and O in tensor memory).
 * No workspace. */
tg_status tg_attn_fwd(const void* Q, const void* K, const void* V, void* O, int64_t heads, int64_t s,
                      int64_t d, float scale, tg_dtype in, tg_dtype out, void* stream);

/* Fused attention backward: the gradients of L = <dO, O> for the forward of
 * tg_attn_fwd, O[h] = softmax(scale . Q[h] K[h]^T) V[h], given Q, K, V and dO:
 *   P = softmax(scale . Q K^T),  D_i = sum_j P_ij (dO V^T)_ij,
 *   dV = P^T dO,  dS = P * (dO V^T - D),  dQ = scale . dS K,  dK = scale . dS^T Q
 * Q, K, V, dO are [heads, s, d] of type `in` (bf16 or fp16); dQ, dK, dV are
 * [heads, s, d] of type `out` (FP32 or `in`), overwritten.  d must be 64;
 * every pointer 16-byte aligned (TG_ERR_MISALIGNED otherwise); scale finite.
 * No mask.  The [s, s] matrices never reach memory: two launches on the
 * tensor cores recompute them per 128 x 64 block (per query tile the row
 * statistics, then dQ; per key tile dK and dV); P and dS enter the
 * products as 16-bit hi + lo parts, each scaled by a power of two that is
 * taken off in FP32, so fp16 neither overflows nor loses small values.
 * Workspace: tg_workspace_size(TG_OP_ATTN_BWD, heads, s, d, 0, in, out)
 * bytes (two FP32 values per row, s rounded up to 128), 16-byte aligned.  Results are bitwise
 * reproducible run to run (no atomics). */
tg_status tg_attn_bwd(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK, void* dV,
                      int64_t heads, int64_t s, int64_t d, float scale, tg_dtype in, tg_dtype out, void* ws,
                      size_t ws_bytes, void* stream);

/* One of the batched products inside attention ("Tuning the kernels";
 * "Checking the results are right": batched attention), see tg_attn_op. */
tg_status tg_bmm_attn(tg_attn_op op, const void* A, const void* B, void* C, int64_t batch,
                      int64_t s, int64_t d, tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes,
                      void* stream);

/* Bytes of `ws` the call with these sizes needs on the current device
 * (0 when none).  Returns SIZE_MAX for invalid arguments. */
size_t tg_workspace_size(tg_op op, int64_t d0, int64_t d1, int64_t d2, int64_t d3, tg_dtype in,
                         tg_dtype out);

/* Synchronises `stream`, then reads and clears the current device's status
 * word: TG_ERR_DEVICE_TIMEOUT if any kernel's bounded wait ran out since the
 * last check, TG_ERR_CUDA if the synchronisation failed, else TG_OK. */
tg_status tg_stream_status(void* stream);

/* Static text for a status code. */
const char* tg_status_string(tg_status s);

/* Load a tile table (the analogue of tuned logic files; section "Tuning the
 * kernels").  Lines: "op dtype_in dtype_out M N K batch bn splits", where op
 * is nt|nn|tn (also accepted: fwd|dgrad|wgrad) -- the operand layout of the
 * product; attention products use the layout of theirs -- and M N K are the
 * product's own output rows, output columns and reduction length; an
 * optional tenth field m|n|auto sets the order in which output tiles are
 * visited.  Replaces any table loaded before; NULL or "" clears it.  At first
 * use the library loads $TG_TABLE if set (empty: none), else the table
 * shipped beside libtg.so (tables/gb300.txt) if present. */
tg_status tg_load_table(const char* path);

/* Library version: major * 10000 + minor * 100 + patch. */
int tg_version(void);

/* Writes a one-line description of the last dispatch decision made on the
 * calling thread (kernel path, tile, splits, whether a table entry was used)
 * into buf (NUL-terminated, truncated to len).  Returns the full length. */
size_t tg_last_call(char* buf, size_t len);

/* Host only (no device needed, nothing launched): writes into buf
 * (NUL-terminated, truncated to len) the plan the tensor-core path would use
 * for a layer product on a device with `sms` SMs -- tile width, CTA pairs /
 * deep ring / cluster split, split count or stream-K grid, tail split, tile
 * order, and whether the tile table or the cost model chose it -- in the
 * format of tg_last_call, "simt <layout>" when contiguous operands of
 * these sizes need the CUDA-core path, or "ffma <layout> splits=S" for FP32
 * operands (the CUDA-core FFMA kernel and its K split).  op is TG_OP_GEMM_FWD, _DGRAD or
 * _WGRAD; M, N, K are the product's output rows, output columns and
 * reduction length (as in the tile table).  Returns the full length, 0 for
 * invalid arguments. */
size_t tg_plan_describe(tg_op op, int64_t M, int64_t N, int64_t K, int64_t batch, tg_dtype in, tg_dtype out,
                        int sms, char* buf, size_t len);

/* Diagnostic of the bounded-wait mechanism every pipelined kernel uses: one
 * CTA waits on a barrier that nothing ever completes, gives up after
 * timeout_us microseconds and records a timeout in the status word, which
 * tg_stream_status then reports as TG_ERR_DEVICE_TIMEOUT.  The context stays
 * usable.  timeout_us must lie in [1, 10,000,000]. */
tg_status tg_wait_probe(int64_t timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TG_H */
