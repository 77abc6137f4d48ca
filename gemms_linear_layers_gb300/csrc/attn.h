// attn.h -- the fused attention forward kernel's launcher (attn_fused.cu),
// kept out of tg_internal.h so that the GEMM units do not see it.
#pragma once
#include "tg_internal.h"

namespace tg {

// O[h][s][d] = softmax(scale * Q[h] K[h]^T) V[h] per head h; Q, K, V 16-bit
// (in_kind), O of out_kind; d must be 64; every pointer 16-byte aligned.
cudaError_t attn_fwd_launch(const void* Q, const void* K, const void* V, void* O, int64_t heads, int64_t s, int64_t d,
                            float scale, int in_kind, int out_kind, cudaStream_t stream);

}  // namespace tg
