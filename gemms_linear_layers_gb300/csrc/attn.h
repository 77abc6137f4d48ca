// attn.h -- the fused attention kernels' launchers (attn_tc.cu forward,
// attn_bwd_tc.cu backward), kept out of tg_internal.h so that the GEMM units
// do not see them.
#pragma once
#include "tg_internal.h"

namespace tg {

// O[h][s][d] = softmax(scale * Q[h] K[h]^T) V[h] per head h: Q, K, V 16-bit
// (in_kind), O of out_kind; d must be 64; every pointer 16-byte aligned.
// tcgen05 MMAs with S, P and O in tensor memory, operands by TMA; every wait
// bounded by timeout_ns (a timeout is recorded in *status).
cudaError_t attn_fwd_tc_launch(const void* Q, const void* K, const void* V, void* O, int64_t heads, int64_t s,
                               int64_t d, float scale, int in_kind, int out_kind, unsigned int* status,
                               unsigned long long timeout_ns, cudaStream_t stream);

// dQ, dK, dV of the forward above given dO; ws holds attn_bwd_ws_bytes(heads,
// s) bytes of row statistics (16-byte aligned).
size_t attn_bwd_ws_bytes(int64_t heads, int64_t s);
cudaError_t attn_bwd_tc_launch(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK,
                               void* dV, int64_t heads, int64_t s, int64_t d, float scale, int in_kind,
                               int out_kind, void* ws, unsigned int* status, unsigned long long timeout_ns,
                               cudaStream_t stream);

}  // namespace tg
