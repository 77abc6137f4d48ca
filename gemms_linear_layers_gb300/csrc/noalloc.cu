// noalloc.cu -- tg_gemm_wgrad_noalloc: the weight-gradient product for
// callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc or hand out a workspace: code that runs
// inside a host framework which owns every byte of device memory through its
// own pool (a cudaMalloc there would fragment that pool and synchronise the
// device behind the framework's back), or a process started with a fixed
// memory budget that forbids allocation after start-up.  For them this entry
// point runs the same kernels as tg_gemm_wgrad, with the split-K scratch in a
// fixed array that is part of the library image instead of a caller buffer.
#include <cuda_runtime.h>

#include <mutex>

#include "tg.h"
#include "tg_internal.h"

namespace tg {

// The scratch: 32 MiB, 256-byte aligned, one copy on every device that loads
// this library, held until the process exits.  Every call shares it.
constexpr size_t kNoallocScratchBytes = static_cast<size_t>(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// The host-side name of g_noalloc_scratch is not a device address: its
// device address is looked up once per device, with that device current.
static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[128];

static tg_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return TG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return TG_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return TG_OK;
}

}  // namespace tg

extern "C" tg_status tg_gemm_wgrad_noalloc(const void* dY, const void* X, void* dW, int64_t T, int64_t d_out,
                                           int64_t d_in, tg_dtype in, tg_dtype out, void* stream) {
  // the same argument checks as tg_gemm_wgrad, before any device work
  if (T < 0 || d_out < 0 || d_in < 0) return TG_ERR_INVALID_ARG;
  const size_t need = tg_workspace_size(TG_OP_GEMM_WGRAD, T, d_out, d_in, 0, in, out);
  if (need == SIZE_MAX) return tg_gemm_wgrad(dY, X, dW, T, d_out, d_in, in, out, nullptr, 0, stream);
  if (need > tg::kNoallocScratchBytes) {
    tg::note_last_call("wgrad_noalloc: this shape needs " + std::to_string(need) +
                       " bytes of split-K scratch, more than the 33554432-byte static array");
    return TG_ERR_WORKSPACE_TOO_SMALL;
  }
  void* scratch = nullptr;
  if (need > 0) {
    const tg_status s = tg::noalloc_scratch(&scratch);
    if (s != TG_OK) return s;
  }
  return tg_gemm_wgrad(dY, X, dW, T, d_out, d_in, in, out, scratch, need > 0 ? tg::kNoallocScratchBytes : 0,
                       stream);
}
