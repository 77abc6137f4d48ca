// tmap.cpp -- TMA tensor-map encoding through the driver entry point, so the
// library needs no link-time dependency on libcuda.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tg_internal.h"

namespace tg {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D tiled map: dims {d0 (contiguous), d1, d2}, byte strides of d1 and d2,
// box {box0, box1, 1}; out-of-range elements of a load read as zero and
// out-of-range elements of a store are skipped.
bool encode_tmap_3d(void* tmap_out, const void* base, int elem_kind, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                    uint32_t box1, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  CUtensorMapDataType dt = elem_kind == EK_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                           : elem_kind == EK_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (d0 == 0 || d1 == 0 || d2 == 0) return false;
  // a batch of one still needs a legal (16-byte multiple, non-zero) stride
  if (d2 == 1 && stride2_bytes < stride1_bytes * d1) stride2_bytes = stride1_bytes * d1;
  if (stride1_bytes % 16 || stride2_bytes % 16) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(static_cast<CUtensorMap*>(tmap_out), dt, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace tg
