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
// out-of-range elements of a store are skipped.  swizzle_bytes: 0 (none),
// 32, 64 or 128 (the box's inner extent in bytes must not exceed it).
bool encode_tmap_3d(void* tmap_out, const void* base, int elem_kind, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                    uint32_t box1, int swizzle_bytes) {
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
  CUtensorMapSwizzle sw;
  switch (swizzle_bytes) {
    case 0: sw = CU_TENSOR_MAP_SWIZZLE_NONE; break;
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    default: return false;
  }
  if (swizzle_bytes != 0 && box0 * static_cast<uint64_t>(elem_bytes(elem_kind)) > static_cast<uint64_t>(swizzle_bytes))
    return false;
  CUresult r = fn(static_cast<CUtensorMap*>(tmap_out), dt, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiled map of rank 2..5 with explicit byte strides of dimensions 1.. (any
// order: a view may walk memory out of order, e.g. [chunk][row][column] over
// a row-major matrix).  Same fill, promotion and swizzle rules as above.
bool encode_tmap_nd(void* tmap_out, const void* base, int elem_kind, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || rank < 2 || rank > 5) return false;
  CUtensorMapDataType dt = elem_kind == EK_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                           : elem_kind == EK_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    if (dims[i] == 0 || box[i] == 0 || box[i] > 256) return false;
    d[i] = dims[i];
    bx[i] = box[i];
    estr[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) {
    if (strides_bytes[i] % 16) return false;
    st[i] = strides_bytes[i];
  }
  CUtensorMapSwizzle sw;
  switch (swizzle_bytes) {
    case 0: sw = CU_TENSOR_MAP_SWIZZLE_NONE; break;
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    default: return false;
  }
  if (swizzle_bytes != 0 && box[0] * static_cast<uint64_t>(elem_bytes(elem_kind)) > static_cast<uint64_t>(swizzle_bytes))
    return false;
  CUresult r = fn(static_cast<CUtensorMap*>(tmap_out), dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d,
                  st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace tg
