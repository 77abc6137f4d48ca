// smem_attr.cpp -- see smem_attr.h.
#include "smem_attr.h"

#include <map>
#include <mutex>
#include <utility>

namespace tg {

cudaError_t raise_smem_limit(const void* kern, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> done;  // the limit set per (device, kernel)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  auto it = done.find({dev, kern});
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[{dev, kern}] = bytes;
  return e;
}

}  // namespace tg
