// smem_attr.h -- raising a kernel's dynamic shared-memory limit, once per
// device and kernel.
#pragma once
#include <cuda_runtime.h>

namespace tg {

// Raises the dynamic shared-memory limit of `kern` on the current device to
// `bytes` the first time this (device, kernel) pair asks for that much, so
// that later launches (including launches under stream capture) make no such
// call.  Safe to call from several host threads.
cudaError_t raise_smem_limit(const void* kern, int bytes);

}  // namespace tg
