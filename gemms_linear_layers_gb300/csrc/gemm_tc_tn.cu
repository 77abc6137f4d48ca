// gemm_tc_tn.cu -- instantiation of the tensor-core GEMM family with
// A MN-major, B MN-major.
#include "gemm_tc_launch.cuh"

namespace tg {
cudaError_t tc_gemm_launch_tn(const TcGemm& g) { return tc_launch_layout<true, true>(g); }
}  // namespace tg
