// gemm_tc_nn.cu -- instantiation of the tensor-core GEMM family with
// A K-major, B MN-major.
#include "gemm_tc_launch.cuh"

namespace tg {
cudaError_t tc_gemm_launch_nn(const TcGemm& g) { return tc_launch_layout<false, true>(g); }
}  // namespace tg
