// gemm_tc_nt.cu -- instantiation of the tensor-core GEMM family with
// A K-major, B K-major.
#include "gemm_tc_launch.cuh"

namespace tg {
cudaError_t tc_gemm_launch_nt(const TcGemm& g) { return tc_launch_layout<false, false>(g); }
}  // namespace tg
