// gemm_grouped.cu -- grouped (mixture-of-experts) instantiations of the
// warp-specialized GEMM.
#include "gemm_ws_launch.cuh"

namespace wst {

int run_gemm_grouped(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t stream) {
  return dispatch<true, 1>(pr, dev, stream);
}

}  // namespace wst
