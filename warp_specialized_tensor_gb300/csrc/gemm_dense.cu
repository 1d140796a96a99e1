// gemm_dense.cu -- dense / strided-batched instantiations of the
// warp-specialized GEMM, and the entry used by the C ABI.
#include "gemm_ws_launch.cuh"

namespace wst {

int run_gemm_grouped(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t stream);

int run_gemm(const GemmProblem& pr, cudaStream_t stream) {
  DeviceInfo dev;
  int st = current_device_info(&dev);
  if (st) return st;
  return pr.grouped ? run_gemm_grouped(pr, dev, stream) : (dense_cta_group(pr.M) == 2 ? dispatch<false, 2>(pr, dev, stream)
                                              : dispatch<false, 1>(pr, dev, stream));
}

}  // namespace wst
