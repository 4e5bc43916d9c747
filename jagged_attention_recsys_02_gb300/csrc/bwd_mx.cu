// MXFP8 backward of jagged softmax attention: the launcher (kernel in
// bwd_mx_kernel.cuh; the dense-bias instantiations compile in
// bwd_mx_dense.cu, in parallel with these).
#include "bwd_mx_kernel.cuh"

namespace gdpa {

cudaError_t launch_bwd_mx(const BwdParams& p, const BwdMxOperands& mx, const CUtensorMap* maps,
                          int grid, cudaStream_t s) {
  if (p.d != kD) return cudaErrorInvalidValue;
  if (p.bias_dense != nullptr) return launch_bwd_mx_dense(p, mx, maps, grid, s);
  return p.window > 0 ? launch_mx_band<true, false>(p, mx, maps, grid, s)
                      : launch_mx_band<false, false>(p, mx, maps, grid, s);
}

}  // namespace gdpa
