// MXFP8 backward of jagged softmax attention with a dense jagged bias (kernel
// in bwd_mx_kernel.cuh).
#include "bwd_mx_kernel.cuh"

namespace gdpa {

cudaError_t launch_bwd_mx_dense(const BwdParams& p, const BwdMxOperands& mx,
                                const CUtensorMap* maps, int grid, cudaStream_t s) {
  if (p.d != kD) return cudaErrorInvalidValue;
  return p.window > 0 ? launch_mx_band<true, true>(p, mx, maps, grid, s)
                      : launch_mx_band<false, true>(p, mx, maps, grid, s);
}

}  // namespace gdpa
