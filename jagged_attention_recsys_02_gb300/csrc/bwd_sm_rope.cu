// Softmax backward with the rotary-embedding backward fused into the dK
// epilogue: the launcher of the rotary instantiations (kernel in
// bwd_sm_kernel.cuh).
#include "bwd_sm_kernel.cuh"

namespace gdpa {

cudaError_t launch_bwd_softmax_rope(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& tdo,
                                    const CUtensorMap& tdq, int grid, cudaStream_t s) {
  return dispatch_sm<true>(p, tq, tk, tv, tdo, tdq, grid, s);
}

}  // namespace gdpa
