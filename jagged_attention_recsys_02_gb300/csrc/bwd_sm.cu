// Softmax backward: the launcher without the rotary backward (the kernel and
// its instantiation dispatch are in bwd_sm_kernel.cuh; the rotary
// instantiations compile in bwd_sm_rope.cu, in parallel with these).
#include "bwd_sm_kernel.cuh"

namespace gdpa {

cudaError_t launch_bwd_softmax_main(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& tdo,
                                    const CUtensorMap& tdq, int grid, cudaStream_t s) {
  return p.rope_base > 0.0f ? launch_bwd_softmax_rope(p, tq, tk, tv, tdo, tdq, grid, s)
                            : dispatch_sm<false>(p, tq, tk, tv, tdo, tdq, grid, s);
}

}  // namespace gdpa
