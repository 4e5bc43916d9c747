// Block-aligned attention forward with a dense jagged bias (kernel in
// block_fwd_kernel.cuh).
#include "block_fwd_kernel.cuh"

namespace gdpa {

cudaError_t launch_block_fwd_dense(const BlockParams& p, int act, const CUtensorMap& tq,
                                   const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                                   cudaStream_t s) {
  return p.d == 64 ? launch_fwd_d<64, true>(p, act, tq, tk, tv, grid, s)
                   : launch_fwd_d<128, true>(p, act, tq, tk, tv, grid, s);
}

}  // namespace gdpa
