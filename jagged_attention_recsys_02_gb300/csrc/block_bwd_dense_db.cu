// Block-aligned attention backward with a dense jagged bias and its gradient
// (kernel in block_bwd_kernel.cuh).
#include "block_bwd_kernel.cuh"

namespace gdpa {

cudaError_t launch_block_bwd_dense_db(const BlockParams& p, int act, const CUtensorMap* maps,
                                      int grid, cudaStream_t s) {
  return p.d == 64 ? launch_bwd_d<64, true, true>(p, act, maps, grid, s)
                   : launch_bwd_d<128, true, true>(p, act, maps, grid, s);
}

}  // namespace gdpa
