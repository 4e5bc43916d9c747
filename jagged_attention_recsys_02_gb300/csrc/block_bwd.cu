// Block-aligned attention backward: the launcher (kernel in
// block_bwd_kernel.cuh; the instantiations with a bias gradient or a dense
// bias compile in block_bwd_db.cu, block_bwd_dense.cu and
// block_bwd_dense_db.cu, in parallel with these).
#include "block_bwd_kernel.cuh"

namespace gdpa {

cudaError_t launch_block_bwd(const BlockParams& p, int act, const CUtensorMap* maps, int grid,
                             cudaStream_t s) {
  if (p.bias_dense != nullptr)
    return p.dbias != nullptr ? launch_block_bwd_dense_db(p, act, maps, grid, s)
                              : launch_block_bwd_dense(p, act, maps, grid, s);
  if (p.dbias != nullptr) return launch_block_bwd_dbias(p, act, maps, grid, s);
  return p.d == 64 ? launch_bwd_d<64, false, false>(p, act, maps, grid, s)
                   : launch_bwd_d<128, false, false>(p, act, maps, grid, s);
}

}  // namespace gdpa
