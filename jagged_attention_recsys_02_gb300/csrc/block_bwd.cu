// Block-aligned attention backward: the launcher (kernel in
// block_bwd_kernel.cuh; the bias-table gradient's instantiations compile in
// block_bwd_db.cu, in parallel with these).
#include "block_bwd_kernel.cuh"

namespace gdpa {

cudaError_t launch_block_bwd(const BlockParams& p, int act, const CUtensorMap* maps, int grid,
                             cudaStream_t s) {
  if (p.dbias != nullptr) return launch_block_bwd_dbias(p, act, maps, grid, s);
  return p.d == 64 ? launch_bwd_d<64, false>(p, act, maps, grid, s)
                   : launch_bwd_d<128, false>(p, act, maps, grid, s);
}

}  // namespace gdpa
