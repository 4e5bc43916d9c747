// Block-aligned attention: the tile list and the forward's launcher (kernel in
// block_fwd_kernel.cuh; the dense-bias instantiations compile in
// block_fwd_dense.cu, in parallel with these).
#include "block_fwd_kernel.cuh"

namespace gdpa {
namespace {

using namespace ptx;

// ---------------------------------------------------------------- tile list
// tiles[t] = {first row, rows of block 2t, rows of block 2t+1 (0 if none) | 1 << 16 if
// that block continues the first one's sample, position of the first row in its sample}.
__global__ void __launch_bounds__(kListThreads, 1)
block_list_kernel(const int32_t* __restrict__ offs, int B, long long T, int4* __restrict__ tiles,
                  int* __restrict__ n_tiles, int* __restrict__ status,
                  const int64_t* __restrict__ bias_off, int H) {
  __shared__ int warp_sum[kListThreads / 32];
  __shared__ int carry;
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry = 0;
    bad = (offs[0] != 0 || offs[B] != T || (bias_off != nullptr && bias_off[0] != 0)) ? 1 : 0;
  }
  __syncthreads();
  // a dense bias must hold H * L_b * L_b values per sample, in sample order
  for (int b = tid; b < B; b += kListThreads) {
    const long long L = static_cast<long long>(offs[b + 1]) - offs[b];
    if (L < 0 || (bias_off != nullptr && bias_off[b + 1] - bias_off[b] != H * L * L)) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      *n_tiles = 0;
      set_status(status, GDPA_ERR_BAD_OFFSETS);
    }
    return;
  }
  // Chunks of 1024 samples: block counts, inclusive scan, scatter.
  for (int base = 0; base < B; base += kListThreads) {
    const int b = base + tid;
    const int L = b < B ? offs[b + 1] - offs[b] : 0;
    const int nb = (L + kBlk - 1) / kBlk;
    int incl = nb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sum[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += v;
      }
      warp_sum[lane] = w;
    }
    __syncthreads();
    const int first = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + incl - nb;  // global block index
    for (int r = 0; r < nb; ++r) {
      const int g = first + r;
      const int len = min(kBlk, L - kBlk * r);
      int* t = reinterpret_cast<int*>(tiles + (g >> 1));
      if ((g & 1) == 0) {
        t[0] = offs[b] + kBlk * r;
        t[1] = len;
        t[3] = kBlk * r;
      } else {
        t[2] = len | (r > 0 ? 1 << 16 : 0);  // block r > 0 follows block r - 1 of its sample
      }
    }
    __syncthreads();
    if (tid == 0) carry += warp_sum[31];
    __syncthreads();
  }
  if (tid == 0) {
    const int total = carry;
    if (total & 1) reinterpret_cast<int*>(tiles + (total >> 1))[2] = 0;
    *n_tiles = (total + 1) >> 1;
  }
}

}  // namespace

cudaError_t launch_block_list(const int32_t* offsets, int B, int64_t T, int4* tiles, int* n_tiles,
                              int* status, cudaStream_t s, const int64_t* bias_off, int H) {
  block_list_kernel<<<1, kListThreads, 0, s>>>(offsets, B, T, tiles, n_tiles, status, bias_off, H);
  return cudaGetLastError();
}

cudaError_t launch_block_fwd(const BlockParams& p, int act, const CUtensorMap& tq,
                             const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                             cudaStream_t s) {
  if (p.bias_dense != nullptr) return launch_block_fwd_dense(p, act, tq, tk, tv, grid, s);
  return p.d == 64 ? launch_fwd_d<64, false>(p, act, tq, tk, tv, grid, s)
                   : launch_fwd_d<128, false>(p, act, tq, tk, tv, grid, s);
}

}  // namespace gdpa
