// Block-aligned attention, sm_103a.
//
// "GEM Training ..." SWA paragraph, its block-aligned part: with fixed
// 64-token blocks each query block attends only to its own key/value block,
// so attention becomes independent 64 x 64 problems.  That removes the
// multi-tile iteration and partial-window masking of sliding windows, and a
// dedicated kernel drops the FlashAttention overheads: no online softmax
// correction (a row's keys all sit in one tile, so the softmax is exact in
// one pass), no logsumexp written to HBM (the backward recomputes the row's
// softmax from its own tile) and no separate D = rowsum(dO * O) pass (the
// backward forms D from P and dP inside the tile).
//
// Blocks start at each sample's first token; a sample's last block may be
// shorter.  Self-attention only (one offsets array).  The work unit is a
// tile of two consecutive blocks in global row order (they may belong to
// two samples): its rows are contiguous, at most 128, and every row's keys
// lie inside the tile, so one 128 x 128 score MMA covers both blocks and the
// off-block quadrants are masked.  The two blocks of a tile waste half of
// the MMA work, but these problems are bound by HBM traffic (64 x 64 x d
// per block: about 32 FLOP per byte at d = 128), far below the tensor ridge.
//
// block_list_kernel turns the offsets into the tile list; the kernels walk
// the (tile, head) items with a static stride over a persistent grid (every
// item costs the same).
//
// This header holds what the forward (block_fwd_kernel.cuh) and backward
// (block_bwd_kernel.cuh) kernels share: the tile descriptor, the row's key
// range, the activation, the bias window and the dense bias's row address.
#pragma once
#include <type_traits>

#include "common.cuh"

namespace gdpa {
namespace {

using namespace ptx;

constexpr int kBlk = kBlockRows;       // 64 tokens per block
constexpr int kTileRows = 2 * kBlk;    // two blocks per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kListThreads = 1024;

struct TileInfo {
  int row0;       // first global row of the tile
  int len_a;      // rows of the first block
  int rows;       // rows of both blocks
  int pos_a;      // position of the first row in its sample
  bool cont;      // the second block belongs to the first one's sample
  // position of tile row r in its sample
  __device__ __forceinline__ int pos(int r) const {
    return (r < len_a || cont) ? pos_a + r : r - len_a;
  }
};

__device__ __forceinline__ TileInfo load_tile(const int4* tiles, int t) {
  const int4 v = tiles[t];
  return TileInfo{v.x, v.y, v.y + (v.z & 0xFFFF), v.w, (v.z >> 16) != 0};
}

// Keys [*c_lo, *c_hi) of tile row r (tile-local columns): the row's own block,
// cut at the diagonal when causal; empty for rows past the tile.
__device__ __forceinline__ void row_keys(const TileInfo& ti, int r, int causal, int* c_lo,
                                         int* c_hi) {
  int lo = r < ti.len_a ? 0 : ti.len_a;
  int hi = r < ti.len_a ? ti.len_a : ti.rows;
  if (r >= ti.rows) hi = lo;
  if (causal) hi = min(hi, r + 1);
  *c_lo = lo;
  *c_hi = hi;
}

// Dense bias of tile row r for one head: the value for (row r, tile column c)
// is p.bias_dense[base + c] for the keys the row sees (its own block, so its
// own sample); -1 for rows past the tile.  The row's sample is the last b
// with offsets[b] <= its global row (empty samples are skipped by that).
__device__ __forceinline__ long long dense_row_base(const BlockParams& p, const TileInfo& ti,
                                                    int r, int head) {
  if (r >= ti.rows) return -1;
  const int gr = ti.row0 + r;
  int lo = 0, hi = p.B;  // offsets[lo] <= gr < offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.offsets + mid) <= gr) lo = mid; else hi = mid;
  }
  const int s0 = __ldg(p.offsets + lo);
  const long long L = __ldg(p.offsets + lo + 1) - s0;
  return __ldg(p.bias_off + lo) + (head * L + (gr - s0)) * L + (ti.row0 - s0);
}

__device__ __forceinline__ float act_fwd(int act, float x) {
  if (act == GDPA_ACT_SILU) {
    const float h = 0.5f * x;
    return fmaf(h, tanh_approx(h), h);
  }
  if (act == GDPA_ACT_GELU_TANH) {
    const float k0 = 0.7978845608028654f, k1 = 0.7978845608028654f * 0.044715f;
    const float u = x * fmaf(k1, x * x, k0);
    const float h = 0.5f * x;
    return fmaf(h, tanh_approx(u), h);
  }
  if (act == GDPA_ACT_GELU_ERF) return 0.5f * x * (1.0f + erff(x * 0.7071067811865476f));
  return x;
}

// Bias window of one head: entry e holds bias(i - j = e - 127), times log2 e
// for softmax (exponents are in log2 units), for the 255 differences a
// 128-row tile can hold.
__device__ __forceinline__ void stage_bias(float* win, const float* table, int head, int max_rel,
                                           float mul, int lane) {
  const int width = 2 * max_rel - 1;
  const float* row = table + static_cast<long long>(head) * width;
  for (int e = lane; e < 2 * kTileRows - 1; e += 32)
    win[e] = __ldg(row + min(max(e - (kTileRows - 1) + max_rel - 1, 0), width - 1)) * mul;
}

}  // namespace
}  // namespace gdpa
