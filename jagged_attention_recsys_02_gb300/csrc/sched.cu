// Varlen tile scheduler: turns per-sample offsets into a cost-sorted list of
// (sample, head, block) work items for the persistent attention kernels.
//
// Jagged inputs break the uniform tiling of dense attention: short samples
// finish early and leave SMs idle ("GEM Training ..." JFA paragraph, and the
// GDPA paragraph on large batches breaking occupancy assumptions).  The fix
// here: estimate every block's cost as the number of inner tiles it will
// visit, counting-sort the samples by their total cost in descending order
// (longest-processing-time first) and let the persistent CTAs pull items in
// that order from an atomic ticket.  A sample's items stay contiguous
// (blocks in descending cost, heads innermost), so the CTAs working at the
// same time share that sample's key/value (forward) or query/dO (backward)
// tiles through L2 instead of refetching them from DRAM.
//
// One CTA of 1024 threads builds the list; it also validates the offsets and
// reports malformed ones through the device status word instead of trapping.
//
// Short-query samples (1 <= Lq_b <= short_q, when short_q > 0) go to a second
// list of (sample, head) items, sorted the same way by their key-tile count,
// for the kernels that stream a whole sample's keys past its few queries; the
// scheduler then also records whether every sample with queries is short.
// In the forward, samples with few keys (1 <= Lkv_b <= max_kv) and more
// queries go to a third list for the kernel that keeps a sample's keys in
// shared memory and streams its queries past them: one item per head and
// chunk of kShortKvChunk queries, sorted by the item's own cost (query tiles
// times 32-key columns), so the short last chunks of long samples come last.
#include "common.cuh"

namespace gdpa {
namespace {

constexpr int kThreads = 1024;

// mode 0 (forward): outer = queries in 256-row blocks, inner = key tiles of 128.
// mode 1 (backward): outer = keys in 128-row blocks, inner = query tiles of 64.
// The cost counts only the inner tiles inside the causal / sliding-window
// band (tiles outside it are skipped by the kernels), plus one for the
// block's fixed work.
__device__ __forceinline__ int block_cost(int mode, int causal, int window, int Lo, int Li,
                                          int blk) {
  int tb, te;
  if (mode == 0) {
    band_key_tiles(blk * kItemRows, min(Lo, (blk + 1) * kItemRows), causal, window, Li, kKvRows,
                   &tb, &te);
  } else {
    band_query_tiles(blk * kBwdKvRows, min(Lo, (blk + 1) * kBwdKvRows), causal, window, Li,
                     kBwdQRows, &tb, &te);
  }
  return te - tb + 1;
}

// Histogram bucket of a sample's total cost: exact below 1024 inner tiles,
// then 64-tile steps (coarser ordering among very long samples is enough for
// the longest-first schedule).
__device__ __forceinline__ int sample_bucket(int mode, int causal, int window, int Lo, int Li,
                                             int nblk) {
  long long total = 0;
  for (int blk = 0; blk < nblk; ++blk) total += block_cost(mode, causal, window, Lo, Li, blk);
  const long long b = total < 1024 ? total : 1024 + (total - 1024) / 64;
  return static_cast<int>(b < kCostBuckets - 1 ? b : kCostBuckets - 1);
}

// Query rows of sample b, for either mode.
__device__ __forceinline__ int query_rows(int mode, int Lo, int Li) { return mode == 0 ? Lo : Li; }

// Short-key items: cost of a chunk of `rows` queries against Li keys (at most
// 16 tiles x 8 columns of 32 keys: below kKvBuckets).
constexpr int kKvBuckets = 256;
__device__ __forceinline__ int kv_cost(int rows, int Li) {
  return ((rows + kHalfRows - 1) / kHalfRows) * ((Li + 31) / 32);
}
static_assert((kShortKvChunk / kHalfRows) * (kShortKv / 32) < kKvBuckets, "short-key cost range");

// Exclusive scan in descending bucket order: base[c] = sum of hist[c'] for
// c' > c; returns the total.  Thread t owns reversed positions 2t and 2t+1.
__device__ int scan_desc(const int* hist, int* base, int* warp_tot) {
  const int tid = threadIdx.x;
  const int c0 = kCostBuckets - 1 - 2 * tid, c1 = c0 - 1;
  const int v0 = hist[c0], v1 = hist[c1];
  int incl = v0 + v1;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += t;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - (v0 + v1);
  base[c0] = before;
  base[c1] = before + v0;
  const int total = warp_tot[kThreads / 32 - 1];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kThreads, 1)
build_worklist_kernel(const int32_t* __restrict__ outer_off, const int32_t* __restrict__ inner_off,
                      int B, int H, long long T_outer, long long T_inner, int causal, int window,
                      int mode,
                      int2* __restrict__ items, int* __restrict__ n_items,
                      int* __restrict__ ticket, int* __restrict__ status,
                      const int64_t* __restrict__ bias_off, ShortList sq, KvList kv) {
  __shared__ int hist[kCostBuckets];
  __shared__ int base[kCostBuckets];
  __shared__ int shist[kCostBuckets];
  __shared__ int sbase[kCostBuckets];
  __shared__ int khist[kKvBuckets];
  __shared__ int kbase[kKvBuckets];
  __shared__ int ktotal;
  __shared__ int warp_tot[kThreads / 32];
  __shared__ int bad;
  const int tid = threadIdx.x;
  const int block_rows = (mode == 0) ? kItemRows : kBwdKvRows;
  const bool split = sq.items != nullptr && sq.max_q > 0;
  const bool kv_split = mode == 0 && kv.items != nullptr && kv.max_kv > 0;
  // a short-key sample (forward): more queries than the short-query list
  // takes, and 1..max_kv keys
  auto short_kv = [&](int Lo, int Li) {
    return kv_split && Li >= 1 && Li <= kv.max_kv && Lo >= 1 && !(split && Lo <= sq.max_q);
  };
  for (int i = tid; i < kCostBuckets; i += kThreads) hist[i] = shist[i] = 0;
  for (int i = tid; i < kKvBuckets; i += kThreads) khist[i] = 0;
  if (tid == 0) {
    bad = (outer_off[0] != 0 || inner_off[0] != 0 || outer_off[B] != T_outer ||
           inner_off[B] != T_inner || (bias_off != nullptr && bias_off[0] != 0)) ? 1 : 0;
  }
  __syncthreads();
  for (int b = tid; b < B; b += kThreads) {
    const int Lo = outer_off[b + 1] - outer_off[b];
    const int Li = inner_off[b + 1] - inner_off[b];
    if (Lo < 0 || Li < 0 || ((causal || window > 0) && Lo != Li) ||
        (bias_off != nullptr &&
         bias_off[b + 1] - bias_off[b] != static_cast<int64_t>(H) * Lo * Li)) {
      bad = 1;
      continue;
    }
    const int nblk = (Lo + block_rows - 1) / block_rows;
    const int lq = query_rows(mode, Lo, Li);
    if (split && lq >= 1 && lq <= sq.max_q) {
      // one item per head; cost: the sample's key tiles
      const int lk = mode == 0 ? Li : Lo;
      const int c = 1 + (lk + kKvRows - 1) / kKvRows;
      atomicAdd(&shist[c < 1024 ? c : min(kCostBuckets - 1, 1024 + (c - 1024) / 64)], 1);
    } else if (short_kv(Lo, Li)) {
      const int nch = (Lo + kShortKvChunk - 1) / kShortKvChunk;
      if (nch > 1) atomicAdd(&khist[kv_cost(kShortKvChunk, Li)], nch - 1);
      atomicAdd(&khist[kv_cost(Lo - (nch - 1) * kShortKvChunk, Li)], 1);
    } else if (nblk > 0) {
      atomicAdd(&hist[sample_bucket(mode, causal, window, Lo, Li, nblk)], nblk);
    }
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      *n_items = 0;
      *ticket = 0;
      if (split) {
        *sq.n_items = 0;
        *sq.ticket = 0;
        *sq.all_short = 0;
      }
      if (kv_split) {
        *kv.n_items = 0;
        *kv.ticket = 0;
      }
      set_status(status, GDPA_ERR_BAD_OFFSETS);
    }
    return;
  }
  const int total = scan_desc(hist, base, warp_tot);
  const int stotal = split ? scan_desc(shist, sbase, warp_tot) : 0;
  if (kv_split && tid == 0) {  // descending exclusive scan of the short-key costs
    int acc = 0;
    for (int c = kKvBuckets - 1; c >= 0; --c) {
      kbase[c] = acc;
      acc += khist[c];
    }
    ktotal = acc;
  }
  __syncthreads();
  for (int b = tid; b < B; b += kThreads) {
    const int Lo = outer_off[b + 1] - outer_off[b];
    const int Li = inner_off[b + 1] - inner_off[b];
    const int nblk = (Lo + block_rows - 1) / block_rows;
    const int lq = query_rows(mode, Lo, Li);
    if (split && lq >= 1 && lq <= sq.max_q) {
      const int lk = mode == 0 ? Li : Lo;
      const int c = 1 + (lk + kKvRows - 1) / kKvRows;
      const int pos = atomicAdd(&sbase[c < 1024 ? c : min(kCostBuckets - 1, 1024 + (c - 1024) / 64)], 1);
      for (int h = 0; h < H; ++h)
        sq.items[static_cast<long long>(pos) * H + h] = make_int2(b, h);
      continue;
    }
    if (short_kv(Lo, Li)) {
      const int nch = (Lo + kShortKvChunk - 1) / kShortKvChunk;
      if (nch > 1) {
        const int pos = atomicAdd(&kbase[kv_cost(kShortKvChunk, Li)], nch - 1);
        for (int ch = 0; ch < nch - 1; ++ch)
          for (int h = 0; h < H; ++h)
            kv.items[static_cast<long long>(pos + ch) * H + h] = make_int2(b, (ch << 8) | h);
      }
      const int pos = atomicAdd(&kbase[kv_cost(Lo - (nch - 1) * kShortKvChunk, Li)], 1);
      for (int h = 0; h < H; ++h)
        kv.items[static_cast<long long>(pos) * H + h] = make_int2(b, ((nch - 1) << 8) | h);
      continue;
    }
    if (nblk == 0) continue;
    const int pos = atomicAdd(&base[sample_bucket(mode, causal, window, Lo, Li, nblk)], nblk);
    // Blocks in descending cost: under the causal mask the forward's last
    // query blocks and the backward's first key blocks visit the most tiles
    // (a sliding window makes the costs nearly flat; the order stays).
    for (int r = 0; r < nblk; ++r) {
      const int blk = (causal && mode == 0) ? nblk - 1 - r : r;
      for (int h = 0; h < H; ++h)
        items[static_cast<long long>(pos + r) * H + h] = make_int2(b, (blk << 8) | h);
    }
  }
  if (tid == 0) {
    *n_items = total * H;
    *ticket = 0;
    if (split) {
      *sq.n_items = stotal * H;
      *sq.ticket = 0;
      *sq.all_short = (total == 0 && stotal > 0) ? 1 : 0;
    }
    if (kv_split) {
      *kv.n_items = ktotal * H;
      *kv.ticket = 0;
    }
  }
}

}  // namespace

cudaError_t launch_build_worklist(const int32_t* outer_off, const int32_t* inner_off, int B, int H,
                                  int64_t T_outer, int64_t T_inner, int causal, int window,
                                  int mode, int2* items, int* n_items, int* ticket, int* status,
                                  cudaStream_t stream, const int64_t* bias_off,
                                  const ShortList& sq, const KvList& kv) {
  build_worklist_kernel<<<1, kThreads, 0, stream>>>(outer_off, inner_off, B, H, T_outer, T_inner,
                                                    causal, window, mode, items, n_items, ticket,
                                                    status, bias_off, sq, kv);
  return cudaGetLastError();
}

}  // namespace gdpa
