// Shared definitions of the jagged attention kernels (host + device).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdpa.h"
#include "ptx.cuh"

namespace gdpa {

// Tile shapes.  A forward work item covers 256 query rows of one (sample,
// head), split in two 128-row halves (the 128 TMEM lanes of one MMA tile);
// key/value tiles have 128 rows.
constexpr int kHalfRows = 128;
constexpr int kItemRows = 256;
constexpr int kKvRows = 128;
// Backward: a work item is one 128-row key/value tile; queries stream past
// it in 64-row tiles.
constexpr int kBwdKvRows = 128;
constexpr int kBwdQRows = 64;
constexpr int kBwdSmQRows = 128;  // query tile of the softmax backward
constexpr int kBwdSmDqRows = 16;  // query rows per dQ reduce box of the softmax backward
constexpr int kBwdMxQRows = 64;   // query tile of the MXFP8 backward

constexpr int kCostBuckets = 2048;

// Block-aligned attention: tokens per block (fixed; blocks start at each
// sample's first token).
constexpr int kBlockRows = 64;

// Work item: x = sample b (or -1 = end of list), y = (block << 8) | head.
__host__ __device__ inline int item_head(int2 it) { return it.y & 0xFF; }
__host__ __device__ inline int item_block(int2 it) { return it.y >> 8; }

// Sliding-window band ("GEM Training ..." SWA paragraph: each token attends
// only to nearby events).  Local key j is visible from local query i when
// j <= i (causal) and |i - j| < window (window > 0); window 0 is no window.
// Both bounds are monotone in i (and in j), so the keys visible from a run
// of consecutive rows, and the queries that see a run of consecutive keys,
// are contiguous ranges.
__host__ __device__ __forceinline__ int band_key_begin(int i, int window) {
  return window > 0 ? max(0, i - window + 1) : 0;
}
__host__ __device__ __forceinline__ int band_key_end(int i, int causal, int window, int Lkv) {
  if (causal) return min(Lkv, i + 1);
  return window > 0 ? min(Lkv, i + window) : Lkv;
}
__host__ __device__ __forceinline__ int band_query_begin(int j, int causal, int window) {
  if (causal) return j;
  return window > 0 ? max(0, j - window + 1) : 0;
}
__host__ __device__ __forceinline__ int band_query_end(int j, int window, int Lq) {
  return window > 0 ? min(Lq, j + window) : Lq;
}
// Tiles of `tile` keys visited by the query rows [r_begin, r_end) (r_begin <
// r_end): [*t_begin, *t_end), empty when no key is visible.
__host__ __device__ __forceinline__ void band_key_tiles(int r_begin, int r_end, int causal,
                                                        int window, int Lkv, int tile,
                                                        int* t_begin, int* t_end) {
  const int kb = band_key_begin(r_begin, window);
  const int ke = band_key_end(r_end - 1, causal, window, Lkv);
  if (ke <= kb) {
    *t_begin = *t_end = 0;
    return;
  }
  *t_begin = kb / tile;
  *t_end = (ke + tile - 1) / tile;
}
// Tiles of `tile` queries that see some key of [c_begin, c_end) (c_begin < c_end).
__host__ __device__ __forceinline__ void band_query_tiles(int c_begin, int c_end, int causal,
                                                          int window, int Lq, int tile,
                                                          int* t_begin, int* t_end) {
  const int qb = band_query_begin(c_begin, causal, window);
  const int qe = band_query_end(c_end - 1, window, Lq);
  if (qe <= qb) {
    *t_begin = *t_end = 0;
    return;
  }
  *t_begin = qb / tile;
  *t_end = (qe + tile - 1) / tile;
}

// GDPA activation and its derivative: SiLU x sigmoid(x) and GELU-tanh
// 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) through tanh.approx (for
// SiLU via sigmoid(x) = 0.5 + 0.5 tanh(x / 2)), GELU-erf x Phi(x) through
// erff; identity otherwise.
template <int ACT>
__device__ __forceinline__ void act_and_grad(float x, float& a, float& g) {
  if (ACT == GDPA_ACT_SILU) {
    const float h = 0.5f * x;
    const float t = ptx::tanh_approx(h);
    const float sg = fmaf(0.5f, t, 0.5f);           // sigmoid(x)
    a = x * sg;
    g = sg * fmaf(x, 1.0f - sg, 1.0f);               // sigmoid * (1 + x (1 - sigmoid))
  } else if (ACT == GDPA_ACT_GELU_TANH) {
    const float k0 = 0.7978845608028654f, k1 = 0.7978845608028654f * 0.044715f;
    const float x2 = x * x;
    const float t = ptx::tanh_approx(x * fmaf(k1, x2, k0));
    const float h = 0.5f * x;
    a = fmaf(h, t, h);
    // 0.5 (1 + t) + 0.5 x (1 - t^2) sqrt(2/pi) (1 + 3 * 0.044715 x^2)
    g = fmaf(0.5f, t, 0.5f) + h * (1.0f - t * t) * fmaf(3.0f * k1, x2, k0);
  } else if (ACT == GDPA_ACT_GELU_ERF) {
    // Phi(x) = 0.5 (1 + erf(x / sqrt 2)); act = x Phi(x), act' = Phi(x) + x phi(x)
    const float cdf = fmaf(0.5f, erff(x * 0.7071067811865476f), 0.5f);
    a = x * cdf;
    g = fmaf(x * 0.3989422804014327f, expf(-0.5f * x * x), cdf);
  } else {
    a = x;
    g = 1.0f;
  }
}

// Rotary-embedding backward of one row ("GEM Training ..." SWA / block
// paragraph: the RoPE backward fused into the attention epilogue, gradients
// kept in fp32).  The row's D fp32 gradient values sit in TMEM columns
// taddr..taddr+D; scaled by `mul`, each channel pair (c, c + D/2) is rotated
// by -pos * theta_c with theta_c = base^(-2c/D) = exp2(c * rope_k), then
// stored as bf16 to dst (when `store`; every lane must call this: the TMEM
// loads are warp-collective).
template <int D>
__device__ __forceinline__ void rope_bwd_row(uint32_t taddr, float mul, int pos, float rope_k,
                                             __nv_bfloat16* dst, bool store) {
#pragma unroll 1
  for (int j = 0; j < D / 64; ++j) {
    uint32_t v1[32], v2[32];
    ptx::tmem_ld32(taddr + 32 * j, v1);
    ptx::tmem_ld32(taddr + 32 * j + D / 2, v2);
    uint32_t pa[16], pb[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float a[2], b[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float g1 = __uint_as_float(v1[i + e]) * mul;
        const float g2 = __uint_as_float(v2[i + e]) * mul;
        float sn, cs;
        sincosf(static_cast<float>(pos) * exp2f(static_cast<float>(32 * j + i + e) * rope_k), &sn, &cs);
        a[e] = fmaf(g1, cs, g2 * sn);
        b[e] = fmaf(g2, cs, -g1 * sn);
      }
      pa[i / 2] = ptx::pack_bf16x2(a[0], a[1]);
      pb[i / 2] = ptx::pack_bf16x2(b[0], b[1]);
    }
    if (store) {
      uint4* d1 = reinterpret_cast<uint4*>(dst + 32 * j);
      uint4* d2 = reinterpret_cast<uint4*>(dst + D / 2 + 32 * j);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        d1[v] = make_uint4(pa[4 * v], pa[4 * v + 1], pa[4 * v + 2], pa[4 * v + 3]);
        d2[v] = make_uint4(pb[4 * v], pb[4 * v + 1], pb[4 * v + 2], pb[4 * v + 3]);
      }
    }
  }
}

// One thread's run of N 32-bit words (N a multiple of 8) to global memory:
// 32-byte stores when `v8` (the address is then 32-byte aligned), else
// 16-byte ones.  Epilogues write one row per thread, so a warp's store
// touches 32 rows: halving the store instructions halves that traffic.
template <int N>
__device__ __forceinline__ void store_words(void* dst, const uint32_t (&w)[N], bool v8) {
  static_assert(N % 8 == 0, "whole 32-byte pieces");
  if (v8) {
#pragma unroll
    for (int i = 0; i < N / 8; ++i)
      ptx::st_global_v8(static_cast<uint8_t*>(dst) + 32 * i,
                        *reinterpret_cast<const uint32_t(*)[8]>(&w[8 * i]));
  } else {
    uint4* d = static_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < N / 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}
// 32-byte stores are possible into rows of D bf16 (a multiple of 32 bytes)
// when every base is 32-byte aligned.
__device__ __forceinline__ bool aligned32(const void* a, const void* b = nullptr) {
  return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 31u) == 0;
}

// Device status word values (same numbering as gdpa_status).
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}


struct FwdParams {
  const int32_t* qo;
  const int32_t* ko;
  int B, H, d;
  int64_t Tq, Tkv;
  const float* bias_table;  // nullptr: no bias
  int max_rel;
  int causal;
  int window;               // 0: no sliding window
  float scale;
  const float* bias_dense;  // dense jagged bias (nullptr: none); sample b's [H][Lq][Lkv]
  const int64_t* bias_off;  //   block starts at element bias_off[b]
  __nv_bfloat16* out;
  float* lse;               // nullptr allowed for GDPA activations
  const int2* items;
  const int* n_items;
  int* ticket;
  int* status;
};

struct BwdParams {
  const int32_t* qo;
  const int32_t* ko;
  int B, H, d;
  int64_t Tq, Tkv;
  const float* bias_table;
  int max_rel;
  int causal;
  int window;
  float scale;
  const float* bias_dense;  // dense jagged bias (nullptr: none), as in FwdParams
  const int64_t* bias_off;
  const __nv_bfloat16* out;
  const float* lse;
  const __nv_bfloat16* dout;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dbias;             // fp32 [H][2*max_rel-1], added to (nullptr: not computed)
  float rope_base;          // > 0: dq, dk go back through the rotary embedding
  float* dq_acc;            // fp32 [Tq][H][d] accumulator (zeroed by the preprocess kernel)
  float* delta;             // fp32 [H][Tq]: rowsum(dO * O) for softmax
  const int* all_short;     // scheduler flag: every sample takes the short-query kernel, so
                            //   the accumulator is neither zeroed nor converted (nullptr: no
                            //   short-query list)
  __nv_bfloat16* dq;        // bf16 dQ output
  int dq_direct_kv;         // > 0: samples with 1..dq_direct_kv keys and more than short_q_max
                            //   queries get dQ written once in bf16 by the main kernel (one key
                            //   block sees every key); their accumulator rows are neither zeroed
                            //   nor converted.  0: every row goes through the accumulator.
  int short_q_max;          // queries of a short-query sample (0: no short-query list)
  const int2* items;
  const int* n_items;
  int* ticket;
  int* status;
};

struct BlockParams {
  const int4* tiles;        // {first row, rows of block A, rows of block B, 0} per tile
  const int* n_tiles;
  int H, d;
  int64_t T;
  const float* bias_table;  // nullptr: no bias
  int max_rel;
  int causal;
  float scale;
  // dense jagged bias instead of the table (nullptr: none): sample b's
  // [H][L_b][L_b] values from bias_dense + bias_off[b]; offsets / B locate a
  // row's sample
  const float* bias_dense;
  const int64_t* bias_off;
  const int32_t* offsets;
  int B;
  __nv_bfloat16* out;             // forward output
  const __nv_bfloat16* dout;      // backward inputs / outputs
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float rope_base;                // > 0: dq, dk go back through the rotary embedding
  float* dbias;                   // backward: the bias's gradient, added to (nullptr: none)
  int* status;
};

// The short-query list of the scheduler: samples with 1 <= Lq_b <= max_q get
// one item {b, head} per head here instead of blocks in the main list
// (max_q 0 or items null: no split).  all_short is set to 1 when every
// sample with query rows went to this list.
struct ShortList {
  int max_q = 0;
  int2* items = nullptr;
  int* n_items = nullptr;
  int* ticket = nullptr;
  int* all_short = nullptr;
};
// Queries of a short-query item (the MMA width of the short-query kernels).
constexpr int kShortQ = 32;

// The short-key list of the forward scheduler: samples with more than kShortQ
// queries and 1 <= Lkv_b <= max_kv keys get items {b, (chunk << 8) | head},
// one per head and chunk of kShortKvChunk queries, here instead of blocks in
// the main list (max_kv 0 or items null: no split).  Items are sorted by
// their own cost, longest first.
struct KvList {
  int max_kv = 0;
  int2* items = nullptr;
  int* n_items = nullptr;
  int* ticket = nullptr;
};
// Keys a short-key sample may have (its K and V stay in shared memory) and
// queries per short-key item.
constexpr int kShortKv = 256;
constexpr int kShortKvChunk = 2048;
inline int64_t max_kv_items(int B, int H, int64_t Tq) {
  return static_cast<int64_t>(H) * (Tq / kShortKvChunk + B);
}

// Host-side launchers (defined in the kernel translation units).
// bias_off (optional): element offsets of a dense jagged bias, checked against
// H * Lq_b * Lkv_b (a mismatch is reported as GDPA_ERR_BAD_OFFSETS).
cudaError_t launch_build_worklist(const int32_t* outer_off, const int32_t* inner_off, int B, int H,
                                  int64_t T_outer, int64_t T_inner, int causal, int window,
                                  int mode,
                                  int2* items, int* n_items, int* ticket, int* status,
                                  cudaStream_t stream, const int64_t* bias_off = nullptr,
                                  const ShortList& sq = ShortList{},
                                  const KvList& kv = KvList{});
cudaError_t launch_fwd(const FwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, int grid, cudaStream_t stream);
// Short-query forward (GDPA activations, no mask or bias): p.items is the
// scheduler's short-query list; tq has kShortQ-row boxes.
cudaError_t launch_fwd_short_q(const FwdParams& p, int act, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                               cudaStream_t stream);
// Short-key forward (GDPA activations, no mask or bias): p.items is the
// scheduler's short-key list; tq has kHalfRows-row boxes, tk and tv kKvRows.
cudaError_t launch_fwd_short_kv(const FwdParams& p, int act, const CUtensorMap& tq,
                                const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                                cudaStream_t stream);
int fwd_smem_bytes(int d);
cudaError_t launch_bwd_softmax_main(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& tdo,
                                    const CUtensorMap& tdq, int grid, cudaStream_t s);
// The rotary-backward instantiations of the softmax backward (p.rope_base > 0).
cudaError_t launch_bwd_softmax_rope(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& tdo,
                                    const CUtensorMap& tdq, int grid, cudaStream_t s);
// The short-query part of a backward call (its own list, maps and grid).
struct ShortBwd {
  BwdParams p;
  CUtensorMap tq, tdo;
  void* dq;
  int grid;
};
cudaError_t launch_bwd(const BwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                       int grid,
                       cudaStream_t stream, int* launches, cudaEvent_t ev_begin,
                       cudaEvent_t ev_end, const ShortBwd* sq = nullptr);
cudaError_t launch_dq_convert(const float* acc, void* dq, long long n, float scale,
                              cudaStream_t stream, const int* skip = nullptr,
                              const BwdParams* direct = nullptr);
// Short-query backward (p.items: the scheduler's short-query list; tq, tdo
// with kShortQ-row boxes).  dQ goes to dq as bf16 when *p.all_short, else
// (unscaled) into the rows of p.dq_acc that the short samples own.
cudaError_t launch_bwd_short_q(const BwdParams& p, int act, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, void* dq, int grid, cudaStream_t stream);
// dq = bf16 of the rotary backward of scale * acc ([T][H][d]); positions are
// local to the samples of `offsets` (B + 1 entries).
cudaError_t launch_dq_convert_rope(const float* acc, void* dq, const int32_t* offsets, int B,
                                   long long T, int H, int d, float scale, float rope_base,
                                   cudaStream_t stream);
// Zeroes p.dq_acc and, for softmax, writes p.delta = rowsum(dO * O).
cudaError_t launch_bwd_preprocess(const BwdParams& p, bool softmax, cudaStream_t stream);

// nosat: the saturation-free block scale (mx::e8m0_nosat) instead of the OCP one.
cudaError_t launch_quant_rows(const void* x, long long rows, int d, void* codes, void* scales,
                              cudaStream_t s, bool nosat = false);
cudaError_t launch_quant_tokens(const void* x, const int32_t* offsets, int B, int H, int d,
                                long long T, void* codes, void* scales, cudaStream_t s,
                                bool nosat = false);

int fwd_mx_tile_rows();
// MXFP8 softmax backward (d = 128): operand codes and scales of each product.
struct BwdMxOperands {
  const uint8_t* qd_sc;   // Q along channels: u32 word of 4 scales per (token, head)
  const uint8_t* kd_sc;
  const uint8_t* vd_sc;
  const uint8_t* dod_sc;
  const uint8_t* qt_sc;   // along tokens: [B + T/32 + 1][H][d] bytes
  const uint8_t* kt_sc;
  const uint8_t* dot_sc;
};
// maps: qd, qt, dod, dot (64-row boxes), kd, kt, vd (128-row boxes), dq (fp32, 16-row boxes)
cudaError_t launch_bwd_mx(const BwdParams& p, const BwdMxOperands& mx, const CUtensorMap* maps,
                          int grid, cudaStream_t s);
// The dense-bias instantiations of the MXFP8 backward (p.bias_dense set).
cudaError_t launch_bwd_mx_dense(const BwdParams& p, const BwdMxOperands& mx,
                                const CUtensorMap* maps, int grid, cudaStream_t s);
cudaError_t launch_fwd_mx(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const uint8_t* q_sc, const uint8_t* k_sc,
                          const uint8_t* v_sc, long long v_sc_rows, int grid, cudaStream_t s);

// bias_off (a dense bias's per-sample offsets, H heads) is checked with the
// offsets: GDPA_ERR_BAD_OFFSETS unless sample b holds H * L_b^2 values.
cudaError_t launch_block_list(const int32_t* offsets, int B, int64_t T, int4* tiles, int* n_tiles,
                              int* status, cudaStream_t s, const int64_t* bias_off = nullptr,
                              int H = 0);
cudaError_t launch_block_fwd(const BlockParams& p, int act, const CUtensorMap& tq,
                             const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                             cudaStream_t s);
// The dense-bias instantiations of the block forward (p.bias_dense set).
cudaError_t launch_block_fwd_dense(const BlockParams& p, int act, const CUtensorMap& tq,
                                   const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                                   cudaStream_t s);
// maps: q, k, v, dout, dq, dk, dv (bf16 [T][H][d], 128-row boxes)
cudaError_t launch_block_bwd(const BlockParams& p, int act, const CUtensorMap* maps, int grid,
                             cudaStream_t s);
// The bias-table gradient's instantiations of the block backward (p.dbias set).
cudaError_t launch_block_bwd_dbias(const BlockParams& p, int act, const CUtensorMap* maps, int grid,
                                   cudaStream_t s);
// The dense-bias instantiations of the block backward, without and with the
// dense bias's gradient (p.bias_dense set; p.dbias selects the gradient).
cudaError_t launch_block_bwd_dense(const BlockParams& p, int act, const CUtensorMap* maps, int grid,
                                   cudaStream_t s);
cudaError_t launch_block_bwd_dense_db(const BlockParams& p, int act, const CUtensorMap* maps,
                                      int grid, cudaStream_t s);

// Upper bound on the number of work items (host-side sizing).
inline int64_t max_fwd_items(int B, int H, int64_t Tq) {
  return static_cast<int64_t>(H) * (Tq / kItemRows + B);
}
inline int64_t max_bwd_items(int B, int H, int64_t Tkv) {
  return static_cast<int64_t>(H) * (Tkv / kBwdKvRows + B);
}
// Tiles of two 64-token blocks: at most (T/64 + B + 1) / 2.
inline int64_t max_block_tiles(int B, int64_t T) { return (T / kBlockRows + B + 2) / 2; }

}  // namespace gdpa
