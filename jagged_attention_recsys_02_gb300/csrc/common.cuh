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

constexpr int kCostBuckets = 2048;

// Work item: x = sample b (or -1 = end of list), y = (block << 8) | head.
__host__ __device__ inline int item_head(int2 it) { return it.y & 0xFF; }
__host__ __device__ inline int item_block(int2 it) { return it.y >> 8; }

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
  float scale;
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
  float scale;
  const __nv_bfloat16* out;
  const float* lse;
  const __nv_bfloat16* dout;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dq_acc;            // fp32 [Tq][H][d] accumulator (zeroed by the preprocess kernel)
  float* delta;             // fp32 [H][Tq]: rowsum(dO * O) for softmax
  const int2* items;
  const int* n_items;
  int* ticket;
  int* status;
};

// Host-side launchers (defined in the kernel translation units).
cudaError_t launch_build_worklist(const int32_t* outer_off, const int32_t* inner_off, int B, int H,
                                  int64_t T_outer, int64_t T_inner, int causal, int mode,
                                  int2* items, int* n_items, int* ticket, int* status,
                                  cudaStream_t stream);
cudaError_t launch_fwd(const FwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, int grid, cudaStream_t stream);
int fwd_smem_bytes(int d);
cudaError_t launch_bwd_softmax_main(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& tdo,
                                    const CUtensorMap& tdq, int grid, cudaStream_t s);
cudaError_t launch_bwd(const BwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                       int grid,
                       cudaStream_t stream, int* launches, cudaEvent_t ev_begin,
                       cudaEvent_t ev_end);
cudaError_t launch_dq_convert(const float* acc, void* dq, long long n, float scale,
                              cudaStream_t stream);

cudaError_t launch_quant_rows(const void* x, long long rows, int d, void* codes, void* scales,
                              cudaStream_t s);
cudaError_t launch_quant_tokens(const void* x, const int32_t* offsets, int B, int H, int d,
                                long long T, void* codes, void* scales, cudaStream_t s);

int fwd_mx_tile_rows();
cudaError_t launch_fwd_mx(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const uint8_t* q_sc, const uint8_t* k_sc,
                          const uint8_t* v_sc, long long v_sc_rows, int grid, cudaStream_t s);

// Upper bound on the number of work items (host-side sizing).
inline int64_t max_fwd_items(int B, int H, int64_t Tq) {
  return static_cast<int64_t>(H) * (Tq / kItemRows + B);
}
inline int64_t max_bwd_items(int B, int H, int64_t Tkv) {
  return static_cast<int64_t>(H) * (Tkv / kBwdKvRows + B);
}

}  // namespace gdpa
