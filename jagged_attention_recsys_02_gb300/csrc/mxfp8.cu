// MXFP8 quantisation of jagged bf16 tensors (OCP Microscaling Formats v1.0):
// E4M3 elements, one E8M0 scale per block of 32 elements.
//
// "GEM Training ..." low-precision paragraph: attention with end-to-end MXFP8
// block-scaled MMA.  A block's shared scale is 2^(floor(log2 amax) - 8)
// (8 = exponent of E4M3's largest normal, 448); elements are divided by it,
// rounded to nearest even and saturated at +-448.  With `nosat` the scale is
// instead the smallest power of two that keeps the block maximum at or below
// 448 (mx::e8m0_nosat), so no element saturates.
//
// Two block shapes, matching the two products of attention:
//   along channels (Q, K: the contraction of S = Q K^T runs over d): each
//     (token, head) row splits into d/32 blocks; scales [T][H][d/32].
//   along tokens (V: the contraction of O = P V runs over keys): blocks of 32
//     consecutive tokens of one sample, the first starting at the sample's
//     first token (the last may be partial); one scale per (block, head,
//     channel).  Block r of sample b is scale row b + floor(offsets[b]/32) + r,
//     an injective index that needs no prefix sum over samples.
#include "common.cuh"
#include "mx.cuh"

namespace gdpa {
namespace {

// E8M0 code of 2^(floor(log2 amax) - 8), clamped to [0, 254]; 0 for amax == 0.
__device__ __forceinline__ int e8m0_code(float amax) {
  const uint32_t u = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (u == 0) return 0;
  int e;
  if ((u >> 23) != 0) {
    e = static_cast<int>(u >> 23) - 127;
  } else {  // subnormal: position of the leading mantissa bit
    e = -127 - (__clz(u) - 9);
  }
  const int code = e - 8 + 127;
  return code < 0 ? 0 : (code > 254 ? 254 : code);
}

// 2^(127 - code) as an exact float (code in [0, 254) for finite bf16 inputs).
__device__ __forceinline__ float inv_scale(int code) {
  return __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One thread per 32-channel block of one (token, head) row.
__global__ void __launch_bounds__(256)
quant_rows_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                  uint8_t* __restrict__ scales, long long nblocks, bool nosat) {
  for (long long blk = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
       blk < nblocks; blk += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(x + blk * 32);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = src[i];
    float f[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        f[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
        f[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
    const int code = nosat ? mx::e8m0_nosat(amax) : e8m0_code(amax);
    const float inv = inv_scale(code);
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      out[i] = e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv) |
               (e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv) << 16);
    uint4* dst = reinterpret_cast<uint4*>(codes + blk * 32);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    scales[blk] = static_cast<uint8_t>(code);
  }
}

// One CTA per scale row s (32-token block r of sample b, s = b + floor(o_b/32) + r;
// g(b) = b + floor(o_b/32) rises by at least 1 per sample, so the sample owning s is
// the last b with g(b) <= s).  Rows in the gaps between samples own no tokens and are
// left untouched; a few CTAs after the last row zero the codes of tokens outside
// every sample.  Each thread takes 4 consecutive (head, channel) columns: 32 8-byte
// loads in flight, a warp covers 256 contiguous bytes of each token row.
__global__ void __launch_bounds__(128)
quant_tokens_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ offsets,
                    int B, int hd, long long T, long long n_rows, uint8_t* __restrict__ codes,
                    uint8_t* __restrict__ scales, bool nosat) {
  const long long s = blockIdx.x;
  if (s >= n_rows) {
    // Tail blocks: tokens before the first sample or after the last one have no
    // scale row; their codes are zeroed so that a tile running past a sample's
    // end never reads stale bytes (an E4M3 NaN code times a zero weight is NaN).
    const long long a = min(static_cast<long long>(max(offsets[0], 0)), T);
    const long long b = max(a, min(static_cast<long long>(offsets[B]), T));
    const long long nthreads = (gridDim.x - n_rows) * static_cast<long long>(blockDim.x);
    const long long tid = (s - n_rows) * blockDim.x + threadIdx.x;
    uint4* c4 = reinterpret_cast<uint4*>(codes);
    const long long per_tok = hd / 16;
    for (long long i = tid; i < a * per_tok; i += nthreads) c4[i] = make_uint4(0u, 0u, 0u, 0u);
    for (long long i = b * per_tok + tid; i < T * per_tok; i += nthreads)
      c4[i] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  int lo = 0, hi = B - 1;  // largest b with g(b) <= s; g(0) = 0 <= s
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mid + offsets[mid] / 32 <= s) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int t0 = offsets[b], L = offsets[b + 1] - t0;
  if (t0 < 0 || L <= 0 || t0 + static_cast<long long>(L) > T) return;  // nothing valid to read
  const int r = static_cast<int>(s - (b + t0 / 32));
  if (r < 0 || 32 * r >= L) return;
  const int n = min(32, L - 32 * r);
  const long long tok = static_cast<long long>(t0) + 32 * r;
  for (int g = threadIdx.x; 4 * g < hd; g += blockDim.x) {
    const __nv_bfloat16* src = x + tok * hd + 4 * g;
    uint2 v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
      v[i] = i < n ? *reinterpret_cast<const uint2*>(src + static_cast<long long>(i) * hd)
                   : make_uint2(0u, 0u);
    float amax[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      amax[0] = fmaxf(amax[0], fabsf(__uint_as_float(v[i].x << 16)));
      amax[1] = fmaxf(amax[1], fabsf(__uint_as_float(v[i].x & 0xFFFF0000u)));
      amax[2] = fmaxf(amax[2], fabsf(__uint_as_float(v[i].y << 16)));
      amax[3] = fmaxf(amax[3], fabsf(__uint_as_float(v[i].y & 0xFFFF0000u)));
    }
    int code[4];
    float inv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      code[c] = nosat ? mx::e8m0_nosat(amax[c]) : e8m0_code(amax[c]);
      inv[c] = inv_scale(code[c]);
    }
    uint8_t* dst = codes + tok * hd + 4 * g;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < n) {
        const uint32_t w =
            e4m3x2(__uint_as_float(v[i].x << 16) * inv[0],
                   __uint_as_float(v[i].x & 0xFFFF0000u) * inv[1]) |
            (e4m3x2(__uint_as_float(v[i].y << 16) * inv[2],
                    __uint_as_float(v[i].y & 0xFFFF0000u) * inv[3]) << 16);
        *reinterpret_cast<uint32_t*>(dst + static_cast<long long>(i) * hd) = w;
      }
    }
    *reinterpret_cast<uint32_t*>(scales + s * hd + 4 * g) =
        static_cast<uint32_t>(code[0]) | (static_cast<uint32_t>(code[1]) << 8) |
        (static_cast<uint32_t>(code[2]) << 16) | (static_cast<uint32_t>(code[3]) << 24);
  }
}

}  // namespace

cudaError_t launch_quant_rows(const void* x, long long rows, int d, void* codes, void* scales,
                              cudaStream_t s, bool nosat) {
  const long long nblocks = rows * (d / 32);
  if (nblocks == 0) return cudaSuccess;
  const long long want = (nblocks + 255) / 256;
  const int grid = static_cast<int>(want < 65536 ? want : 65536);
  quant_rows_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                         static_cast<uint8_t*>(codes),
                                         static_cast<uint8_t*>(scales), nblocks, nosat);
  return cudaGetLastError();
}

cudaError_t launch_quant_tokens(const void* x, const int32_t* offsets, int B, int H, int d,
                                long long T, void* codes, void* scales, cudaStream_t s,
                                bool nosat) {
  if (B == 0) return cudaSuccess;
  // Scale rows as counted by the buffer size: B + T/32 + 1 covers g(B-1) + ceil(L/32).
  const long long rows = static_cast<long long>(B) + T / 32 + 1;
  if (rows > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  constexpr int kTailBlocks = 16;  // zero the codes of tokens outside every sample
  quant_tokens_kernel<<<static_cast<unsigned>(rows + kTailBlocks), 128, 0, s>>>(
      static_cast<const __nv_bfloat16*>(x), offsets, B, H * d, T, rows,
      static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales), nosat);
  return cudaGetLastError();
}

}  // namespace gdpa
