// MXFP8 quantisation of jagged bf16 tensors (OCP Microscaling Formats v1.0):
// E4M3 elements, one E8M0 scale per block of 32 elements.
//
// "GEM Training ..." low-precision paragraph: attention with end-to-end MXFP8
// block-scaled MMA.  A block's shared scale is 2^(floor(log2 amax) - 8)
// (8 = exponent of E4M3's largest normal, 448); elements are divided by it,
// rounded to nearest even and saturated at +-448.
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
                  uint8_t* __restrict__ scales, long long nblocks) {
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
    const int code = e8m0_code(amax);
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

// One CTA per sample; threads cover (head, channel) pairs, one block of 32
// tokens at a time (consecutive threads read consecutive channels).
__global__ void __launch_bounds__(256)
quant_tokens_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ offsets,
                    int H, int d, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int b = blockIdx.x;
  const int t0 = offsets[b], L = offsets[b + 1] - t0;
  const int hd = H * d;
  const long long srow0 = static_cast<long long>(b) + t0 / 32;
  for (int r = 0; 32 * r < L; ++r) {
    const int n = min(32, L - 32 * r);
    const long long tok = static_cast<long long>(t0) + 32 * r;
    for (int c = threadIdx.x; c < hd; c += blockDim.x) {
      float f[32];
      float amax = 0.0f;
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        f[i] = i < n ? __bfloat162float(x[(tok + i) * hd + c]) : 0.0f;
        amax = fmaxf(amax, fabsf(f[i]));
      }
      const int code = e8m0_code(amax);
      const float inv = inv_scale(code);
#pragma unroll 8
      for (int i = 0; i < 32; ++i)
        if (i < n) codes[(tok + i) * hd + c] = static_cast<uint8_t>(e4m3x2(f[i] * inv, 0.0f));
      scales[(srow0 + r) * hd + c] = static_cast<uint8_t>(code);
    }
  }
}

}  // namespace

cudaError_t launch_quant_rows(const void* x, long long rows, int d, void* codes, void* scales,
                              cudaStream_t s) {
  const long long nblocks = rows * (d / 32);
  if (nblocks == 0) return cudaSuccess;
  const long long want = (nblocks + 255) / 256;
  const int grid = static_cast<int>(want < 65536 ? want : 65536);
  quant_rows_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                         static_cast<uint8_t*>(codes),
                                         static_cast<uint8_t*>(scales), nblocks);
  return cudaGetLastError();
}

cudaError_t launch_quant_tokens(const void* x, const int32_t* offsets, int B, int H, int d,
                                void* codes, void* scales, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  quant_tokens_kernel<<<B, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), offsets, H, d,
                                        static_cast<uint8_t*>(codes),
                                        static_cast<uint8_t*>(scales));
  return cudaGetLastError();
}

}  // namespace gdpa
