// Block-scaled MXFP8 MMA helpers (sm_103a), shared by the MXFP8 forward and
// backward kernels: E4M3 operands with one E8M0 scale per 32 elements of
// the contraction (OCP Microscaling v1.0), fp32 accumulation in TMEM.
#pragma once

#include "ptx.cuh"

namespace gdpa {
namespace mx {

// Instruction descriptor of kind::mxf8f6f4, E4M3 x E4M3 with E8M0 scales,
// M = 128: B scale-factor byte (bits 4-5), A / B MN-major (15 / 16), N >> 3
// (17-22), E8M0 scale type (23), M >> 4 (24-28), A scale-factor byte (29-30).
__device__ __forceinline__ uint32_t idesc(int N, bool a_mn, bool b_mn, int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (8u << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

// D[tmem] (+)= A[smem] * B[smem] with the scale words at sfa / sfb (TMEM).
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}\n"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem].
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%4], [%5], p;\n}\n"
      ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

// E8M0 code of the smallest power of two X with amax / X <= 448 (E4M3's
// largest normal), clamped to [0, 254]; amax is a non-negative float.  For
// values made inside a kernel (P, dS) this saturation-free choice is used
// instead of 2^(floor(log2 amax) - 8), which maps the block maximum into
// [256, 512) and would clip it by up to 12.5% when its mantissa exceeds 1.75.
__device__ __forceinline__ int e8m0_nosat(float amax) {
  const uint32_t u = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (u == 0) return 0;
  int e = (u >> 23) != 0 ? static_cast<int>(u >> 23) - 127 : -127 - (__clz(u) - 9);
  if ((u >> 23) != 0 && (u & 0x7FFFFFu) > 0x600000u) ++e;  // mantissa above 1.75
  const int code = e - 8 + 127;
  return code < 0 ? 0 : (code > 254 ? 254 : code);
}

// Four E4M3 codes (round to nearest even, saturating), a in the low byte.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

}  // namespace mx
}  // namespace gdpa
