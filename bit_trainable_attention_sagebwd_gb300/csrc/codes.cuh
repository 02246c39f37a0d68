// Quantization codes without a division per element.
//
// The scheme's codes are roundings of a correctly rounded quotient: the INT8 code
// rint(RN(x / s)) (ties to even) and the e4m3 code e4m3(RN(x / s)).  With inv = RN(1 / s),
// q = RN(x * inv) is within 2 ulps of x / s, and so within 2.5 ulps of RN(x / s).  Both
// round to the same code unless a rounding boundary (a half-integer, or an e4m3 midpoint)
// lies within that distance of q; such elements (a few in a million) are recomputed with
// the IEEE division.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace sage {
namespace {  // internal linkage: each translation unit keeps its own copy

__device__ __noinline__ uint32_t e4m3_code_exact(float x, float s) {
  return (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E4M3);
}

// e4m3 (round to nearest even, saturating) of RN(x / s); inv = RN(1 / s), or 0 when s == 0.
// A normal e4m3 midpoint has fp32 mantissa bit 19 set and bits 18..0 clear; the key below is
// at most 16 << 12 exactly when q is within 8 ulps of one.  Below 2^-6 e4m3 is subnormal with
// coarser midpoints, so any nonzero q there takes the division too (it is rare: values that
// small are under 2^-6 / 448 of the channel maximum).
__device__ __forceinline__ uint32_t e4m3_code(float x, float s, float inv) {
  const float q = __fmul_rn(x, inv);
  const uint32_t key = __float_as_uint(q) * 4096u + ((8u - 0x80000u) << 12);
  const float aq = fabsf(q);
  if (key <= (16u << 12) || (aq < 0.015625f && aq != 0.f)) return e4m3_code_exact(x, s);
  return (uint32_t)__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
}

// Eight INT8 codes with one scale: the doubt test costs no branch per element; when any of
// the eight is in doubt all eight take the (inlined) division, which is rare.
__device__ __forceinline__ void int_codes8(const float (&x)[8], float s, float inv, float (&c)[8]) {
  bool doubt = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float q = __fmul_rn(x[i], inv);
    const float r = rintf(q);
    doubt |= fabsf(__fsub_rn(q, r)) > 0.49993896484375f;
    c[i] = fminf(fmaxf(r, -127.f), 127.f);
  }
  if (doubt) {
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = fminf(fmaxf(rintf(__fdiv_rn(x[i], s)), -127.f), 127.f);
  }
}

// Eight e4m3 codes with per-element scales, same scheme as e4m3_code.
__device__ __forceinline__ void e4m3_codes8(const float (&x)[8], const float (&s)[8], const float (&inv)[8],
                                            uint32_t (&c)[8]) {
  bool doubt = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float q = __fmul_rn(x[i], inv[i]);
    const uint32_t key = __float_as_uint(q) * 4096u + ((8u - 0x80000u) << 12);
    const float aq = fabsf(q);
    doubt |= (key <= (16u << 12)) | ((aq < 0.015625f) & (aq != 0.f));
    c[i] = (uint32_t)__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
  }
  if (doubt) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      c[i] = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[i], s[i]), __NV_SATFINITE, __NV_E4M3);
  }
}

}  // namespace
}  // namespace sage
