// INT8 codes without a division per element.
//
// The scheme's INT8 code is the rounding of a correctly rounded quotient, rint(RN(x / s))
// (ties to even).  With inv = RN(1 / s), q = RN(x * inv) is within 2 ulps of x / s, and so
// within 2.5 ulps of RN(x / s).  Both round to the same code unless a half-integer lies
// within that distance of q; such elements (a few in a million) are recomputed with the
// IEEE division.  (The e4m3 codes follow the same scheme in stage.cuh.)
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace sage {
namespace {  // internal linkage: each translation unit keeps its own copy

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

}  // namespace
}  // namespace sage
