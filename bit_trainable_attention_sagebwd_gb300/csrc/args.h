// Softmax-scale argument of the C ABI, shared by every entry point that takes one.
#pragma once

#include <math.h>

namespace sage {

// NaN and infinities are refused; every finite value is accepted.
inline bool scale_ok(float sm_scale) { return sm_scale == sm_scale && !isinf(sm_scale); }

// A scale <= 0 selects the default 1/sqrt(D).
inline float resolve_scale(float sm_scale, int D) { return sm_scale > 0.f ? sm_scale : 1.0f / sqrtf((float)D); }

}  // namespace sage
