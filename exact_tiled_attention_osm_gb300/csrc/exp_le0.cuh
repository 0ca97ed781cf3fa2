// exp_le0.cuh — exp(d) for d <= 0 in FP32, for the kernels whose outputs are
// held to a relative error of 1e-5 (row softmax, softmax + top-k).
//
// The hardware's ex2.approx is accurate for a base-2 argument of small
// magnitude; a large argument d*log2(e) computed in FP32 would lose the low
// bits of its fractional part.  So the argument is split (Cody & Waite range
// reduction): n = round(d * log2e_hi), f = d * log2e_hi - n + d * log2e_lo with
// log2(e) held as an FP32 head and its remainder, r = 2^f by ex2.approx, and
// the result is r * 2^n built from the exponent bits.  Results below the
// normal FP32 range flush to 0.
#pragma once
#include "ptx.cuh"

namespace osm {

// log2(e) split into an FP32 head and its remainder
constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963033500011079e-8f;

__device__ __forceinline__ float exp_le0(float d) {
  d = fmaxf(d, -100.f);  // also maps -inf (and -inf - -inf) to a flushed 0
  const float n = rintf(d * kLog2eHi);
  float f = fmaf(d, kLog2eHi, -n);
  f = fmaf(d, kLog2eLo, f);
  const float r = ptx::ex2(f);
  const int ni = static_cast<int>(n);
  return ni < -125 ? 0.f : r * __int_as_float((ni + 127) << 23);
}

}  // namespace osm
