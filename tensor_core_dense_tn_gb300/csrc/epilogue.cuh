// Fused epilogue operations applied after alpha * acc + beta * c:
//
//   v = act(v + bias[n])
//
// The bias is a per-output-column vector (the N dimension: one value per row
// of B, i.e. per output feature of an MLP layer), in bf16 or fp32.  The
// activations are the usual MLP ones: ReLU, GELU (erf form and tanh
// approximation) and SiLU, evaluated in fp32.
//
// The tanh form of GELU is computed as a logistic.  Since
// 1 + tanh(u) = 2 / (1 + e^(-2u)) exactly, 0.5 x (1 + tanh(u)) = x / (1 + e^(-2u)),
// so that it and SiLU (x / (1 + e^(-x))) both take one expf, an add and a fast
// divide, with no branch.  The exponent is capped at 80 so that the divisor
// stays below 2^126, where __fdividef is accurate to 2 ulp; where the cap
// applies the result is x / (1 + e^80) instead of a value nearer zero, a
// difference below 2^-115 |x|.
// Error of either form: expf (2 ulp), the add and the divide (2 ulp) on the
// result, plus the rounding of the argument, which moves the result by at
// most 0.23 |x| times the argument's relative error.  The erf form keeps erff.
#pragma once

#include <cstdint>

#include "kernels.h"

namespace gtn {

__device__ __forceinline__ float load_bias(const Epilogue& e, int n) {
  if (e.bias_f32) return static_cast<const float*>(e.bias)[n];
  return __uint_as_float((uint32_t) static_cast<const uint16_t*>(e.bias)[n] << 16);
}

template <int ACT>
__device__ __forceinline__ float act_of(float v) {
  if constexpr (ACT == kActRelu) {
    return fmaxf(v, 0.0f);
  } else if constexpr (ACT == kActGelu) {  // x * Phi(x)
    return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
  } else if constexpr (ACT == kActGeluTanh) {  // x / (1 + exp(-2 sqrt(2/pi) (x + 0.044715 x^3)))
    const float t = fminf(-1.5957691216057308f * fmaf(0.044715f * v, v * v, v), 80.0f);
    return __fdividef(v, 1.0f + expf(t));
  } else if constexpr (ACT == kActSilu) {  // x / (1 + exp(-x))
    return __fdividef(v, 1.0f + expf(fminf(-v, 80.0f)));
  } else {
    return v;
  }
}

__device__ __forceinline__ float activate(float v, int act) {
  switch (act) {
    case kActRelu: return act_of<kActRelu>(v);
    case kActGelu: return act_of<kActGelu>(v);
    case kActGeluTanh: return act_of<kActGeluTanh>(v);
    case kActSilu: return act_of<kActSilu>(v);
    default: return v;
  }
}

// One activation over an unrolled row chunk: the switch on the activation is
// taken once per chunk, not once per value.
template <int ACT, int N>
__device__ __forceinline__ void act_chunk(float (&v)[N]) {
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] = act_of<ACT>(v[j]);
}

template <int N>
__device__ __forceinline__ void activate_chunk(float (&v)[N], int act) {
  switch (act) {
    case kActRelu: act_chunk<kActRelu>(v); break;
    case kActGelu: act_chunk<kActGelu>(v); break;
    case kActGeluTanh: act_chunk<kActGeluTanh>(v); break;
    case kActSilu: act_chunk<kActSilu>(v); break;
    default: break;
  }
}

}  // namespace gtn
