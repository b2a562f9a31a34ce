// Fused epilogue operations applied after alpha * acc + beta * c:
//
//   v = act(v + bias[n])
//
// The bias is a per-output-column vector (the N dimension: one value per row
// of B, i.e. per output feature of an MLP layer), in bf16 or fp32.  The
// activations are the usual MLP ones: ReLU, GELU (erf form and tanh
// approximation) and SiLU.  They evaluate in fp32 with CUDA's erff, tanhf
// and expf.
#pragma once

#include <cstdint>

#include "kernels.h"

namespace gtn {

__device__ __forceinline__ float load_bias(const Epilogue& e, int n) {
  if (e.bias_f32) return static_cast<const float*>(e.bias)[n];
  return __uint_as_float((uint32_t) static_cast<const uint16_t*>(e.bias)[n] << 16);
}

__device__ __forceinline__ float activate(float v, int act) {
  switch (act) {
    case kActRelu:
      return fmaxf(v, 0.0f);
    case kActGelu:  // x * Phi(x)
      return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
    case kActGeluTanh: {  // 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
      const float u = 0.79788456080286536f * fmaf(0.044715f * v, v * v, v);
      return 0.5f * v * (1.0f + tanhf(u));
    }
    case kActSilu:  // x * sigmoid(x)
      return v / (1.0f + expf(-v));
    default:
      return v;
  }
}

}  // namespace gtn
