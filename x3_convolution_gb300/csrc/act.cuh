// act.cuh -- derivative of the epilogue activations, for the fused backward
// through a layer's activation (dgrad epilogue: dz_in = act'(z_in) * dx).
#pragma once

#include <cuda_runtime.h>

#include "../../include/conv3x3.h"

namespace c3 {

// SiLU'(z) = s (1 + z (1 - s)) with s the logistic sigmoid; leaky ReLU' = 1
// above zero and 0.2 at or below it (the lower one-sided derivative at the
// kink, as PyTorch takes it); none: 1.  For z far below zero e^{-z} is +inf,
// s is 0 and the SiLU derivative is (-)0, its limit.
__device__ __forceinline__ float act_grad_f32(int act, float z) {
  if (act == CONV3X3_ACT_SILU) {
    const float s = __fdividef(1.0f, 1.0f + __expf(-z));
    return s * (1.0f + z * (1.0f - s));
  }
  if (act == CONV3X3_ACT_LRELU) return z > 0.0f ? 1.0f : 0.2f;
  return 1.0f;
}

}  // namespace c3
