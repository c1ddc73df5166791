// act.cuh -- the MLP activations and their derivatives in fp32, as used by
// the fused epilogues.
//   silu(z)  = z * sigmoid(z)            silu'(z)  = s (1 + z (1 - s)),  s = sigmoid(z)
//   relu2(z) = max(z,0)^2                relu2'(z) = 2 max(z,0)
//   gelu_tanh(z) = 0.5 z (1 + t),  t = tanh(c (z + 0.044715 z^3)),  c = sqrt(2/pi)
//   gelu_tanh'(z) = 0.5 (1 + t) + 0.5 z (1 - t^2) c (1 + 3*0.044715 z^2)
//   relu(z)  = max(z,0)                  relu'(z)  = 1 for z > 0, else 0
//   sigmoid(z) = 1 / (1 + e^-z)          sigmoid'(z) = s (1 - s)
// (tanh approximation of GELU: Hendrycks & Gimpel, 2016).  The sigmoid is
// taken from the hardware tanh, sigmoid(z) = (1 + tanh(z/2)) / 2, one
// tanh.approx.f32 instead of an exponential and a reciprocal (measured on a
// GB300 over z in [-20, 20]: at most 4e-6 from the fp64 sigmoid, 1e-5 for
// silu and silu'; the epilogues' arithmetic is bound by instruction issue,
// and this takes SwiGLU's fused epilogues from two special-function
// instructions per element to one).  The GELU's tanh is CUDA's tanhf.
#pragma once
#include "gemm_params.h"

namespace mlpk {

__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float sigmoid_f(float z) {
  return fmaf(0.5f, tanh_hw(0.5f * z), 0.5f);
}

template <int ACT>
__device__ __forceinline__ float act_f(float z) {
  if constexpr (ACT == ACT_SILU) {
    return z * sigmoid_f(z);
  } else if constexpr (ACT == ACT_RELU_SQ) {
    float r = fmaxf(z, 0.0f);
    return r * r;
  } else if constexpr (ACT == ACT_RELU) {
    return fmaxf(z, 0.0f);
  } else if constexpr (ACT == ACT_SIGMOID) {
    return sigmoid_f(z);
  } else {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    float t = tanhf(c * fmaf(0.044715f * z, z * z, z));
    return 0.5f * z * (1.0f + t);
  }
}

// act(z) and act'(z) together.
template <int ACT>
__device__ __forceinline__ void act_and_grad(float z, float& a, float& da) {
  if constexpr (ACT == ACT_SILU) {
    float s = sigmoid_f(z);
    a = z * s;
    da = s * fmaf(z, 1.0f - s, 1.0f);
  } else if constexpr (ACT == ACT_RELU_SQ) {
    float r = fmaxf(z, 0.0f);
    a = r * r;
    da = 2.0f * r;
  } else if constexpr (ACT == ACT_RELU) {
    a = fmaxf(z, 0.0f);
    da = z > 0.0f ? 1.0f : 0.0f;
  } else if constexpr (ACT == ACT_SIGMOID) {
    const float s = sigmoid_f(z);
    a = s;
    da = s * (1.0f - s);
  } else {
    const float c = 0.7978845608028654f;
    const float k = 0.044715f;
    float z2 = z * z;
    float t = tanhf(c * fmaf(k * z, z2, z));
    a = 0.5f * z * (1.0f + t);
    da = 0.5f * (1.0f + t) + 0.5f * z * (1.0f - t * t) * c * fmaf(3.0f * k, z2, 1.0f);
  }
}

}  // namespace mlpk
