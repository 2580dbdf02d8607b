// gdn_math.cuh -- the scalar gate and activation functions of the prepare
// step, shared by the prepare kernels and the packed decode kernel, and the
// gate and scale of the gated output norm, shared by the norm kernel and the
// kernels that apply the norm where they store their output.
//
// [cpu.rs] (ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs) sigmoid,
// softplus and silu: a two-branch sigmoid, softplus equal to x above 20 and to
// e^x below -20, silu(x) = x sigmoid(x).
#pragma once

#include <cuda_runtime.h>

namespace gdn {
namespace math {

__device__ __forceinline__ float sigmoid_f(float x) {
  if (x >= 0.0f) {
    const float z = expf(-x);
    return 1.0f / (1.0f + z);
  }
  const float z = expf(x);
  return z / (1.0f + z);
}

__device__ __forceinline__ float softplus_f(float x) {
  if (x > 20.0f) return x;
  if (x < -20.0f) return expf(x);
  return log1pf(expf(x));
}

// 1 / y: the hardware's approximate reciprocal refined by one Newton-Raphson
// step, r <- r + r (1 - y r), which roughly doubles its correct bits (to
// within about one ulp of the correctly rounded value).  A lone approximate
// reciprocal is biased enough to shift bf16 roundings of whole tensors the
// same way.  For finite y >= 1.
__device__ __forceinline__ float recip_nr(float y) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return fmaf(r, fmaf(-y, r, 1.0f), r);
}

// e^x as 2^{x log2(e)} on the hardware's approximate base-2 exponential
// (flush-to-zero form: results below 2^-126 read 0).  About two ulp; used
// where an exponential is evaluated per state column.
__device__ __forceinline__ float exp_ex2(float x) {
  constexpr float kLog2e = 1.4426950408889634f;
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * kLog2e));
  return y;
}

// silu(x) = x / (1 + e^{-x}).  e^{-x} is capped at e^80 (the result is then
// below 1e-32 in magnitude either way) so that the reciprocal's operand stays
// finite.
__device__ __forceinline__ float silu_f(float x) {
  return x * recip_nr(1.0f + __expf(fminf(-x, 80.0f)));
}

// The gate of the gated RMSNorm ([cpu.rs] gated_rms_norm_f32: silu(z);
// [cpu_ops.cpp] RmsNormGatedKernel's option: sigmoid(z)), with sigmoid(z) =
// 1 / (1 + e^{-z}) on the refined reciprocal (e^{-z} capped at e^80).
__device__ __forceinline__ float norm_gate(float z, bool sigmoid_gate) {
  const float sg = recip_nr(1.0f + __expf(fminf(-z, 80.0f)));
  return sigmoid_gate ? sg : z * sg;
}

// 1 / sqrt(mean + eps) of a row of n values whose squares sum to ss.
__device__ __forceinline__ float rms_inv(float ss, float inv_n, float eps) {
  return rsqrtf(fmaf(ss, inv_n, eps));
}

}  // namespace math
}  // namespace gdn
