// gdn_rowstep.cuh -- the register-resident row update of the gated delta
// rule, shared by the recurrent kernels and the packed decode kernel.
//
// [cpu_ops.cpp] (vllm.cpp, src/vt/cpu/cpu_ops.cpp) GdnHeadTokenStep, per row i
// of the [Dv, Dk] state S with a = S_i.k and b = S_i.q taken on the old row:
//   u_i = beta (v_i - e^g a),  S_i <- e^g S_i + u_i k,  o_i = e^g b + u_i (k.q)
// (o_i before the q scale).  A row of Dk floats is split over LPR = Dk/16
// lanes, each holding 16 floats as 4 float4 at columns 4*lr + 4*LPR*m.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace gdn {
namespace rows {

template <typename TA>
__device__ __forceinline__ float ld_act(const TA* p);
template <>
__device__ __forceinline__ float ld_act<float>(const float* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ float ld_act<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}
template <typename TA>
__device__ __forceinline__ void st_act(TA* p, float v);
template <>
__device__ __forceinline__ void st_act<float>(float* p, float v) {
  *p = v;
}
template <>
__device__ __forceinline__ void st_act<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

// 4 consecutive activations starting at p (16-byte aligned for f32, 8 for bf16).
template <typename TA>
__device__ __forceinline__ float4 ld_act4(const TA* p);
template <>
__device__ __forceinline__ float4 ld_act4<float>(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
template <>
__device__ __forceinline__ float4 ld_act4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}

template <int LPR>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int m = 1; m < LPR; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

__device__ __forceinline__ float dot4(const float4& a, const float4& b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// The row update for one token.  Returns o_i (before scale) for this row.
template <int LPR>
__device__ __forceinline__ float row_step(float4 (&s)[4], const float4 (&k)[4],
                                          const float4 (&q)[4], float kq, float decay,
                                          float beta, float v) {
  float a = 0.f, b = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    a += dot4(s[m], k[m]);
    b += dot4(s[m], q[m]);
  }
  a = row_sum<LPR>(a);
  b = row_sum<LPR>(b);
  const float u = beta * (v - decay * a);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    s[m].x = fmaf(decay, s[m].x, u * k[m].x);
    s[m].y = fmaf(decay, s[m].y, u * k[m].y);
    s[m].z = fmaf(decay, s[m].z, u * k[m].z);
    s[m].w = fmaf(decay, s[m].w, u * k[m].w);
  }
  return fmaf(decay, b, u * kq);
}

}  // namespace rows
}  // namespace gdn
