// gdn_norm.cu -- gated RMSNorm of the recurrence output.
//
// Defines: [cpu.rs] (ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs)
// gated_rms_norm_f32; [cpu_ops.cpp] (vllm.cpp, src/vt/cpu/cpu_ops.cpp)
// RmsNormGatedKernel (sigmoid-gate option, token-strided gate rows).  Per
// (token, head) row of dim values:
//   out = core / sqrt(mean(core^2) + eps) * weight * act(z),  act = silu | sigmoid.
//
// HBM-bound (read core and z, write out).  A row is handled by a group of
// lpr = min(32, pow2 >= dim / V) lanes, V = 16-byte vector width (8 bf16 or 4
// f32), each lane taking vectors lane, lane + lpr, ... of the row; a warp
// handles 32 / lpr rows at a time and walks rows with a grid stride, keeping
// its slice of the weight vector in registers.  The sum of squares is a
// shuffle reduction inside the group.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "gdn_math.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxVec = 4;  // vectors per lane and row: dim <= 32 * V * kMaxVec

template <typename TA>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ static void load(const void* p, float (&o)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(void* p, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Vec<float> {
  static constexpr int kN = 4;
  __device__ static void load(const void* p, float (&o)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x;
    o[1] = v.y;
    o[2] = v.z;
    o[3] = v.w;
  }
  __device__ static void store(void* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};

// math::norm_gate of two values with paired f32 arithmetic: e^{-z} as
// 2^{-z log2(e)} on the hardware's base-2 exponential (capped at e^80), 1 / (1
// + e^{-z}) on the approximate reciprocal refined by one Newton-Raphson step;
// silu multiplies by z.  The same operations, two values an instruction.
__device__ __forceinline__ float2 norm_gate2(float2 z, bool sigmoid_gate) {
  constexpr float kNegLog2e = -1.4426950408889634f;
  constexpr float kCap = 80.0f * 1.4426950408889634f;
  const float2 m = __fmul2_rn(z, make_float2(kNegLog2e, kNegLog2e));
  float e0, e1;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(fminf(m.x, kCap)));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(fminf(m.y, kCap)));
  const float2 d = __fadd2_rn(make_float2(1.0f, 1.0f), make_float2(e0, e1));
  float r0, r1;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(d.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(d.y));
  float2 r = make_float2(r0, r1);
  const float2 t = __ffma2_rn(make_float2(-d.x, -d.y), r, make_float2(1.0f, 1.0f));
  r = __ffma2_rn(r, t, r);
  return sigmoid_gate ? r : __fmul2_rn(z, r);
}

template <typename TA, int NV>
__global__ void __launch_bounds__(kThreads) gated_rmsnorm_kernel(const NormLaunch p, int lpr) {
  constexpr int V = Vec<TA>::kN;
  constexpr int es = sizeof(TA);
  const int lane = threadIdx.x & 31;
  const int sub = lane % lpr;                    // lane inside the row group
  const int rows_per_warp = 32 / lpr;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) / 32;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * kThreads / 32;
  const int nvec = p.dim / V;
  const uint8_t* w8 = static_cast<const uint8_t*>(p.weight);
  float w[NV][V];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int vi = sub + j * lpr;
    if (vi < nvec) {
      Vec<TA>::load(w8 + static_cast<int64_t>(vi) * V * es, w[j]);
    } else {
#pragma unroll
      for (int e = 0; e < V; ++e) w[j][e] = 0.0f;
    }
  }
  const float inv_dim = 1.0f / static_cast<float>(p.dim);
  const uint8_t* core8 = static_cast<const uint8_t*>(p.core);
  const uint8_t* z8 = static_cast<const uint8_t*>(p.z);
  uint8_t* out8 = static_cast<uint8_t*>(p.out);
  for (int64_t base = warp_global * rows_per_warp; base < p.rows; base += n_warps * rows_per_warp) {
    const int64_t row = base + lane / lpr;
    const bool live = row < p.rows;
    const int64_t t = live ? row / p.heads : 0, h = live ? row % p.heads : 0;
    const uint8_t* xr = core8 + (live ? row : 0) * p.dim * es;
    const uint8_t* zr = z8 + (t * p.z_stride + h * p.dim) * es;
    float x[NV][V], zz[NV][V];
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vi = sub + j * lpr;
      if (live && vi < nvec) {
        Vec<TA>::load(xr + static_cast<int64_t>(vi) * V * es, x[j]);
        Vec<TA>::load(zr + static_cast<int64_t>(vi) * V * es, zz[j]);
      } else {
#pragma unroll
        for (int e = 0; e < V; ++e) x[j][e] = zz[j][e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < V; ++e) ss = fmaf(x[j][e], x[j][e], ss);
    }
    for (int m = 1; m < lpr; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float inv = math::rms_inv(ss, inv_dim, p.eps);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vi = sub + j * lpr;
      if (live && vi < nvec) {
        float o[V];
#pragma unroll
        for (int e = 0; e < V; e += 2) {
          const float2 g = norm_gate2(make_float2(zz[j][e], zz[j][e + 1]), p.sigmoid_gate);
          const float2 xs = __fmul2_rn(make_float2(x[j][e], x[j][e + 1]), make_float2(inv, inv));
          const float2 oo = __fmul2_rn(__fmul2_rn(xs, make_float2(w[j][e], w[j][e + 1])), g);
          o[e] = oo.x;
          o[e + 1] = oo.y;
        }
        Vec<TA>::store(out8 + (row * p.dim + static_cast<int64_t>(vi) * V) * es, o);
      }
    }
  }
}

template <typename TA>
cudaError_t launch_t(const NormLaunch& p, cudaStream_t s) {
  constexpr int V = Vec<TA>::kN;
  const int nvec = p.dim / V;
  int lpr = 1;
  while (lpr < 32 && lpr < nvec) lpr <<= 1;
  const int nv = (nvec + lpr - 1) / lpr;  // vectors per lane (<= kMaxVec for dim <= 4096)
  const int rows_per_block = (kThreads / 32) * (32 / lpr);
  int64_t blocks = (p.rows + rows_per_block - 1) / rows_per_block;
  blocks = blocks < 152 * 16 ? blocks : 152 * 16;  // grid stride beyond 16 CTAs per SM
  const unsigned grid = static_cast<unsigned>(blocks > 0 ? blocks : 1);
  if (nv <= 1)
    gated_rmsnorm_kernel<TA, 1><<<grid, kThreads, 0, s>>>(p, lpr);
  else if (nv <= 2)
    gated_rmsnorm_kernel<TA, 2><<<grid, kThreads, 0, s>>>(p, lpr);
  else
    gated_rmsnorm_kernel<TA, kMaxVec><<<grid, kThreads, 0, s>>>(p, lpr);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const NormLaunch& p, cudaStream_t s) {
  return p.bf16 ? launch_t<__nv_bfloat16>(p, s) : launch_t<float>(p, s);
}

}  // namespace gdn
