// gdn_packed.cu -- decode in one launch from the packed projections: conv
// update + SiLU + q/k L2 norm + gates + the gated delta rule.
//
// Defines: [cpu_ops.cpp] (vllm.cpp, src/vt/cpu/cpu_ops.cpp)
// GdnPackedDecodeKernel -- the split of the packed row, q and k normalised in
// f32 and never stored, the gates per value head and the recurrence -- with
// the conv update of [cpu_ops.cpp] CausalConv1dUpdateKernel folded in, on the
// packed layouts of [cpu.rs] (ferrum-kernels 0.8.0,
// src/ferrum_kernels/backend/cpu.rs)
// linear_attention_prepare_varlen_packed_qkvz_ba_f32 (rows of q, k, v then z;
// gate rows of b then a), which the caller describes with row strides.
//
// One CTA per (row b, key head hk).  It owns the conv channels of hk's q and k
// and of the value heads hk*ratio .. hk*ratio + ratio - 1, so every conv tail
// is read and rewritten by exactly one CTA and nothing but the inputs is
// shared between CTAs.  Phase 1 puts those channels' conv outputs (f32) in
// shared memory, with the two norms and the ratio gates.  Phase 2 streams the
// value heads' state rows through registers, one head at a time, with the
// row update of the recurrent kernels (LPR = Dk/16 lanes per row, 256/LPR rows
// per pass), and writes out = scale * o.  The first head's rows are requested
// before phase 1.  Nothing is rounded to the activation type between the
// steps; only out is stored in it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "gdn_internal.h"
#include "gdn_math.cuh"
#include "gdn_rowstep.cuh"

namespace gdn {
namespace {

using namespace rows;

constexpr int kThreads = 256;

template <typename TA, int DK, int KW>
__global__ void __launch_bounds__(kThreads) packed_decode_kernel(const PackedDecodeLaunch p) {
  constexpr int LPR = DK / 16;
  constexpr int RPP = kThreads / LPR;   // rows per pass
  constexpr int PASSES = (128 + RPP - 1) / RPP;  // covers Dv <= 128
  constexpr int W = KW - 1;
  extern __shared__ float sm[];
  const int ratio = p.Hv / p.Hk;
  const int hk = blockIdx.x % p.Hk, b = blockIdx.x / p.Hk;
  const int h0 = hk * ratio;
  const int tid = threadIdx.x;
  // shared: q [DK] | k [DK] | v [ratio*Dv] | decay [ratio] | beta [ratio] | inv [2]
  float* y = sm;
  float* decay_s = sm + 2 * DK + ratio * p.Dv;
  float* beta_s = decay_s + ratio;
  float* inv_s = beta_s + ratio;

  int slot = __ldg(p.sidx + b);
  if (slot < -1 || slot >= p.slots) {
    if (tid == 0) atomicOr(p.status, kStatusBadIndex);
    slot = -1;
  }
  TA* out = static_cast<TA*>(p.out) + ((int64_t)b * p.Hv + h0) * p.Dv;
  if (slot < 0) {  // padding row: zero outputs, neither pool touched
    for (int e = tid; e < ratio * p.Dv; e += kThreads) st_act<TA>(out + e, 0.0f);
    return;
  }

  // The first value head's state rows are requested before phase 1, so their
  // latency overlaps the conv; later heads load at the top of their turn.
  const int lr = tid % LPR, rg = tid / LPR;
  float4 st[PASSES][4];
  auto load_state = [&](int hh) {
    const float* S = p.pool + ((int64_t)slot * p.Hv + h0 + hh) * p.Dv * DK;
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = rg + ps * RPP;
#pragma unroll
      for (int m = 0; m < 4; ++m)
        st[ps][m] = r < p.Dv ? __ldcs(reinterpret_cast<const float4*>(S + (int64_t)r * DK + 4 * lr +
                                                                        4 * LPR * m))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load_state(0);

  // ---- phase 1: conv update of this CTA's channels, gates, norms -----------
  const int qk_total = p.Hk * DK;
  const int C = 2 * qk_total + p.Hv * p.Dv;
  const int nch = 2 * DK + ratio * p.Dv;
  const TA* __restrict__ x = static_cast<const TA*>(p.x) + (int64_t)b * p.x_stride;
  float* __restrict__ tails = p.conv_pool + (int64_t)slot * C * W;
  for (int e = tid; e < nch; e += kThreads) {
    const int c = e < DK       ? hk * DK + e
                  : e < 2 * DK ? qk_total + hk * DK + (e - DK)
                               : 2 * qk_total + h0 * p.Dv + (e - 2 * DK);
    const float xv = ld_act<TA>(x + c);
    float* tr = tails + (int64_t)c * W;
    float old[W > 0 ? W : 1];
#pragma unroll
    for (int j = 0; j < W; ++j) old[j] = tr[j];
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < W; ++j) acc = fmaf(old[j], __ldg(p.w + (int64_t)c * KW + j), acc);
    acc = fmaf(xv, __ldg(p.w + (int64_t)c * KW + W), acc);
    y[e] = math::silu_f(acc);
#pragma unroll
    for (int j = 0; j + 1 < W; ++j) tr[j] = old[j + 1];  // new tail: old[1..W-1], x
    if (W > 0) tr[W - 1] = xv;
  }
  if (tid < ratio) {
    const int h = h0 + tid;
    const float av = ld_act<TA>(static_cast<const TA*>(p.a) + (int64_t)b * p.a_stride + h);
    const float bv = ld_act<TA>(static_cast<const TA*>(p.b) + (int64_t)b * p.b_stride + h);
    const float g = -expf(__ldg(p.A_log + h)) * math::softplus_f(av + __ldg(p.dt_bias + h));
    decay_s[tid] = expf(g);
    // [cpu_ops.cpp] GdnPackedDecodeKernel rounds beta through b's storage type
    // (nearest even), as the unfused path stores it; f32 keeps it exact.
    float beta = math::sigmoid_f(bv);
    if constexpr (std::is_same<TA, __nv_bfloat16>::value)
      beta = __bfloat162float(__float2bfloat16_rn(beta));
    beta_s[tid] = beta;
  }
  __syncthreads();
  if (tid < 64) {  // warp 0: |q|^2, warp 1: |k|^2
    const float* src = y + (tid >> 5) * DK;
    float ss = 0.0f;
    for (int d = tid & 31; d < DK; d += 32) ss = fmaf(src[d], src[d], ss);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if ((tid & 31) == 0) inv_s[tid >> 5] = p.norm ? rsqrtf(ss + 1e-6f) : 1.0f;
  }
  __syncthreads();

  // ---- phase 2: the value heads' rows ---------------------------------------
  float4 q4[4], k4[4];
  {
    const float qi = inv_s[0], ki = inv_s[1];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float* qs = y + 4 * lr + 4 * LPR * m;
      const float* ks = y + DK + 4 * lr + 4 * LPR * m;
      q4[m] = make_float4(qs[0] * qi, qs[1] * qi, qs[2] * qi, qs[3] * qi);
      k4[m] = make_float4(ks[0] * ki, ks[1] * ki, ks[2] * ki, ks[3] * ki);
    }
  }
  float kq = 0.0f;
#pragma unroll
  for (int m = 0; m < 4; ++m) kq += dot4(k4[m], q4[m]);
  kq = row_sum<LPR>(kq);

#pragma unroll 1
  for (int hh = 0; hh < ratio; ++hh) {
    float* S = p.pool + ((int64_t)slot * p.Hv + h0 + hh) * p.Dv * DK;
    if (hh > 0) load_state(hh);
    const float decay = decay_s[hh], beta = beta_s[hh];
    const float* v = y + 2 * DK + hh * p.Dv;
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = rg + ps * RPP;
      const float vv = r < p.Dv ? v[r] : 0.0f;
      const float o = row_step<LPR>(st[ps], k4, q4, kq, decay, beta, vv);
      if (r < p.Dv) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
          __stcs(reinterpret_cast<float4*>(S + (int64_t)r * DK + 4 * lr + 4 * LPR * m), st[ps][m]);
        if (lr == 0) st_act<TA>(out + hh * p.Dv + r, o * p.scale);
      }
    }
  }
}

template <typename TA, int DK, int KW>
cudaError_t launch_k(const PackedDecodeLaunch& p, cudaStream_t s) {
  const int ratio = p.Hv / p.Hk;
  const size_t smem = (size_t)(2 * DK + ratio * p.Dv + 2 * ratio + 2) * sizeof(float);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  const int64_t blocks = (int64_t)p.B * p.Hk;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  packed_decode_kernel<TA, DK, KW><<<(unsigned)blocks, kThreads, smem, s>>>(p);
  note_launch();
  return cudaGetLastError();
}

template <typename TA, int DK>
cudaError_t launch_dk(const PackedDecodeLaunch& p, cudaStream_t s) {
  switch (p.K) {
    case 2: return launch_k<TA, DK, 2>(p, s);
    case 3: return launch_k<TA, DK, 3>(p, s);
    case 4: return launch_k<TA, DK, 4>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename TA>
cudaError_t launch_dtype(const PackedDecodeLaunch& p, cudaStream_t s) {
  switch (p.Dk) {
    case 64: return launch_dk<TA, 64>(p, s);
    case 128: return launch_dk<TA, 128>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool packed_decode_supported(int Dk, int Dv, int K) {
  return (Dk == 64 || Dk == 128) && Dv >= 1 && Dv <= 128 && K >= 2 && K <= 4;
}

cudaError_t launch_packed_decode(const PackedDecodeLaunch& p, cudaStream_t s) {
  if (!packed_decode_supported(p.Dk, p.Dv, p.K) || p.Hk <= 0 || p.Hv % p.Hk != 0)
    return cudaErrorInvalidValue;
  return p.bf16 ? launch_dtype<__nv_bfloat16>(p, s) : launch_dtype<float>(p, s);
}

}  // namespace gdn
