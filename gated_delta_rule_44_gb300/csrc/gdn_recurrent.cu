// gdn_recurrent.cu -- the gated delta rule one token at a time, on CUDA cores.
//
// Defines: [cpu_ops.cpp] (vllm.cpp, src/vt/cpu/cpu_ops.cpp) GdnHeadTokenStep,
// GdnDecodeKernel and GdnPrefillKernel; [cpu.rs] (ferrum-kernels 0.8.0,
// src/ferrum_kernels/backend/cpu.rs) recurrent_gated_delta_rule_batch_f32 and
// recurrent_gated_delta_rule_varlen_f32.
//
// Per value head h and token, with S = [Dv, Dk] f32:
//   S *= exp(g);  u = beta (v - S k);  S += u k^T;  o = S (scale q)
// Row i of S evolves on its own given k, q, v_i: with a = S_i.k and b = S_i.q
// taken on the OLD row,
//   u_i = beta (v_i - e^g a),  S_i <- e^g S_i + u_i k,  o_i = scale (e^g b + u_i (k.q))
// which is the same update, so each row is read once and written once.
//
// Thread layout.  A row of Dk floats is split over LPR = Dk/16 lanes, each
// holding 16 floats as 4 float4 at columns 4*lr + 4*LPR*m (m = 0..3): one
// load instruction of a warp covers 32/LPR rows x 128 contiguous bytes.  The
// two dots are xor-shuffle reductions over the LPR lanes of a row.  A CTA of
// 128 threads holds PASSES x (128/LPR) rows of one (sequence, head).
//
// gdn_decode: one CTA per (row b, head, row slice); the state slice streams
// HBM -> registers -> HBM once (evict-first loads and stores).
// recurrent prefill: one CTA per (sequence, head, row slice) keeps its slice in
// registers across the sequence's tokens, prefetching the next token's q/k/v.
//
// Speculative decode ([cpu_ops.cpp] GdnSpecDecodeKernel): sequence s is a
// request whose draft tokens run from the slot of column num_accepted[s] - 1
// of its state_indices row; after token t the CTA stores its rows of S into
// the slot of column t - cu[s] (negative: no store).  The initial slot is not
// written back, so a request can later resume from any of its snapshots.
//
// KDA ([cpu_ops.cpp] KdaHeadTokenStep, KdaGatedDeltaRuleKernel): the decay is
// per key channel, e_d = exp(g[t, h, d]).  With a = S_i.(e k) and b = S_i.(e q)
// on the old row, u_i = beta (v_i - a), S_i <- e S_i + u_i k and
// o_i = scale (b + u_i (k.q)): the same single pass over the row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "gdn_math.cuh"
#include "gdn_rowstep.cuh"

namespace gdn {
namespace {

using namespace rows;

constexpr int kThreads = 128;

// The stored value of x: x rounded to the activation type.
template <typename TA>
__device__ __forceinline__ float round_act(float x);
template <>
__device__ __forceinline__ float round_act<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float round_act<__nv_bfloat16>(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// q and k columns of one lane (16 each), optionally L2-normalised, plus k.q.
template <typename TA, int DK>
struct QK {
  static constexpr int LPR = DK / 16;
  float4 k[4], q[4];
  float kq;
  __device__ __forceinline__ void load(const TA* kp, const TA* qp, int lr) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      k[m] = ld_act4<TA>(kp + 4 * lr + 4 * LPR * m);
      q[m] = ld_act4<TA>(qp + 4 * lr + 4 * LPR * m);
    }
  }
  __device__ __forceinline__ void finish(bool norm) {
    if (norm) {
      float kk = 0.f, qq = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        kk += dot4(k[m], k[m]);
        qq += dot4(q[m], q[m]);
      }
      kk = row_sum<LPR>(kk);
      qq = row_sum<LPR>(qq);
      const float ki = 1.0f / sqrtf(kk + 1e-6f), qi = 1.0f / sqrtf(qq + 1e-6f);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        k[m].x *= ki; k[m].y *= ki; k[m].z *= ki; k[m].w *= ki;
        q[m].x *= qi; q[m].y *= qi; q[m].z *= qi; q[m].w *= qi;
      }
    }
    float d = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) d += dot4(k[m], q[m]);
    kq = row_sum<LPR>(d);
  }
};

// The KDA row update: per-column decay e (the lane's 16 columns), ek = e k and
// eq = e q.  Returns o_i (before scale).
template <int LPR>
__device__ __forceinline__ float row_step_kda(float4 (&s)[4], const float4 (&e)[4],
                                              const float4 (&ek)[4], const float4 (&eq)[4],
                                              const float4 (&k)[4], float kq, float beta,
                                              float v) {
  float a = 0.f, b = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    a += dot4(s[m], ek[m]);
    b += dot4(s[m], eq[m]);
  }
  a = row_sum<LPR>(a);
  b = row_sum<LPR>(b);
  const float u = beta * (v - a);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    s[m].x = fmaf(e[m].x, s[m].x, u * k[m].x);
    s[m].y = fmaf(e[m].y, s[m].y, u * k[m].y);
    s[m].z = fmaf(e[m].z, s[m].z, u * k[m].z);
    s[m].w = fmaf(e[m].w, s[m].w, u * k[m].w);
  }
  return fmaf(u, kq, b);
}

__device__ __forceinline__ float4 exp4(const float4& g) {
  return make_float4(math::exp_ex2(g.x), math::exp_ex2(g.y), math::exp_ex2(g.z),
                     math::exp_ex2(g.w));
}
__device__ __forceinline__ float4 mul4(const float4& a, const float4& b) {
  return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
}

// ---------------------------------------------------------------------------
// Decode: grid.x = B * Hv * slices, one 128-thread CTA per value-dimension
// slice.  KDA: the one-token sequences of a KDA call (T == N), with the
// per-key-channel decay and has_initial_state.
// NS > 0: the gated RMSNorm of each output row is applied before the store.
// Then one CTA holds all slices of a (row, head), NS groups of 128 threads
// (NS = the slice count rounded up to a power of two, <= 4; groups past the
// last slice own no rows); the squares of the stored outputs are summed per
// warp and the warp sums added in order, so the whole row gets one norm.
// (NS > 0 caps the registers at 128 a thread, 512 threads an SM as the plain
// decode's four CTAs of 128: the state stream needs the warps in flight.)
template <typename TA, int DK, int PASSES, bool KDA, int NS>
__global__ void __launch_bounds__(kThreads * (NS > 0 ? NS : 1), 4 / (NS > 0 ? NS : 4))
    decode_kernel(const RecurLaunch p, int slices) {
  constexpr bool ONORM = NS > 0;
  constexpr int LPR = DK / 16;
  constexpr int RPP = kThreads / LPR;  // rows per pass
  const int tid = ONORM ? threadIdx.x % kThreads : threadIdx.x;
  const int lr = tid % LPR, rg = tid / LPR;
  const int slice = ONORM ? threadIdx.x / kThreads : blockIdx.x % slices;
  const int bh = ONORM ? blockIdx.x : blockIdx.x / slices;
  const int h = bh % p.Hv, b = bh / p.Hv;
  const int row0 = slice * (RPP * PASSES) + rg;
  TA* out = static_cast<TA*>(p.out) + ((int64_t)b * p.Hv + h) * p.Dv;

  if constexpr (KDA) {  // row b must be sequence b
    if (__ldg(p.cu + b) != b || __ldg(p.cu + b + 1) != b + 1) {
      if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
  }
  int slot = p.sidx != nullptr ? __ldg(p.sidx + b) : b;
  if (slot < -1 || slot >= p.slots) {
    if (tid == 0) atomicOr(p.status, kStatusBadIndex);
    slot = -1;
  }
  if (slot < 0) {  // padding row: zero output, state untouched
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = row0 + ps * RPP;
      if (lr == 0 && r < p.Dv) st_act<TA>(out + r, 0.0f);
    }
    return;
  }
  const int hk = h / (p.Hv / p.Hk);
  float* S = p.pool + ((int64_t)slot * p.Hv + h) * p.Dv * DK;

  const bool init = !KDA || p.has_init == nullptr || __ldg(p.has_init + b) != 0;
  // Issue every state load of the slice first (memory-level parallelism).
  float4 st[PASSES][4];
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    const int r = row0 + ps * RPP;
#pragma unroll
    for (int m = 0; m < 4; ++m)
      st[ps][m] = (init && r < p.Dv) ? __ldcs(reinterpret_cast<const float4*>(
                                           S + (int64_t)r * DK + 4 * lr + 4 * LPR * m))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // ONORM: the row's gate and weight values, requested with the state so that
  // their latency is not paid again after the reduction.
  float zv[ONORM ? PASSES : 1], wv[ONORM ? PASSES : 1];
  if constexpr (ONORM) {
    const TA* zr = static_cast<const TA*>(p.onorm_z) + (int64_t)b * p.onorm_z_stride +
                   (int64_t)h * p.Dv;
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = row0 + ps * RPP;
      const bool mine = lr == 0 && r < p.Dv;
      zv[ps] = mine ? ld_act<TA>(zr + r) : 0.0f;
      wv[ps] = mine ? ld_act<TA>(static_cast<const TA*>(p.onorm_w) + r) : 0.0f;
    }
  }
  QK<TA, DK> qk;
  const TA* kp = static_cast<const TA*>(p.k) + ((int64_t)b * p.Hk + hk) * DK;
  const TA* qp = static_cast<const TA*>(p.q) + ((int64_t)b * p.Hk + hk) * DK;
  qk.load(kp, qp, lr);
  qk.finish(p.norm);
  const float beta = __ldg(p.beta + (int64_t)b * p.Hv + h);
  const TA* vp = static_cast<const TA*>(p.v) + ((int64_t)b * p.Hv + h) * p.Dv;
  float decay = 0.0f;
  float4 e[KDA ? 4 : 1], ek[KDA ? 4 : 1], eq[KDA ? 4 : 1];
  if constexpr (KDA) {  // this lane's 16 columns of e^{g[b, h, :]}
    const float* gr = p.g + ((int64_t)b * p.Hv + h) * DK;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      e[m] = exp4(__ldg(reinterpret_cast<const float4*>(gr + 4 * lr + 4 * LPR * m)));
      ek[m] = mul4(e[m], qk.k[m]);
      eq[m] = mul4(e[m], qk.q[m]);
    }
  } else {
    decay = expf(__ldg(p.g + (int64_t)b * p.Hv + h));
  }

  float core[PASSES];  // ONORM: this row's output as stored, before the norm
  float ss = 0.0f;
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    const int r = row0 + ps * RPP;
    const float vv = r < p.Dv ? ld_act<TA>(vp + r) : 0.0f;
    float o;
    if constexpr (KDA)
      o = row_step_kda<LPR>(st[ps], e, ek, eq, qk.k, qk.kq, beta, vv);
    else
      o = row_step<LPR>(st[ps], qk.k, qk.q, qk.kq, decay, beta, vv);
    core[ps] = 0.0f;
    if (r < p.Dv) {
#pragma unroll
      for (int m = 0; m < 4; ++m)
        __stcs(reinterpret_cast<float4*>(S + (int64_t)r * DK + 4 * lr + 4 * LPR * m), st[ps][m]);
      if constexpr (ONORM) {
        core[ps] = round_act<TA>(o * p.scale);
        if (lr == 0) ss = fmaf(core[ps], core[ps], ss);
      } else {
        if (lr == 0) st_act<TA>(out + r, o * p.scale);
      }
    }
  }
  if constexpr (ONORM) {
    constexpr int kWarps = kThreads * (ONORM ? NS : 1) / 32;
    __shared__ float wpart[kWarps];
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if ((threadIdx.x & 31) == 0) wpart[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += wpart[w];
    const float inv = math::rms_inv(tot, 1.0f / static_cast<float>(p.Dv), p.onorm_eps);
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = row0 + ps * RPP;
      if (lr == 0 && r < p.Dv)
        st_act<TA>(out + r, core[ps] * inv * wv[ps] * math::norm_gate(zv[ps], p.onorm_sigmoid));
    }
  }
}

// ---------------------------------------------------------------------------
// Recurrent prefill: grid.x = N * Hv * slices; tokens of the sequence in order.
// SPEC: the speculative decode (per-token snapshots, see the file header).
template <typename TA, int DK, int PASSES, bool KDA, bool SPEC>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(const RecurLaunch p, int slices) {
  constexpr int LPR = DK / 16;
  constexpr int RPP = kThreads / LPR;
  const int tid = threadIdx.x;
  const int lr = tid % LPR, rg = tid / LPR;
  const int slice = blockIdx.x % slices;
  const int sh = blockIdx.x / slices;
  const int h = sh % p.Hv, s = sh / p.Hv;
  const int row0 = slice * (RPP * PASSES) + rg;

  const int t0 = __ldg(p.cu + s), t1 = __ldg(p.cu + s + 1);
  // a speculative request may be empty but holds at most num_cols tokens
  const bool bad_range = SPEC ? (t1 < t0 || t1 - t0 > p.num_cols) : t1 <= t0;
  if (__ldg(p.cu) != 0 || __ldg(p.cu + p.N) != p.T || t0 < 0 || bad_range || t1 > p.T) {
    if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }
  if (SPEC && t1 == t0) return;
  const int32_t* spec_row = SPEC ? p.sidx + (int64_t)s * p.num_cols : nullptr;
  int slot;
  if constexpr (SPEC) {
    const int accepted = __ldg(p.num_accepted + s);
    const bool ok = accepted >= 1 && accepted <= p.num_cols;
    slot = ok ? __ldg(spec_row + accepted - 1) : -1;
    if (!ok || slot >= p.slots) {
      if (tid == 0) atomicOr(p.status, kStatusBadIndex);
      slot = -1;
    }
  } else {
    slot = p.sidx != nullptr ? __ldg(p.sidx + s) : s;
    if (slot < -1 || slot >= p.slots) {
      if (tid == 0) atomicOr(p.status, kStatusBadIndex);
      slot = -1;
    }
  }
  if (slot < 0) {  // padded sequence: zero outputs, pool untouched
    for (int t = t0; t < t1; ++t) {
      TA* out = static_cast<TA*>(p.out) + ((int64_t)t * p.Hv + h) * p.Dv;
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        const int r = row0 + ps * RPP;
        if (lr == 0 && r < p.Dv) st_act<TA>(out + r, 0.0f);
      }
    }
    return;
  }
  const int hk = h / (p.Hv / p.Hk);
  float* S = p.pool + ((int64_t)slot * p.Hv + h) * p.Dv * DK;
  const bool init = SPEC || p.has_init == nullptr || __ldg(p.has_init + s) != 0;

  float4 st[PASSES][4];
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    const int r = row0 + ps * RPP;
#pragma unroll
    for (int m = 0; m < 4; ++m)
      st[ps][m] = (init && r < p.Dv)
                      ? *reinterpret_cast<const float4*>(S + (int64_t)r * DK + 4 * lr + 4 * LPR * m)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const TA* kbase = static_cast<const TA*>(p.k) + (int64_t)hk * DK;
  const TA* qbase = static_cast<const TA*>(p.q) + (int64_t)hk * DK;
  const TA* vbase = static_cast<const TA*>(p.v) + (int64_t)h * p.Dv;
  const int64_t qk_row = (int64_t)p.Hk * DK, v_row = (int64_t)p.Hv * p.Dv;

  // Software pipeline: operands of token t+1 load while token t computes.
  QK<TA, DK> cur, nxt;
  float v_cur[PASSES], v_nxt[PASSES];
  float g_cur, b_cur, g_nxt = 0.f, b_nxt = 0.f;
  // KDA: this lane's 16 log decays of the token (g [T, Hv, Dk]).
  float4 gk_cur[KDA ? 4 : 1], gk_nxt[KDA ? 4 : 1];
  auto load_gk = [&](int t, float4 (&dst)[KDA ? 4 : 1]) {
    if constexpr (KDA) {
      const float* gr = p.g + ((int64_t)t * p.Hv + h) * DK;
#pragma unroll
      for (int m = 0; m < 4; ++m) dst[m] = __ldg(reinterpret_cast<const float4*>(gr + 4 * lr + 4 * LPR * m));
    }
  };
  cur.load(kbase + (int64_t)t0 * qk_row, qbase + (int64_t)t0 * qk_row, lr);
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    const int r = row0 + ps * RPP;
    v_cur[ps] = r < p.Dv ? ld_act<TA>(vbase + (int64_t)t0 * v_row + r) : 0.f;
  }
  if constexpr (KDA) {
    load_gk(t0, gk_cur);
    g_cur = 0.f;
  } else {
    g_cur = __ldg(p.g + (int64_t)t0 * p.Hv + h);
  }
  b_cur = __ldg(p.beta + (int64_t)t0 * p.Hv + h);

  // A speculative request has a few tokens only: it loads each token's
  // operands after the previous token instead of keeping a second set in
  // registers, which leaves room for a fourth CTA per SM.
  for (int t = t0; t < t1; ++t) {
    if (!SPEC && t + 1 < t1) {
      nxt.load(kbase + (int64_t)(t + 1) * qk_row, qbase + (int64_t)(t + 1) * qk_row, lr);
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        const int r = row0 + ps * RPP;
        v_nxt[ps] = r < p.Dv ? ld_act<TA>(vbase + (int64_t)(t + 1) * v_row + r) : 0.f;
      }
      if constexpr (KDA)
        load_gk(t + 1, gk_nxt);
      else
        g_nxt = __ldg(p.g + (int64_t)(t + 1) * p.Hv + h);
      b_nxt = __ldg(p.beta + (int64_t)(t + 1) * p.Hv + h);
    }
    cur.finish(p.norm);
    TA* out = static_cast<TA*>(p.out) + ((int64_t)t * p.Hv + h) * p.Dv;
    if constexpr (KDA) {
      float4 e[4], ek[4], eq[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        e[m] = exp4(gk_cur[m]);
        ek[m] = mul4(e[m], cur.k[m]);
        eq[m] = mul4(e[m], cur.q[m]);
      }
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        const int r = row0 + ps * RPP;
        const float o = row_step_kda<LPR>(st[ps], e, ek, eq, cur.k, cur.kq, b_cur, v_cur[ps]);
        if (lr == 0 && r < p.Dv) st_act<TA>(out + r, o * p.scale);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) gk_cur[m] = gk_nxt[m];
    } else {
      const float decay = expf(g_cur);
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        const int r = row0 + ps * RPP;
        const float o = row_step<LPR>(st[ps], cur.k, cur.q, cur.kq, decay, b_cur, v_cur[ps]);
        if (lr == 0 && r < p.Dv) st_act<TA>(out + r, o * p.scale);
      }
      g_cur = g_nxt;
    }
    if constexpr (SPEC) {  // snapshot after token t
      int snap = __ldg(spec_row + (t - t0));
      if (snap >= p.slots) {
        if (tid == 0) atomicOr(p.status, kStatusBadIndex);
        snap = -1;
      }
      if (snap >= 0) {
        float* D = p.pool + ((int64_t)snap * p.Hv + h) * p.Dv * DK;
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
          const int r = row0 + ps * RPP;
          if (r < p.Dv)
#pragma unroll
            for (int m = 0; m < 4; ++m)
              __stcs(reinterpret_cast<float4*>(D + (int64_t)r * DK + 4 * lr + 4 * LPR * m),
                     st[ps][m]);
        }
      }
    }
    if constexpr (SPEC) {
      if (t + 1 < t1) {
        cur.load(kbase + (int64_t)(t + 1) * qk_row, qbase + (int64_t)(t + 1) * qk_row, lr);
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
          const int r = row0 + ps * RPP;
          v_cur[ps] = r < p.Dv ? ld_act<TA>(vbase + (int64_t)(t + 1) * v_row + r) : 0.f;
        }
        g_cur = __ldg(p.g + (int64_t)(t + 1) * p.Hv + h);
        b_cur = __ldg(p.beta + (int64_t)(t + 1) * p.Hv + h);
      }
    } else {
      cur = nxt;
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) v_cur[ps] = v_nxt[ps];
      b_cur = b_nxt;
    }
  }

  if constexpr (!SPEC) {
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = row0 + ps * RPP;
      if (r < p.Dv)
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *reinterpret_cast<float4*>(S + (int64_t)r * DK + 4 * lr + 4 * LPR * m) = st[ps][m];
    }
  }
}

enum class Mode { kDecode, kRecurrent, kKda, kKdaDecode, kSpec };

// Slices of one row in one CTA (512 threads: 128 registers a thread, as the
// plain decode; wider rows take the norm kernel after the decode).
constexpr int kMaxNormSlices = 4;

// Rows of the value dimension one CTA holds: PASSES chosen so that a CTA
// holds 64 rows at Dk = 128 (32 floats of state per thread).
constexpr int passes_for(int dk) { return dk <= 32 ? 1 : dk == 64 ? 2 : 4; }
constexpr int rows_per_cta_for(int dk) { return (kThreads / (dk / 16)) * passes_for(dk); }

template <typename TA, int DK, int PASSES>
cudaError_t launch_dk(const RecurLaunch& p, cudaStream_t s, Mode mode) {
  constexpr int rows_per_cta = (kThreads / (DK / 16)) * PASSES;
  static_assert(rows_per_cta == rows_per_cta_for(DK), "one place for the slice rule");
  const int slices = (p.Dv + rows_per_cta - 1) / rows_per_cta;
  const bool per_row = mode == Mode::kDecode || mode == Mode::kKdaDecode;
  const int64_t blocks = (int64_t)(per_row ? p.T : p.N) * p.Hv * slices;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const unsigned grid = (unsigned)blocks;
  switch (mode) {
    case Mode::kDecode:
      if (p.onorm_w != nullptr) {  // one CTA per (row, head) holding all its slices
        const unsigned rows = static_cast<unsigned>(grid / slices);
        if (slices == 1)
          decode_kernel<TA, DK, PASSES, false, 1><<<rows, kThreads, 0, s>>>(p, slices);
        else if (slices == 2)
          decode_kernel<TA, DK, PASSES, false, 2><<<rows, 2 * kThreads, 0, s>>>(p, slices);
        else if (slices <= kMaxNormSlices)
          decode_kernel<TA, DK, PASSES, false, 4><<<rows, 4 * kThreads, 0, s>>>(p, slices);
        else
          return cudaErrorInvalidConfiguration;
        break;
      }
      decode_kernel<TA, DK, PASSES, false, 0><<<grid, kThreads, 0, s>>>(p, slices);
      break;
    case Mode::kKdaDecode:
      decode_kernel<TA, DK, PASSES, true, 0><<<grid, kThreads, 0, s>>>(p, slices);
      break;
    case Mode::kRecurrent:
      recurrent_kernel<TA, DK, PASSES, false, false><<<grid, kThreads, 0, s>>>(p, slices);
      break;
    case Mode::kKda:
      recurrent_kernel<TA, DK, PASSES, true, false><<<grid, kThreads, 0, s>>>(p, slices);
      break;
    case Mode::kSpec:
      recurrent_kernel<TA, DK, PASSES, false, true><<<grid, kThreads, 0, s>>>(p, slices);
      break;
  }
  note_launch();
  return cudaGetLastError();
}

// PASSES chosen so a CTA holds 64 rows (32 floats of state per thread at
// Dk = 128); decode issues all of them before the first use.
template <typename TA>
cudaError_t launch_any(const RecurLaunch& p, cudaStream_t s, Mode mode) {
  switch (p.Dk) {
    case 16: return launch_dk<TA, 16, 1>(p, s, mode);
    case 32: return launch_dk<TA, 32, 1>(p, s, mode);
    case 64: return launch_dk<TA, 64, 2>(p, s, mode);
    case 128: return launch_dk<TA, 128, 4>(p, s, mode);
    case 256: return launch_dk<TA, 256, 4>(p, s, mode);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool recurrent_supported(int Dk) {
  return Dk == 16 || Dk == 32 || Dk == 64 || Dk == 128 || Dk == 256;
}

bool decode_norm_in_kernel(int Dk, int Dv) {
  if (!recurrent_supported(Dk) || Dv < 1) return false;
  const int rows = rows_per_cta_for(Dk);
  return (Dv + rows - 1) / rows <= kMaxNormSlices;
}

static cudaError_t launch_mode(const RecurLaunch& p, cudaStream_t s, Mode mode) {
  return p.bf16 ? launch_any<__nv_bfloat16>(p, s, mode) : launch_any<float>(p, s, mode);
}

cudaError_t launch_decode(const RecurLaunch& p, cudaStream_t s) {
  return launch_mode(p, s, Mode::kDecode);
}

cudaError_t launch_recurrent(const RecurLaunch& p, cudaStream_t s) {
  return launch_mode(p, s, Mode::kRecurrent);
}

cudaError_t launch_kda(const RecurLaunch& p, cudaStream_t s) {
  if (p.norm) return cudaErrorInvalidValue;
  // T == N: every sequence holds exactly one token (cu_seqlens must be 0..N,
  // which the decode form checks on the device), so run the decode form.
  return launch_mode(p, s, p.T == p.N ? Mode::kKdaDecode : Mode::kKda);
}

cudaError_t launch_spec_decode(const RecurLaunch& p, cudaStream_t s) {
  if (p.norm || p.sidx == nullptr || p.num_accepted == nullptr || p.num_cols < 1)
    return cudaErrorInvalidValue;
  return launch_mode(p, s, Mode::kSpec);
}

}  // namespace gdn
