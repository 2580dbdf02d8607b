// gdn_prepare.cu -- fused prepare kernel: causal depthwise conv1d + SiLU +
// q/k/v split + q/k L2 norm + gates, with the conv tail carried in a slot pool.
//
// Defines: [cpu.rs] (ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs)
// linear_attention_prepare_varlen_f32 and linear_attention_decode_prepare_
// batch_f32; [cpu_ops.cpp] (vllm.cpp, src/vt/cpu/cpu_ops.cpp)
// CausalConv1dFwdKernel, CausalConv1dUpdateKernel, CausalConv1dSpecUpdateKernel
// and GdnPostConvKernel.
//
// Work decomposition.  A thread owns one 16-byte vector of channels (8 bf16 or
// 4 f32) and walks the tokens of a tile in order, keeping the last K-1 raw
// inputs of its channels in registers (the conv window).  A warp therefore
// reads 512 contiguous bytes of a token row per step; a CTA of 4 warps covers
// 2 KB of the row.  grid.x = channel blocks (+1 for the gates), grid.y = token
// tiles of `tile` tokens.  The L2 norm of a key head (Dk channels =
// Dk/8 lanes) is a shuffle reduction inside the warp.
//
// Conv-tail ownership.  The old tail of a sequence is read by the outputs of
// its first K-1 tokens, and the new tail replaces it in place.  Both are done
// by the tile that holds the sequence's first token: it also computes the
// first K-1 tokens of the sequence when they spill past its end, and the next
// tile skips them.  So no tail is written while another CTA may still read it,
// and no grid-wide synchronisation is needed (tile >= K-1).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "gdn_math.cuh"

namespace gdn {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

using math::sigmoid_f;
using math::silu_f;
using math::softplus_f;

template <typename TA>
struct Act;

template <>
struct Act<float> {
  static constexpr int kVec = 4;  // channels per 16-byte vector
  __device__ static void load(const float* p, float (&o)[4]) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    o[0] = v.x;
    o[1] = v.y;
    o[2] = v.z;
    o[3] = v.w;
  }
  __device__ static void store(float* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
  __device__ static float scalar(const float* p) { return __ldg(p); }
  __device__ static uint4 load_raw(const float* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ static void unpack(const uint4& v, float (&o)[4]) {
    o[0] = __uint_as_float(v.x);
    o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z);
    o[3] = __uint_as_float(v.w);
  }
};

template <>
struct Act<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&o)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static float scalar(const __nv_bfloat16* p) { return __bfloat162float(p[0]); }
  __device__ static uint4 load_raw(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
  }
  __device__ static void unpack(const uint4& v, float (&o)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

// silu of two values with paired f32 arithmetic (the prepare's hot loop):
// e^{-x} as 2^{-x log2(e)} on the hardware's approximate base-2 exponential,
// capped at e^80 as in silu_f, then x / (1 + e^{-x}) on the refined reciprocal.
__device__ __forceinline__ float2 silu2(float2 x) {
  constexpr float kNegLog2e = -1.4426950408889634f;
  constexpr float kCap = 80.0f * 1.4426950408889634f;
  const float2 m = __fmul2_rn(x, make_float2(kNegLog2e, kNegLog2e));
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
  return __fmul2_rn(x, r);
}

// conv + SiLU of one token's V channels from its window (win[j] = the input
// W - j tokens back, oldest first) and its own input xt, with channel pairs in
// paired f32 arithmetic; returns the sum of the squares of y (even and odd
// channels summed apart, then added).  The conv of each channel is the same
// chain of fused multiply-adds, oldest tap first, as a scalar loop.
template <int V, int KW, int WV>
__device__ __forceinline__ float conv_silu_row(const float (&win)[WV][V], const float (&xt)[V],
                                               const float (&wt)[V][KW], float (&y)[V]) {
  constexpr int W = KW - 1;
  float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < V; i += 2) {
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < W; ++j)
      acc = __ffma2_rn(make_float2(win[j][i], win[j][i + 1]), make_float2(wt[i][j], wt[i + 1][j]), acc);
    acc = __ffma2_rn(make_float2(xt[i], xt[i + 1]), make_float2(wt[i][W], wt[i + 1][W]), acc);
    const float2 yy = silu2(acc);
    y[i] = yy.x;
    y[i + 1] = yy.y;
    ss2 = __ffma2_rn(yy, yy, ss2);
  }
  return ss2.x + ss2.y;
}

// Largest s in [0, n) with cu[s] <= t (cu assumed non-decreasing; callers
// re-check the bracket, so a malformed cu only yields a bounded wrong guess).
// A 32-way search by the whole warp: each round the lanes read 32 evenly
// spaced entries of the remaining range and keep the span after the last one
// <= t, so n = 1024 takes two dependent reads.  Called by every lane.
__device__ __forceinline__ int find_seq(const int32_t* __restrict__ cu, int n, int t, int lane) {
  int lo = 0, len = n;
  while (len > 1) {
    const int step = (len + 31) >> 5;
    const int idx = lo + lane * step;
    const bool le = lane * step < len && __ldg(cu + idx) <= t;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    const int last = m != 0u ? 31 - __clz(static_cast<int>(m)) : 0;
    lo += last * step;
    len = min(step, len - last * step);
  }
  return lo;
}

template <typename TA, int KW>
__global__ void __launch_bounds__(kThreads, 4) prepare_kernel(const PrepareLaunch p, int tile,
                                                              int chan_blocks, bool tiles_on_y) {
  // blockIdx.x runs over the channel blocks (and the gate block), blockIdx.y
  // over the tiles: the hardware hands out CTAs with x fastest, so every
  // channel block of a tile goes out before the next tile (the one-token
  // sequences, which take longest, come first in a mixed batch).  Above
  // 65535 tiles the two swap.
  const int tile_idx = tiles_on_y ? blockIdx.y : blockIdx.x;
  const int cblk = tiles_on_y ? blockIdx.x : blockIdx.y;
  constexpr int V = Act<TA>::kVec;
  constexpr int W = KW - 1;  // conv tail length
  constexpr int WV = W > 0 ? W : 1;
  const int qk_total = p.Hk * p.Dk;
  const int C = 2 * qk_total + p.Hv * p.Dv;
  const int t_begin = tile_idx * tile;
  const int t_end = min(p.T, t_begin + tile);
  const TA* __restrict__ x = static_cast<const TA*>(p.x);

  if (cblk == chan_blocks) {  // gates: g, beta per (token, value head)
    const TA* __restrict__ a = static_cast<const TA*>(p.a);
    const TA* __restrict__ b = static_cast<const TA*>(p.b);
    const int n = (t_end - t_begin) * p.Hv;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const int t = t_begin + i / p.Hv, h = i % p.Hv;
      const float av = Act<TA>::scalar(a + (int64_t)t * p.a_stride + h);
      const float bv = Act<TA>::scalar(b + (int64_t)t * p.b_stride + h);
      p.g[(int64_t)t * p.Hv + h] = -expf(__ldg(p.A_log + h)) * softplus_f(av + __ldg(p.dt_bias + h));
      p.beta[(int64_t)t * p.Hv + h] = sigmoid_f(bv);
    }
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Stream this CTA's rows (the tile and the W rows before it, its channel
  // block) into L2 up front, one bulk prefetch per row: the per-thread loads
  // below then wait on L2 rather than on HBM, without holding registers.
  {
    const int cb = cblk * kThreads * V;
    const int bytes = min(kThreads * V, C - cb) * static_cast<int>(sizeof(TA));
    const int r = t_begin - W + static_cast<int>(threadIdx.x);
    if (r >= 0 && r < t_end && bytes > 0)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(x + (int64_t)r * p.x_stride + cb),
                   "r"(bytes)
                   : "memory");
  }
  const int c0 = ((cblk * kWarps + warp) * 32 + lane) * V;
  const bool active = c0 < C;
  const bool is_qk = c0 < 2 * qk_total;
  const int group = p.Dk / V;  // lanes per key head (power of two <= 32)
  constexpr int kG = 4;  // interior tiles: rows per group (their norms share shuffle rounds)

  // Loads that need nothing but the tile go out before anything waits: the
  // bounds of cu_seqlens, the W rows before the tile and its first kG rows (what
  // an interior tile reads first; other tiles drop them) and the conv weights
  // (V * KW consecutive floats, 16-byte aligned).
  const int cu_first = __ldg(p.cu), cu_last = __ldg(p.cu + p.N);
  const TA* xrow = x + (int64_t)t_begin * p.x_stride + c0;
  const bool spec = active && t_begin >= W;
  uint4 pre_w[WV], pre_x[kG];
#pragma unroll
  for (int j = 0; j < WV; ++j)
    pre_w[j] = (spec && j < W) ? Act<TA>::load_raw(xrow - (int64_t)(W - j) * p.x_stride)
                               : make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int u = 0; u < kG; ++u)
    pre_x[u] = (spec && t_begin + u < t_end) ? Act<TA>::load_raw(xrow + (int64_t)u * p.x_stride)
                                             : make_uint4(0, 0, 0, 0);
  float wt[V][KW];
  {
    static_assert((V * KW) % 4 == 0, "weights as float4");
    float wf[V * KW];
    const float4* wsrc = reinterpret_cast<const float4*>(p.w + (int64_t)c0 * KW);
#pragma unroll
    for (int q4 = 0; q4 < V * KW / 4; ++q4) {
      const float4 f = active ? __ldg(wsrc + q4) : make_float4(0.f, 0.f, 0.f, 0.f);
      wf[4 * q4] = f.x;
      wf[4 * q4 + 1] = f.y;
      wf[4 * q4 + 2] = f.z;
      wf[4 * q4 + 3] = f.w;
    }
#pragma unroll
    for (int i = 0; i < V; ++i)
#pragma unroll
      for (int j = 0; j < KW; ++j) wt[i][j] = wf[i * KW + j];
  }

  TA* __restrict__ out_ptr;  // row base of this thread's output vector
  int64_t out_stride;
  if (c0 < qk_total) {
    out_ptr = static_cast<TA*>(p.q) + c0;
    out_stride = qk_total;
  } else if (c0 < 2 * qk_total) {
    out_ptr = static_cast<TA*>(p.k) + (c0 - qk_total);
    out_stride = qk_total;
  } else {
    out_ptr = static_cast<TA*>(p.v) + (c0 - 2 * qk_total);
    out_stride = (int64_t)p.Hv * p.Dv;
  }

  // conv + SiLU + (norm) + store of token t, given its window (oldest first)
  // and its own input.  Uniform across the warp: every lane joins the shuffles.
  auto emit = [&](int t, const float (&win)[WV][V], const float (&xt)[V]) {
    float y[V];
    float ss = conv_silu_row<V, KW, WV>(win, xt, wt, y);
    if (p.norm) {
      for (int m = 1; m < group; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      if (is_qk) {
        const float inv = rsqrtf(ss + 1e-6f);
#pragma unroll
        for (int i = 0; i < V; ++i) y[i] *= inv;
      }
    }
    if (active) Act<TA>::store(out_ptr + (int64_t)t * out_stride, y);
  };

  // Sequence bracket of the tile's first token.
  int s = find_seq(p.cu, p.N, t_begin, lane);
  int seq_lo = __ldg(p.cu + s), seq_hi = __ldg(p.cu + s + 1);
  if (cu_first != 0 || cu_last != p.T || !(seq_lo <= t_begin && t_begin < seq_hi) ||
      seq_lo < 0 || seq_hi > p.T) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }

  // ---- interior tile: every token's window lies inside one sequence --------------
  // Groups of kG rows: the next group's loads are issued as this group's rows
  // are consumed; the L2 norms of a group's kG tokens share their shuffle
  // rounds.  The shuffles run on every warp that holds a q or k channel (a
  // warp-uniform test: with 2*Hk*Dk below a multiple of the warp's channels a
  // warp holds k and v lanes), and the scaling on q and k lanes only; warps of
  // v channels alone skip both.
  if (seq_lo + W <= t_begin && t_end <= seq_hi) {  // here t_begin >= W: the early loads hold
    const int n = t_end - t_begin;
    const bool norm_warp = p.norm && (c0 - lane * V) < 2 * qk_total;  // lane 0's channel
    float win[WV][V];
#pragma unroll
    for (int j = 0; j < W; ++j) Act<TA>::unpack(pre_w[j], win[j]);
    uint4 nxt[kG];
#pragma unroll
    for (int u = 0; u < kG; ++u) nxt[u] = pre_x[u];
#pragma unroll 1
    for (int r0 = 0; r0 < n; r0 += kG) {
      float y[kG][V];
      float ss[kG];
#pragma unroll
      for (int u = 0; u < kG; ++u) {
        float xt[V];
        Act<TA>::unpack(nxt[u], xt);
        const int r = r0 + kG + u;
        nxt[u] = (active && r < n) ? Act<TA>::load_raw(xrow + (int64_t)r * p.x_stride)
                                   : make_uint4(0, 0, 0, 0);
        ss[u] = conv_silu_row<V, KW, WV>(win, xt, wt, y[u]);
#pragma unroll
        for (int j = 0; j + 1 < W; ++j)
#pragma unroll
          for (int i = 0; i < V; ++i) win[j][i] = win[j + 1][i];
        if (W > 0)
#pragma unroll
          for (int i = 0; i < V; ++i) win[WV - 1][i] = xt[i];
      }
      if (norm_warp) {
        for (int m = 1; m < group; m <<= 1)
#pragma unroll
          for (int u = 0; u < kG; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], m);
        if (is_qk)
#pragma unroll
          for (int u = 0; u < kG; ++u) {
            const float inv = rsqrtf(ss[u] + 1e-6f);
#pragma unroll
            for (int i = 0; i < V; ++i) y[u][i] *= inv;
          }
      }
#pragma unroll
      for (int u = 0; u < kG; ++u)
        if (active && r0 + u < n) Act<TA>::store(out_ptr + (int64_t)(t_begin + r0 + u) * out_stride, y[u]);
    }
    return;
  }

  // Resolves the pool slot of sequence sq (bad index -> reported, treated as padding).
  auto slot_of = [&](int sq) {
    int slot = p.sidx != nullptr ? __ldg(p.sidx + sq) : sq;
    if (slot < -1 || slot >= p.slots) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatusBadIndex);
      slot = -1;
    }
    return slot;
  };

  // ---- decode tile: every token is a sequence of length one ----------------------
  {
    const int n = t_end - t_begin;
    bool one = true;
    if (seq_lo != t_begin) {
      one = false;
    } else if (lane < n) {
      one = s + lane < p.N && __ldg(p.cu + s + lane + 1) == t_begin + lane + 1;
    }
    if (__all_sync(0xffffffffu, one) && W > 0) {
      // The slot and has_init of row i, read once by lane i of every warp (n <= 32).
      int my_slot = -1;
      bool my_init = false;
      if (lane < n) {
        my_slot = p.sidx != nullptr ? __ldg(p.sidx + s + lane) : s + lane;
        if (my_slot < -1 || my_slot >= p.slots) {
          atomicOr(p.status, kStatusBadIndex);
          my_slot = -1;
        }
        my_init = my_slot >= 0 && (p.has_init == nullptr || __ldg(p.has_init + s + lane) != 0);
      }
      constexpr int kBatch = 2;
      for (int b0 = 0; b0 < n; b0 += kBatch) {
        float tails[kBatch][WV][V];
        uint4 xr[kBatch];
        float* tp[kBatch];
#pragma unroll
        for (int bi = 0; bi < kBatch; ++bi) {
          const int i = b0 + bi;
          tp[bi] = nullptr;
          xr[bi] = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int j = 0; j < W; ++j)
#pragma unroll
            for (int e = 0; e < V; ++e) tails[bi][j][e] = 0.0f;
          const int slot = __shfl_sync(0xffffffffu, my_slot, i & 31);
          const bool init = __shfl_sync(0xffffffffu, my_init ? 1 : 0, i & 31) != 0;
          if (i < n) {
            if (slot >= 0 && active) tp[bi] = p.conv_pool + ((int64_t)slot * C + c0) * W;
            if (active) xr[bi] = Act<TA>::load_raw(x + (int64_t)(t_begin + i) * p.x_stride + c0);
            if (init && active) {
              // V*W consecutive floats, channel-major: element (e, j) at e*W + j.
              const float4* src = reinterpret_cast<const float4*>(tp[bi]);
#pragma unroll
              for (int q4 = 0; q4 < V * W / 4; ++q4) {
                const float4 f = src[q4];
                const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int idx = q4 * 4 + u;
                  tails[bi][idx % WV][idx / WV] = fv[u];
                }
              }
            }
          }
        }
#pragma unroll
        for (int bi = 0; bi < kBatch; ++bi) {
          const int i = b0 + bi;
          if (i < n) {
            float xt[V];
            Act<TA>::unpack(xr[bi], xt);
            emit(t_begin + i, tails[bi], xt);
            if (tp[bi] != nullptr) {  // new tail: old[1..W-1], x
              float nt[V * WV];
#pragma unroll
              for (int e = 0; e < V; ++e) {
#pragma unroll
                for (int j = 0; j + 1 < W; ++j) nt[e * W + j] = tails[bi][j + 1][e];
                nt[e * W + W - 1] = xt[e];
              }
              float4* dst = reinterpret_cast<float4*>(tp[bi]);
#pragma unroll
              for (int q4 = 0; q4 < V * W / 4; ++q4)
                dst[q4] = make_float4(nt[4 * q4], nt[4 * q4 + 1], nt[4 * q4 + 2], nt[4 * q4 + 3]);
            }
          }
        }
      }
      return;
    }
  }

  // ---- general tile: sequence starts, tails, short sequences --------------------
  float win[WV][V];  // win[j] = input at token t - W + j
#pragma unroll
  for (int j = 0; j < WV; ++j)
#pragma unroll
    for (int i = 0; i < V; ++i) win[j][i] = 0.0f;

  // Starts sequence s at its first token: loads the old tail into the window
  // and writes the new tail (last W raw inputs of tail || x) to the slot.
  auto begin_sequence = [&]() {
    const int slot = slot_of(s);
    const bool live = slot >= 0;
    const bool init = live && (p.has_init == nullptr || __ldg(p.has_init + s) != 0);
    float* tail = live ? p.conv_pool + ((int64_t)slot * C + c0) * W : nullptr;
#pragma unroll
    for (int j = 0; j < W; ++j)
#pragma unroll
      for (int i = 0; i < V; ++i) win[j][i] = (init && active) ? tail[i * W + j] : 0.0f;
    if (live && active) {
      const int len = seq_hi - seq_lo;
#pragma unroll
      for (int pos = 0; pos < W; ++pos) {
        const int src = len + pos - W;  // token index inside the sequence
        float nv[V];
        if (src >= 0) {
          Act<TA>::load(x + (int64_t)(seq_lo + src) * p.x_stride + c0, nv);
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) {
            float o = 0.0f;
#pragma unroll
            for (int j = 0; j < W; ++j) o = (j == W + src) ? win[j][i] : o;
            nv[i] = o;
          }
        }
#pragma unroll
        for (int i = 0; i < V; ++i) tail[i * W + pos] = nv[i];
      }
    }
  };

  int t = t_begin;
  if (t > seq_lo && t < seq_lo + W) t = min(seq_lo + W, seq_hi);  // owned by the previous tile
  if (t == seq_lo) {
    begin_sequence();
  } else if (t < seq_hi) {  // mid-sequence: the window comes from earlier raw inputs
#pragma unroll
    for (int j = 0; j < W; ++j)
      if (active) Act<TA>::load(x + (int64_t)(t - W + j) * p.x_stride + c0, win[j]);
  }

  for (;;) {
    if (t == seq_hi) {  // sequence s is finished
      if (t >= t_end || s + 1 >= p.N) break;
      ++s;
      seq_lo = seq_hi;
      seq_hi = __ldg(p.cu + s + 1);
      if (seq_hi <= seq_lo || seq_hi > p.T) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeqlens);
        break;
      }
      begin_sequence();
    }
    if (t >= t_end && t >= seq_lo + W) break;

    float xt[V];
    if (active) {
      Act<TA>::load(x + (int64_t)t * p.x_stride + c0, xt);
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) xt[i] = 0.0f;
    }
    emit(t, win, xt);
#pragma unroll
    for (int j = 0; j + 1 < W; ++j)
#pragma unroll
      for (int i = 0; i < V; ++i) win[j][i] = win[j + 1][i];
    if (W > 0)
#pragma unroll
      for (int i = 0; i < V; ++i) win[W - 1][i] = xt[i];
    ++t;
  }
}

// ---------------------------------------------------------------------------
// Speculative prepare ([cpu_ops.cpp] CausalConv1dSpecUpdateKernel, then the
// split, norm and gates above).  grid = (requests, channel blocks + 1).
// Request i's conv row holds state_len raw inputs per channel; the window
// before its first draft is row[off .. off+W-1], off = num_accepted[i] - 1,
// and the row becomes row[off+1 .. off+keep] || drafts (keep = state_len -
// drafts; entries past the row read 0).
//
// The CTA's rows (its channels x state_len floats, channel-major in HBM) are
// staged in shared memory transposed -- entry j of channel c at
// rows[j * kPitch + c] -- with coalesced 16-byte loads and stores, so that
// each thread reads and rewrites its V channels' entry j as 16-byte vectors.
// The pitch is padded by 4 floats to spread the transposing accesses over the
// banks.  A thread only touches its own columns between the two barriers,
// and the in-place shift walks j upwards (it reads entry off+1+j > j).
template <typename TA, int KW>
__global__ void __launch_bounds__(kThreads) spec_prepare_kernel(const PrepareLaunch p,
                                                                int chan_blocks) {
  constexpr int V = Act<TA>::kVec;
  constexpr int W = KW - 1;
  static_assert(W >= 1, "the speculative conv row needs a tail");
  constexpr int kPitch = kThreads * V + 4;
  extern __shared__ float4 rows4[];
  float* rows = reinterpret_cast<float*>(rows4);
  const int SL = p.state_len, max_q = SL - W + 1;
  const int qk_total = p.Hk * p.Dk;
  const int C = 2 * qk_total + p.Hv * p.Dv;
  const int req = blockIdx.x;
  const bool gate_block = blockIdx.y == chan_blocks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cb = blockIdx.y * kThreads * V;
  const int col = (warp * 32 + lane) * V;  // this thread's first column in the block
  const int c0 = cb + col;
  const bool active = !gate_block && c0 < C;
  // Everything that needs only the request and the channel block is read
  // before anything waits: cu_seqlens, the slot, the accepted count and the
  // conv weights; the request's inputs and conv row follow in one more trip.
  const int lo = __ldg(p.cu + req), hi = __ldg(p.cu + req + 1);
  const int cu_first = __ldg(p.cu), cu_last = __ldg(p.cu + p.N);
  const int slot_in = gate_block ? -1 : __ldg(p.sidx + req);
  const int accepted = gate_block ? 1 : __ldg(p.num_accepted + req);
  float wt[V][KW];
  {
    static_assert((V * KW) % 4 == 0, "weights as float4");
    float wf[V * KW];
    const float4* wsrc = reinterpret_cast<const float4*>(p.w + (int64_t)c0 * KW);
#pragma unroll
    for (int q4 = 0; q4 < V * KW / 4; ++q4) {
      const float4 f = active ? __ldg(wsrc + q4) : make_float4(0.f, 0.f, 0.f, 0.f);
      wf[4 * q4] = f.x;
      wf[4 * q4 + 1] = f.y;
      wf[4 * q4 + 2] = f.z;
      wf[4 * q4 + 3] = f.w;
    }
#pragma unroll
    for (int e = 0; e < V; ++e)
#pragma unroll
      for (int j = 0; j < KW; ++j) wt[e][j] = wf[e * KW + j];
  }
  if (cu_first != 0 || cu_last != p.T || lo < 0 || hi < lo || hi > p.T || hi - lo > max_q) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }
  const int len = hi - lo;
  if (len == 0) return;  // an empty request reads and writes nothing

  if (gate_block) {  // gates: g, beta per (token, value head)
    const TA* __restrict__ a = static_cast<const TA*>(p.a);
    const TA* __restrict__ b = static_cast<const TA*>(p.b);
    for (int e = threadIdx.x; e < len * p.Hv; e += kThreads) {
      const int t = lo + e / p.Hv, h = e % p.Hv;
      const float av = Act<TA>::scalar(a + (int64_t)t * p.a_stride + h);
      const float bv = Act<TA>::scalar(b + (int64_t)t * p.b_stride + h);
      p.g[(int64_t)t * p.Hv + h] = -expf(__ldg(p.A_log + h)) * softplus_f(av + __ldg(p.dt_bias + h));
      p.beta[(int64_t)t * p.Hv + h] = sigmoid_f(bv);
    }
    return;
  }

  int slot = slot_in;
  if (slot >= p.slots || (slot >= 0 && (accepted < 1 || accepted > max_q))) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadIndex);
    slot = -1;
  }
  const bool live = slot >= 0;  // uniform across the CTA
  const int off = live ? accepted - 1 : 0;
  const int nch = min(kThreads * V, C - cb);
  const int n4 = nch * SL / 4;  // nch is a multiple of V >= 4
  float* grow = live ? p.conv_pool + ((int64_t)slot * C + cb) * SL : nullptr;

  // The first kPre drafts' inputs are requested before the rows, so their
  // latency overlaps the staging.
  constexpr int kPre = 4;
  const TA* __restrict__ x = static_cast<const TA*>(p.x) + c0;
  uint4 xpre[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u)
    xpre[u] = (active && u < len) ? Act<TA>::load_raw(x + (int64_t)(lo + u) * p.x_stride)
                                  : make_uint4(0, 0, 0, 0);

  if (live) {  // rows -> shared memory, transposed; kB loads in flight per thread
    constexpr int kB = 4;
    const float4* src = reinterpret_cast<const float4*>(grow);
    for (int f0 = threadIdx.x; f0 < n4; f0 += kB * kThreads) {
      float4 v[kB];
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int f4 = f0 + b * kThreads;
        v[b] = f4 < n4 ? src[f4] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int f4 = f0 + b * kThreads;
        if (f4 < n4) {
          const float vv[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int f = 4 * f4 + u, c = f / SL;
            rows[(f - c * SL) * kPitch + c] = vv[u];
          }
        }
      }
    }
  }
  __syncthreads();
  const bool is_qk = c0 < 2 * qk_total;
  const bool norm_warp = p.norm && (c0 - lane * V) < 2 * qk_total;  // warp-uniform
  const int group = p.Dk / V;                        // lanes per key head
  const bool mine = live && active;

  TA* __restrict__ out_ptr;
  int64_t out_stride;
  if (c0 < qk_total) {
    out_ptr = static_cast<TA*>(p.q) + c0;
    out_stride = qk_total;
  } else if (c0 < 2 * qk_total) {
    out_ptr = static_cast<TA*>(p.k) + (c0 - qk_total);
    out_stride = qk_total;
  } else {
    out_ptr = static_cast<TA*>(p.v) + (c0 - 2 * qk_total);
    out_stride = (int64_t)p.Hv * p.Dv;
  }

  // entry j of this thread's channels, as V/4 float4 (j < SL)
  auto entry = [&](int j) { return rows4 + (j * kPitch + col) / 4; };
  float win[W][V];
#pragma unroll
  for (int j = 0; j < W; ++j) {
#pragma unroll
    for (int q4 = 0; q4 < V / 4; ++q4) {
      const float4 v = mine ? entry(off + j)[q4] : make_float4(0.f, 0.f, 0.f, 0.f);
      win[j][4 * q4] = v.x;
      win[j][4 * q4 + 1] = v.y;
      win[j][4 * q4 + 2] = v.z;
      win[j][4 * q4 + 3] = v.w;
    }
  }
  const int keep = SL - len;  // >= W - 1 >= 0
  if (mine) {
    for (int j = 0; j < keep; ++j) {
      const int src = off + 1 + j;
#pragma unroll
      for (int q4 = 0; q4 < V / 4; ++q4)
        entry(j)[q4] = src < SL ? entry(src)[q4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  // one draft: conv + SiLU + norm + store, then the row and window updates
  auto step = [&](int u, const float (&xt)[V]) {
    const int t = lo + u;
    float y[V];
    float ss = conv_silu_row<V, KW, W>(win, xt, wt, y);
    if (norm_warp) {
      for (int m = 1; m < group; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      if (is_qk) {
        const float inv = rsqrtf(ss + 1e-6f);
#pragma unroll
        for (int e = 0; e < V; ++e) y[e] *= inv;
      }
    }
    if (active) Act<TA>::store(out_ptr + (int64_t)t * out_stride, y);
    if (mine)
#pragma unroll
      for (int q4 = 0; q4 < V / 4; ++q4)
        entry(keep + u)[q4] = make_float4(xt[4 * q4], xt[4 * q4 + 1], xt[4 * q4 + 2], xt[4 * q4 + 3]);
#pragma unroll
    for (int j = 0; j + 1 < W; ++j)
#pragma unroll
      for (int e = 0; e < V; ++e) win[j][e] = win[j + 1][e];
#pragma unroll
    for (int e = 0; e < V; ++e) win[W - 1][e] = xt[e];
  };
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    if (u < len) {  // uniform across the CTA
      float xt[V];
      Act<TA>::unpack(xpre[u], xt);
      step(u, xt);
    }
  }
#pragma unroll 1
  for (int u = kPre; u < len; ++u) {
    float xt[V];
    if (active) {
      Act<TA>::load(x + (int64_t)(lo + u) * p.x_stride, xt);
    } else {
#pragma unroll
      for (int e = 0; e < V; ++e) xt[e] = 0.0f;
    }
    step(u, xt);
  }
  __syncthreads();

  if (live) {
    float4* dst = reinterpret_cast<float4*>(grow);
    for (int f4 = threadIdx.x; f4 < n4; f4 += kThreads) {
      float vv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int f = 4 * f4 + u, c = f / SL;
        vv[u] = rows[(f - c * SL) * kPitch + c];
      }
      dst[f4] = make_float4(vv[0], vv[1], vv[2], vv[3]);
    }
  }
}

template <typename TA, int KW>
cudaError_t launch_spec_k(const PrepareLaunch& p, cudaStream_t s) {
  constexpr int V = Act<TA>::kVec;
  const int C = 2 * p.Hk * p.Dk + p.Hv * p.Dv;
  const int chan_blocks = (C + kThreads * V - 1) / (kThreads * V);
  const size_t smem = (size_t)p.state_len * (kThreads * V + 4) * sizeof(float);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(spec_prepare_kernel<TA, KW>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(p.N, chan_blocks + 1);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  spec_prepare_kernel<TA, KW><<<grid, kThreads, smem, s>>>(p, chan_blocks);
  note_launch();
  return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_spec_dtype(const PrepareLaunch& p, cudaStream_t s) {
  switch (p.K) {
    case 2: return launch_spec_k<TA, 2>(p, s);
    case 3: return launch_spec_k<TA, 3>(p, s);
    case 4: return launch_spec_k<TA, 4>(p, s);
    case 5: return launch_spec_k<TA, 5>(p, s);
    case 6: return launch_spec_k<TA, 6>(p, s);
    case 7: return launch_spec_k<TA, 7>(p, s);
    case 8: return launch_spec_k<TA, 8>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename TA, int KW>
cudaError_t launch_k(const PrepareLaunch& p, cudaStream_t s) {
  constexpr int V = Act<TA>::kVec;
  const int C = 2 * p.Hk * p.Dk + p.Hv * p.Dv;
  const int chan_blocks = (C + kThreads * V - 1) / (kThreads * V);
  // Tiles of at least K-1 tokens (tail ownership) and at most 32 (a decode
  // tile reads its rows' slots one per lane); shrink them while the grid is
  // short of ~8 CTAs per SM.
  int tile = 32;
  while (tile > 2 && (int64_t)((p.T + tile - 1) / tile) * chan_blocks < 8 * 152) tile >>= 1;
  if (tile < KW - 1) tile = KW - 1;  // >= K-1 for the tail ownership rule (K <= 8: <= 16)
  const int64_t n_tiles = (p.T + tile - 1) / tile;
  const bool tiles_on_y = n_tiles <= 65535;
  if (chan_blocks + 1 > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid = tiles_on_y ? dim3(chan_blocks + 1, static_cast<unsigned>(n_tiles))
                               : dim3(static_cast<unsigned>(n_tiles), chan_blocks + 1);
  prepare_kernel<TA, KW><<<grid, kThreads, 0, s>>>(p, tile, chan_blocks, tiles_on_y);
  note_launch();
  return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_dtype(const PrepareLaunch& p, cudaStream_t s) {
  switch (p.K) {
    case 1: return launch_k<TA, 1>(p, s);
    case 2: return launch_k<TA, 2>(p, s);
    case 3: return launch_k<TA, 3>(p, s);
    case 4: return launch_k<TA, 4>(p, s);
    case 5: return launch_k<TA, 5>(p, s);
    case 6: return launch_k<TA, 6>(p, s);
    case 7: return launch_k<TA, 7>(p, s);
    case 8: return launch_k<TA, 8>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prepare(const PrepareLaunch& p, cudaStream_t s) {
  return p.bf16 ? launch_dtype<__nv_bfloat16>(p, s) : launch_dtype<float>(p, s);
}

cudaError_t launch_spec_prepare(const PrepareLaunch& p, cudaStream_t s) {
  if (p.state_len < p.K - 1 || p.state_len > 16 || p.sidx == nullptr || p.num_accepted == nullptr)
    return cudaErrorInvalidValue;
  return p.bf16 ? launch_spec_dtype<__nv_bfloat16>(p, s) : launch_spec_dtype<float>(p, s);
}

}  // namespace gdn
