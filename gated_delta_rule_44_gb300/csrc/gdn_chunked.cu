// gdn_chunked.cu -- chunked (C = 64) WY/UT-form varlen prefill on tcgen05
// tensor cores, bf16 operands with f32 TMEM accumulators and an f32 state.
//
// Defines the recurrence of [cpu.rs] (ferrum-kernels 0.8.0, src/ferrum_kernels/
// backend/cpu.rs) recurrent_gated_delta_rule_varlen_f32 / [cpu_ops.cpp]
// (vllm.cpp, src/vt/cpu/cpu_ops.cpp) GdnPrefillKernel, evaluated chunk by
// chunk.  The pages name a chunked GPU form but do not print it; the algebra
// below is derived from the recurrence.  For one chunk of L <= 64 tokens of a
// (sequence, value head) with state S0 = [Dv, Dk] at its start:
//   gam_i = sum_{t <= i} g_t                        (cumulative decay, <= 0)
//   A_ij  = beta_i e^{gam_i - gam_j} k_i.k_j         (j < i)
//   T     = (I + A)^-1                               (unit lower triangular)
//   W     = T diag(beta e^gam) K,    Ut = T diag(beta) V
//   U     = Ut - W S0^T
//   O     = diag(e^gam) scale Q S0^T + P U,  P_ij = scale e^{gam_i - gam_j} q_i.k_j (j <= i)
//   S_L^T = e^{gam_L} S0^T + K^T diag(e^{gam_L - gam}) U
// Every exponent is <= 0, so nothing overflows however strong the decay.
//
// Precision.  q, k, v are exact bf16 inputs.  Every operand the kernels compute
// (T, S, U, U', P) enters the tensor core as a pair of bf16 values hi + lo
// with hi = bf16(x), lo = bf16(x - hi), and products use hi*y + lo*y (or
// hi*hi + hi*lo + lo*hi): about 16 significant bits, so the result tracks the
// f32 recurrence instead of picking up one bf16 rounding per step.  Ut is kept
// in f32, W as one bf16 value (its error reaches the output only through the
// small W S^T correction).
//
// In-kernel q/k L2 norm: with kn_i = 1/|k_i|, qn_i = 1/|q_i| (eps 1e-6 inside
// the sqrt; 1 when the norm is off) the normalised rows are never stored: the
// factors fold into A, the columns of Tw, the rows of U' and P.
//
// Two launches on the caller's stream:
//  1. chunk_prep (one CTA per (chunk, value head), all chunks in parallel):
//     G = K K^T (tcgen05, M = 64), A from G, T by column-parallel forward
//     substitution (f32), W = Tw K and Ut = Tu V (tcgen05, hi + lo).  Writes W
//     (as the swizzled shared-memory image the second kernel copies), Ut
//     (f32), gam and 1/|k| to the workspace.
//  2. chunk_scan (one CTA per (sequence, value head, 64-row slice of Dv), its
//     chunks in order; TMA double-buffers W, Q, K, gam):
//        D1 = [W; Q] S^T     (M = 128: rows 0..63 W S^T, rows 64..127 Q S^T)
//        Dp = [W; Q] K^T     (rows 64..127: Q K^T, for P)
//        warps 0-1: U = Ut - W S^T, U' = diag(e^{gam_L - gam} kn) U   (hi + lo)
//        warps 2-3: P from Q K^T (hi + lo); the previous chunk's output
//        D2 = K^T U'         (M = 128 dk rows: the state increment)
//        D3 = [0; P] U       (rows 64..127: P U)
//        S = e^{gam_L} S + D2 in f32 registers; S^T hi + lo images
//     The output of chunk c (e^{gam} scale qn Q S^T + P U) is emitted by warps
//     2-3 while chunk c+1's D1 runs; D1 and D3 are double-buffered in TMEM.
//
// Partial chunks: K and V rows past the chunk end are zeroed in shared memory
// and their g, beta taken as 0, so every derived row is exactly zero.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gdn_internal.h"
#include "tcgen05.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kC = 64;      // chunk length
constexpr int kD = 128;     // Dk = Dv
constexpr int kThreads = 128;
constexpr long long kWaitBudget = 2000000000LL;  // ~1 s of SM clock per wait

// Workspace blob of one (chunk, value head).
constexpr uint32_t kBlobW = 0;       // W image: K-major SW128, 2 boxes of [64 x 64] bf16
constexpr uint32_t kBlobU = 16384;   // Ut: [2 slices][64 tokens][64] f32, see ut_offset
constexpr uint32_t kBlobG = 49152;   // gam: 64 f32
constexpr uint32_t kBlobKn = 49408;  // 1/|k_i| (or 1): 64 f32
constexpr uint32_t kBlobBytes = 49664;

// Byte offset of Ut element (row i, column c < 64) inside one 16 KB slice: 256-byte
// rows whose 16-byte chunks are XOR-swizzled by (i % 16), so that threads reading
// the same chunk of consecutive rows hit different shared-memory banks.
__device__ __forceinline__ uint32_t ut_offset(int i, int c) {
  return i * 256 + ((((c >> 2) ^ (i & 15))) << 4) + (c & 3) * 4;
}

// TMEM row of an M = 64 accumulator held by (warp, lane): rows 16w .. 16w+15
// sit in lanes 0..15 of warp w's 32-lane quarter.
__device__ __forceinline__ int m64_row(int warp, int lane) {
  return lane < 16 ? 16 * warp + lane : -1;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Stores 8 floats as bf16 into one 16-byte chunk.
__device__ __forceinline__ void st_bf16x8(void* p, const float* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

// hi = bf16(v), lo = bf16(v - hi) for 8 values, each into one 16-byte chunk.
__device__ __forceinline__ void st_split8(void* hi, void* lo, const float* v) {
  float h[8], l[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    h[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
    l[e] = v[e] - h[e];
  }
  st_bf16x8(hi, h);
  st_bf16x8(lo, l);
}

__device__ __forceinline__ void ld_bf16x8(const void* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(mbar)
      : "memory");
}

// Sequence and chunk-in-sequence of global chunk `gc`, from cu_seqlens (warp 0).
// Returns false when gc is past the last chunk or cu_seqlens is malformed.
__device__ bool locate_chunk(const int32_t* __restrict__ cu, int N, int T, int gc, int& s_out,
                             int& j_out, bool& bad) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  bad = false;
  for (int s0 = 0; s0 < N; s0 += 32) {
    const int s = s0 + lane;
    int nc = 0;
    if (s < N) {
      const int lo = __ldg(cu + s), hi = __ldg(cu + s + 1);
      if (lo < 0 || hi <= lo || hi > T) bad = true;
      nc = hi > lo ? (hi - lo + kC - 1) / kC : 0;
    }
    int incl = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int excl = incl - nc;
    const unsigned hit =
        __ballot_sync(0xffffffffu, nc > 0 && gc >= base + excl && gc < base + incl);
    bad = __any_sync(0xffffffffu, bad);
    if (hit) {
      const int src = __ffs(hit) - 1;
      s_out = s0 + src;
      j_out = gc - base - __shfl_sync(0xffffffffu, excl, src);
      return !bad;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return false;
}

// First global chunk of sequence s (sum of earlier sequences' chunk counts);
// `bad` reports an empty or decreasing earlier range (warp 0).
__device__ int chunk_base(const int32_t* __restrict__ cu, int s, bool& bad) {
  int b = 0;
  bool nb = false;
  for (int i = threadIdx.x & 31; i < s; i += 32) {
    const int len = __ldg(cu + i + 1) - __ldg(cu + i);
    nb |= len <= 0;
    b += len > 0 ? (len + kC - 1) / kC : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) b += __shfl_xor_sync(0xffffffffu, b, o);
  bad = __any_sync(0xffffffffu, nb);
  return b;
}

// ---------------------------------------------------------------------------
// Kernel 1: per (chunk, value head).
struct PrepSmem {
  static constexpr uint32_t K = 0;           // [K box0 | K box1], 16 KB
  static constexpr uint32_t V = 16384;       // [V box0 | V box1], 16 KB
  static constexpr uint32_t TWH = 32768;     // Tw hi image [64 x 64] bf16, 8 KB
  static constexpr uint32_t TWL = 40960;     // Tw lo
  static constexpr uint32_t TUH = 49152;     // Tu hi
  static constexpr uint32_t TUL = 57344;     // Tu lo
  static constexpr uint32_t A = 65536;       // A, f32 [64][68]
  static constexpr uint32_t kAStride = 68;
  static constexpr uint32_t TT = A + 64 * kAStride * 4;   // T = (I + A)^-1, f32 [64][68]
  static constexpr uint32_t X = TT + 64 * kAStride * 4;   // block scratch, f32 [3][16][17]
  static constexpr uint32_t GB = X + 3 * 16 * 17 * 4;     // g, beta, gam, kn, wj, uj: 6 x 64 f32
  static constexpr uint32_t BYTES = GB + 6 * 64 * 4;
};

__global__ void __launch_bounds__(kThreads) chunk_prep_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const RecurLaunch p, uint8_t* __restrict__ ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t mbar_tma, mbar_mma;
  __shared__ uint32_t tslot;
  __shared__ int s_seq, s_chunk, s_ok;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gc = blockIdx.x, h = blockIdx.y;

  if (warp == 0) {
    int s = 0, j = 0;
    bool bad = false;
    const bool ok = locate_chunk(p.cu, p.N, p.T, gc, s, j, bad);
    if (lane == 0) {
      s_seq = s;
      s_chunk = j;
      s_ok = ok ? 1 : 0;
      if (bad && gc == 0 && h == 0) atomicOr(p.status, kStatusBadSeqlens);
    }
  }
  __syncthreads();
  if (!s_ok) return;  // uniform: past the last chunk (or malformed cu_seqlens)
  const int s = s_seq;
  const int t0 = __ldg(p.cu + s) + kC * s_chunk;
  const int L = min(kC, __ldg(p.cu + s + 1) - t0);
  const int hk = h / (p.Hv / p.Hk);
  float* sg = reinterpret_cast<float*>(sm + PrepSmem::GB);
  float* sb = sg + 64;
  float* sgam = sb + 64;
  float* skn = sgam + 64;
  float* sA = reinterpret_cast<float*>(sm + PrepSmem::A);
  const uint32_t base = smem_u32(sm);
  const uint32_t mb_tma = smem_u32(&mbar_tma), mb_mma = smem_u32(&mbar_mma);

  if (tid == 0) {
    mbar_init(mb_tma, 1);
    mbar_init(mb_mma, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_expect_tx(mb_tma, 4 * 8192);
    tma_load_3d(base + PrepSmem::K + 0, &tm_k, mb_tma, 0, hk, t0);
    tma_load_3d(base + PrepSmem::K + 8192, &tm_k, mb_tma, 64, hk, t0);
    tma_load_3d(base + PrepSmem::V + 0, &tm_v, mb_tma, 0, h, t0);
    tma_load_3d(base + PrepSmem::V + 8192, &tm_v, mb_tma, 64, h, t0);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tslot), 256);
  if (tid < 64) {
    const bool in = tid < L;
    sg[tid] = in ? __ldg(p.g + (int64_t)(t0 + tid) * p.Hv + h) : 0.0f;
    sb[tid] = in ? __ldg(p.beta + (int64_t)(t0 + tid) * p.Hv + h) : 0.0f;
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tslot;
  if (warp == 0) {  // inclusive scan of g over the chunk (2 tokens per lane)
    const float a = sg[2 * lane], b = sg[2 * lane + 1];
    float x = a + b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    sgam[2 * lane + 1] = x;
    sgam[2 * lane] = x - b;
  }
  bool ok = mbar_wait(mb_tma, 0, kWaitBudget);
  if (L < kC) {  // zero K and V rows past the chunk end
    for (int i = tid; i < (kC - L) * 8; i += kThreads) {
      const int r = L + i / 8, q16 = i % 8;
#pragma unroll
      for (int box = 0; box < 4; ++box)
        *reinterpret_cast<uint4*>(sm + box * 8192 + r * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async();
  }
  __syncthreads();
  if (!__syncthreads_and(ok)) {
    if (tid == 0) atomicOr(p.status, kStatusTimeout);
    if (warp == 0) tmem_dealloc(tmem, 256);
    return;
  }
  if (tid < 64) {  // inverse k row norms
    float ss = 0.0f;
    if (p.norm) {
#pragma unroll
      for (int box = 0; box < 2; ++box)
#pragma unroll
        for (int q16 = 0; q16 < 8; ++q16) {
          float v[8];
          ld_bf16x8(sm + PrepSmem::K + box * 8192 + tid * 128 + ((q16 ^ (tid & 7)) << 4), v);
#pragma unroll
          for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
        }
    }
    skn[tid] = p.norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
  }
  fence_after_sync();
  // G = K K^T  (M = 64, N = 64, K = 128; both operands the K tile, K-major).
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(64, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < kD; kk += 16) {
      const uint32_t off = (kk / 64) * 8192 + (kk % 64) * 2;
      mma_bf16(tmem, desc_sw128(base + PrepSmem::K + off, 16, 1024),
               desc_sw128(base + PrepSmem::K + off, 16, 1024), idesc, kk > 0);
    }
    mma_commit(mb_mma);
  }
  __syncthreads();  // also publishes skn
  ok = mbar_wait(mb_mma, 0, kWaitBudget);
  fence_after_sync();
  uint8_t* blob = ws + ((int64_t)gc * p.Hv + h) * kBlobBytes;
  {
    const int i = m64_row(warp, lane);
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const float gi = i >= 0 ? sgam[i] : 0.0f;
    const float fi = i >= 0 ? sb[i] * skn[i] : 0.0f;
#pragma unroll
    for (int c = 0; c < kC; c += 16) {
      float v[16];
      tmem_ld16(tmem + lane_addr + c, v);
      tmem_ld_wait();
      if (i >= 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int jj = c + e;
          v[e] = jj < i ? fi * skn[jj] * __expf(gi - sgam[jj]) * v[e] : 0.0f;
        }
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(sA + i * PrepSmem::kAStride + c + e) =
              make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  float* sT = reinterpret_cast<float*>(sm + PrepSmem::TT);
  float* sX = reinterpret_cast<float*>(sm + PrepSmem::X);
  float* swj = skn + 64;
  float* suj = swj + 64;
  constexpr int S_ = PrepSmem::kAStride;
  for (int e = tid; e < 64 * S_; e += kThreads) sT[e] = 0.0f;  // blocks above the diagonal
  if (tid < 64) {
    swj[tid] = sb[tid] * skn[tid] * __expf(sgam[tid]);
    suj[tid] = sb[tid];
  }
  fence_before_sync();
  __syncthreads();
  // T = (I + A)^-1 in 16 x 16 blocks, A strictly lower triangular.
  // (1) diagonal blocks D_b = (I + A_bb)^-1, column c of block b per thread:
  //     x_i = [i == c] - sum_{m < i} A[16b+i][16b+m] x_m.
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15, r0 = 16 * b;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = 0.0f;
#pragma unroll
      for (int m = 0; m < i; ++m) acc = fmaf(sA[(r0 + i) * S_ + r0 + m], x[m], acc);
      x[i] = (i == c ? 1.0f : 0.0f) - acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sT[(r0 + i) * S_ + r0 + c] = x[i];
  }
  __syncthreads();
  // (2) below-diagonal blocks by distance L = I - J:
  //     Y = sum_{K=J}^{I-1} A_IK T_KJ,   T_IJ = -D_I Y.
#pragma unroll
  for (int L = 1; L < 4; ++L) {
    const int nblk = 4 - L;
    for (int e = tid; e < nblk * 256; e += kThreads) {
      const int J = e >> 8, i = (e >> 4) & 15, j = e & 15, I = J + L;
      float y = 0.0f;
      for (int K = J; K < I; ++K) {
        const float* arow = sA + (16 * I + i) * S_ + 16 * K;
        const float* tcol = sT + (16 * K) * S_ + 16 * J + j;
#pragma unroll
        for (int m = 0; m < 16; ++m) y = fmaf(arow[m], tcol[m * S_], y);
      }
      sX[(J * 16 + i) * 17 + j] = y;
    }
    __syncthreads();
    for (int e = tid; e < nblk * 256; e += kThreads) {
      const int J = e >> 8, i = (e >> 4) & 15, j = e & 15, I = J + L;
      const float* drow = sT + (16 * I + i) * S_ + 16 * I;
      float t = 0.0f;
#pragma unroll
      for (int m = 0; m < 16; ++m) t = fmaf(drow[m], sX[(J * 16 + m) * 17 + j], t);
      sT[(16 * I + i) * S_ + 16 * J + j] = -t;
    }
    __syncthreads();
  }
  // Tw = T diag(beta e^gam kn), Tu = T diag(beta) as hi + lo bf16 images:
  // one (row, 8-column chunk) per thread and step, 16-byte stores.
  for (int item = tid; item < 64 * 8; item += kThreads) {
    const int i = item >> 3, q = item & 7;
    float tw[8], tu[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float t = sT[i * S_ + 8 * q + e];
      tw[e] = t * swj[8 * q + e];
      tu[e] = t * suj[8 * q + e];
    }
    const uint32_t off = swz128_offset(i, 8 * q, 8192);
    st_split8(sm + PrepSmem::TWH + off, sm + PrepSmem::TWL + off, tw);
    st_split8(sm + PrepSmem::TUH + off, sm + PrepSmem::TUL + off, tu);
  }
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // W = (Tw_hi + Tw_lo) K, Ut = (Tu_hi + Tu_lo) V  (M = 64, N = 128, K = 64): B is
  // the K (V) tile, MN-major: token rows, dk (dv) contiguous, boxes 8 KB apart.
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(64, 128, false, true);
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int kk = 0; kk < kC; kk += 16) {
        const uint32_t a_off = (part ? PrepSmem::TWL : PrepSmem::TWH) + (kk % 64) * 2;
        mma_bf16(tmem, desc_sw128(base + a_off, 16, 1024),
                 desc_sw128(base + PrepSmem::K + (kk / 8) * 1024, 8192, 1024), idesc,
                 part > 0 || kk > 0);
      }
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int kk = 0; kk < kC; kk += 16) {
        const uint32_t a_off = (part ? PrepSmem::TUL : PrepSmem::TUH) + (kk % 64) * 2;
        mma_bf16(tmem + 128, desc_sw128(base + a_off, 16, 1024),
                 desc_sw128(base + PrepSmem::V + (kk / 8) * 1024, 8192, 1024), idesc,
                 part > 0 || kk > 0);
      }
    mma_commit(mb_mma);
  }
  __syncwarp();
  ok = ok && mbar_wait(mb_mma, 1, kWaitBudget);
  fence_after_sync();
  {
    const int i = m64_row(warp, lane);
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
    for (int c = 0; c < kD; c += 16) {
      float v[16];
      tmem_ld16(tmem + lane_addr + c, v);
      tmem_ld_wait();
      if (i >= 0) {
        st_bf16x8(blob + kBlobW + swz128_offset(i, c, 8192), v);
        st_bf16x8(blob + kBlobW + swz128_offset(i, c + 8, 8192), v + 8);
      }
    }
#pragma unroll
    for (int c = 0; c < kD; c += 16) {
      float v[16];
      tmem_ld16(tmem + lane_addr + 128 + c, v);
      tmem_ld_wait();
      if (i >= 0) {
        uint8_t* slice_base = blob + kBlobU + (c / 64) * 16384;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          *reinterpret_cast<float4*>(slice_base + ut_offset(i, (c % 64) + 4 * e)) =
              make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
      }
    }
  }
  if (tid < 64) {
    reinterpret_cast<float*>(blob + kBlobG)[tid] = sgam[tid];
    reinterpret_cast<float*>(blob + kBlobKn)[tid] = skn[tid];
  }
  if (!ok && tid == 0) atomicOr(p.status, kStatusTimeout);
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// Kernel 2: per (sequence, value head, 64-row slice of Dv), chunks in order.
//
// 8 warps.  TMEM lane quadrant q = warp % 4 is shared by warps q and q + 4,
// which split every 64-column tile into halves hf = warp / 4.
//   U warps (q = 0, 1):  token rows 0..63 of W S^T -> U, U'
//   P warps (q = 2, 3):  token rows 0..63 of Q S^T, Q K^T -> P, outputs
//   all warps:           dk rows 0..127 of the state increment
// MMAs (thread 0), hi and lo operands side by side along N = 128:
//   D1 = [W; Q] [S_hi | S_lo]^T      rows 0..63 W S^T, 64..127 Q S^T
//   Dp = [W; Q] K^T                  rows 64..127 Q K^T
//   D2 = K^T [U'_hi | U'_lo]         rows = dk
//   D3 = [0; P_hi] [U_hi | U_lo] + [0; P_lo] [U_hi | U_lo]   rows 64..127 P U
// Each result's two column halves are added in the epilogue.  D3 of chunk c is
// issued with D1 of chunk c + 1, so building P (and the output) stays off the
// serial path D1 -> U -> D2 -> S; Q S^T is kept in registers until then.
struct ScanSmem {
  // pipeline stage (x2): A1 = [W; Q] as a 128-row K-major tile, K tile, gam, kn
  static constexpr uint32_t A1 = 0;           // [W box0 | Q box0 | W box1 | Q box1], 32 KB
  static constexpr uint32_t K = 32768;        // [K box0 | K box1], 16 KB
  static constexpr uint32_t GAM = 49152;      // gam (64 f32), kn (64 f32)
  static constexpr uint32_t KN = GAM + 256;
  static constexpr uint32_t STAGE = 50176;    // 49 KB (1 KB aligned)
  static constexpr uint32_t TX = 32768 + 16384 + 512;
  // single buffers
  static constexpr uint32_t UT = 2 * STAGE;   // Ut slice f32 [64 tokens][64] (ut_offset), 16 KB
  static constexpr uint32_t SH = UT + 16384;  // S^T hi image [128 dk x 64 dv], 16 KB, then
  static constexpr uint32_t SL = SH + 16384;  //   S^T lo: one MN-major B operand of N = 128
  static constexpr uint32_t UH = SL + 16384;  // U hi image [64 tok x 64 dv], 8 KB, then U lo
  static constexpr uint32_t UL = UH + 8192;
  static constexpr uint32_t U2H = UL + 8192;  // U' hi, then U' lo
  static constexpr uint32_t U2L = U2H + 8192;
  static constexpr uint32_t PH = U2L + 8192;  // [0; P hi] as a 128-row K-major tile, 16 KB
  static constexpr uint32_t PL = PH + 16384;  // [0; P lo]
  static constexpr uint32_t BYTES = PL + 16384;
};

constexpr int kScanThreads = 256;

__global__ void __launch_bounds__(kScanThreads, 1) chunk_scan_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const RecurLaunch p, const uint8_t* __restrict__ ws, int n_chunks_max) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t mb_ld[2], mb_ut, mb_a, mb_p, mb_c, mb_d, mb_e;
  __shared__ uint32_t tslot;
  __shared__ int s_base, s_bad;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half
  const int slice = blockIdx.x & 1;
  const int sh = blockIdx.x >> 1;
  const int h = sh % p.Hv, s = sh / p.Hv;
  const int hk = h / (p.Hv / p.Hk);

  const int lo = __ldg(p.cu + s), hi = __ldg(p.cu + s + 1);
  if (lo < 0 || hi <= lo || hi > p.T || __ldg(p.cu) != 0 || __ldg(p.cu + p.N) != p.T) {
    if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }
  int slot = p.sidx != nullptr ? __ldg(p.sidx + s) : s;
  if (slot < -1 || slot >= p.slots) {
    if (tid == 0) atomicOr(p.status, kStatusBadIndex);
    slot = -1;
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  if (slot < 0) {  // padded sequence: zero outputs, pool untouched
    for (int idx = tid; idx < (hi - lo) * 8; idx += kScanThreads) {
      const int t = lo + idx / 8, q16 = idx % 8;
      *reinterpret_cast<uint4*>(out + ((int64_t)t * p.Hv + h) * kD + slice * 64 + q16 * 8) =
          make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int nchunks = (hi - lo + kC - 1) / kC;
  if (warp == 0) {
    bool bad = false;
    const int b = chunk_base(p.cu, s, bad);
    if (lane == 0) {
      s_base = b;
      s_bad = (bad || b + nchunks > n_chunks_max) ? 1 : 0;
    }
  }
  __syncthreads();
  if (s_bad) {  // uniform; the workspace holds no chunks for this sequence
    if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }
  const uint32_t base = smem_u32(sm);
  if (tid == 0) {
    mbar_init(smem_u32(&mb_ld[0]), 1);
    mbar_init(smem_u32(&mb_ld[1]), 1);
    mbar_init(smem_u32(&mb_ut), 1);
    mbar_init(smem_u32(&mb_a), 1);
    mbar_init(smem_u32(&mb_p), 1);
    mbar_init(smem_u32(&mb_c), 1);
    mbar_init(smem_u32(&mb_d), 1);
    mbar_init(smem_u32(&mb_e), 1);
    fence_mbar_init();
  }
  for (int i = tid; i < 2 * 512; i += kScanThreads) {  // the zero halves of [0; P]
    const uint32_t off = (i < 512 ? ScanSmem::PH : ScanSmem::PL);
    *reinterpret_cast<uint4*>(sm + off + (i % 512) * 16) = make_uint4(0, 0, 0, 0);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tslot), 512);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tslot;
  const int gc0 = s_base;
  auto blob_of = [&](int c) {
    return ws + ((int64_t)(gc0 + c) * p.Hv + h) * kBlobBytes;
  };
  // Loads W, Q, K, gam, kn of chunk c into stage c & 1 (thread 0 only).
  auto issue_load = [&](int c) {
    const uint32_t sb = base + (c & 1) * ScanSmem::STAGE;
    const uint32_t mb = smem_u32(&mb_ld[c & 1]);
    const uint8_t* blob = blob_of(c);
    const int t0 = lo + c * kC;
    mbar_expect_tx(mb, ScanSmem::TX);
    bulk_g2s(sb + ScanSmem::A1, blob + kBlobW, 8192, mb);
    bulk_g2s(sb + ScanSmem::A1 + 16384, blob + kBlobW + 8192, 8192, mb);
    bulk_g2s(sb + ScanSmem::GAM, blob + kBlobG, 512, mb);  // gam, kn
    tma_load_3d(sb + ScanSmem::A1 + 8192, &tm_q, mb, 0, hk, t0);
    tma_load_3d(sb + ScanSmem::A1 + 24576, &tm_q, mb, 64, hk, t0);
    tma_load_3d(sb + ScanSmem::K, &tm_k, mb, 0, hk, t0);
    tma_load_3d(sb + ScanSmem::K + 8192, &tm_k, mb, 64, hk, t0);
  };
  auto issue_ut = [&](int c) {  // thread 0 only
    const uint32_t mb = smem_u32(&mb_ut);
    mbar_expect_tx(mb, 16384);
    bulk_g2s(base + ScanSmem::UT, blob_of(c) + kBlobU + slice * 16384, 16384, mb);
  };
  // D3 = [0; P_hi][U_hi | U_lo] + [0; P_lo][U_hi | U_lo]  (M = 128, N = 128, K = 64)
  auto issue_d3 = [&]() {  // thread 0 only
    const uint32_t id3 = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int kk = 0; kk < kC; kk += 16)
        mma_bf16(tmem + 320,
                 desc_sw128(base + (part ? ScanSmem::PL : ScanSmem::PH) + (kk % 64) * 2, 16, 1024),
                 desc_sw128(base + ScanSmem::UH + (kk / 8) * 1024, 8192, 1024), id3,
                 part > 0 || kk > 0);
    mma_commit(smem_u32(&mb_d));
  };
  // Loads issued so far (thread 0), for the error path.
  int issued_ld = 0, issued_ut = 0;
  if (tid == 0) {
    issue_load(0);
    issued_ld = 1;
    if (nchunks > 1) {
      issue_load(1);
      issued_ld = 2;
    }
    issue_ut(0);
    issued_ut = 1;
  }

  // State: thread (quad, hf, lane) owns dk = 32 quad + lane and dv columns
  // 32 hf .. 32 hf + 31 of this slice, in f32.
  const int dk = quad * 32 + lane;
  float S[32];
  float* pool = p.pool + ((int64_t)slot * p.Hv + h) * kD * kD;
  const bool init = p.has_init == nullptr || __ldg(p.has_init + s) != 0;
#pragma unroll
  for (int e = 0; e < 32; ++e)
    S[e] = init ? pool[(int64_t)(slice * 64 + hf * 32 + e) * kD + dk] : 0.0f;
  auto write_s = [&]() {  // S^T hi / lo images: row dk, 32 dv columns (MN-major B operand)
#pragma unroll
    for (int e = 0; e < 32; e += 8) {
      const uint32_t off = swz128_offset(dk, hf * 32 + e, 16384);
      st_split8(sm + ScanSmem::SH + off, sm + ScanSmem::SL + off, S + e);
    }
  };
  write_s();
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tm_d1 = tmem, tm_dp = tmem + 128, tm_d2 = tmem + 192, tm_d3 = tmem + 320;
  const bool u_warp = quad < 2;
  const int row = (quad & 1) * 32 + lane;  // token row of U and P warps
  // P warps carry the previous chunk's Q S^T and output factor to its output.
  float qs_prev[32];
  float fo_prev = 0.0f;

  // Output of chunk cc by the P warps: O = e^{gam} scale qn Q S^T + P U.
  auto emit_output = [&](int cc) {
    const int t0 = lo + cc * kC;
    const int L = min(kC, hi - t0);
    float a[32], b[32];
    tmem_ld32(tm_d3 + lane_addr + hf * 32, a);
    tmem_ld32(tm_d3 + lane_addr + 64 + hf * 32, b);
    tmem_ld_wait();
    if (row < L) {
#pragma unroll
      for (int e = 0; e < 32; ++e) a[e] = fmaf(fo_prev, qs_prev[e], a[e] + b[e]);
      __nv_bfloat16* dst = out + ((int64_t)(t0 + row) * p.Hv + h) * kD + slice * 64 + hf * 32;
#pragma unroll
      for (int e = 0; e < 32; e += 8) st_bf16x8(dst + e, a + e);
    }
  };

  bool ok = true;
  int c = 0;
  int last_mma = -1;  // thread 0: last chunk whose MMAs were issued
  for (; c < nchunks; ++c) {
    const int st = c & 1;
    uint8_t* sst = sm + st * ScanSmem::STAGE;
    const uint32_t sb = base + st * ScanSmem::STAGE;
    const int t0 = lo + c * kC;
    const int L = min(kC, hi - t0);
    ok = mbar_wait(smem_u32(&mb_ld[st]), (c >> 1) & 1, kWaitBudget);
    if (!__syncthreads_and(ok)) break;
    if (L < kC) {  // zero K rows past the chunk end (they meet U rows that are 0)
      for (int i = tid; i < (kC - L) * 8; i += kScanThreads) {
        const int r = L + i / 8, q16 = i % 8;
        *reinterpret_cast<uint4*>(sst + ScanSmem::K + r * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sst + ScanSmem::K + 8192 + r * 128 + q16 * 16) =
            make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async();
      __syncthreads();
    }
    if (tid == 0) {
      fence_after_sync();
      // D1 = [W; Q] [S_hi | S_lo]^T  (M = 128, N = 128, K = 128)
      const uint32_t id1 = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
      for (int kk = 0; kk < kD; kk += 16)
        mma_bf16(tm_d1, desc_sw128(sb + ScanSmem::A1 + (kk / 64) * 16384 + (kk % 64) * 2, 16, 1024),
                 desc_sw128(base + ScanSmem::SH + (kk / 8) * 1024, 16384, 1024), id1, kk > 0);
      mma_commit(smem_u32(&mb_a));
      if (c > 0) issue_d3();  // previous chunk's P U (its P and U images are intact)
      // Dp = [W; Q] K^T  (M = 128, N = 64 tokens, K = 128; B = K tile, K-major)
      const uint32_t idp = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
      for (int kk = 0; kk < kD; kk += 16)
        mma_bf16(tm_dp, desc_sw128(sb + ScanSmem::A1 + (kk / 64) * 16384 + (kk % 64) * 2, 16, 1024),
                 desc_sw128(sb + ScanSmem::K + (kk / 64) * 8192 + (kk % 64) * 2, 16, 1024), idp,
                 kk > 0);
      mma_commit(smem_u32(&mb_p));
      last_mma = c;
    }
    __syncwarp();
    const float* gam = reinterpret_cast<const float*>(sst + ScanSmem::GAM);
    const float* kn = reinterpret_cast<const float*>(sst + ScanSmem::KN);
    if (u_warp) {
      // U = Ut - W S^T and U' = diag(e^{gam_L - gam} kn) U, this thread's row and
      // column half, written as hi + lo images once D3 of the previous chunk is done.
      ok = mbar_wait(smem_u32(&mb_ut), c & 1, kWaitBudget);
      ok = mbar_wait(smem_u32(&mb_a), c & 1, kWaitBudget) && ok;
      fence_after_sync();
      float wa[32], wb[32];
      tmem_ld32(tm_d1 + lane_addr + hf * 32, wa);
      tmem_ld32(tm_d1 + lane_addr + 64 + hf * 32, wb);
      tmem_ld_wait();
      const float fu = __expf(gam[kC - 1] - gam[row]) * kn[row];
      const uint8_t* ut = sm + ScanSmem::UT;
      float u[32];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 f = *reinterpret_cast<const float4*>(ut + ut_offset(row, hf * 32 + e));
        u[e] = f.x - (wa[e] + wb[e]);
        u[e + 1] = f.y - (wa[e + 1] + wb[e + 1]);
        u[e + 2] = f.z - (wa[e + 2] + wb[e + 2]);
        u[e + 3] = f.w - (wa[e + 3] + wb[e + 3]);
      }
      if (c > 0) ok = mbar_wait(smem_u32(&mb_d), (c - 1) & 1, kWaitBudget) && ok;
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        float u2[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) u2[x] = fu * u[e + x];
        const uint32_t off = swz128_offset(row, hf * 32 + e, 8192);
        st_split8(sm + ScanSmem::UH + off, sm + ScanSmem::UL + off, u + e);
        st_split8(sm + ScanSmem::U2H + off, sm + ScanSmem::U2L + off, u2);
      }
      fence_proxy_async();
      named_bar(1, 128);  // Ut consumed: fetch the next chunk's
      if (tid == 0 && c + 1 < nchunks) {
        fence_proxy_async();
        issue_ut(c + 1);
        issued_ut = c + 2;
      }
    } else {
      // The previous chunk's output (needs its D3), then Q S^T of this chunk into
      // registers, then P = scale e^{gam_i - gam_j} qn_i kn_j Q K^T (j <= i) as hi + lo.
      if (c > 0) {
        ok = mbar_wait(smem_u32(&mb_d), (c - 1) & 1, kWaitBudget) && ok;
        fence_after_sync();
        emit_output(c - 1);
      }
      float ss = 0.0f;
      if (p.norm) {
#pragma unroll
        for (int box = 0; box < 2; ++box)
#pragma unroll
          for (int q16 = 0; q16 < 8; ++q16) {
            float v[8];
            ld_bf16x8(sst + ScanSmem::A1 + box * 16384 + 8192 + row * 128 +
                          ((q16 ^ (row & 7)) << 4), v);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
          }
      }
      const float qn = p.norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
      ok = mbar_wait(smem_u32(&mb_a), c & 1, kWaitBudget) && ok;
      fence_after_sync();
      {
        float qa[32], qb[32];
        tmem_ld32(tm_d1 + lane_addr + hf * 32, qa);
        tmem_ld32(tm_d1 + lane_addr + 64 + hf * 32, qb);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) qs_prev[e] = qa[e] + qb[e];
      }
      fo_prev = p.scale * __expf(gam[row]) * qn;  // consumed by emit_output(c) next time
      ok = mbar_wait(smem_u32(&mb_p), c & 1, kWaitBudget) && ok;
      fence_after_sync();
      float qk[32];
      tmem_ld32(tm_dp + lane_addr + hf * 32, qk);
      tmem_ld_wait();
      const float gi = gam[row], fi = p.scale * qn;
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        float v[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const int jj = hf * 32 + e + x;
          v[x] = jj <= row ? fi * kn[jj] * __expf(gi - gam[jj]) * qk[e + x] : 0.0f;
        }
        const uint32_t off = swz128_offset(64 + row, hf * 32 + e, 16384);
        st_split8(sm + ScanSmem::PH + off, sm + ScanSmem::PL + off, v);
      }
      fence_proxy_async();
    }
    fence_before_sync();
    if (!__syncthreads_and(ok)) break;
    fence_after_sync();
    if (tid == 0) {
      // D2 = K^T [U'_hi | U'_lo]  (M = 128 dk, N = 128, K = 64 tokens; A = K tile MN-major)
      const uint32_t id2 = idesc_bf16_f32(128, 128, true, true);
#pragma unroll
      for (int kk = 0; kk < kC; kk += 16)
        mma_bf16(tm_d2, desc_sw128(sb + ScanSmem::K + (kk / 8) * 1024, 8192, 1024),
                 desc_sw128(base + ScanSmem::U2H + (kk / 8) * 1024, 8192, 1024), id2, kk > 0);
      mma_commit(smem_u32(&mb_c));
    }
    __syncwarp();
    ok = mbar_wait(smem_u32(&mb_c), c & 1, kWaitBudget) && ok;
    fence_after_sync();
    {
      // S = e^{gam_L} S + D2  (f32, registers), new S^T hi / lo images.
      const float dL = __expf(gam[kC - 1]);
      float da[32], db[32];
      tmem_ld32(tm_d2 + lane_addr + hf * 32, da);
      tmem_ld32(tm_d2 + lane_addr + 64 + hf * 32, db);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) S[e] = fmaf(dL, S[e], da[e] + db[e]);
    }
    write_s();
    fence_proxy_async();
    fence_before_sync();
    if (!__syncthreads_and(ok)) break;
    fence_after_sync();
    // Every reader of this stage (D1, Dp, D2 and the generic reads) is done:
    // refill it with chunk c + 2.
    if (tid == 0 && c + 2 < nchunks) {
      fence_proxy_async();
      issue_load(c + 2);
      issued_ld = c + 3;
    }
  }
  if (c == nchunks) {
    if (tid == 0) issue_d3();  // the last chunk's P U
    if (!u_warp) {
      ok = mbar_wait(smem_u32(&mb_d), (nchunks - 1) & 1, kWaitBudget) && ok;
      fence_after_sync();
      emit_output(nchunks - 1);
    }
  }
  ok = __syncthreads_and(ok);
  if (c < nchunks || !ok) {
    // A wait ran out: report; let in-flight MMAs and loads finish (bounded); free TMEM.
    if (tid == 0) {
      atomicOr(p.status, kStatusTimeout);
      if (last_mma >= 0) {
        mma_commit(smem_u32(&mb_e));
        mbar_wait(smem_u32(&mb_e), 0, kWaitBudget);
      }
      for (int k = c; k < issued_ld; ++k)
        mbar_wait(smem_u32(&mb_ld[k & 1]), (k >> 1) & 1, kWaitBudget);
      for (int k = c; k < issued_ut; ++k) mbar_wait(smem_u32(&mb_ut), k & 1, kWaitBudget);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
    return;
  }
#pragma unroll
  for (int e = 0; e < 32; ++e) pool[(int64_t)(slice * 64 + hf * 32 + e) * kD + dk] = S[e];
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---- host ------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [rows, heads, 128] bf16 tensor; box = 64 rows x 1 head x 64 elements, SW128.
bool make_map(CUtensorMap* m, const void* ptr, int rows, int heads) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                           static_cast<cuuint64_t>(heads) * kD * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t max_chunks(int64_t T, int64_t N) { return T / kC + N; }

}  // namespace

bool chunked_supported(int Dk, int Dv, bool bf16) { return bf16 && Dk == kD && Dv == kD; }

size_t chunked_workspace_bytes(int64_t T, int64_t N, int64_t Hv, int64_t Dk, int64_t Dv) {
  if (Dk != kD || Dv != kD) return 0;
  return static_cast<size_t>(max_chunks(T, N) * Hv) * kBlobBytes;
}

cudaError_t launch_chunked(const ChunkedLaunch& c, cudaStream_t s) {
  const RecurLaunch& p = c.r;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, p.q, p.T, p.Hk) || !make_map(&tk, p.k, p.T, p.Hk) ||
      !make_map(&tv, p.v, p.T, p.Hv))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    PrepSmem::BYTES + 1024);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(chunk_scan_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      ScanSmem::BYTES + 1024);
  });
  if (attr_err != cudaSuccess) return attr_err;
  uint8_t* ws = static_cast<uint8_t*>(c.workspace);
  const int64_t nch = max_chunks(p.T, p.N);
  if (nch > 0x7fffffff || p.Hv > 65535) return cudaErrorInvalidConfiguration;
  chunk_prep_kernel<<<dim3(static_cast<unsigned>(nch), p.Hv), kThreads, PrepSmem::BYTES + 1024,
                      s>>>(tk, tv, p, ws);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t blocks = static_cast<int64_t>(p.N) * p.Hv * 2;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  chunk_scan_kernel<<<static_cast<unsigned>(blocks), kScanThreads, ScanSmem::BYTES + 1024, s>>>(
      tq, tk, p, ws, static_cast<int>(nch));
  note_launch();
  return cudaGetLastError();
}

}  // namespace gdn
