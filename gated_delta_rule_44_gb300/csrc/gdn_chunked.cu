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
// with hi = x rounded to 8 significant bits (a bf16 value), lo = bf16(x - hi),
// and products use hi*y + lo*y (or
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
//     [K; Q] K^T (tcgen05, M = 128) gives A and P; T by 32 x 32 blocks (f32);
//     W = Tw K and Ut = Tu V (tcgen05, hi + lo).  Writes everything of the
//     chunk that does not depend on the state: W and P as the swizzled
//     shared-memory images the second kernel copies, Ut (f32) and the row
//     factors fo = scale qn e^gam, fu = kn e^{gam_L - gam}, e^{gam_L}.
//  2. chunk_scan (one CTA per (sequence, value head, 64-column slice of Dv), its
//     chunks in order; TMA double-buffers W, Q, K and the factors, and P).
//     Per chunk, the serial path is D1 -> U' -> D2 -> S:
//        D1 = [W; Q] [S_hi | S_lo]^T  (M = 128: rows 0..63 W S^T, 64..127 Q S^T)
//        U warps: U = Ut - W S^T; U' = diag(fu) U images, then U images (hi + lo)
//        D2 = K^T [U'_hi | U'_lo]    (M = 128 dk rows: the state increment)
//        D3 = [*; P_hi] U + [*; P_lo] U   (rows 64..127: P U; rows 0..63 unused)
//        all warps: S = e^{gam_L} S + D2 in f32 registers; S^T hi + lo images
//     D3 of chunk c runs behind D2 of chunk c + 1, and the output warps emit
//     chunk c (fo Q S^T + P U) while chunk c + 2 runs; the U images and D3
//     are double-buffered.  One extra warp issues every MMA.
//
// Partial chunks: K, Q and V rows past the chunk end are zeroed in shared
// memory and their g, beta taken as 0, so every derived row is exactly zero.
#include <cuda.h>
#include <algorithm>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_chunk_common.cuh"
#include "gdn_internal.h"
#include "tcgen05.cuh"

namespace gdn {
namespace {

using namespace umma;
using namespace chunk;

constexpr long long kWaitBudget = 2000000000LL;  // ~1 s of SM clock per wait


// Workspace blob of one (chunk, value head): everything of the chunk that does
// not depend on the state.
constexpr uint32_t kBlobW = 0;        // W image: K-major SW128, 2 boxes of [64 x 64] bf16
constexpr uint32_t kBlobP = 16384;    // P hi image, then P lo: K-major SW128 [64 x 64] bf16
constexpr uint32_t kBlobF = 32768;    // fo[64], fu[64], e^{gam_L}, 3 x 0 (f32)
constexpr uint32_t kBlobFBytes = 528;
constexpr uint32_t kBlobU = 33792;    // Ut: [2 slices][64 tokens][64] f32, see ut_offset
constexpr uint32_t kBlobBytes = 66560;

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

// ---------------------------------------------------------------------------
// Kernel 1: per (chunk, key head), its value heads in turn (K, Q, their norms
// and [K; Q] K^T are the same for all of them).  8 warps; TMEM lane quadrant
// q = warp % 4 is shared by warps q and q + 4, which split columns into halves
// hf = warp / 4.
struct PrepSmem {
  static constexpr uint32_t KQ = 0;          // [K box0 | Q box0 | K box1 | Q box1], 32 KB
  static constexpr uint32_t V = 32768;       // [V box0 | V box1], 16 KB
  static constexpr uint32_t TWH = 49152;     // Tw hi image [64 x 64] bf16, 8 KB
  static constexpr uint32_t TWL = 57344;     // Tw lo
  static constexpr uint32_t TUH = 65536;     // Tu hi
  static constexpr uint32_t TUL = 73728;     // Tu lo
  static constexpr uint32_t AT = 81920;      // A, then T = (I + A)^-1 in place, f32 [64][68]
  static constexpr uint32_t kAStride = 68;
  static constexpr uint32_t Y = AT + 64 * kAStride * 4;   // A21 T11, f32 [32][36]
  static constexpr uint32_t kYStride = 36;
  static constexpr uint32_t GB = Y + 32 * kYStride * 4;   // g, beta, gam, kn, qn, wj, uj
  static constexpr uint32_t BYTES = GB + 7 * 64 * 4;
};
constexpr int kPrepThreads = 256;
constexpr int kBarP = 1;  // chunk_prep: warp 0 and the 4 P warps -- the P image space is free

__global__ void __launch_bounds__(kPrepThreads, 2) chunk_prep_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const RecurLaunch p, uint8_t* __restrict__ ws,
    int j0, int j1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  __shared__ uint64_t mbar_tma, mbar_v, mbar_mma;
  __shared__ uint32_t tslot;
  __shared__ int s_seq, s_chunk, s_gc, s_ok;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, hf = warp >> 2;
  const int hk = blockIdx.y;
  const int G = p.Hv / p.Hk;  // value heads of this key head: hk G .. hk G + G - 1

  if (warp == 0) {  // this launch's piece: the chunks with index in [j0, j1) of every sequence
    int s = 0, j = 0;
    bool bad = false;
    const bool ok = locate_chunk(p.cu, p.N, p.T, blockIdx.x, s, j, bad, j0, j1);
    bool bad2 = false;
    const int sbase = ok ? chunk_base(p.cu, s, bad2) : 0;  // the sequence's first global chunk
    if (lane == 0) {
      s_seq = s;
      s_chunk = j;
      s_gc = sbase + j;
      s_ok = ok ? 1 : 0;
      if (bad && blockIdx.x == 0 && hk == 0) atomicOr(p.status, kStatusBadSeqlens);
    }
  }
  __syncthreads();
  // When the chunks are prepared in pieces, the piece's launch runs beside the
  // scan of the piece before it (programmatic dependent launch) and must not
  // complete before that scan has: CTA (0, 0) waits for it on every way out.
  const bool waiter = blockIdx.x == 0 && blockIdx.y == 0;
  if (!s_ok) {  // uniform: outside this piece, past the last chunk, or malformed cu_seqlens
    if (waiter) griddep_wait();
    return;
  }
  const int s = s_seq;
  const int t0 = __ldg(p.cu + s) + kC * s_chunk;
  const int L = min(kC, __ldg(p.cu + s + 1) - t0);
  float* sg = reinterpret_cast<float*>(sm + PrepSmem::GB);
  float* sb = sg + 64;
  float* sgam = sb + 64;
  float* skn = sgam + 64;
  float* sqn = skn + 64;
  float* swj = sqn + 64;
  float* suj = swj + 64;
  float* sA = reinterpret_cast<float*>(sm + PrepSmem::AT);
  float* sY = reinterpret_cast<float*>(sm + PrepSmem::Y);
  constexpr int S_ = PrepSmem::kAStride;
  constexpr int SY = PrepSmem::kYStride;
  const uint32_t base = smem_u32(sm);
  const uint32_t mb_tma = smem_u32(&mbar_tma), mb_v = smem_u32(&mbar_v),
                 mb_mma = smem_u32(&mbar_mma);

  if (tid == 0) {
    mbar_init(mb_tma, 1);
    mbar_init(mb_v, 1);
    mbar_init(mb_mma, 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto load_v = [&](int h) {  // thread 0
    mbar_expect_tx(mb_v, 2 * 8192);
    tma_load_3d(base + PrepSmem::V + 0, &tm_v, mb_v, 0, h, t0);
    tma_load_3d(base + PrepSmem::V + 8192, &tm_v, mb_v, 64, h, t0);
  };
  if (tid == 0) {
    mbar_expect_tx(mb_tma, 4 * 8192);
    tma_load_3d(base + PrepSmem::KQ + 0, &tm_k, mb_tma, 0, hk, t0);
    tma_load_3d(base + PrepSmem::KQ + 8192, &tm_q, mb_tma, 0, hk, t0);
    tma_load_3d(base + PrepSmem::KQ + 16384, &tm_k, mb_tma, 64, hk, t0);
    tma_load_3d(base + PrepSmem::KQ + 24576, &tm_q, mb_tma, 64, hk, t0);
    load_v(hk * G);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tslot), 256);
  // Gates of the current value head, read ahead of their use (the first
  // head's here, the next head's during the solve of the current one).
  float g_next = 0.0f, b_next = 0.0f;
  auto load_gates = [&](int h) {  // threads 0..63
    if (tid < L) {
      g_next = __ldg(p.g + (int64_t)(t0 + tid) * p.Hv + h);
      b_next = __ldg(p.beta + (int64_t)(t0 + tid) * p.Hv + h);
    } else {
      g_next = b_next = 0.0f;
    }
  };
  if (tid < 64) load_gates(hk * G);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tslot;
  // TMEM: columns 0..63 [K; Q] K^T (kept for every value head), 64..191 the
  // M = 64 results W, then Ut, of the current head.
  const uint32_t tm_g = tmem, tm_wu = tmem + 64;
  const bool ok_kq = __syncthreads_and(mbar_wait(mb_tma, 0, kWaitBudget));
  if (!ok_kq) {  // the K, Q tiles did not land: touch none of their bytes
    if (tid == 0) {
      atomicOr(p.status, kStatusTimeout);
      // wait (bounded) for the copies still in flight before the CTA exits
      mbar_wait(mb_tma, 0, kWaitBudget);
      mbar_wait(mb_v, 0, kWaitBudget);  // the first V load
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
    if (waiter) griddep_wait();
    return;
  }
  if (L < kC) {  // zero K and Q rows past the chunk end
    for (int i = tid; i < (kC - L) * 8; i += kPrepThreads) {
      const int r = L + i / 8, q16 = i % 8;
#pragma unroll
      for (int box = 0; box < 4; ++box)
        *reinterpret_cast<uint4*>(sm + box * 8192 + r * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async();
  }
  __syncthreads();
  fence_after_sync();
  // [K; Q] K^T  (M = 128, N = 64, K = 128): A is the 128-row K-major tile
  // [K; Q] (boxes 16 KB apart), B the K tile (its first 64 rows).  Shared by
  // every value head of this key head.
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < kD; kk += 16) {
      const uint32_t off = (kk / 64) * 16384 + (kk % 64) * 2;
      mma_bf16(tm_g, desc_sw128(base + PrepSmem::KQ + off, 16, 1024),
               desc_sw128(base + PrepSmem::KQ + off, 16, 1024), idesc, kk > 0);
    }
    mma_commit(mb_mma);
  }
  if (tid < 128) {  // inverse row norms: threads 0..63 rows of K, 64..127 rows of Q
    const int r = tid & 63;
    float ss = 0.0f;
    if (p.norm) {
      const uint8_t* row = sm + PrepSmem::KQ + (tid < 64 ? 0 : 8192) + r * 128;
#pragma unroll
      for (int box = 0; box < 2; ++box)
#pragma unroll
        for (int q16 = 0; q16 < 8; ++q16) {
          float v[8];
          ld_bf16x8(row + box * 16384 + ((q16 ^ (r & 7)) << 4), v);
#pragma unroll
          for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
        }
    }
    (tid < 64 ? skn : sqn)[r] = p.norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
  }
  bool ok = mbar_wait(mb_mma, 0, kWaitBudget);
  uint32_t mma_phase = 1;
  fence_after_sync();
  __syncthreads();  // publishes skn, sqn; the Q tile is free from here on

  for (int jh = 0; jh < G; ++jh) {
    const int h = hk * G + jh;
    uint8_t* blob = ws + ((int64_t)s_gc * p.Hv + h) * kBlobBytes;
    if (tid < 64) {
      sg[tid] = g_next;
      sb[tid] = b_next;
    }
    __syncthreads();
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
      sg[2 * lane] = __expf(a);  // e^{g_j}: the step between neighbouring decays
      sg[2 * lane + 1] = __expf(b);
    }
    __syncthreads();
    if (tid < 64) {
      swj[tid] = sb[tid] * skn[tid] * __expf(sgam[tid]);
      suj[tid] = sb[tid];
      float* F = reinterpret_cast<float*>(blob + kBlobF);
      F[tid] = p.scale * sqn[tid] * __expf(sgam[tid]);           // fo
      F[64 + tid] = __expf(sgam[kC - 1] - sgam[tid]) * skn[tid];  // fu
      if (tid < 4) F[128 + tid] = tid == 0 ? __expf(sgam[kC - 1]) : 0.0f;
    }
    {
      // Lanes 0..63 hold K K^T -> A (f32, shared); lanes 64..127 hold Q K^T -> P
      // (hi + lo images, staged in the Tw image space).  Row i, columns 32 hf ...
      // The previous head's Ut store must have read the image space the P
      // images use: warp 0 waits for it and releases the P warps, which block
      // only right before their stores.
      if (warp == 0) {
        if (lane == 0) bulk_wait_read();
        __syncwarp();
        named_bar_arrive(kBarP, 5 * 32);
      }
      // Rows 0..31 x columns 32..63 lie above the diagonal: all zero.
      const int i = (quad & 1) * 32 + lane;
      const bool upper = (quad & 1) == 0 && hf == 1;  // uniform across the warp
      float v[32];
      if (!upper) {
        tmem_ld32(tm_g + (static_cast<uint32_t>(quad * 32) << 16) + hf * 32, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0.0f;
      }
      // Decays e^{gam_i - gam_j} (j <= i) along the row, leftward from the
      // block's last column: e^{gam_i - gam_j} = e^{gam_i - gam_{j+1}} e^{g_{j+1}},
      // one exponential per row and block instead of one per entry.  0 right
      // of the diagonal, 1 on it.
      float dec[32];
      if (!upper) {
        const int jr = hf * 32 + 31;
        float cur = jr <= i ? __expf(sgam[i] - sgam[jr]) : 0.0f;
        dec[31] = cur;
#pragma unroll
        for (int e = 30; e >= 0; --e) {
          const int j = hf * 32 + e;
          cur = j == i ? 1.0f : cur * sg[j + 1];
          dec[e] = cur;
        }
      }
      if (quad < 2) {
        const float fi = sb[i] * skn[i];
        if (!upper) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = hf * 32 + e;
            v[e] = j < i ? fi * skn[j] * dec[e] * v[e] : 0.0f;
          }
        }
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(sA + i * S_ + hf * 32 + e) =
              make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      } else {
        const float fi = p.scale * sqn[i];
        if (!upper) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = hf * 32 + e;
            v[e] = fi * skn[j] * dec[e] * v[e];  // dec is 0 right of the diagonal
          }
        }
        named_bar(kBarP, 5 * 32);
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          const uint32_t off = swz128_offset(i, hf * 32 + e, 8192);
          st_split8(sm + PrepSmem::TWH + off, sm + PrepSmem::TWL + off, v + e);
        }
        fence_proxy_async();
      }
    }
    __syncthreads();
    if (tid == 0) {  // P hi, P lo images: one 16 KB store
      bulk_s2g(blob + kBlobP, base + PrepSmem::TWH, 16384);
      bulk_commit();
    }
    if (tid < 64 && jh + 1 < G) load_gates(h + 1);  // consumed at the next head's start
    // T = (I + A)^-1, A strictly lower triangular, by blocks:
    // (1) the four 16 x 16 diagonal blocks by forward substitution, two per
    //     warp of warps 0..1 (lanes 0..15 and 16..31), lane = column c:
    //     x_i = [i == c] - sum_{m < i} A[16b+i][16b+m] x_m;
    // (1b) the 32 x 32 diagonal blocks from them: lower-left 16 x 16 block
    //     X = -D1 (A10 D0) of each, D0 and D1 its two inverted diagonal blocks;
    // (2), (3) below: the 64 x 64 inverse from the two 32 x 32 ones.
    if (warp < 2) {
      const int b0 = 16 * (2 * warp + (lane >> 4)), c = lane & 15;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float* arow = sA + (b0 + i) * S_ + b0;
        float a0 = i == c ? 1.0f : 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
        for (int m = 0; m < i; m += 4) {
          const float4 av = *reinterpret_cast<const float4*>(arow + m);
          a0 = fmaf(-av.x, x[m], a0);
          if (m + 1 < i) a1 = fmaf(-av.y, x[m + 1], a1);
          if (m + 2 < i) a2 = fmaf(-av.z, x[m + 2], a2);
          if (m + 3 < i) a3 = fmaf(-av.w, x[m + 3], a3);
        }
        x[i] = (a0 + a1) + (a2 + a3);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 16; ++i) sA[(b0 + i) * S_ + b0 + c] = x[i];
    }
    __syncthreads();
    {  // (1b) Z = A10 D0 into sY rows 16 B .. 16 B + 15: thread -> block B, row r, 2 columns
      const int B = tid >> 7, r = (tid >> 3) & 15, c0 = (tid & 7) * 2;
      const float* arow = sA + (32 * B + 16 + r) * S_ + 32 * B;
      float z0 = 0.0f, z1 = 0.0f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float a = arow[m];
        const float2 d = *reinterpret_cast<const float2*>(sA + (32 * B + m) * S_ + 32 * B + c0);
        z0 = fmaf(a, d.x, z0);
        z1 = fmaf(a, d.y, z1);
      }
      *reinterpret_cast<float2*>(sY + (16 * B + r) * SY + c0) = make_float2(z0, z1);
    }
    __syncthreads();
    {  // X = -D1 Z into the lower-left 16 x 16 block of each 32 x 32 diagonal block
      const int B = tid >> 7, r = (tid >> 3) & 15, c0 = (tid & 7) * 2;
      const float* drow = sA + (32 * B + 16 + r) * S_ + 32 * B + 16;
      float x0 = 0.0f, x1 = 0.0f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float d = drow[m];
        const float2 z = *reinterpret_cast<const float2*>(sY + (16 * B + m) * SY + c0);
        x0 = fmaf(d, z.x, x0);
        x1 = fmaf(d, z.y, x1);
      }
      *reinterpret_cast<float2*>(sA + (32 * B + 16 + r) * S_ + 32 * B + c0) = make_float2(-x0, -x1);
    }
    __syncthreads();
    // (2) Y = A21 T11, (3) T21 = -T22 Y: thread -> row i, columns j0 .. j0 + 3.
    const int bi = tid >> 3, bj = (tid & 7) * 4;
    {
      const float* arow = sA + (32 + bi) * S_;
      float y[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 a = *reinterpret_cast<const float4*>(arow + k);
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 t = *reinterpret_cast<const float4*>(sA + (k + q) * S_ + bj);
          y[0] = fmaf(av[q], t.x, y[0]);
          y[1] = fmaf(av[q], t.y, y[1]);
          y[2] = fmaf(av[q], t.z, y[2]);
          y[3] = fmaf(av[q], t.w, y[3]);
        }
      }
      *reinterpret_cast<float4*>(sY + bi * SY + bj) = make_float4(y[0], y[1], y[2], y[3]);
    }
    __syncthreads();
    {
      const float* trow = sA + (32 + bi) * S_ + 32;
      float y[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 a = *reinterpret_cast<const float4*>(trow + k);
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 t = *reinterpret_cast<const float4*>(sY + (k + q) * SY + bj);
          y[0] = fmaf(av[q], t.x, y[0]);
          y[1] = fmaf(av[q], t.y, y[1]);
          y[2] = fmaf(av[q], t.z, y[2]);
          y[3] = fmaf(av[q], t.w, y[3]);
        }
      }
      *reinterpret_cast<float4*>(sA + (32 + bi) * S_ + bj) =
          make_float4(-y[0], -y[1], -y[2], -y[3]);
    }
    if (tid == 0) bulk_wait_read();  // the P store has read the Tw image space
    __syncthreads();
    // Tw = T diag(beta e^gam kn), Tu = T diag(beta) as hi + lo bf16 images:
    // one (row, 8-column chunk) per thread and step, 16-byte stores.
    for (int item = tid; item < 64 * 8; item += kPrepThreads) {
      const int i = item >> 3, q = item & 7;
      float tw[8], tu[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float t = sA[i * S_ + 8 * q + e];
        tw[e] = t * swj[8 * q + e];
        tu[e] = t * suj[8 * q + e];
      }
      const uint32_t off = swz128_offset(i, 8 * q, 8192);
      st_split8(sm + PrepSmem::TWH + off, sm + PrepSmem::TWL + off, tw);
      st_split8(sm + PrepSmem::TUH + off, sm + PrepSmem::TUL + off, tu);
    }
    fence_proxy_async();
    fence_before_sync();
    ok = __syncthreads_and(ok);
    fence_after_sync();
    const int i64 = m64_row(quad, lane);  // M = 64 rows: row 16 q + l in lane l < 16
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    // W = (Tw_hi + Tw_lo) K  (M = 64, N = 128, K = 64): B is the K tile,
    // MN-major: token rows, dk contiguous, boxes 16 KB apart.
    if (tid == 0 && ok) {
      const uint32_t idesc = idesc_bf16_f32(64, 128, false, true);
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < kC; kk += 16) {
          const uint32_t a_off = (part ? PrepSmem::TWL : PrepSmem::TWH) + kk * 2;
          mma_bf16(tm_wu, desc_sw128(base + a_off, 16, 1024),
                   desc_sw128(base + PrepSmem::KQ + (kk / 8) * 1024, 16384, 1024), idesc,
                   part > 0 || kk > 0);
        }
      mma_commit(mb_mma);
    }
    __syncwarp();
    ok = ok && mbar_wait(mb_mma, mma_phase & 1, kWaitBudget);
    ++mma_phase;
    fence_after_sync();
    {
      // W image staged in the (free) Q boxes of the K/Q tile, in its workspace
      // layout: box b of W at the Q box b.  Warp halves hf take columns 64 hf ..
      uint8_t* w_box = sm + PrepSmem::KQ + 8192 + hf * 16384;
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        float v[16];
        tmem_ld16(tm_wu + lane_addr + hf * 64 + c, v);
        tmem_ld_wait();
        if (i64 >= 0) {
          st_bf16x8(w_box + swz128_offset(i64, c, 8192), v);
          st_bf16x8(w_box + swz128_offset(i64, c + 8, 8192), v + 8);
        }
      }
      fence_proxy_async();
    }
    // V of this head (loaded during the previous head), rows past the chunk end zeroed.
    ok = mbar_wait(mb_v, jh & 1, kWaitBudget) && ok;
    if (L < kC) {
      for (int i = tid; i < (kC - L) * 8; i += kPrepThreads) {
        const int r = L + i / 8, q16 = i % 8;
        *reinterpret_cast<uint4*>(sm + PrepSmem::V + r * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sm + PrepSmem::V + 8192 + r * 128 + q16 * 16) =
            make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async();
    }
    fence_before_sync();
    ok = __syncthreads_and(ok);
    fence_after_sync();
    if (tid == 0) {
      bulk_s2g(blob + kBlobW, base + PrepSmem::KQ + 8192, 8192);
      bulk_s2g(blob + kBlobW + 8192, base + PrepSmem::KQ + 24576, 8192);
      bulk_commit();
      // Ut = (Tu_hi + Tu_lo) V  (M = 64, N = 128, K = 64): B is the V tile, MN-major.
      if (ok) {
        const uint32_t idesc = idesc_bf16_f32(64, 128, false, true);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int kk = 0; kk < kC; kk += 16) {
            const uint32_t a_off = (part ? PrepSmem::TUL : PrepSmem::TUH) + kk * 2;
            mma_bf16(tm_wu, desc_sw128(base + a_off, 16, 1024),
                     desc_sw128(base + PrepSmem::V + (kk / 8) * 1024, 8192, 1024), idesc,
                     part > 0 || kk > 0);
          }
        mma_commit(mb_mma);
      }
    }
    __syncwarp();
    ok = ok && mbar_wait(mb_mma, mma_phase & 1, kWaitBudget);
    ++mma_phase;
    fence_after_sync();
    __syncthreads();  // the Ut MMA has read V and the Tu images
    if (tid == 0 && jh + 1 < G) load_v(h + 1);  // next head's V, during this epilogue
    {
      // Ut staged in the (free) Tw/Tu image space, both slices, in the workspace
      // layout; warp halves hf take the Ut slice hf.
      uint8_t* slice_base = sm + PrepSmem::TWH + hf * 16384;
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        float v[16];
        tmem_ld16(tm_wu + lane_addr + hf * 64 + c, v);
        tmem_ld_wait();
        if (i64 >= 0) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<float4*>(slice_base + ut_offset(i64, c + 4 * e)) =
                make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        }
      }
      fence_proxy_async();
    }
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      bulk_s2g(blob + kBlobU, base + PrepSmem::TWH, 32768);
      bulk_commit();
    }
  }
  if (!ok && tid == 0) atomicOr(p.status, kStatusTimeout);
  if (tid == 0) bulk_wait_all();
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
  if (waiter) griddep_wait();
}

// ---------------------------------------------------------------------------
// Kernel 2: per (sequence, value head, 64-column slice of Dv), chunks in order.
//
// 17 warps.  TMEM lane quadrant q = warp % 4 is shared by warps q, q+4, q+8,
// q+12, which split every 64-column tile into 16-column groups cg = warp / 4:
//   U warps (q = 0, 1):       token rows 0..63 of W S^T -> U, U'
//   output warps (q = 2, 3):  token rows 0..63 of Q S^T and P U -> outputs
//   warps 0..15:             dk rows 0..127 of the state, 16 columns each
//   warp 16 (lane 0):        every MMA
//   thread 64 (output warp): every copy (W, Q, K, factors; P; Ut)
// MMAs, hi and lo operands side by side along N = 128:
//   D1 = [W; Q] [S_hi | S_lo]^T      rows 0..63 W S^T, 64..127 Q S^T
//   D2 = K^T [U'_hi | U'_lo]         rows = dk
//   D3 = [*; P_hi] [U_hi | U_lo] + [*; P_lo] [U_hi | U_lo]   rows 64..127 P U,
//        accumulated onto [fo Q S^T | 0], which the output warps store there
// Each result's two column halves are added in the epilogue.  The A tiles of
// D3 are 128-row windows that end with P_hi (P_lo): their first 64 rows are
// whatever precedes it in shared memory and only fill TMEM lanes 0..63, which
// nobody reads.
//
// Per chunk c the tensor pipe runs D1(c), D2(c), D3(c - 1): D3 never delays
// the serial path D1 -> U' -> D2 -> S.  The U and P images and the D3
// accumulator are double-buffered by chunk parity; P of chunk c is fetched
// while chunk c runs, chunk c's output is emitted while chunk c + 2 runs.
struct ScanSmem {
  // pipeline stage (x2): W, Q, K tiles; the stage's factors are at F0 / F1
  static constexpr uint32_t A1 = 0;         // [W box0 | Q box0 | W box1 | Q box1], 32 KB
  static constexpr uint32_t K = 32768;      // [K box0 | K box1], 16 KB
  static constexpr uint32_t STAGE = 49152;
  static constexpr uint32_t TX = 32768 + 16384 + kBlobFBytes;
  // single and parity buffers (1 KB aligned operand tiles)
  static constexpr uint32_t UT = 2 * STAGE;    // Ut slice f32 [64 tokens][64] (ut_offset), 16 KB
  static constexpr uint32_t SH = UT + 16384;   // S^T hi image [128 dk x 64 dv], 16 KB, then
  static constexpr uint32_t SL = SH + 16384;   //   S^T lo: one MN-major B operand of N = 128
  static constexpr uint32_t U2H = SL + 16384;  // U' hi image [64 tok x 64 dv], 8 KB, then U' lo
  static constexpr uint32_t U2L = U2H + 8192;
  static constexpr uint32_t U0 = U2L + 8192;   // U images of even chunks: hi, then lo
  static constexpr uint32_t P0 = U0 + 16384;   // P images of even chunks: hi, then lo
  static constexpr uint32_t U1 = P0 + 16384;   // U images of odd chunks
  static constexpr uint32_t P1 = U1 + 16384;   // P images of odd chunks
  static constexpr uint32_t F0 = P1 + 16384;   // fo[64], fu[64], e^{gam_L} of stage 0, then stage 1
  static constexpr uint32_t BYTES = F0 + 2 * kBlobFBytes;
};
// D3's first A window starts 8 KB before P_hi (the lo half of the U images
// before it), its second at P_hi.
static_assert(ScanSmem::P0 == ScanSmem::U0 + 16384 && ScanSmem::P1 == ScanSmem::U1 + 16384,
              "each P buffer must follow 8 KB of other tiles");
static_assert(ScanSmem::BYTES + 1024 <= 232448, "shared memory per CTA");
static_assert(PrepSmem::BYTES + 1024 <= 116736 - 2048, "two chunk_prep CTAs per SM");

constexpr int kScanWorkers = 512;               // warps 0..15
constexpr int kScanThreads = kScanWorkers + 32;  // + the issuing warp
constexpr int kBarU = 1;  // named barrier of the U warps and the issuer: U' images ready
constexpr int kBarW = 2;  // end-of-chunk barrier of the worker warps (not the issuer)

__global__ void __launch_bounds__(kScanThreads, 1) chunk_scan_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const RecurLaunch p, const uint8_t* __restrict__ ws, int n_chunks_max, int j0, int j1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  __shared__ uint64_t mb_ld[2], mb_p[2], mb_ut, mb_utfree, mb_a, mb_c, mb_d[2], mb_s, mb_e;
  __shared__ uint32_t tslot;
  __shared__ int s_base, s_bad;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, cg = warp >> 2;  // TMEM lane quadrant, 16-column group
  const bool issuer_warp = warp == 16;
  const bool issuer = tid == kScanWorkers;
  const bool loader = tid == 64;
  const int slice = blockIdx.x & 1;
  const int sh = blockIdx.x >> 1;
  const int h = sh % p.Hv, s = sh / p.Hv;
  const int hk = h / (p.Hv / p.Hk);

  const int slo = __ldg(p.cu + s), shi = __ldg(p.cu + s + 1);
  if (slo < 0 || shi <= slo || shi > p.T || __ldg(p.cu) != 0 || __ldg(p.cu + p.N) != p.T) {
    if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }
  // This launch's piece of the sequence: chunks [cb, ce) (all of them unless
  // the chunks are processed in pieces); it starts from the state the
  // previous piece left in the slot.
  const int nch_seq = (shi - slo + kC - 1) / kC;
  const int cb = min(j0, nch_seq), ce = min(j1, nch_seq);
  if (cb >= ce) return;
  const int lo = slo + cb * kC, hi = min(shi, slo + ce * kC);
  griddep_wait();               // the piece's blobs (and the previous piece's state) are complete
  griddep_launch_dependents();  // the next piece's preparation may start
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
      s_base = b + cb;
      s_bad = (bad || b + nch_seq > n_chunks_max) ? 1 : 0;
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
    mbar_init(smem_u32(&mb_p[0]), 1);
    mbar_init(smem_u32(&mb_p[1]), 1);
    mbar_init(smem_u32(&mb_ut), 1);
    mbar_init(smem_u32(&mb_utfree), 8);  // one arrival per U warp
    mbar_init(smem_u32(&mb_a), 1);
    mbar_init(smem_u32(&mb_c), 1);
    mbar_init(smem_u32(&mb_d[0]), 1);
    mbar_init(smem_u32(&mb_d[1]), 1);
    mbar_init(smem_u32(&mb_s), 1);
    mbar_init(smem_u32(&mb_e), 1);
    fence_mbar_init();
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
  // Loads W, Q, K and the factors of chunk c into stage c & 1 (loader only).
  auto issue_load = [&](int c) {
    const uint32_t sb = base + (c & 1) * ScanSmem::STAGE;
    const uint32_t mb = smem_u32(&mb_ld[c & 1]);
    const uint8_t* blob = blob_of(c);
    const int t0 = lo + c * kC;
    mbar_expect_tx(mb, ScanSmem::TX);
    bulk_g2s(sb + ScanSmem::A1, blob + kBlobW, 8192, mb);
    bulk_g2s(sb + ScanSmem::A1 + 16384, blob + kBlobW + 8192, 8192, mb);
    bulk_g2s(base + ScanSmem::F0 + (c & 1) * kBlobFBytes, blob + kBlobF, kBlobFBytes, mb);
    tma_load_3d(sb + ScanSmem::A1 + 8192, &tm_q, mb, 0, hk, t0);
    tma_load_3d(sb + ScanSmem::A1 + 24576, &tm_q, mb, 64, hk, t0);
    tma_load_3d(sb + ScanSmem::K, &tm_k, mb, 0, hk, t0);
    tma_load_3d(sb + ScanSmem::K + 8192, &tm_k, mb, 64, hk, t0);
  };
  auto issue_p = [&](int c) {  // P of chunk c into P buffer c & 1 (loader only)
    const uint32_t mb = smem_u32(&mb_p[c & 1]);
    mbar_expect_tx(mb, 16384);
    bulk_g2s(base + ((c & 1) ? ScanSmem::P1 : ScanSmem::P0), blob_of(c) + kBlobP, 16384, mb);
  };
  auto issue_ut = [&](int c) {  // loader only
    const uint32_t mb = smem_u32(&mb_ut);
    mbar_expect_tx(mb, 16384);
    bulk_g2s(base + ScanSmem::UT, blob_of(c) + kBlobU + slice * 16384, 16384, mb);
  };
  // D3 of chunk cc += [*; P_hi] [U_hi | U_lo] + [*; P_lo] [U_hi | U_lo]  (M = 128,
  // N = 128, K = 64) from U buffer cc & 1 onto TMEM buffer cc & 1, which holds
  // [fo Q S^T | 0] of that chunk (issuer only).
  auto issue_d3 = [&](int cc) {
    if (!mbar_wait(smem_u32(&mb_p[cc & 1]), (cc >> 1) & 1, kWaitBudget)) return false;
    fence_after_sync();
    const uint32_t id3 = idesc_bf16_f32(128, 128, false, true);
    const uint32_t ub = base + ((cc & 1) ? ScanSmem::U1 : ScanSmem::U0);
    const uint32_t pb = base + ((cc & 1) ? ScanSmem::P1 : ScanSmem::P0);
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int kk = 0; kk < kC; kk += 16)
        mma_bf16(tmem + 256 + (cc & 1) * 128, desc_sw128(pb + part * 8192 - 8192 + kk * 2, 16, 1024),
                 desc_sw128(ub + (kk / 8) * 1024, 8192, 1024), id3, true);
    mma_commit(smem_u32(&mb_d[cc & 1]));
    return true;
  };
  // Copies issued so far (loader), for the error path.  Write-after-read
  // hazards on the destinations are ordered by the mbarrier and barrier waits
  // before each copy; writers of generic data that a copy overwrites (the
  // K-tail zeros) fence their own stores.
  int issued_ld = 0, issued_ut = 0, issued_p = 0;
  if (loader) {
    issue_ut(0);
    issue_load(0);
    issue_p(0);
    issued_ut = issued_ld = issued_p = 1;
    if (nchunks > 1) {
      issue_load(1);
      issue_p(1);
      issued_ld = issued_p = 2;
    }
  }

  // State: worker (quad, cg, lane) owns dk = 32 quad + lane and dv columns
  // 16 cg .. 16 cg + 15 of this slice, in f32.
  const int dk = quad * 32 + lane;
  float S[16];
  float* pool = p.pool + ((int64_t)slot * p.Hv + h) * kD * kD;
  const bool init = cb > 0 || p.has_init == nullptr || __ldg(p.has_init + s) != 0;
  if (!issuer_warp) {
#pragma unroll
    for (int e = 0; e < 16; ++e)
      S[e] = init ? pool[(int64_t)(slice * 64 + cg * 16 + e) * kD + dk] : 0.0f;
  }
  auto write_s = [&]() {  // S^T hi / lo images: row dk, 16 dv columns (MN-major B operand)
#pragma unroll
    for (int e = 0; e < 16; e += 8) {
      const uint32_t off = swz128_offset(dk, cg * 16 + e, 16384);
      st_split8(sm + ScanSmem::SH + off, sm + ScanSmem::SL + off, S + e);
    }
  };
  if (!issuer_warp) write_s();
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tm_d1 = tmem, tm_d2 = tmem + 128, tm_d3 = tmem + 256;  // D3: 2 x 128
  const bool u_warp = !issuer_warp && quad < 2;
  const int row = (quad & 1) * 32 + lane;  // token row of U and output warps
  // Output of chunk cc by the output warps: O = fo Q S^T + P U, the sum of
  // D3's two column halves.
  auto emit_output = [&](int cc) {
    const int t0 = lo + cc * kC;
    const int L = min(kC, hi - t0);
    const uint32_t d3 = tm_d3 + (cc & 1) * 128 + lane_addr + cg * 16;
    float a[16], b[16];
    tmem_ld16(d3, a);
    tmem_ld16(d3 + 64, b);
    tmem_ld_wait();
    if (row < L) {
#pragma unroll
      for (int e = 0; e < 16; ++e) a[e] += b[e];
      __nv_bfloat16* dst = out + ((int64_t)(t0 + row) * p.Hv + h) * kD + slice * 64 + cg * 16;
      st_bf16x8(dst, a);
      st_bf16x8(dst + 8, a + 8);
    }
  };

  bool ok = true;
  int c = 0;
  int last_mma = -1;  // issuer: last chunk whose MMAs were issued
  for (; c < nchunks; ++c) {
    const int st = c & 1;
    uint8_t* sst = sm + st * ScanSmem::STAGE;
    const uint32_t sb = base + st * ScanSmem::STAGE;
    const int t0 = lo + c * kC;
    const int L = min(kC, hi - t0);
    const float* F = reinterpret_cast<const float*>(sm + ScanSmem::F0 + st * kBlobFBytes);
    ok = mbar_wait(smem_u32(&mb_ld[st]), (c >> 1) & 1, kWaitBudget) && ok;
    if (issuer_warp) {
      // The workers finished chunk c - 1: S images of chunk c, U images and the
      // D3 preload of chunk c - 1 are in place.  No signal in time means they
      // have stopped (they leave the loop only at their end-of-chunk barrier,
      // so none of them will reach the U barrier again).
      const bool go = c < 1 || mbar_wait(smem_u32(&mb_s), (c - 1) & 1, kWaitBudget);
      if (!__all_sync(0xffffffffu, go)) {  // leave the loop as a whole warp
        ok = false;
        break;
      }
      if (issuer && ok) {
        fence_after_sync();
        // D1 = [W; Q] [S_hi | S_lo]^T  (M = 128, N = 128, K = 128)
        const uint32_t id1 = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
        for (int kk = 0; kk < kD; kk += 16)
          mma_bf16(tm_d1,
                   desc_sw128(sb + ScanSmem::A1 + (kk / 64) * 16384 + (kk % 64) * 2, 16, 1024),
                   desc_sw128(base + ScanSmem::SH + (kk / 8) * 1024, 16384, 1024), id1, kk > 0);
        mma_commit(smem_u32(&mb_a));
        last_mma = c;
      }
      __syncwarp();
      named_bar(kBarU, 256 + 32);  // U' images written, K tail zeroed, Ut consumed
      if (issuer) {
        if (ok) {
          fence_after_sync();
          // D2 = K^T [U'_hi | U'_lo]  (M = 128 dk, N = 128, K = 64 tokens; A = K tile MN-major)
          const uint32_t id2 = idesc_bf16_f32(128, 128, true, true);
#pragma unroll
          for (int kk = 0; kk < kC; kk += 16)
            mma_bf16(tm_d2, desc_sw128(sb + ScanSmem::K + (kk / 8) * 1024, 8192, 1024),
                     desc_sw128(base + ScanSmem::U2H + (kk / 8) * 1024, 8192, 1024), id2,
                     kk > 0);
          mma_commit(smem_u32(&mb_c));
        }
        // The previous chunk's P U, behind D2.
        if (c >= 1 && ok) ok = issue_d3(c - 1);
      }
    } else if (u_warp) {
      // U = Ut - W S^T and U' = diag(fu) U, this thread's row and 16 columns,
      // written as hi + lo images (U' first: D2 waits for it).
      if (L < kC) {  // zero K rows past the chunk end (D2 meets them with U' rows of 0)
        const int ui = (cg * 2 + quad) * 32 + lane;  // 0 .. 255 over the U warps
        for (int i = ui; i < (kC - L) * 16; i += 256) {
          const int r = L + i / 16, q16 = i % 16;
          *reinterpret_cast<uint4*>(sst + ScanSmem::K + (q16 >> 3) * 8192 + r * 128 +
                                    (q16 & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      ok = mbar_wait(smem_u32(&mb_ut), c & 1, kWaitBudget) && ok;
      float u[16];
      {
        const uint8_t* ut = sm + ScanSmem::UT;
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const float4 f = *reinterpret_cast<const float4*>(ut + ut_offset(row, cg * 16 + e));
          u[e] = f.x;
          u[e + 1] = f.y;
          u[e + 2] = f.z;
          u[e + 3] = f.w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&mb_utfree));  // this warp is done with Ut
      const float fu = F[64 + row];
      ok = mbar_wait(smem_u32(&mb_a), c & 1, kWaitBudget) && ok;
      fence_after_sync();
      {
        float wa[16], wb[16];
        tmem_ld16(tm_d1 + lane_addr + cg * 16, wa);
        tmem_ld16(tm_d1 + lane_addr + 64 + cg * 16, wb);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) u[e] -= wa[e] + wb[e];
      }
#pragma unroll
      for (int e = 0; e < 16; e += 8) {
        float u2[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) u2[x] = fu * u[e + x];
        const uint32_t off = swz128_offset(row, cg * 16 + e, 8192);
        st_split8(sm + ScanSmem::U2H + off, sm + ScanSmem::U2L + off, u2);
      }
      fence_proxy_async();
      fence_before_sync();
      named_bar(kBarU, 256 + 32);
      // U buffer c & 1 was last read by D3 of chunk c - 2.
      if (c >= 2) ok = mbar_wait(smem_u32(&mb_d[st]), ((c - 2) >> 1) & 1, kWaitBudget) && ok;
      uint8_t* ub = sm + (st ? ScanSmem::U1 : ScanSmem::U0);
#pragma unroll
      for (int e = 0; e < 16; e += 8) {
        const uint32_t off = swz128_offset(row, cg * 16 + e, 8192);
        st_split8(ub + off, ub + 8192 + off, u + e);
      }
      fence_proxy_async();
    } else {
      // The output of chunk c - 2 (its D3 ran during chunk c - 1), which frees
      // D3 buffer c & 1; then [fo Q S^T | 0] of this chunk into that buffer,
      // for D3 of this chunk to accumulate onto.
      if (c >= 2) {
        ok = mbar_wait(smem_u32(&mb_d[st]), ((c - 2) >> 1) & 1, kWaitBudget) && ok;
        if (loader && c < nchunks) {  // P buffer c & 1 is free: fetch P of this chunk
          issue_p(c);
          issued_p = c + 1;
        }
        fence_after_sync();
        emit_output(c - 2);
      }
      const float fo = F[row];
      ok = mbar_wait(smem_u32(&mb_a), c & 1, kWaitBudget) && ok;
      fence_after_sync();
      float qa[16], qb[16];
      tmem_ld16(tm_d1 + lane_addr + cg * 16, qa);
      tmem_ld16(tm_d1 + lane_addr + 64 + cg * 16, qb);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        qa[e] = fo * (qa[e] + qb[e]);
        qb[e] = 0.0f;
      }
      const uint32_t d3 = tm_d3 + st * 128 + lane_addr + cg * 16;
      tmem_st16(d3, qa);
      tmem_st16(d3 + 64, qb);
      tmem_st_wait();
      // Once the U warps have read Ut, fetch the next chunk's.
      if (loader && c + 1 < nchunks) {
        ok = mbar_wait(smem_u32(&mb_utfree), c & 1, kWaitBudget) && ok;
        issue_ut(c + 1);
        issued_ut = c + 2;
      }
    }
    if (!issuer_warp) {
      // S = e^{gam_L} S + D2  (f32, registers), new S^T hi / lo images.
      ok = mbar_wait(smem_u32(&mb_c), c & 1, kWaitBudget) && ok;
      fence_after_sync();
      const float dL = F[128];
      float da[16], db[16];
      tmem_ld16(tm_d2 + lane_addr + cg * 16, da);
      tmem_ld16(tm_d2 + lane_addr + 64 + cg * 16, db);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) S[e] = fmaf(dL, S[e], da[e] + db[e]);
      write_s();
      fence_proxy_async();
      fence_before_sync();
      ok = named_bar_and(kBarW, kScanWorkers, ok);
      if (!ok) break;
      if (tid == 0) mbar_arrive(smem_u32(&mb_s));  // chunk c done: the issuer may go on
      fence_after_sync();
      // Every reader of this stage (D1, D2 and the factor reads) is done:
      // refill it with chunk c + 2.
      if (loader && c + 2 < nchunks) {
        issue_load(c + 2);
        issued_ld = c + 3;
      }
    }
  }
  if (c == nchunks) {
    if (issuer_warp) {  // the last chunk's P U, once the workers are done with it
      const bool go = mbar_wait(smem_u32(&mb_s), (nchunks - 1) & 1, kWaitBudget);
      if (issuer) ok = go && issue_d3(nchunks - 1) && ok;
      else ok = go && ok;
    }
    if (!u_warp && !issuer_warp) {                  // the last two chunks' outputs
      if (nchunks >= 2) {
        const int cc = nchunks - 2;
        ok = mbar_wait(smem_u32(&mb_d[cc & 1]), (cc >> 1) & 1, kWaitBudget) && ok;
        fence_after_sync();
        emit_output(cc);
      }
      const int cc = nchunks - 1;
      ok = mbar_wait(smem_u32(&mb_d[cc & 1]), (cc >> 1) & 1, kWaitBudget) && ok;
      fence_after_sync();
      emit_output(cc);
    }
  }
  ok = __syncthreads_and(ok);
  if (c < nchunks || !ok) {
    // A wait ran out: report; let in-flight MMAs and loads finish (bounded); free TMEM.
    if (issuer) {
      atomicOr(p.status, kStatusTimeout);
      if (last_mma >= 0) {
        mma_commit(smem_u32(&mb_e));
        mbar_wait(smem_u32(&mb_e), 0, kWaitBudget);
      }
    }
    if (loader) {
      for (int k = c; k < issued_ld; ++k)
        mbar_wait(smem_u32(&mb_ld[k & 1]), (k >> 1) & 1, kWaitBudget);
      for (int k = c; k < issued_ut; ++k) mbar_wait(smem_u32(&mb_ut), k & 1, kWaitBudget);
      for (int k = max(0, issued_p - 2); k < issued_p; ++k)
        mbar_wait(smem_u32(&mb_p[k & 1]), (k >> 1) & 1, kWaitBudget);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
    return;
  }
  if (!issuer_warp) {
#pragma unroll
    for (int e = 0; e < 16; ++e) pool[(int64_t)(slice * 64 + cg * 16 + e) * kD + dk] = S[e];
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---- host ------------------------------------------------------------------------

constexpr int kPieces = 4;  // pieces of chunk indices when the chains are few

}  // namespace

bool chunked_supported(int Dk, int Dv, bool bf16) { return bf16 && Dk == kD && Dv == kD; }

size_t chunked_workspace_bytes(int64_t T, int64_t N, int64_t Hv, int64_t Dk, int64_t Dv) {
  if (Dk != kD || Dv != kD) return 0;
  return static_cast<size_t>(max_chunks(T, N) * Hv) * kBlobBytes;
}

// Few chains (the scan would leave most SMs idle behind the preparation): the
// chunks are taken in pieces of consecutive chunk indices.  Piece i's scan
// runs beside piece i + 1's preparation on the other SMs; each launch after
// the first is a programmatic dependent launch, the scan waits for its
// piece's blobs (and, through the preparation's last CTA, for the previous
// scan), and every launch keeps the stream's order for what follows.
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
  const int64_t blocks = static_cast<int64_t>(p.N) * p.Hv * 2;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const int64_t cmax = (p.T + kC - 1) / kC;  // chunks of the longest possible sequence
  const bool pieces = 2 * blocks <= sm_count() && cmax >= 16;
  const int step = pieces ? static_cast<int>((cmax + kPieces - 1) / kPieces) : 0x7fffffff;
  const int n_pieces = pieces ? static_cast<int>((cmax + step - 1) / step) : 1;
  for (int i = 0; i < n_pieces; ++i) {
    const int j0 = pieces ? i * step : 0, j1 = pieces ? j0 + step : 0x7fffffff;
    // chunks of the piece: at most `step` of each sequence, and no more than all
    const int64_t n_piece = pieces ? std::min<int64_t>(nch, (int64_t)p.N * step) : nch;
    cudaError_t e = launch_maybe_pdl(chunk_prep_kernel, dim3(static_cast<unsigned>(n_piece), p.Hk),
                                     dim3(kPrepThreads), PrepSmem::BYTES + 1024, s, i > 0, tq, tk,
                                     tv, p, ws, j0, j1);
    if (e != cudaSuccess) return e;
    e = launch_maybe_pdl(chunk_scan_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kScanThreads),
                         ScanSmem::BYTES + 1024, s, pieces, tq, tk, p,
                         static_cast<const uint8_t*>(ws), static_cast<int>(nch), j0, j1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace gdn
