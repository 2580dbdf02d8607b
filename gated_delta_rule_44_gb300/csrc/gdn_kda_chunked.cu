// gdn_kda_chunked.cu -- chunked (C = 64) varlen prefill of the KDA recurrence
// (one log decay per KEY CHANNEL) on tcgen05 tensor cores.
//
// [cpu_ops.cpp] (vllm.cpp, src/vt/cpu/cpu_ops.cpp) KdaHeadTokenStep /
// KdaGatedDeltaRuleKernel define the recurrence token by token, per (sequence,
// value head) with state S = [Dv, Dk]:
//   S[:, d] *= e^{g_t[d]};  u = beta_t (v_t - S k_t);  S += u k_t^T;  o_t = S (scale q_t)
// and the KdaChunkPrefillKernel comment names a chunked GPU form without
// printing it.  The chunk form below is derived from the recurrence.  For one
// chunk of L <= 64 tokens with state S0 at its start, E_t = e^{g_t} (per
// channel) and products of E over token ranges, every one a decay from an
// earlier token to a later one (so none exceeds 1 when g <= 0):
//   A_ts = beta_t sum_d k_t[d] k_s[d] prod_{s<u<=t} E_u[d]     (s < t)
//   P_ts = scale  sum_d q_t[d] k_s[d] prod_{s<u<=t} E_u[d]     (s <= t)
//   T = (I + A)^-1,  Tb = T diag(beta)
//   Ke_t = k_t . prod_{u<=t} E_u,  Qe_t = q_t . prod_{u<=t} E_u,  Kd_s = k_s . prod_{u>s} E_u
//   W = Tb Ke,  Ut = Tb V,  U = Ut - W S0^T
//   O = scale Qe S0^T + P U
//   S_L = S0 diag(prod_u E_u) + U^T Kd
//
// A and P.  The decay inside each dot product depends on the channel, so it
// cannot be taken out as in the scalar-decay form.  They are split by 16-token
// sub-chunks.  For t in sub-chunk I and s in an earlier one,
//   prod_{s<u<=t} E_u = prod_{s<u<16I} E_u . prod_{16I<=u<=t} E_u
// (both decays, <= 1), so those blocks are dot products of pre-scaled rows and
// go to the tensor core as hi + lo bf16 images.  Pairs inside one sub-chunk
// take running products of E from s to t on CUDA cores in f32.
//
// Two launches on the caller's stream:
//  1. kda_prep (one CTA per (chunk, value head), all chunks in parallel): E, A
//     and P (f32), T by blocks, W^T = Ke^T Tb^T (tcgen05); writes the
//     chunk's blob: the -W^T, P, Tb, Qe and Kd images (hi + lo bf16 pairs but
//     W) in the shared-memory layouts the second kernel feeds to the tensor
//     core, and prod_u E_u.
//  2. kda_scan (one CTA per (sequence, value head), its chunks in order): per
//     chunk, loads the blob and V, then
//        D1 = [Ut^T - S W^T | S Qe^T]   (M = 128 dv; Ut^T = V^T Tb^T on the tensor core)
//        U^T (hi + lo) into TMEM; D2: S += U^T Kd;  D3: O^T += U^T P^T
//        S' images for the next D1; S' diag(prod E of the next chunk) in TMEM,
//        onto which the next D2 accumulates; the output rows.
//
// Precision: as the scalar-decay chunked form -- T, S, U, P, Qe and Kd enter
// the tensor core as hi + lo bf16 pairs (hi = x rounded to 8 significant bits,
// lo = bf16(x - hi)) with products hi*hi + hi*lo + lo*hi; W and Ke as single
// bf16 values (W reaches the output only through the W S^T correction).
//
// Partial chunks: g and beta of rows past the chunk end are taken as 0, so
// those rows of T are unit rows, their Tb, W, Ut and U rows are zero, and the
// K, Q, V rows there (the next sequence's tokens, or zeros past the tensor
// end) never reach a stored value.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "gdn_chunk_common.cuh"
#include "gdn_internal.h"
#include "tcgen05.cuh"

namespace gdn {
namespace {

using namespace umma;
using namespace chunk;

constexpr long long kWaitBudget = 2000000000LL;  // ~1 s of SM clock per wait

// Blob of one (chunk, value head) in the workspace.
constexpr uint32_t kBW = 0;          // -W^T image [128 dk][64 tok], MN-major B operand (16 KB)
constexpr uint32_t kBP = 16384;      // P hi, P lo: K-major [64 i][64 j] (8 KB each)
constexpr uint32_t kBT = 32768;      // Tb hi, Tb lo: K-major [64 i][64 s] (8 KB each)
constexpr uint32_t kBQ = 49152;      // Qe hi, Qe lo: K-major [64 tok][128 dk] (16 KB each)
constexpr uint32_t kBK = 81920;      // Kd hi, Kd lo: same layout (16 KB each)
constexpr uint32_t kBImg = 114688;   // the images above: copied to the scan's stage as they are
constexpr uint32_t kBE = 114688;     // prod_u E_u per channel, f32 [128]
constexpr uint32_t kBlob = 115712;   // 113 KB
constexpr int kPrepWaves = 3;        // pieces: ~3 waves of preparation CTAs beside each scan piece

// bf16 element (t, d) of a [64 tok][128] tile stored as two SW128 boxes of 64 columns.
__device__ __forceinline__ float tile_at(const uint8_t* tile, int t, int d) {
  return __bfloat162float(
      *reinterpret_cast<const __nv_bfloat16*>(tile + swz128_offset(t, d, 8192)));
}

// Four consecutive bf16 values (8 bytes, 8-byte aligned) as f32.
__device__ __forceinline__ void ld_bf16x4(const uint8_t* p, float* v) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(u.x << 16);
  v[1] = __uint_as_float(u.x & 0xffff0000u);
  v[2] = __uint_as_float(u.y << 16);
  v[3] = __uint_as_float(u.y & 0xffff0000u);
}

// hi + lo bf16 pair of x into two images at the same offset.
__device__ __forceinline__ void st_split1(uint8_t* hi, uint8_t* lo, float x) {
  const float h = split_hi(x);
  *reinterpret_cast<uint16_t*>(hi) = static_cast<uint16_t>(__float_as_uint(h) >> 16);
  *reinterpret_cast<__nv_bfloat16*>(lo) = __float2bfloat16_rn(__fsub_rn(x, h));
}

// ---------------------------------------------------------------------------
// Kernel 1: per (chunk, value head).  16 warps.
struct KPrep {
  static constexpr uint32_t K = 0;           // K tile [64 tok][128 dk], 2 SW128 boxes (TMA)
  static constexpr uint32_t Q = 16384;       // Q tile
  static constexpr uint32_t E = 32768;       // e^{g}, f32 [64][128]; then the P hi, lo images
  static constexpr uint32_t OP = 65536;      // bf16 operand images of the off-diagonal A, P:
  static constexpr uint32_t kBox = 12288;    //   96 rows of 128 B per 64-channel box
  static constexpr uint32_t RBH = OP;                   //   R hi: rows 0-15 R_1, 16-47 R_2, 48-95 R_3
  static constexpr uint32_t RBL = OP + 2 * kBox;        //   R lo
  static constexpr uint32_t LBH = OP + 4 * kBox;        //   L hi: rows 32 (I - 1) + [0, 16) k, + [16, 32) q
  static constexpr uint32_t LBL = OP + 6 * kBox;        //   L lo
  static constexpr uint32_t KE = OP;                    // then: Ke image (16 KB), later -W^T
  static constexpr uint32_t QE = OP + 16384;            //       Qe hi, lo (16 KB each)
  static constexpr uint32_t KD = OP + 49152;            //       Kd hi, lo (16 KB each)
  static constexpr uint32_t TB = OP + 8 * kBox;         // Tb hi, lo images (8 KB each)
  static constexpr uint32_t AT = TB + 16384;            // A, then T in place, f32 [64][kAs]
  static constexpr uint32_t kAs = 68;
  static constexpr uint32_t PM = AT + 64 * kAs * 4;     // P, f32 [64][kAs]
  static constexpr uint32_t Z = PM + 64 * kAs * 4;      // T solve scratch [32][kZs]
  static constexpr uint32_t kZs = 36;
  static constexpr uint32_t BLK = Z + 32 * kZs * 4;     // sub-chunk products [4][128]
  static constexpr uint32_t BETA = BLK + 4 * 128 * 4;   // [64]
  static constexpr uint32_t EL = BETA + 64 * 4;         // prod_u E_u [128]
  static constexpr uint32_t BYTES = EL + 128 * 4;
};
static_assert(KPrep::KD + 32768 <= KPrep::TB, "images fit before Tb");
// The M = 128 product reads 32 rows past each 96-row R box; they exist in
// shared memory (the next box or image) and only feed unread rows of D.
static_assert(KPrep::RBL + 2 * KPrep::kBox + 32 * 128 <= KPrep::TB, "R reads stay in bounds");
static_assert(KPrep::BYTES + 1024 <= 232448, "shared memory per CTA");

constexpr int kPrepThreads = 512;

__global__ void __launch_bounds__(kPrepThreads, 1) kda_prep_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_g, const RecurLaunch p, uint8_t* __restrict__ ws, int j0,
    int j1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  __shared__ uint64_t mbar_tma, mbar_mma;
  __shared__ uint32_t tslot;
  __shared__ int s_seq, s_chunk, s_gc, s_ok;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  const int hk = h / (p.Hv / p.Hk);

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
      if (bad && blockIdx.x == 0 && h == 0) atomicOr(p.status, kStatusBadSeqlens);
    }
  }
  __syncthreads();
  // In pieces, this launch runs beside the scan of the previous piece and
  // must not complete before it: CTA (0, 0) waits for it on every way out.
  const bool waiter = blockIdx.x == 0 && blockIdx.y == 0;
  if (!s_ok) {  // uniform: outside this piece, past the last chunk, or malformed cu_seqlens
    if (waiter) griddep_wait();
    return;
  }
  const int t0 = __ldg(p.cu + s_seq) + kC * s_chunk;
  const int L = min(kC, __ldg(p.cu + s_seq + 1) - t0);
  const uint32_t base = smem_u32(sm);
  const uint32_t mb_tma = smem_u32(&mbar_tma), mb_mma = smem_u32(&mbar_mma);
  uint8_t* blob = ws + ((int64_t)s_gc * p.Hv + h) * kBlob;

  if (tid == 0) {
    mbar_init(mb_tma, 1);
    mbar_init(mb_mma, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_expect_tx(mb_tma, 4 * 8192 + 64 * kD * 4);
    tma_load_3d(base + KPrep::E, &tm_g, mb_tma, 0, h, t0);
    tma_load_3d(base + KPrep::K, &tm_k, mb_tma, 0, hk, t0);
    tma_load_3d(base + KPrep::K + 8192, &tm_k, mb_tma, 64, hk, t0);
    tma_load_3d(base + KPrep::Q, &tm_q, mb_tma, 0, hk, t0);
    tma_load_3d(base + KPrep::Q + 8192, &tm_q, mb_tma, 64, hk, t0);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tslot), 128);

  const uint8_t* sK = sm + KPrep::K;
  const uint8_t* sQ = sm + KPrep::Q;
  float* sE = reinterpret_cast<float*>(sm + KPrep::E);
  float* sA = reinterpret_cast<float*>(sm + KPrep::AT);
  float* sP = reinterpret_cast<float*>(sm + KPrep::PM);
  float* sZ = reinterpret_cast<float*>(sm + KPrep::Z);
  float* sBlk = reinterpret_cast<float*>(sm + KPrep::BLK);
  float* sBeta = reinterpret_cast<float*>(sm + KPrep::BETA);
  float* sEL = reinterpret_cast<float*>(sm + KPrep::EL);
  constexpr int AS = KPrep::kAs;
  const int d = tid & 127, quarter = tid >> 7;

  if (tid < 64) sBeta[tid] = tid < L ? __ldg(p.beta + (int64_t)(t0 + tid) * p.Hv + h) : 0.0f;
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tslot;
  bool ok = __syncthreads_and(mbar_wait(mb_tma, 0, kWaitBudget));
  if (!ok) {  // the g, K, Q tiles did not land: touch none of their bytes
    if (tid == 0) {
      atomicOr(p.status, kStatusTimeout);
      mbar_wait(mb_tma, 0, kWaitBudget);  // let the copies in flight finish
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
    if (waiter) griddep_wait();
    return;
  }

  // Off-diagonal operands.  For t in sub-chunk I and s in an earlier one,
  // prod_{s<u<=t} E_u = prod_{s<u<16I} E_u . prod_{16I<=u<=t} E_u, so
  //   A_ts = beta_t R_I[s] . L_k[t],  P_ts = scale R_I[s] . L_q[t]
  // with R_I[s] = k_s . prod_{s<u<16I} E_u and L_k[t], L_q[t] = k_t, q_t .
  // prod_{16I<=u<=t} E_u (every factor a decay).  They go to the tensor core
  // as hi + lo bf16 images (products hi.hi + hi.lo + lo.hi, about 16
  // significant bits) in one product D = R L^T over all of them: M = 128
  // (the R rows, 96 of them read), N = 96 (the L rows); the entries of
  // sub-chunk I are D[r_I + s][32 (I - 1) + x] with r_I = 0, 16, 48.
  // Pass 1: thread (d, b) turns its g entries of sub-chunk b into E = e^{g}
  // in place (g taken as 0 past the chunk end, where the rows are the next
  // sequence's or the tensor's zero fill), runs the product from the
  // sub-chunk start to t and, for b >= 1, writes the L rows of sub-chunk b.
  {
    const int b = quarter;
    float f = 1.0f;
#pragma unroll 4
    for (int r = 0; r < 16; ++r) {
      const int t = 16 * b + r;
      const float e = t < L ? expf(sE[t * kD + d]) : 1.0f;
      sE[t * kD + d] = e;
      f *= e;
      if (b > 0) {
        const uint32_t ok_k = swz128_offset(32 * (b - 1) + r, d, KPrep::kBox);
        const uint32_t ok_q = swz128_offset(32 * (b - 1) + 16 + r, d, KPrep::kBox);
        st_split1(sm + KPrep::LBH + ok_k, sm + KPrep::LBL + ok_k, tile_at(sK, t, d) * f);
        st_split1(sm + KPrep::LBH + ok_q, sm + KPrep::LBL + ok_q, tile_at(sQ, t, d) * f);
      }
    }
    sBlk[b * kD + d] = f;
  }
  __syncthreads();
  // Pass 2: the R rows.  Warp w < 12 takes the sub-chunk pair (J, I) =
  // (0,1), (0,2), (0,3), (1,2), (1,3), (2,3) for w / 2 and rows
  // 16 J + 8 (w % 2) .. + 7; lane = channel quad.  It runs prod_{s<u<16I} E_u
  // backward from the end of its rows, started from the products of the rows
  // after them in J and of the whole sub-chunks between J and I.
  if (warp < 12) {
    const int u = warp >> 1, hh = warp & 1, c0 = 4 * lane;
    const int J = u < 3 ? 0 : u < 5 ? 1 : 2;
    const int I = u < 3 ? u + 1 : u < 5 ? u - 1 : 3;
    float w[4] = {1.0f, 1.0f, 1.0f, 1.0f};
    for (int bb = J + 1; bb < I; ++bb) {
      const float4 bl = *reinterpret_cast<const float4*>(sBlk + bb * kD + c0);
      w[0] *= bl.x;
      w[1] *= bl.y;
      w[2] *= bl.z;
      w[3] *= bl.w;
    }
    if (hh == 0) {
#pragma unroll
      for (int r = 8; r < 16; ++r) {
        const float4 e = *reinterpret_cast<const float4*>(sE + (16 * J + r) * kD + c0);
        w[0] *= e.x;
        w[1] *= e.y;
        w[2] *= e.z;
        w[3] *= e.w;
      }
    }
    const int rbase = I == 1 ? 0 : I == 2 ? 16 : 48;
#pragma unroll
    for (int r = 7; r >= 0; --r) {
      const int t = 16 * J + 8 * hh + r;
      float kv[4];
      ld_bf16x4(sK + swz128_offset(t, c0, 8192), kv);
      uint32_t h0, l0, h1, l1;
      split2(kv[0] * w[0], kv[1] * w[1], h0, l0);
      split2(kv[2] * w[2], kv[3] * w[3], h1, l1);
      const uint32_t o = swz128_offset(rbase + t, c0, KPrep::kBox);
      *reinterpret_cast<uint2*>(sm + KPrep::RBH + o) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(sm + KPrep::RBL + o) = make_uint2(l0, l1);
      const float4 e = *reinterpret_cast<const float4*>(sE + t * kD + c0);
      w[0] *= e.x;
      w[1] *= e.y;
      w[2] *= e.z;
      w[3] *= e.w;
    }
  }
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (tid == 0) {  // D into TMEM columns 0-95; the diagonal blocks run meanwhile
    const uint32_t idesc = idesc_bf16_f32(128, 96, false, false);
#pragma unroll
    for (int part = 0; part < 3; ++part)  // hi.hi, hi.lo, lo.hi
#pragma unroll
      for (int kk = 0; kk < kD; kk += 16) {
        const uint32_t ko = (kk >> 6) * KPrep::kBox + (kk & 63) * 2;
        mma_bf16(tmem, desc_sw128(base + (part == 2 ? KPrep::RBL : KPrep::RBH) + ko, 16, 1024),
                 desc_sw128(base + (part == 1 ? KPrep::LBL : KPrep::LBH) + ko, 16, 1024), idesc,
                 part > 0 || kk > 0);
      }
    mma_commit(mb_mma);
  }

  // Diagonal sub-blocks (s <= t inside one sub-chunk).  Warp w takes the
  // columns s = w % 8 and s = 15 - w % 8 of sub-chunks 2 (w / 8) and
  // 2 (w / 8) + 1: 17 rows per column pair, so the warps carry equal work and
  // every trip count is warp-uniform.  Lane (b2, c) = (lane / 16, lane % 16)
  // holds 8 channels of sub-chunk b = 2 (w / 8) + b2, the quads
  // c + 16 ((j + b2) mod 2) for j < 2, and carries R = k_s . prod_{s<u<=t} E_u
  // over them down the column.  The rows after the first go two at a time:
  // the 16 lanes of a sub-chunk reduce the four partial dot products (A and P
  // of both rows) by halving, so lane c ends with the full sum of value
  // 2 (c / 8) + (c / 4) % 2.
  {
    const int b2 = lane >> 4, c = lane & 15;
    const int b = 2 * (warp >> 3) + b2;
    int ch[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) ch[j] = 4 * (c + 16 * ((j + b2) & 1));
    const bool up8 = (c & 8) != 0, up4 = (c & 4) != 0;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const int s = pass == 0 ? (warp & 7) : 15 - (warp & 7);
      float R[8];
      {  // row t = s: P only, R = k_s
        const int t = 16 * b + s;
        float qt[8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          ld_bf16x4(sK + swz128_offset(t, ch[j], 8192), R + 4 * j);
          ld_bf16x4(sQ + swz128_offset(t, ch[j], 8192), qt + 4 * j);
        }
        float2 p2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int e = 0; e < 8; e += 2)
          p2 = __ffma2_rn(make_float2(qt[e], qt[e + 1]), make_float2(R[e], R[e + 1]), p2);
        float pv = p2.x + p2.y;
#pragma unroll
        for (int m = 1; m < 16; m <<= 1) pv += __shfl_xor_sync(0xffffffffu, pv, m);
        if (c == 0) sP[t * AS + 16 * b + s] = p.scale * pv;
      }
#pragma unroll 1
      for (int tt = s + 1; tt < 16; tt += 2) {
        const bool two = tt + 1 < 16;  // warp-uniform
        const int t = 16 * b + tt;
        float v[4];
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          float2 a2 = make_float2(0.0f, 0.0f), p2 = make_float2(0.0f, 0.0f);
          if (x == 0 || two) {
            const int tx = t + x;
            float kt[8], qt[8];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              ld_bf16x4(sK + swz128_offset(tx, ch[j], 8192), kt + 4 * j);
              ld_bf16x4(sQ + swz128_offset(tx, ch[j], 8192), qt + 4 * j);
              const float4 e = *reinterpret_cast<const float4*>(sE + tx * kD + ch[j]);
              const float2 r0 = __fmul2_rn(make_float2(R[4 * j], R[4 * j + 1]), make_float2(e.x, e.y));
              const float2 r1 =
                  __fmul2_rn(make_float2(R[4 * j + 2], R[4 * j + 3]), make_float2(e.z, e.w));
              R[4 * j] = r0.x;
              R[4 * j + 1] = r0.y;
              R[4 * j + 2] = r1.x;
              R[4 * j + 3] = r1.y;
            }
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float2 r = make_float2(R[e], R[e + 1]);
              a2 = __ffma2_rn(make_float2(kt[e], kt[e + 1]), r, a2);
              p2 = __ffma2_rn(make_float2(qt[e], qt[e + 1]), r, p2);
            }
          }
          v[2 * x] = a2.x + a2.y;
          v[2 * x + 1] = p2.x + p2.y;
        }
        // Halving: keep two of four (xor 8), one of two (xor 4), then add (xor 2, 1).
        const float k0 = up8 ? v[2] : v[0], k1 = up8 ? v[3] : v[1];
        const float s0 = up8 ? v[0] : v[2], s1 = up8 ? v[1] : v[3];
        const float h0 = k0 + __shfl_xor_sync(0xffffffffu, s0, 8);
        const float h1 = k1 + __shfl_xor_sync(0xffffffffu, s1, 8);
        float w = (up4 ? h1 : h0) + __shfl_xor_sync(0xffffffffu, up4 ? h0 : h1, 4);
        w += __shfl_xor_sync(0xffffffffu, w, 2);
        w += __shfl_xor_sync(0xffffffffu, w, 1);
        if ((c & 3) == 0 && (!up8 || two)) {
          const int tw = t + (up8 ? 1 : 0);
          if (up4)
            sP[tw * AS + 16 * b + s] = p.scale * w;
          else
            sA[tw * AS + 16 * b + s] = sBeta[tw] * w;
        }
      }
    }
  }
  // The off-diagonal blocks from D: warp w < 12 reads columns 32 (I - 1) ..
  // 32 I - 1, I = w / 4 + 1, over its TMEM lane quarter (row m of D in lane
  // m); the lanes whose row is a key row of R_I write theirs.
  ok = __syncthreads_and(mbar_wait(mb_mma, 0, kWaitBudget));  // uniform: tcgen05.ld is warp-wide
  fence_after_sync();
  if (!ok) {  // the MMAs did not complete: drain them (bounded) and leave
    if (tid == 0) {
      atomicOr(p.status, kStatusTimeout);
      mbar_wait(mb_mma, 0, kWaitBudget);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
    if (waiter) griddep_wait();
    return;
  }
  if (warp < 12) {
    const int qd = warp & 3, I = (warp >> 2) + 1;
    float v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(qd * 32) << 16) + 32 * (I - 1), v);
    tmem_ld_wait();
    const int sc = 32 * qd + lane - (I == 1 ? 0 : I == 2 ? 16 : 48);
    if (sc >= 0 && sc < 16 * I) {
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const int t = 16 * I + x;
        sA[t * AS + sc] = sBeta[t] * v[x];
        sP[t * AS + sc] = p.scale * v[16 + x];
      }
    }
  }
  fence_before_sync();
  __syncthreads();  // A and P complete; the operand images are dead
  fence_after_sync();

  // Warps 8-15 write the images over the operand space while warps 0-7
  // solve for T (its barriers are named barrier 1 over those 256 threads).
  if (warp >= 8) {
    // Thread (dir, seg, quad) covers channels 4 quad .. 4 quad + 3 of the
    // 16 rows of sub-chunk seg: forward (dir 0) with prod_{u<=t} E_u, started
    // from the products of the sub-chunks before (Ke, Qe and, from the last
    // sub-chunk, prod_u E_u), or backward (dir 1) with prod_{u>s} E_u started
    // from the products of the sub-chunks after (Kd).
    const int item = tid - 256, dir = item >> 7, seg = (item >> 5) & 3, c0 = 4 * (item & 31);
    float run[4];
    {
      const float4 one = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
      float4 acc = one;
      for (int b = dir ? seg + 1 : 0; b < (dir ? 4 : seg); ++b) {
        const float4 bl = *reinterpret_cast<const float4*>(sBlk + b * kD + c0);
        acc.x *= bl.x;
        acc.y *= bl.y;
        acc.z *= bl.z;
        acc.w *= bl.w;
      }
      run[0] = acc.x;
      run[1] = acc.y;
      run[2] = acc.z;
      run[3] = acc.w;
    }
    if (dir == 0) {
#pragma unroll 4
      for (int r = 0; r < 16; ++r) {
        const int t = 16 * seg + r;
        const float4 e = *reinterpret_cast<const float4*>(sE + t * kD + c0);
        run[0] *= e.x;
        run[1] *= e.y;
        run[2] *= e.z;
        run[3] *= e.w;
        float kv[4], qv[4];
        const uint32_t off = swz128_offset(t, c0, 8192);
        ld_bf16x4(sK + off, kv);
        ld_bf16x4(sQ + off, qv);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          kv[x] *= run[x];
          qv[x] *= run[x];
        }
        *reinterpret_cast<uint2*>(sm + KPrep::KE + off) =
            make_uint2(pack_bf16x2(kv[0], kv[1]), pack_bf16x2(kv[2], kv[3]));
        uint32_t h0, l0, h1, l1;
        split2(qv[0], qv[1], h0, l0);
        split2(qv[2], qv[3], h1, l1);
        *reinterpret_cast<uint2*>(sm + KPrep::QE + off) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(sm + KPrep::QE + 16384 + off) = make_uint2(l0, l1);
      }
      if (seg == 3)
        *reinterpret_cast<float4*>(sEL + c0) = make_float4(run[0], run[1], run[2], run[3]);
    } else {
#pragma unroll 4
      for (int r = 15; r >= 0; --r) {
        const int t = 16 * seg + r;
        float kv[4];
        const uint32_t off = swz128_offset(t, c0, 8192);
        ld_bf16x4(sK + off, kv);
#pragma unroll
        for (int x = 0; x < 4; ++x) kv[x] *= run[x];
        uint32_t h0, l0, h1, l1;
        split2(kv[0], kv[1], h0, l0);
        split2(kv[2], kv[3], h1, l1);
        *reinterpret_cast<uint2*>(sm + KPrep::KD + off) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(sm + KPrep::KD + 16384 + off) = make_uint2(l0, l1);
        const float4 e = *reinterpret_cast<const float4*>(sE + t * kD + c0);
        run[0] *= e.x;
        run[1] *= e.y;
        run[2] *= e.z;
        run[3] *= e.w;
      }
    }
  } else {
    // T = (I + A)^-1 (A strictly lower triangular) by blocks, on warps 0-7:
    // (1) the four 16 x 16 diagonal blocks by forward substitution, a
    //     half-warp per block with lane = column c:
    //     x_i = [i == c] - sum_{m < i} A[16b+i][16b+m] x_m;
    // (2) each 32 x 32 diagonal block from its two: lower-left block
    //     X = -D1 (A10 D0), D0 and D1 the inverted diagonal blocks;
    // (3) the lower-left 32 x 32 block T21 = -T22 (A21 T11).
    constexpr int ZS = KPrep::kZs;
    if (warp < 2) {
      const int b0 = 16 * (2 * warp + (lane >> 4)), c = lane & 15;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float* arow = sA + (b0 + i) * AS + b0;
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
      for (int i = 0; i < 16; ++i) sA[(b0 + i) * AS + b0 + c] = x[i];
    }
    named_bar(1, 256);
    {  // (2) Z = A10 D0 (thread: block B, row r, two columns), then X = -D1 Z
      const int B = tid >> 7, r = (tid >> 3) & 15, c0 = (tid & 7) * 2;
      const float* arow = sA + (32 * B + 16 + r) * AS + 32 * B;
      float z0 = 0.0f, z1 = 0.0f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float a = arow[m];
        const float2 dv = *reinterpret_cast<const float2*>(sA + (32 * B + m) * AS + 32 * B + c0);
        z0 = fmaf(a, dv.x, z0);
        z1 = fmaf(a, dv.y, z1);
      }
      *reinterpret_cast<float2*>(sZ + (16 * B + r) * ZS + c0) = make_float2(z0, z1);
      named_bar(1, 256);
      const float* drow = sA + (32 * B + 16 + r) * AS + 32 * B + 16;
      float x0 = 0.0f, x1 = 0.0f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float dv = drow[m];
        const float2 z = *reinterpret_cast<const float2*>(sZ + (16 * B + m) * ZS + c0);
        x0 = fmaf(dv, z.x, x0);
        x1 = fmaf(dv, z.y, x1);
      }
      *reinterpret_cast<float2*>(sA + (32 * B + 16 + r) * AS + 32 * B + c0) =
          make_float2(-x0, -x1);
      // The upper-right 16 x 16 block of each 32 x 32 inverse is zero (nothing
      // above the diagonal of A was written); step (3) reads whole rows.
      *reinterpret_cast<float2*>(sA + (32 * B + r) * AS + 32 * B + 16 + c0) =
          make_float2(0.0f, 0.0f);
    }
    named_bar(1, 256);
    {  // (3) Y = A21 T11, then T21 = -T22 Y: thread -> row i, columns j0 .. j0 + 3
      const int bi = tid >> 3, bj = (tid & 7) * 4;
      float y[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const float* arow = sA + (32 + bi) * AS;
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 av4 = *reinterpret_cast<const float4*>(arow + k);
        const float av[4] = {av4.x, av4.y, av4.z, av4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 tv = *reinterpret_cast<const float4*>(sA + (k + q) * AS + bj);
          y[0] = fmaf(av[q], tv.x, y[0]);
          y[1] = fmaf(av[q], tv.y, y[1]);
          y[2] = fmaf(av[q], tv.z, y[2]);
          y[3] = fmaf(av[q], tv.w, y[3]);
        }
      }
      *reinterpret_cast<float4*>(sZ + bi * ZS + bj) = make_float4(y[0], y[1], y[2], y[3]);
      named_bar(1, 256);
      const float* trow = sA + (32 + bi) * AS + 32;
      float w[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 tv4 = *reinterpret_cast<const float4*>(trow + k);
        const float tv[4] = {tv4.x, tv4.y, tv4.z, tv4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 yv = *reinterpret_cast<const float4*>(sZ + (k + q) * ZS + bj);
          w[0] = fmaf(tv[q], yv.x, w[0]);
          w[1] = fmaf(tv[q], yv.y, w[1]);
          w[2] = fmaf(tv[q], yv.z, w[2]);
          w[3] = fmaf(tv[q], yv.w, w[3]);
        }
      }
      *reinterpret_cast<float4*>(sA + (32 + bi) * AS + bj) = make_float4(-w[0], -w[1], -w[2], -w[3]);
    }
  }
  __syncthreads();

  // Tb = T diag(beta) and P as hi + lo images (zero above the diagonal); the P
  // images take the space of E, which is dead.
  for (int item = tid; item < 64 * 8; item += kPrepThreads) {
    const int i = item >> 3, q = item & 7;
    float tv[8], pv[8], bv[8];
    *reinterpret_cast<float4*>(tv) = *reinterpret_cast<const float4*>(sA + i * AS + 8 * q);
    *reinterpret_cast<float4*>(tv + 4) = *reinterpret_cast<const float4*>(sA + i * AS + 8 * q + 4);
    *reinterpret_cast<float4*>(pv) = *reinterpret_cast<const float4*>(sP + i * AS + 8 * q);
    *reinterpret_cast<float4*>(pv + 4) = *reinterpret_cast<const float4*>(sP + i * AS + 8 * q + 4);
    *reinterpret_cast<float4*>(bv) = *reinterpret_cast<const float4*>(sBeta + 8 * q);
    *reinterpret_cast<float4*>(bv + 4) = *reinterpret_cast<const float4*>(sBeta + 8 * q + 4);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const bool lower = 8 * q + e <= i;
      tv[e] = lower ? tv[e] * bv[e] : 0.0f;
      pv[e] = lower ? pv[e] : 0.0f;
    }
    const uint32_t off = swz128_offset(i, 8 * q, 8192);
    st_split8(sm + KPrep::TB + off, sm + KPrep::TB + 8192 + off, tv);
    st_split8(sm + KPrep::E + off, sm + KPrep::E + 8192 + off, pv);
  }
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (tid == 0) {
    // W^T = Ke^T Tb^T (M = 128 dk, N = 64 tokens, K = 64 tokens): A = Ke MN-major,
    // B = Tb hi, lo (K-major).
    const uint32_t idesc = idesc_bf16_f32(128, 64, true, false);
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int kk = 0; kk < kC; kk += 16)
        mma_bf16(tmem, desc_sw128(base + KPrep::KE + (kk / 8) * 1024, 8192, 1024),
                 desc_sw128(base + KPrep::TB + part * 8192 + kk * 2, 16, 1024), idesc,
                 part > 0 || kk > 0);
    mma_commit(mb_mma);
  } else if (tid == 32) {  // the images that are final go out meanwhile
    bulk_s2g(blob + kBP, base + KPrep::E, 16384);
    bulk_s2g(blob + kBT, base + KPrep::TB, 16384);
    bulk_s2g(blob + kBQ, base + KPrep::QE, 32768);
    bulk_s2g(blob + kBK, base + KPrep::KD, 32768);
    bulk_s2g(blob + kBE, base + KPrep::EL, 512);
    bulk_commit();
  }
  ok = __syncthreads_and(mbar_wait(mb_mma, 1, kWaitBudget));  // uniform: tcgen05.ld is warp-wide
  fence_after_sync();
  if (ok && warp < 4) {  // -W^T image over Ke (the MMA has read Ke)
    const uint32_t la = static_cast<uint32_t>(warp * 32) << 16;
    const int dk = tid;
#pragma unroll 1
    for (int j0 = 0; j0 < kC; j0 += 32) {
      float w[32];
      tmem_ld32(tmem + la + j0, w);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        float nv[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) nv[x] = -w[e + x];
        st_bf16x8(sm + KPrep::KE + swz128_offset(dk, j0 + e, 16384), nv);
      }
    }
  }
  fence_proxy_async();
  fence_before_sync();
  ok = __syncthreads_and(ok);
  if (tid == 32) {
    if (ok) {
      bulk_s2g(blob + kBW, base + KPrep::KE, 16384);
      bulk_commit();
    }
    bulk_wait_all();  // the blob is complete (and the shared memory read) before exit
  }
  if (!ok && tid == 0) {
    atomicOr(p.status, kStatusTimeout);
    mbar_wait(mb_mma, 1, kWaitBudget);  // the MMA in flight
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
  if (waiter) griddep_wait();
}

// ---------------------------------------------------------------------------
// Kernel 2: per (sequence, value head), its chunks in order.  4 warps; thread
// dv owns TMEM lane dv (row dv of the state).
struct KScan {
  static constexpr uint32_t SH = 0;                 // S hi image [128 dv][128 dk], K-major
  static constexpr uint32_t SL = 32768;             // S lo image
  static constexpr uint32_t ST = 65536;             // the chunk's blob images (kBImg bytes)
  static constexpr uint32_t V = ST + kBImg;         // V tile [64 tok][128 dv], 2 SW128 boxes
  static constexpr uint32_t OST = V + 16384;        // output staging [32 tok][128 dv] bf16
  static constexpr uint32_t ELB = OST + 8192;       // prod_u E_u of two chunks, f32 [2][128]
  static constexpr uint32_t BYTES = ELB + 1024;
};
static_assert(KScan::V % 1024 == 0, "swizzled tiles are 1024-byte aligned");
static_assert(KScan::BYTES + 1024 <= 232448, "shared memory per CTA");
constexpr uint32_t kSD1 = 0;    // TMEM: D1 = [U^T | O^T] (128 columns; O^T of odd chunks at kSO1)
constexpr uint32_t kSS = 128;   //       the f32 state S[dv][dk] (128)
constexpr uint32_t kSU = 256;   //       U^T hi | lo as packed bf16 pairs (32 + 32)
constexpr uint32_t kSO1 = 320;  //       O^T of odd chunks (64): a chunk's output leaves while
                                //       the next chunk's D1 runs
__device__ __forceinline__ uint32_t o_col(int c) { return (c & 1) ? kSO1 : kSD1 + 64; }
constexpr int kScanThreads = 128;

__global__ void __launch_bounds__(kScanThreads, 1) kda_scan_kernel(
    const __grid_constant__ CUtensorMap tm_v, const RecurLaunch p, const uint8_t* __restrict__ ws,
    int j0, int j1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  __shared__ uint64_t mbar_ld, mbar_ldb, mbar_el, mbar_mma;
  __shared__ uint32_t tslot;
  __shared__ int s_gc0, s_bad;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % p.Hv, s = blockIdx.x / p.Hv;

  const int slo = __ldg(p.cu + s), shi = __ldg(p.cu + s + 1);
  if (slo < 0 || shi <= slo || shi > p.T || __ldg(p.cu) != 0 || __ldg(p.cu + p.N) != p.T) {
    if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }
  // This launch's piece of the sequence: chunks [cb, ce); it starts from the
  // state the previous piece left in the slot.
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
    for (int idx = tid; idx < (hi - lo) * 16; idx += kScanThreads) {
      const int t = lo + idx / 16, q16 = idx % 16;
      *reinterpret_cast<uint4*>(out + ((int64_t)t * p.Hv + h) * kD + q16 * 8) =
          make_uint4(0, 0, 0, 0);
    }
    return;
  }
  if (warp == 0) {
    bool bad = false;
    const int b = chunk_base(p.cu, s, bad);
    if (lane == 0) {
      s_gc0 = b + cb;
      s_bad = bad ? 1 : 0;
    }
  }
  const uint32_t base = smem_u32(sm);
  const uint32_t mb_ld = smem_u32(&mbar_ld), mb_ldb = smem_u32(&mbar_ldb),
                 mb_el = smem_u32(&mbar_el), mb_mma = smem_u32(&mbar_mma);
  if (tid == 0) {
    mbar_init(mb_ld, 1);
    mbar_init(mb_ldb, 1);
    mbar_init(mb_el, 1);
    mbar_init(mb_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tslot), 512);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tslot;
  if (s_bad) {  // an earlier sequence's range is empty or decreasing
    if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
    return;
  }
  const int nch = (hi - lo + kC - 1) / kC;
  auto blob = [&](int c) { return ws + ((int64_t)(s_gc0 + c) * p.Hv + h) * kBlob; };
  const float* elb = reinterpret_cast<const float*>(sm + KScan::ELB);
  const int dv = tid;
  const uint32_t la = static_cast<uint32_t>(warp * 32) << 16;
  float* prow = p.pool + (((int64_t)slot * p.Hv + h) * kD + dv) * kD;
  const bool init = cb > 0 || p.has_init == nullptr || __ldg(p.has_init + s) != 0;
  // Copies and MMAs issued but not yet seen complete (thread 0's books, for a
  // clean exit after a wait that gave up).
  int pend_ld = -1, pend_ldb = -1, pend_el = -1, n_mma = 0;
  bool pend_mma = false;
  // A chunk's stage in two parts: A (Tb, -W^T, Qe and V: read by D1 only) and
  // B (P and Kd: read by D2 / D3), each on its own mbarrier, so the next
  // chunk's part A lands while this chunk's state update runs, and part B
  // after D2 / D3 have read this chunk's.
  auto load_a = [&](int cc) {
    const uint8_t* b = blob(cc);
    mbar_expect_tx(mb_ld, 4 * 16384 + 2 * 8192);
    bulk_g2s(base + KScan::ST + kBW, b + kBW, 16384, mb_ld);
    bulk_g2s(base + KScan::ST + kBT, b + kBT, 16384, mb_ld);
    bulk_g2s(base + KScan::ST + kBQ, b + kBQ, 16384, mb_ld);
    bulk_g2s(base + KScan::ST + kBQ + 16384, b + kBQ + 16384, 16384, mb_ld);
    tma_load_3d(base + KScan::V, &tm_v, mb_ld, 0, h, lo + cc * kC);
    tma_load_3d(base + KScan::V + 8192, &tm_v, mb_ld, 64, h, lo + cc * kC);
    pend_ld = cc;
  };
  auto load_b = [&](int cc) {
    const uint8_t* b = blob(cc);
    mbar_expect_tx(mb_ldb, 3 * 16384);
    bulk_g2s(base + KScan::ST + kBP, b + kBP, 16384, mb_ldb);
    bulk_g2s(base + KScan::ST + kBK, b + kBK, 16384, mb_ldb);
    bulk_g2s(base + KScan::ST + kBK + 16384, b + kBK + 16384, 16384, mb_ldb);
    pend_ldb = cc;
  };
  __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + KScan::OST);
  // Output rows of chunk cc from its O^T columns: 32 tokens at a time through
  // the staging rows (called by every thread).
  auto emit_out = [&](int cc) {
    const int t0c = lo + cc * kC, Lc = min(kC, hi - t0c);
#pragma unroll 1
    for (int j0 = 0; j0 < Lc; j0 += 32) {
      float o[32];
      tmem_ld32(tmem + o_col(cc) + la + j0, o);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) ost[e * kD + dv] = __float2bfloat16_rn(o[e]);
      __syncthreads();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int idx = q * kScanThreads + tid;  // 16-byte vector: token idx / 16
        const int r = idx >> 4, c16 = idx & 15;
        if (j0 + r < Lc)
          *reinterpret_cast<uint4*>(out + ((int64_t)(t0c + j0 + r) * p.Hv + h) * kD + c16 * 8) =
              *reinterpret_cast<const uint4*>(ost + r * kD + c16 * 8);
      }
      __syncthreads();
    }
  };

  if (tid == 0) {
    mbar_expect_tx(mb_el, 512);
    bulk_g2s(base + KScan::ELB, blob(0) + kBE, 512, mb_el);
    pend_el = 0;
    load_a(0);
    load_b(0);
  }
  bool ok = mbar_wait(mb_el, 0, kWaitBudget);
  if (tid == 0 && ok) pend_el = -1;
  // Initial state: its hi + lo images, and S0 diag(prod E) in TMEM.
  for (int j = 0; j < kD; j += 16) {
    float v[16];
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
      float4 f = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (init) f = *reinterpret_cast<const float4*>(prow + j + e);
      v[e] = f.x;
      v[e + 1] = f.y;
      v[e + 2] = f.z;
      v[e + 3] = f.w;
    }
#pragma unroll
    for (int e = 0; e < 16; e += 8) {
      const uint32_t off = swz128_offset(dv, j + e, 16384);
      st_split8(sm + KScan::SH + off, sm + KScan::SL + off, v + e);
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] *= elb[j + e];
    tmem_st16(tmem + kSS + la + j, v);
  }
  tmem_st_wait();
  fence_proxy_async();
  fence_before_sync();
  ok = __syncthreads_and(ok);

  const uint32_t id_ut = idesc_bf16_f32(128, 64, true, false);
  const uint32_t id_w = idesc_bf16_f32(128, 64, false, true);
  const uint32_t id_q = idesc_bf16_f32(128, 64, false, false);
  const uint32_t id_d2 = idesc_bf16_f32(128, 128, false, true);
  const uint32_t id_d3 = idesc_bf16_f32(128, 64, false, false);

  for (int c = 0; c < nch && ok; ++c) {
    const bool last = c + 1 == nch;
    if (tid == 0 && !last) {
      // prod E of the next chunk, for the state update of this one
      mbar_expect_tx(mb_el, 512);
      bulk_g2s(base + KScan::ELB + ((c + 1) & 1) * 512, blob(c + 1) + kBE, 512, mb_el);
      pend_el = c + 1;

    }
    ok = __syncthreads_and(mbar_wait(mb_ld, c & 1, kWaitBudget) &&
                           mbar_wait(mb_ldb, c & 1, kWaitBudget));
    if (!ok) break;
    if (tid == 0) {
      pend_ld = -1;
      pend_ldb = -1;
      fence_after_sync();
      // Ut^T = V^T Tb^T into D1[:, 0:64]  (A = V MN-major, M = dv; B = Tb hi, lo)
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < kC; kk += 16)
          mma_bf16(tmem + kSD1, desc_sw128(base + KScan::V + (kk / 8) * 1024, 8192, 1024),
                   desc_sw128(base + KScan::ST + kBT + part * 8192 + kk * 2, 16, 1024), id_ut,
                   part > 0 || kk > 0);
      // D1[:, 0:64] += S (-W)^T  (A = S hi, lo; B = the -W^T image, MN-major)
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < kD; kk += 16)
          mma_bf16(tmem + kSD1,
                   desc_sw128(base + (part ? KScan::SL : KScan::SH) + (kk / 64) * 16384 +
                                  (kk % 64) * 2,
                              16, 1024),
                   desc_sw128(base + KScan::ST + kBW + (kk / 8) * 1024, 8192, 1024), id_w, true);
      // O^T = S Qe^T (this chunk's O columns): S hi Qe hi, S lo Qe hi, S hi Qe lo
#pragma unroll
      for (int pr = 0; pr < 3; ++pr) {
        const uint32_t sa = pr == 1 ? KScan::SL : KScan::SH;
        const uint32_t qo = pr == 2 ? 16384 : 0;
#pragma unroll
        for (int kk = 0; kk < kD; kk += 16)
          mma_bf16(tmem + o_col(c),
                   desc_sw128(base + sa + (kk / 64) * 16384 + (kk % 64) * 2, 16, 1024),
                   desc_sw128(base + KScan::ST + kBQ + qo + (kk / 64) * 8192 + (kk % 64) * 2, 16,
                              1024),
                   id_q, pr > 0 || kk > 0);
      }
      mma_commit(mb_mma);
      pend_mma = true;
    }
    if (c > 0) emit_out(c - 1);  // the previous chunk's output, beside D1
    ok = mbar_wait(mb_mma, n_mma & 1, kWaitBudget);
    ++n_mma;
    if (tid == 0 && ok) pend_mma = false;
    ok = __syncthreads_and(ok);  // uniform: tcgen05.ld / st are warp-wide
    if (!ok) break;
    fence_after_sync();
    if (tid == 0 && !last) load_a(c + 1);  // D1 has read Tb, -W^T, Qe and V
    // U^T = D1[:, 0:64] as hi + lo pairs into TMEM; the O^T columns scaled in
    // place: O^T starts as scale (Qe S^T)^T, onto which P U accumulates.
    {
#pragma unroll 1
      for (int j0 = 0; j0 < kC; j0 += 32) {
        float u[32], qs[32];
        tmem_ld32(tmem + kSD1 + la + j0, u);
        tmem_ld32(tmem + o_col(c) + la + j0, qs);
        tmem_ld_wait();
#pragma unroll
        for (int j1 = 0; j1 < 32; j1 += 16) {
          uint32_t uh[8], ul[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) split2(u[j1 + e], u[j1 + e + 1], uh[e / 2], ul[e / 2]);
          tmem_st8u(tmem + kSU + la + (j0 + j1) / 2, uh);
          tmem_st8u(tmem + kSU + 32 + la + (j0 + j1) / 2, ul);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) qs[e] *= p.scale;
        tmem_st32(tmem + o_col(c) + la + j0, qs);
      }
      tmem_st_wait();
    }
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      fence_after_sync();
      // S += U^T Kd: U hi Kd hi, U lo Kd hi, U hi Kd lo (A = U^T from TMEM; B = Kd MN-major)
#pragma unroll
      for (int pr = 0; pr < 3; ++pr) {
        const uint32_t ua = pr == 1 ? 32 : 0;
        const uint32_t ko = pr == 2 ? 16384 : 0;
#pragma unroll
        for (int kk = 0; kk < kC; kk += 16)
          mma_bf16_ta(tmem + kSS, tmem + kSU + ua + kk / 2,
                      desc_sw128(base + KScan::ST + kBK + ko + (kk / 8) * 1024, 8192, 1024), id_d2,
                      true);
      }
      // O^T += U^T P^T: U hi P hi, U hi P lo, U lo P hi (B = P, K-major)
#pragma unroll
      for (int pr = 0; pr < 3; ++pr) {
        const uint32_t ua = pr == 2 ? 32 : 0;
        const uint32_t po = pr == 1 ? 8192 : 0;
#pragma unroll
        for (int kk = 0; kk < kC; kk += 16)
          mma_bf16_ta(tmem + o_col(c), tmem + kSU + ua + kk / 2,
                      desc_sw128(base + KScan::ST + kBP + po + kk * 2, 16, 1024), id_d3, true);
      }
      mma_commit(mb_mma);
      pend_mma = true;
    }
    ok = mbar_wait(mb_mma, n_mma & 1, kWaitBudget);
    ++n_mma;
    if (tid == 0 && ok) pend_mma = false;
    if (!last) {
      const bool el_ok = mbar_wait(mb_el, (c + 1) & 1, kWaitBudget);
      if (tid == 0 && el_ok) pend_el = -1;
      ok = el_ok && ok;
    }
    ok = __syncthreads_and(ok);
    if (!ok) break;
    fence_after_sync();
    if (tid == 0 && !last) load_b(c + 1);  // D2 / D3 have read P and Kd
    // S' = S0 diag(prod E) + U^T Kd: its images for the next D1 and S' diag(prod
    // E of the next chunk) back into TMEM; the last chunk's S' goes to the pool.
    const float* eln = elb + ((c + 1) & 1) * 128;
#pragma unroll 1
    for (int j0 = 0; j0 < kD; j0 += 32) {
      float v[32];
      tmem_ld32(tmem + kSS + la + j0, v);
      tmem_ld_wait();
      if (last) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(prow + j0 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      } else {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          const uint32_t off = swz128_offset(dv, j0 + e, 16384);
          st_split8(sm + KScan::SH + off, sm + KScan::SL + off, v + e);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] *= eln[j0 + e];
        tmem_st32(tmem + kSS + la + j0, v);
      }
    }
    if (!last) tmem_st_wait();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
  }

  if (ok) emit_out(nch - 1);
  // teardown: copies and MMAs still in flight (after a wait that gave up) land
  // first, then the TMEM is freed.
  if (!ok && tid == 0) {
    atomicOr(p.status, kStatusTimeout);
    if (pend_ld >= 0) mbar_wait(mb_ld, pend_ld & 1, kWaitBudget);
    if (pend_ldb >= 0) mbar_wait(mb_ldb, pend_ldb & 1, kWaitBudget);
    if (pend_el >= 0) mbar_wait(mb_el, pend_el & 1, kWaitBudget);
    if (pend_mma) mbar_wait(mb_mma, (n_mma - 1) & 1, kWaitBudget);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// g [rows, heads, 128] f32; box = 64 rows x 1 head x 128 channels, unswizzled
// (row-major [64][128] in shared memory).  Rows past `rows` read as zeros.
bool make_g_map(CUtensorMap* m, const float* g, int rows, int heads) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 4,
                           static_cast<cuuint64_t>(heads) * kD * 4};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kD), 1, static_cast<cuuint32_t>(kC)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(g), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool kda_chunked_supported(int Dk, int Dv, bool bf16) { return bf16 && Dk == kD && Dv == kD; }

size_t kda_chunked_workspace_bytes(int64_t T, int64_t N, int64_t Hv, int64_t Dk, int64_t Dv) {
  if (Dk != kD || Dv != kD) return 0;
  return static_cast<size_t>(max_chunks(T, N) * Hv) * kBlob;
}

// In pieces of chunk indices when the chains are few, as the scalar-decay
// two-launch form: each piece's preparation runs beside the previous piece's
// scan (programmatic dependent launch).
cudaError_t launch_kda_chunked(const ChunkedLaunch& c, cudaStream_t s) {
  const RecurLaunch& p = c.r;
  CUtensorMap tq, tk, tv, tg;
  if (!make_map(&tq, p.q, p.T, p.Hk) || !make_map(&tk, p.k, p.T, p.Hk) ||
      !make_map(&tv, p.v, p.T, p.Hv) || !make_g_map(&tg, p.g, p.T, p.Hv))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(kda_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    KPrep::BYTES + 1024);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(kda_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      KScan::BYTES + 1024);
  });
  if (attr_err != cudaSuccess) return attr_err;
  uint8_t* ws = static_cast<uint8_t*>(c.workspace);
  const int64_t nch = max_chunks(p.T, p.N);
  if (nch > 0x7fffffff || p.Hv > 65535) return cudaErrorInvalidConfiguration;
  const int64_t blocks = static_cast<int64_t>(p.N) * p.Hv;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const int64_t cmax = (p.T + kC - 1) / kC;
  const bool pieces = 2 * blocks <= sm_count() && cmax >= 16;
  // A piece's preparation (one CTA per chunk of each sequence and value head,
  // one per SM) fills about kPrepWaves waves of the SMs the scan leaves free,
  // and holds at least 8 chunk indices (each piece restarts the scan).
  const int64_t per_chunk = static_cast<int64_t>(p.N) * p.Hv;
  const int64_t free_sms = std::max<int64_t>(1, sm_count() - blocks);
  const int step = pieces ? static_cast<int>(std::min<int64_t>(
                                cmax, std::max<int64_t>(8, kPrepWaves * free_sms / per_chunk)))
                          : 0x7fffffff;
  const int n_pieces = pieces ? static_cast<int>((cmax + step - 1) / step) : 1;
  for (int i = 0; i < n_pieces; ++i) {
    const int j0 = pieces ? i * step : 0, j1 = pieces ? j0 + step : 0x7fffffff;
    const int64_t n_piece = pieces ? std::min<int64_t>(nch, (int64_t)p.N * step) : nch;
    cudaError_t e = launch_maybe_pdl(kda_prep_kernel, dim3(static_cast<unsigned>(n_piece), p.Hv),
                                     dim3(kPrepThreads), KPrep::BYTES + 1024, s, i > 0, tq, tk, tg, p,
                                     ws, j0, j1);
    if (e != cudaSuccess) return e;
    e = launch_maybe_pdl(kda_scan_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kScanThreads),
                         KScan::BYTES + 1024, s, pieces, tv, p, static_cast<const uint8_t*>(ws), j0,
                         j1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace gdn
