// gdn_fused.cu -- chunked (C = 64) WY/UT-form varlen prefill in ONE launch:
// a CTA carries a (sequence, value head) chain's f32 state through the
// sequence's chunks while its own warps prepare the next chunk, so nothing of
// a chunk but its output (and, where a chain moves between CTAs, its state)
// leaves the SM.  One CTA per chain, or, with more chains than SMs and the
// optional workspace, one CTA per SM over even ranges of the chains' chunks
// (the wrap-around schedule below).
//
// Defines the recurrence of [cpu.rs] (ferrum-kernels 0.8.0, src/ferrum_kernels/
// backend/cpu.rs) recurrent_gated_delta_rule_varlen_f32 / [cpu_ops.cpp]
// (vllm.cpp, src/vt/cpu/cpu_ops.cpp) GdnPrefillKernel, evaluated chunk by
// chunk in the form derived from it (the pages name a chunked GPU form but do
// not print it).  For one chunk of L <= 64 tokens with state S = [Dv, Dk] at
// its start (gam_i = sum_{t <= i} g_t):
//   A_ij = beta_i e^{gam_i - gam_j} k_i.k_j (j < i),   T = (I + A)^-1
//   W    = T diag(beta e^gam) K,   Ut = T diag(beta) V,   U = Ut - W S^T
//   O    = diag(e^gam) scale Q S^T + P U,   P_ij = scale e^{gam_i - gam_j} q_i.k_j (j <= i)
//   S'   = e^{gam_L} S + U^T diag(e^{gam_L - gam}) K
// with every exponent <= 0.
//
// Orientation.  The state-side products run transposed, with TMEM lanes = the
// value dimension dv, so that one thread owns one row S[dv, :]:
//   G    = [K; Q] K^T                 (M = 128 token rows, N = 64)     prep
//   W^T  = K^T Tw^T                   (M = 128 dk, N = 64 tokens)      prep
//   D1   = V^T Tu^T - S W^T | S Q^T   (M = 128 dv, N = 64 + 64)
//          so D1[:, 0:64] = U^T and D1[:, 64:128] = (Q S^T)^T directly
//   dS   = U'^T K   onto  e^{gam_L} S (M = 128 dv, N = 128 dk), U' = diag(fu) U
//   O^T  = U^T P^T  onto  (fo Q S^T)^T, in place in D1's second half
//          (M = 128 dv, N = 64 tokens)
// U'^T and U^T enter the tensor core from TMEM (A operand in tensor memory),
// the f32 state lives in TMEM as dS's accumulator, its hi + lo bf16 images in
// shared memory as D1's A operand.
//
// Precision.  q, k, v are exact bf16 inputs.  T, S, U', U and P enter the
// tensor core as hi + lo bf16 pairs (hi = x rounded to 8 significant bits, lo
// = bf16(x - hi)), about 16 significant bits; W as one bf16 value (it reaches
// the output only through the W S^T correction).  Products of two split
// operands take hi*hi + hi*lo + lo*hi.
//
// Roles (14 warps):
//   warp 0      TMA loads: K, Q of chunk c into stage c % 2; V of chunk c into
//               the region W^T(c - 1) held once D1(c - 1) has read it
//   warp 1      every MMA, issued in dependency order as their inputs appear
//   warps 2-9   prep of chunk c: norms, gates, A and P from G, T by 16 x 16
//               blocks, the Tw / Tu / P images
//   warps 10-13 the state chain of chunk c: the W^T image, U from D1 (U', U
//               into TMEM, fo Q S^T in place), the state update S' and its
//               images, the output rows
// Prep of chunk c + 1 overlaps the chain of chunk c.  Every hand-off is an
// mbarrier; every wait is bounded and, once any wait gives up, every role
// leaves at its next wait, in-flight copies and MMAs are drained (bounded) and
// the TMEM is freed.
//
// Partial chunks: g and beta of rows past the chunk end are taken as 0, so
// those rows of W, Ut, U and U' are exactly zero and their K, Q, V rows (the
// next sequence's tokens, or zeros past the tensor end) never contribute.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gdn_chunk_common.cuh"
#include "gdn_internal.h"
#include "tcgen05.cuh"

namespace gdn {
namespace {

using namespace umma;
using namespace chunk;

constexpr long long kWaitBudget = 2000000000LL;  // ~1 s of SM clock per wait

struct FusedSmem {
  static constexpr uint32_t KQ = 0;             // 2 stages x [K box0 | Q box0 | K box1 | Q box1]
  static constexpr uint32_t kStage = 32768;
  static constexpr uint32_t SH = 65536;         // S hi image [128 dv][128 dk], K-major, 2 x 16 KB
  static constexpr uint32_t SL = SH + 32768;    // S lo image
  static constexpr uint32_t WV = SL + 32768;    // W^T image [128 dk][64 tok] MN-major, or V [V0|V1]
  static constexpr uint32_t PI = WV + 16384;    // P hi [64 i][64 j] K-major, then P lo
  static constexpr uint32_t TI = PI + 16384;    // Tw hi, Tw lo, Tu hi, Tu lo (8 KB each); Y aliases
  static constexpr uint32_t AT = TI + 32768;    // A, then T in place, f32 [64][68]
  static constexpr uint32_t kAStride = 68;
  static constexpr uint32_t kYStride = 36;      // Y = A21 T11, f32 [32][36] at TI
  static constexpr uint32_t GB = AT + 64 * kAStride * 4;  // g, beta, gam, kn, qn, wj, uj
  static constexpr uint32_t FAC = GB + 7 * 64 * 4;        // 2 x {fo[64], fu[64], e^{gam_L}, 0, 0, 0}
  static constexpr uint32_t kFac = 132;                   // floats per factor buffer
  static constexpr uint32_t OST = FAC + 2 * kFac * 4;     // output staging [32 tok][128 dv] bf16
  static constexpr uint32_t BYTES = OST + 32 * 128 * 2;
};
static_assert(FusedSmem::BYTES + 1024 + 1024 <= 232448, "shared memory per CTA");
static_assert(32 * FusedSmem::kYStride * 4 <= 8192, "Y fits in the Tw hi image space");

// TMEM columns (512 allocated).
constexpr uint32_t kTG = 0;     // G = [K;Q] K^T (64)
constexpr uint32_t kTW = 64;    // W^T (64)
constexpr uint32_t kTD1 = 128;  // D1: U^T | (Q S^T)^T, the second half then fo-scaled and the
                                // output accumulator O^T (128)
constexpr uint32_t kTS = 256;   // f32 state S[dv][dk], dS accumulates onto it (128)
constexpr uint32_t kTU2 = 384;  // U'^T hi | lo as packed bf16 pairs (32 + 32)
constexpr uint32_t kTU = 448;   // U^T hi | lo (32 + 32)

constexpr int kThreads = 448;
constexpr int kPrepThreads = 256;
constexpr int kScanThreads = 128;
constexpr int kBarPrep = 1;
constexpr int kBarScan = 2;

enum Mb : int {
  kMbKq0 = 0, kMbKq1, kMbKqFree0, kMbKqFree1, kMbV, kMbG, kMbGRead, kMbTwTu, kMbWu, kMbWImg,
  kMbPImg, kMbFac, kMbD1, kMbD1Free, kMbUReady, kMbSImg, kMbD2, kMbD3, kMbOFree, kMbEnd, kMbState,
  kNumMb
};

// Chains spread over the SMs when they outnumber them (McNaughton's
// wrap-around rule for preemptive jobs on identical machines).  The machines
// are gangs of grp = Hv / Hk CTAs (of a grid of one CTA per SM) and the jobs
// are the (sequence, key head) pairs: member m of a gang runs value head
// hk * grp + m of every pair, so the heads that share K and Q run in step and
// read each tile once from DRAM.  The pairs' chunks, in (sequence, key head)
// order, are cut into consecutive ranges of C = max(ceil(total / gangs),
// longest sequence) chunks, one per gang.  A pair cut between gangs g and
// g + 1 runs its first chunks at the start of gang g + 1's range and the
// rest at the end of gang g's (in that rule the two parts of a job never
// overlap in time because C is at least the longest job), so gang g resumes
// its chains from the states gang g + 1 stored long before and no CTA's start
// waits for anything (one flag per chain, waited for with a bound; the launch
// is cooperative, so every CTA is resident).  Two waves of 152 + 104 equal
// chains become one range of ceil(4 * 16 * 32 / 38) = 54 chunks instead of 64.
constexpr int kMaxSchedCtas = 1024;
struct FusedSched {
  int32_t* seq_chunks;  // [N] chunks of each live sequence (0: padded, invalid or empty)
  int32_t* prefix;      // [N + 1] exclusive prefix of seq_chunks
  int4* starts;         // [grid] per CTA: its first (sequence, value head), the chunks of that
                        // chain the gang before holds, and the CTA's chunk count
  unsigned* flags;      // [N * Hv] 1 once a chain's state was stored for the CTA that resumes it
};

// A chain's f32 state moves between the pool and the SM by TMA, staged where
// the S hi / lo images live (free whenever a chain starts or ends): four boxes
// of [128 dv][32 dk] with the 128-byte swizzle, so that each thread's row is
// read and written without bank conflicts.  Byte offset of column c (a
// multiple of 4) of row r:
__device__ __forceinline__ uint32_t stage_off(uint32_t r, uint32_t c) {
  return (c >> 5) * 16384u + r * 128u + ((((c & 31u) >> 2) ^ (r & 7u)) << 4);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst_smem, const void* tmap, uint32_t mbar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst_smem),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src_smem, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1), "r"(src_smem)
               : "memory");
}
// Orders this thread's global accesses of the generic proxy against those of
// the async proxy (the TMA copies of a handed-over state and its flag).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One CTA: the chunks of every sequence (padded, invalid and empty ones get
// none and their errors go to the status word), their prefix, C, each CTA's
// start (CTAs past the last whole gang get none), and the flags cleared.
__global__ void __launch_bounds__(1024, 1) fused_schedule_kernel(const RecurLaunch p,
                                                                 const FusedSched sc, int grid) {
  __shared__ int s_warp[32];
  __shared__ int s_carry, s_max;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    s_carry = 0;
    s_max = 0;
    if (__ldg(p.cu) != 0 || __ldg(p.cu + p.N) != p.T) atomicOr(p.status, kStatusBadSeqlens);
  }
  __syncthreads();
  for (int b0 = 0; b0 < p.N; b0 += 1024) {
    const int sq = b0 + tid;
    int n = 0;
    if (sq < p.N) {
      const int lo = __ldg(p.cu + sq), hi = __ldg(p.cu + sq + 1);
      int slot = p.sidx != nullptr ? __ldg(p.sidx + sq) : sq;
      const bool bad = lo < 0 || hi <= lo || hi > p.T;
      if (bad) atomicOr(p.status, kStatusBadSeqlens);
      if (slot < -1 || slot >= p.slots) {
        atomicOr(p.status, kStatusBadIndex);
        slot = -1;
      }
      n = (!bad && slot >= 0) ? (hi - lo + kC - 1) / kC : 0;
      sc.seq_chunks[sq] = n;
      atomicMax(&s_max, n);
    }
    int x = n;  // inclusive scan: the warp, then the warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    const int incl = s_carry + x + (warp > 0 ? s_warp[warp - 1] : 0);
    if (sq < p.N) sc.prefix[sq] = incl - n;
    __syncthreads();
    if (tid == 1023) s_carry = incl;
    __syncthreads();
  }
  if (tid == 0) sc.prefix[p.N] = s_carry;
  __syncthreads();
  const int grp = p.Hv / p.Hk, gangs = grid / grp;
  const int64_t total = static_cast<int64_t>(s_carry) * p.Hk;
  const int64_t C = max((total + gangs - 1) / gangs, static_cast<int64_t>(s_max));
  for (int j = tid; j < grid; j += 1024) {
    int4 st = make_int4(0, 0, 0, 0);
    const int g = j / grp, m = j % grp;
    const int64_t g0 = static_cast<int64_t>(g) * C;
    if (g < gangs && g0 < total) {  // the sequence holding chunk g0: the last with Hk * prefix <= g0
      int lo = 0, hi = p.N - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(sc.prefix[mid]) * p.Hk <= g0)
          lo = mid;
        else
          hi = mid - 1;
      }
      const int n = sc.seq_chunks[lo];
      const int64_t r = g0 - static_cast<int64_t>(sc.prefix[lo]) * p.Hk;
      st = make_int4(lo, static_cast<int>(r / n) * grp + m, static_cast<int>(r % n),
                     static_cast<int>(min(C, total - g0)));
    }
    sc.starts[j] = st;
  }
  for (int64_t q = tid; q < static_cast<int64_t>(p.N) * p.Hv; q += 1024) sc.flags[q] = 0u;
}

// Bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool wait_mb(uint32_t mb, uint32_t parity, volatile int* abort,
                                        unsigned* status) {
  if (mbar_try_wait(mb, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(mb, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitBudget) {
      if (atomicExch(const_cast<int*>(abort), 1) == 0) atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// A role's position in the CTA's chunks: chain (s, h), chunk k of its n (the
// CTA runs chunks up to e of it), the sequence's token range [lo, hi), and the
// chunks left.  The prep and chain roles keep theirs in shared memory (one
// thread advances it between two barriers), which keeps it out of the
// registers of a kernel at its 128-register cap.
struct ChunkIt {
  int s, h, k, e, n, lo, hi, left;
};

// kSpread: the CTA runs the range the schedule gave it, else the one chain
// (sequence, value head) = blockIdx.x (that instance keeps none of the
// range's bookkeeping in registers).
template <bool kSpread>
__global__ void __launch_bounds__(kThreads, 1) fused_prefill_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_s,
    const RecurLaunch p, const FusedSched sc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  __shared__ uint64_t mbs[kNumMb];
  __shared__ uint32_t tslot;
  __shared__ ChunkIt s_igt, s_it;  // the prep's gate chunk; the chain's chunk
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  // This CTA's chunks: cnt of them through the chains of its gang member's
  // value heads, in (sequence, key head) order, from chain (s0, h0), of which
  // the gang before holds the last k0 (this CTA runs the first n - k0); a
  // last chain cut by the range's end runs its last chunks here.
  int s0, h0, k0, cnt;
  if constexpr (!kSpread) {
    h0 = blockIdx.x % p.Hv;
    s0 = blockIdx.x / p.Hv;
    k0 = 0;
    const int lo = __ldg(p.cu + s0), hi = __ldg(p.cu + s0 + 1);
    if (lo < 0 || hi <= lo || hi > p.T || __ldg(p.cu) != 0 || __ldg(p.cu + p.N) != p.T) {
      if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
    int slot = p.sidx != nullptr ? __ldg(p.sidx + s0) : s0;
    if (slot < -1 || slot >= p.slots) {
      if (tid == 0) atomicOr(p.status, kStatusBadIndex);
      slot = -1;
    }
    if (slot < 0) {  // padded sequence: zero outputs, pool untouched
      for (int idx = tid; idx < (hi - lo) * 16; idx += kThreads) {
        const int t = lo + idx / 16, q16 = idx % 16;
        *reinterpret_cast<uint4*>(out + ((int64_t)t * p.Hv + h0) * kD + q16 * 8) =
            make_uint4(0, 0, 0, 0);
      }
      return;
    }
    cnt = (hi - lo + kC - 1) / kC;
  } else {
    const int4 st = sc.starts[blockIdx.x];
    s0 = st.x;
    h0 = st.y;
    k0 = st.z;
    cnt = st.w;
    // The outputs of padded sequences (no chunks): chain q by CTA q % grid.
    for (int64_t q = blockIdx.x; q < static_cast<int64_t>(p.N) * p.Hv; q += gridDim.x) {
      const int sq = static_cast<int>(q / p.Hv), hq = static_cast<int>(q % p.Hv);
      if (sc.seq_chunks[sq] != 0) continue;
      const int lo = __ldg(p.cu + sq), hi = __ldg(p.cu + sq + 1);
      if (lo < 0 || hi <= lo || hi > p.T) continue;  // malformed: reported, nothing written
      for (int idx = tid; idx < (hi - lo) * 16; idx += kThreads) {
        const int t = lo + idx / 16, q16 = idx % 16;
        *reinterpret_cast<uint4*>(out + ((int64_t)t * p.Hv + hq) * kD + q16 * 8) =
            make_uint4(0, 0, 0, 0);
      }
    }
    if (cnt <= 0) return;
  }
  auto it_start = [&]() {
    ChunkIt x;
    x.s = s0;
    x.h = h0;
    x.k = 0;
    x.left = cnt;
    x.lo = __ldg(p.cu + s0);
    x.hi = __ldg(p.cu + s0 + 1);
    x.n = kSpread ? sc.seq_chunks[s0] : cnt;
    x.e = x.n - k0;
    return x;
  };
  auto it_next = [&](ChunkIt& x) {
    if constexpr (!kSpread) {
      ++x.k;
      return;
    }
    if (--x.left <= 0) return;
    if (++x.k < x.e) return;
    x.h += p.Hv / p.Hk;  // the gang member's head of the next key head
    if (x.h >= p.Hv) {
      x.h -= p.Hv;
      do {
        ++x.s;
      } while (sc.seq_chunks[x.s] == 0);
      x.lo = __ldg(p.cu + x.s);
      x.hi = __ldg(p.cu + x.s + 1);
      x.n = sc.seq_chunks[x.s];
    }
    x.e = x.n;
    x.k = x.n - min(x.n, x.left);  // cut by the range's end: its last chunks
  };
  const int nch = cnt;
  const uint32_t base = smem_u32(sm);
  auto MB = [&](int i) { return smem_u32(&mbs[i]); };
  volatile int* abort = &s_abort;

  if (tid == 0) {
    for (int i = 0; i < kNumMb; ++i) mbar_init(MB(i), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tslot), 512);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tslot;
  float* fac = reinterpret_cast<float*>(sm + FusedSmem::FAC);

  if (warp == 0) {
    // ---------------------------------------------------------------- loader
    if (lane == 0) {
      int last_kq[2] = {-1, -1}, n_v = 0;
      ChunkIt ikq = it_start(), iv = it_start();  // the chunks of the K/Q and of the V loads
      const int grp = p.Hv / p.Hk;
      auto load_kq = [&](int c) {  // chunks in order
        const uint32_t st = base + FusedSmem::KQ + (c & 1) * FusedSmem::kStage;
        const uint32_t mb = MB(kMbKq0 + (c & 1));
        const int t0 = ikq.lo + ikq.k * kC, hk = ikq.h / grp;
        mbar_expect_tx(mb, 4 * 8192);
        tma_load_3d(st + 0, &tm_k, mb, 0, hk, t0);
        tma_load_3d(st + 8192, &tm_q, mb, 0, hk, t0);
        tma_load_3d(st + 16384, &tm_k, mb, 64, hk, t0);
        tma_load_3d(st + 24576, &tm_q, mb, 64, hk, t0);
        last_kq[c & 1] = c;
        it_next(ikq);
      };
      auto load_v = [&](int c) {  // chunks in order
        const uint32_t mb = MB(kMbV);
        const int t0 = iv.lo + iv.k * kC;
        mbar_expect_tx(mb, 2 * 8192);
        tma_load_3d(base + FusedSmem::WV, &tm_v, mb, 0, iv.h, t0);
        tma_load_3d(base + FusedSmem::WV + 8192, &tm_v, mb, 64, iv.h, t0);
        n_v = c + 1;
        it_next(iv);
      };
      load_kq(0);
      if (nch > 1) load_kq(1);
      load_v(0);
      for (int c = 1; c < nch; ++c) {
        // V(c) replaces W^T(c - 1) once D1(c - 1) has read it.
        if (!wait_mb(MB(kMbD1), (c - 1) & 1, abort, p.status)) break;
        load_v(c);
        if (c + 1 < nch) {  // stage (c + 1) % 2 is free once D2(c - 1) has read K(c - 1)
          if (!wait_mb(MB(kMbKqFree0 + ((c + 1) & 1)), ((c - 1) >> 1) & 1, abort, p.status))
            break;
          load_kq(c + 1);
        }
      }
      __syncwarp(1u);
      if (*abort) {  // let the copies in flight land before the CTA exits
        for (int st = 0; st < 2; ++st)
          if (last_kq[st] >= 0) mbar_wait(MB(kMbKq0 + st), (last_kq[st] >> 1) & 1, kWaitBudget);
        if (n_v > 0) mbar_wait(MB(kMbV), (n_v - 1) & 1, kWaitBudget);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_g = idesc_bf16_f32(128, 64, false, false);
      const uint32_t id_wu = idesc_bf16_f32(128, 64, true, false);
      const uint32_t id_d1w = idesc_bf16_f32(128, 64, false, true);
      const uint32_t id_d1q = idesc_bf16_f32(128, 64, false, false);
      const uint32_t id_d2 = idesc_bf16_f32(128, 128, false, true);
      const uint32_t id_d3 = idesc_bf16_f32(128, 64, false, false);
      // Chunks whose MMAs of each group have been issued, in priority order:
      // D2 + D3 (the state chain and the output), D1, the prep's W / Ut, G.
      int cg = 0, cwu = 0, cd1 = 0, cd23 = 0;
      long long last = clock64();
      while (cd23 < nch) {
        if (*abort) break;
        bool went = false;
        if (cd23 < cd1 && mbar_test_wait(MB(kMbUReady), cd23 & 1) &&
            mbar_test_wait(MB(kMbPImg), cd23 & 1)) {
          fence_after_sync();
          const int c = cd23;
          const uint32_t st = base + FusedSmem::KQ + (c & 1) * FusedSmem::kStage;
          // dS = U'^T K onto e^{gam_L} S  (A = U'^T hi, lo from TMEM; B = K MN-major)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < kC; kk += 16)
              mma_bf16_ta(tmem + kTS, tmem + kTU2 + part * 32 + kk / 2,
                          desc_sw128(st + (kk / 8) * 1024, 16384, 1024), id_d2, true);
          mma_commit(MB(kMbD2));
          mma_commit(MB(kMbKqFree0 + (c & 1)));
          // O^T += U^T P^T onto fo (Q S^T)^T: hi*hi, hi*lo, lo*hi (A = U^T from TMEM;
          // B = P, K-major)
#pragma unroll
          for (int pr = 0; pr < 3; ++pr) {
            const uint32_t ua = kTU + (pr == 2 ? 32 : 0);
            const uint32_t pb = base + FusedSmem::PI + (pr == 1 ? 8192 : 0);
#pragma unroll
            for (int kk = 0; kk < kC; kk += 16)
              mma_bf16_ta(tmem + kTD1 + 64, tmem + ua + kk / 2,
                          desc_sw128(pb + kk * 2, 16, 1024), id_d3, true);
          }
          mma_commit(MB(kMbD3));
          ++cd23;
          went = true;
        } else if (cd1 < cwu && mbar_test_wait(MB(kMbWImg), cd1 & 1) &&
                   mbar_test_wait(MB(kMbSImg), cd1 & 1) &&
                   (cd1 == 0 || mbar_test_wait(MB(kMbOFree), (cd1 - 1) & 1))) {
          fence_after_sync();
          const int c = cd1;
          const uint32_t st = base + FusedSmem::KQ + (c & 1) * FusedSmem::kStage;
          // D1[:, 0:64] += S (-W)^T onto Ut^T;  D1[:, 64:128] = S Q^T (the previous
          // chunk's output rows have been read).  A = S hi, lo.
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < kD; kk += 16) {
              const uint64_t a = desc_sw128(base + (part ? FusedSmem::SL : FusedSmem::SH) +
                                                (kk / 64) * 16384 + (kk % 64) * 2,
                                            16, 1024);
              mma_bf16(tmem + kTD1, a,
                       desc_sw128(base + FusedSmem::WV + (kk / 8) * 1024, 8192, 1024), id_d1w,
                       true);
              mma_bf16(tmem + kTD1 + 64, a,
                       desc_sw128(st + 8192 + (kk / 64) * 16384 + (kk % 64) * 2, 16, 1024),
                       id_d1q, part > 0 || kk > 0);
            }
          mma_commit(MB(kMbD1));
          ++cd1;
          went = true;
        } else if (cwu < cg && mbar_test_wait(MB(kMbTwTu), cwu & 1) &&
                   mbar_test_wait(MB(kMbV), cwu & 1) &&
                   (cwu == 0 || mbar_test_wait(MB(kMbD1Free), (cwu - 1) & 1))) {
          fence_after_sync();
          const int c = cwu;
          const uint32_t st = base + FusedSmem::KQ + (c & 1) * FusedSmem::kStage;
          // W^T = K^T Tw^T (A = K, MN-major, M = dk), hi + lo of Tw.
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < kC; kk += 16)
              mma_bf16(tmem + kTW, desc_sw128(st + (kk / 8) * 1024, 16384, 1024),
                       desc_sw128(base + FusedSmem::TI + part * 8192 + kk * 2, 16, 1024), id_wu,
                       part > 0 || kk > 0);
          // Ut^T = V^T Tu^T into D1[:, 0:64] (A = V, MN-major, M = dv).
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < kC; kk += 16)
              mma_bf16(tmem + kTD1, desc_sw128(base + FusedSmem::WV + (kk / 8) * 1024, 8192, 1024),
                       desc_sw128(base + FusedSmem::TI + 16384 + part * 8192 + kk * 2, 16, 1024),
                       id_wu, part > 0 || kk > 0);
          mma_commit(MB(kMbWu));
          ++cwu;
          went = true;
        } else if (cg < nch && mbar_test_wait(MB(kMbKq0 + (cg & 1)), (cg >> 1) & 1) &&
                   (cg == 0 || mbar_test_wait(MB(kMbGRead), (cg - 1) & 1))) {
          fence_after_sync();
          const uint32_t st = base + FusedSmem::KQ + (cg & 1) * FusedSmem::kStage;
          // G = [K; Q] K^T  (M = 128, N = 64, K = 128)
#pragma unroll
          for (int kk = 0; kk < kD; kk += 16) {
            const uint32_t off = (kk / 64) * 16384 + (kk % 64) * 2;
            mma_bf16(tmem + kTG, desc_sw128(st + off, 16, 1024), desc_sw128(st + off, 16, 1024),
                     id_g, kk > 0);
          }
          mma_commit(MB(kMbG));
          ++cg;
          went = true;
        }
        if (went) {
          last = clock64();
        } else if (clock64() - last > kWaitBudget) {
          if (atomicExch(const_cast<int*>(abort), 1) == 0) atomicOr(p.status, kStatusTimeout);
          break;
        }
      }
    }
  } else if (warp < 10) {
    // ---------------------------------------------------------------- prep
    const int ptid = tid - 64, pw = warp - 2;
    const int quad = warp & 3, hf = pw >> 2;
    float* sg = reinterpret_cast<float*>(sm + FusedSmem::GB);
    float* sb = sg + 64;
    float* sgam = sb + 64;
    float* skn = sgam + 64;
    float* sqn = skn + 64;
    float* swj = sqn + 64;
    float* suj = swj + 64;
    float* sA = reinterpret_cast<float*>(sm + FusedSmem::AT);
    float* sY = reinterpret_cast<float*>(sm + FusedSmem::TI);
    constexpr int S_ = FusedSmem::kAStride;
    constexpr int SY = FusedSmem::kYStride;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    float g_next = 0.0f, b_next = 0.0f;
    if (ptid == 0) s_igt = it_start();
    named_bar(kBarPrep, kPrepThreads);
    auto load_gates = [&]() {  // ptid < 64; the chunk s_igt is on
      const int t0 = s_igt.lo + s_igt.k * kC, L = min(kC, s_igt.hi - t0), hg = s_igt.h;
      if (ptid < L) {
        g_next = __ldg(p.g + (int64_t)(t0 + ptid) * p.Hv + hg);
        b_next = __ldg(p.beta + (int64_t)(t0 + ptid) * p.Hv + hg);
      } else {
        g_next = b_next = 0.0f;
      }
    };
    if (ptid < 64) load_gates();
    float pv[32];  // this thread's P values (P-row warps) until the images go out
    const int i = (quad & 1) * 32 + lane;
    for (int c = 0; c < nch; ++c) {
      const uint8_t* sst = sm + FusedSmem::KQ + (c & 1) * FusedSmem::kStage;
      float* F = fac + (c & 1) * FusedSmem::kFac;
      bool ok = true;
      if (ptid < 64) {
        sg[ptid] = g_next;
        sb[ptid] = b_next;
      }
      ok = wait_mb(MB(kMbKq0 + (c & 1)), (c >> 1) & 1, abort, p.status) && ok;
      if (ptid < 128) {  // inverse row norms: rows of K (ptid < 64), of Q (64..127)
        const int r = ptid & 63;
        float ss = 0.0f;
        if (p.norm) {
          const uint8_t* row = sst + (ptid < 64 ? 0 : 8192) + r * 128;
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
        (ptid < 64 ? skn : sqn)[r] = p.norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
      }
      named_bar(kBarPrep, kPrepThreads);
      if (ptid == 0 && c + 1 < nch) it_next(s_igt);  // read for chunk c before this barrier
      if (pw == 0) {  // inclusive scan of g over the chunk (2 tokens per lane)
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
      // FAC[c % 2] was last read by the chain's U step of chunk c - 2 and its
      // state update of chunk c - 1 ... and fac(c) must not complete before the
      // chain has taken fac(c - 1): both hold once the chain has published the
      // state images of chunk c - 1.
      if (c >= 1) ok = wait_mb(MB(kMbSImg), (c - 1) & 1, abort, p.status) && ok;
      named_bar(kBarPrep, kPrepThreads);
      if (ptid < 64) {
        swj[ptid] = sb[ptid] * skn[ptid] * __expf(sgam[ptid]);
        suj[ptid] = sb[ptid];
        F[ptid] = p.scale * sqn[ptid] * __expf(sgam[ptid]);              // fo
        F[64 + ptid] = __expf(sgam[kC - 1] - sgam[ptid]) * skn[ptid];    // fu
        if (ptid < 4) F[128 + ptid] = ptid == 0 ? __expf(sgam[kC - 1]) : 0.0f;  // e^{gam_L}
      }
      named_bar(kBarPrep, kPrepThreads);
      if (ptid == 0) mbar_arrive(MB(kMbFac));
      if (ptid < 64 && c + 1 < nch) load_gates();  // chunk c + 1, consumed next chunk
      ok = wait_mb(MB(kMbG), c & 1, abort, p.status) && ok;
      fence_after_sync();
      // Lanes 0..63 of G hold K K^T -> A (f32, shared); lanes 64..127 hold
      // Q K^T -> P.  Row i, columns 32 hf ... 32 hf + 31.
      const bool upper = (quad & 1) == 0 && hf == 1;  // rows 0..31 x columns 32..63: zero
      {
        float v[32];
        if (!upper) {
          tmem_ld32(tmem + kTG + lane_addr + hf * 32, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.0f;
        }
        // Decays e^{gam_i - gam_j} (j <= i) as a running product leftward from
        // the block's last column; 0 right of the diagonal, 1 on it.
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
#pragma unroll
          for (int e = 0; e < 32; ++e) pv[e] = 0.0f;
        } else {
          const float fi = p.scale * sqn[i];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = hf * 32 + e;
            pv[e] = upper ? 0.0f : fi * skn[j] * dec[e] * v[e];
          }
        }
      }
      fence_before_sync();
      named_bar(kBarPrep, kPrepThreads);  // A complete; G read: the next chunk's G may go
      if (ptid == 0) mbar_arrive(MB(kMbGRead));
      // T = (I + A)^-1 by blocks: the four 16 x 16 diagonal blocks by forward
      // substitution (the two A-row warps of column half 0, lane = column),
      // the two 32 x 32 diagonal blocks from them (X = -D1 A10 D0), then
      // T21 = -T22 (A21 T11).
      if (quad < 2 && hf == 0) {
        const int b0 = 16 * (2 * quad + (lane >> 4)), cc = lane & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const float* arow = sA + (b0 + r) * S_ + b0;
          float a0 = r == cc ? 1.0f : 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
          for (int m = 0; m < r; m += 4) {
            const float4 av = *reinterpret_cast<const float4*>(arow + m);
            a0 = fmaf(-av.x, x[m], a0);
            if (m + 1 < r) a1 = fmaf(-av.y, x[m + 1], a1);
            if (m + 2 < r) a2 = fmaf(-av.z, x[m + 2], a2);
            if (m + 3 < r) a3 = fmaf(-av.w, x[m + 3], a3);
          }
          x[r] = (a0 + a1) + (a2 + a3);
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 16; ++r) sA[(b0 + r) * S_ + b0 + cc] = x[r];
      }
      // Y lives in the Tw / Tu image space: the previous chunk's W and Ut
      // MMAs must have read it.
      if (c >= 1) ok = wait_mb(MB(kMbWu), (c - 1) & 1, abort, p.status) && ok;
      named_bar(kBarPrep, kPrepThreads);
      {  // Z = A10 D0 into sY rows 16 B .. 16 B + 15
        const int Bq = ptid >> 7, r = (ptid >> 3) & 15, c0 = (ptid & 7) * 2;
        const float* arow = sA + (32 * Bq + 16 + r) * S_ + 32 * Bq;
        float z0 = 0.0f, z1 = 0.0f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float a = arow[m];
          const float2 d = *reinterpret_cast<const float2*>(sA + (32 * Bq + m) * S_ + 32 * Bq + c0);
          z0 = fmaf(a, d.x, z0);
          z1 = fmaf(a, d.y, z1);
        }
        *reinterpret_cast<float2*>(sY + (16 * Bq + r) * SY + c0) = make_float2(z0, z1);
      }
      named_bar(kBarPrep, kPrepThreads);
      {  // X = -D1 Z into the lower-left 16 x 16 block of each 32 x 32 diagonal block
        const int Bq = ptid >> 7, r = (ptid >> 3) & 15, c0 = (ptid & 7) * 2;
        const float* drow = sA + (32 * Bq + 16 + r) * S_ + 32 * Bq + 16;
        float x0 = 0.0f, x1 = 0.0f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float d = drow[m];
          const float2 z = *reinterpret_cast<const float2*>(sY + (16 * Bq + m) * SY + c0);
          x0 = fmaf(d, z.x, x0);
          x1 = fmaf(d, z.y, x1);
        }
        *reinterpret_cast<float2*>(sA + (32 * Bq + 16 + r) * S_ + 32 * Bq + c0) =
            make_float2(-x0, -x1);
      }
      named_bar(kBarPrep, kPrepThreads);
      const int bi = ptid >> 3, bj = (ptid & 7) * 4;
      {  // Y = A21 T11
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
      named_bar(kBarPrep, kPrepThreads);
      {  // T21 = -T22 Y
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
      named_bar(kBarPrep, kPrepThreads);  // T complete, Y dead
      // The P-row warps store the P images (once D3 of the previous chunk has
      // read them); the A-row warps store Tw = T diag(beta e^gam kn) and
      // Tu = T diag(beta) as hi + lo images.
      if (quad >= 2) {
        if (c >= 1) ok = wait_mb(MB(kMbD3), (c - 1) & 1, abort, p.status) && ok;
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          const uint32_t off = swz128_offset(i, hf * 32 + e, 8192);
          st_split8(sm + FusedSmem::PI + off, sm + FusedSmem::PI + 8192 + off, pv + e);
        }
      }
      const int atid = (quad & 1) * 32 + lane + hf * 64;  // 0..127 over the A-row warps
      for (int item = atid; item < 64 * 8 && quad < 2; item += 128) {
        const int r = item >> 3, q = item & 7;
        float tw[8], tu[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float t = sA[r * S_ + 8 * q + e];
          tw[e] = t * swj[8 * q + e];
          tu[e] = t * suj[8 * q + e];
        }
        const uint32_t off = swz128_offset(r, 8 * q, 8192);
        st_split8(sm + FusedSmem::TI + off, sm + FusedSmem::TI + 8192 + off, tw);
        st_split8(sm + FusedSmem::TI + 16384 + off, sm + FusedSmem::TI + 24576 + off, tu);
      }
      fence_proxy_async();
      ok = named_bar_and(kBarPrep, kPrepThreads, ok);
      if (ptid == 0) {
        mbar_arrive(MB(kMbTwTu));
        mbar_arrive(MB(kMbPImg));
      }
      if (!ok) break;
    }
  } else {
    // ---------------------------------------------------------------- state chain
    const int quad = warp & 3;
    const int dv = quad * 32 + lane;
    const bool lead = warp == 10 && lane == 0;
    const uint32_t la = static_cast<uint32_t>(quad * 32) << 16;
    if (lead) s_it = it_start();  // the chain and chunk this role is on
    named_bar(kBarScan, kScanThreads);
    // The pool slot of sequence sq.
    auto chain_slot = [&](int sq) { return p.sidx != nullptr ? __ldg(p.sidx + sq) : sq; };
    int n_state = 0, st_issued = 0, st_seen = 0;  // state loads (the counts on the lead)
    // A chain's initial state into the S images and, times e^{gam_L} of its
    // first chunk here, into TMEM.  A chain that starts mid-way here resumes
    // from the state its gang member in the next gang stored (its flag
    // waited for first).
    auto init_chain = [&](const ChunkIt& x, float eL, bool okr) {
      bool init = p.has_init == nullptr || __ldg(p.has_init + x.s) != 0;
      if (kSpread && x.k > 0) {
        if (lead) {
          const unsigned* flag = sc.flags + (int64_t)x.s * p.Hv + x.h;
          const long long t0 = clock64();
          while (ld_acquire_u32(flag) == 0u) {
            if (*abort) {
              okr = false;
              break;
            }
            if (clock64() - t0 > kWaitBudget) {
              if (atomicExch(const_cast<int*>(abort), 1) == 0) atomicOr(p.status, kStatusTimeout);
              okr = false;
              break;
            }
          }
          __threadfence();
        }
        okr = named_bar_and(kBarScan, kScanThreads, okr);
        init = true;
      }
      if (init) {
        // The state by TMA into the staging, each row into TMEM, and once
        // every row is out of the staging, its images over it.
        if (lead && okr) {
          fence_proxy_async_global();
          mbar_expect_tx(MB(kMbState), 4 * 16384);
          const int row0 = (chain_slot(x.s) * p.Hv + x.h) * kD;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            tma_load_2d(base + FusedSmem::SH + b * 16384, &tm_s, MB(kMbState), 32 * b, row0);
          ++st_issued;
        }
        const bool got = wait_mb(MB(kMbState), n_state & 1, abort, p.status);
        if (lead && got) ++st_seen;
        okr = got && okr;
        ++n_state;
#pragma unroll 1
        for (int j0 = 0; j0 < kD; j0 += 32) {
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 f = *reinterpret_cast<const float4*>(sm + FusedSmem::SH + stage_off(dv, j0 + e));
            v[e] = f.x;
            v[e + 1] = f.y;
            v[e + 2] = f.z;
            v[e + 3] = f.w;
          }
          tmem_st32(tmem + kTS + la + j0, v);
        }
        tmem_st_wait();
        named_bar(kBarScan, kScanThreads);
#pragma unroll 1
        for (int j0 = 0; j0 < kD; j0 += 32) {
          float v[32];
          tmem_ld32(tmem + kTS + la + j0, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            const uint32_t off = swz128_offset(dv, j0 + e, 16384);
            st_split8(sm + FusedSmem::SH + off, sm + FusedSmem::SL + off, v + e);
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] *= eL;
          tmem_st32(tmem + kTS + la + j0, v);
        }
      } else {  // a fresh chain: zero images and state
#pragma unroll 1
        for (int j0 = 0; j0 < kD; j0 += 32) {
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.0f;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            const uint32_t off = swz128_offset(dv, j0 + e, 16384);
            st_split8(sm + FusedSmem::SH + off, sm + FusedSmem::SL + off, v + e);
          }
          tmem_st32(tmem + kTS + la + j0, v);
        }
      }
      return okr;
    };
    bool ok = wait_mb(MB(kMbFac), 0, abort, p.status);
    // With ranges a chain's state comes in at the top of its first chunk here
    // (one place in the code for the first chain and every later one).
    bool need_init = kSpread;
    float eL_init = fac[128];  // e^{gam_L} of that chunk
    if constexpr (!kSpread) {
      const ChunkIt x0 = s_it;
      ok = init_chain(x0, eL_init, ok);
      tmem_st_wait();
      fence_proxy_async();
      fence_before_sync();
      ok = named_bar_and(kBarScan, kScanThreads, ok);
      if (lead) mbar_arrive(MB(kMbSImg));
    }
    // Per chunk: the W^T image (D1 waits), U (D2 and D3 wait), the state update
    // (the next D1 waits), the output rows (the next D1's Q half waits).
    for (int c = 0; c < nch && ok; ++c) {
      if (kSpread && need_init) {
        const ChunkIt x0 = s_it;
        ok = init_chain(x0, eL_init, ok);
        tmem_st_wait();
        fence_proxy_async();
        fence_before_sync();
        ok = named_bar_and(kBarScan, kScanThreads, ok);
        if (lead) mbar_arrive(MB(kMbSImg));
        need_init = false;
        if (!ok) break;
      }
      const int t0 = s_it.lo + s_it.k * kC;
      const int L = min(kC, s_it.hi - t0);
      const int hc = s_it.h;
      const float* F = fac + (c & 1) * FusedSmem::kFac;
      // W^T (TMEM lanes = dk, 64 token columns) -> the -W^T image, the MN-major
      // B operand of this chunk's D1 (V, which shared the space, is consumed).
      ok = wait_mb(MB(kMbWu), c & 1, abort, p.status) && ok;
      fence_after_sync();
#pragma unroll 1
      for (int j0 = 0; j0 < kC; j0 += 32) {
        float w[32];
        tmem_ld32(tmem + kTW + la + j0, w);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float nv[8];
#pragma unroll
          for (int x = 0; x < 8; ++x) nv[x] = -w[e + x];
          st_bf16x8(sm + FusedSmem::WV + swz128_offset(dv, j0 + e, 16384), nv);
        }
      }
      fence_proxy_async();
      fence_before_sync();
      ok = named_bar_and(kBarScan, kScanThreads, ok);
      if (lead) mbar_arrive(MB(kMbWImg));
      if (!ok) break;
      // U^T = D1[:, 0:64] (Ut^T - W S^T); U'^T = U^T diag(fu) and U^T into TMEM
      // as hi + lo bf16 pairs; D1[:, 64:128] scaled in place to fo (Q S^T)^T,
      // onto which P U accumulates.  Two rounds of 32 token columns.
      ok = wait_mb(MB(kMbD1), c & 1, abort, p.status) && ok;
      fence_after_sync();
#pragma unroll 1
      for (int j0 = 0; j0 < kC; j0 += 32) {
        float u[32], qs[32];
        tmem_ld32(tmem + kTD1 + la + j0, u);
        tmem_ld32(tmem + kTD1 + 64 + la + j0, qs);
        tmem_ld_wait();
#pragma unroll
        for (int j1 = 0; j1 < 32; j1 += 16) {
          const int j = j0 + j1;
          uint32_t u2h[8], u2l[8], uh[8], ul[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            split2(u[j1 + e] * F[64 + j + e], u[j1 + e + 1] * F[64 + j + e + 1], u2h[e / 2],
                   u2l[e / 2]);
            split2(u[j1 + e], u[j1 + e + 1], uh[e / 2], ul[e / 2]);
          }
          tmem_st8u(tmem + kTU2 + la + j / 2, u2h);
          tmem_st8u(tmem + kTU2 + 32 + la + j / 2, u2l);
          tmem_st8u(tmem + kTU + la + j / 2, uh);
          tmem_st8u(tmem + kTU + 32 + la + j / 2, ul);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) qs[e] *= F[j0 + e];
        tmem_st32(tmem + kTD1 + 64 + la + j0, qs);
      }
      tmem_st_wait();
      fence_before_sync();
      ok = named_bar_and(kBarScan, kScanThreads, ok);
      if (lead) {
        mbar_arrive(MB(kMbUReady));
        mbar_arrive(MB(kMbD1Free));
      }
      if (!ok) break;
      // S' = e^{gam_L} S + dS (in TMEM): its images for D1 of the next chunk,
      // then S' e^{gam_L'} back (the next dS accumulates onto it).  At the
      // chain's last chunk here S' goes to the pool instead (with its flag when
      // the gang before resumes the chain); the next chain's state comes in
      // at the top of the next chunk.
      ok = wait_mb(MB(kMbD2), c & 1, abort, p.status) && ok;
      const bool last = c + 1 == nch;
      const bool chain_end = last || (kSpread && s_it.k + 1 == s_it.e);
      float eLn = 0.0f;
      if (!last) {
        ok = wait_mb(MB(kMbFac), (c + 1) & 1, abort, p.status) && ok;
        eLn = fac[((c + 1) & 1) * FusedSmem::kFac + 128];
      }
      fence_after_sync();
#pragma unroll 1
      for (int j0 = 0; j0 < kD; j0 += 32) {
        float v[32];
        tmem_ld32(tmem + kTS + la + j0, v);
        tmem_ld_wait();
        if (chain_end) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(sm + FusedSmem::SH + stage_off(dv, j0 + e)) =
                make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            const uint32_t off = swz128_offset(dv, j0 + e, 16384);
            st_split8(sm + FusedSmem::SH + off, sm + FusedSmem::SL + off, v + e);
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] *= eLn;
          tmem_st32(tmem + kTS + la + j0, v);
        }
      }
      if (chain_end) {  // the staged S' to the pool by TMA (and the flag when the gang before resumes it)
        fence_proxy_async();
        named_bar(kBarScan, kScanThreads);
        if (lead) {
          const int row0 = (chain_slot(s_it.s) * p.Hv + s_it.h) * kD;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            tma_store_2d(&tm_s, base + FusedSmem::SH + b * 16384, 32 * b, row0);
          bulk_commit();
          if (kSpread && s_it.e < s_it.n) {
            bulk_wait_all();
            fence_proxy_async_global();
            __threadfence();
            atomicExch(sc.flags + (int64_t)s_it.s * p.Hv + s_it.h, 1u);
          } else if (last) {
            bulk_wait_all();
          } else {
            bulk_wait_read();
          }
        }
        named_bar(kBarScan, kScanThreads);  // the staging is free again
      }
      // Past a chain's end here the next chain (mid-way if cut by the range's
      // end) comes in at the top of the next chunk.
      const bool next_init = kSpread && chain_end && !last;
      if (next_init) {
        need_init = true;
        eL_init = eLn;
      }
      if (!last && !next_init) {
        tmem_st_wait();
        fence_proxy_async();
      }
      fence_before_sync();
      ok = named_bar_and(kBarScan, kScanThreads, ok);
      if (lead && !last && !next_init) mbar_arrive(MB(kMbSImg));
      if (!ok) break;
      // Output rows of the chunk: O^T[dv, i] = fo Q S^T + P U, then the
      // columns are free for the next chunk's D1.
      ok = wait_mb(MB(kMbD3), c & 1, abort, p.status) && ok;
      fence_after_sync();
      {
        // 32 tokens at a time through the staging rows: each thread writes its
        // dv of every token, then the rows leave as 16-byte vectors.
        __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + FusedSmem::OST);
        const int stid = tid - 320;  // 0..127
        const int c16 = stid & 15;   // this thread's 16-byte vector of every row it copies
#pragma unroll 1
        for (int j0 = 0; j0 < kC && j0 < L; j0 += 32) {
          float o[32];
          tmem_ld32(tmem + kTD1 + 64 + la + j0, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ost[e * kD + dv] = __float2bfloat16_rn(o[e]);
          named_bar(kBarScan, kScanThreads);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = (q * kScanThreads + stid) >> 4;  // the vector's token row
            __nv_bfloat16* dst = out + ((int64_t)(t0 + j0 + r) * p.Hv + hc) * kD + c16 * 8;
            if (j0 + r < L) {
              *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(ost + r * kD + c16 * 8);
            }
          }
          named_bar(kBarScan, kScanThreads);
        }
      }
      if (lead) it_next(s_it);  // every read of this chunk's s_it was before the S' barrier
      fence_before_sync();
      ok = named_bar_and(kBarScan, kScanThreads, ok);
      if (lead) mbar_arrive(MB(kMbOFree));
      if (!ok) break;
    }
    if (lead && st_issued != st_seen)  // a state load still landing (after an abort)
      mbar_wait(MB(kMbState), (n_state - 1) & 1, kWaitBudget);
  }

  // ---- teardown: every thread arrives here exactly once --------------------
  fence_before_sync();
  __syncthreads();
  if (*abort) {  // drain the MMAs in flight (their copies were drained by the loader)
    if (warp == 1 && lane == 0) {
      mma_commit(MB(kMbEnd));
      mbar_wait(MB(kMbEnd), 0, kWaitBudget);
    }
    __syncthreads();
  }
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

bool fused_supported(int Dk, int Dv, bool bf16) { return bf16 && Dk == kD && Dv == kD; }

namespace {
// Workspace of the schedule: seq_chunks [N], prefix [N + 1], starts
// [kMaxSchedCtas], flags [N * Hv], each 256-byte aligned.
constexpr size_t ws_align(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
struct SchedLayout {
  size_t chunks, prefix, starts, flags, bytes;
};
SchedLayout sched_layout(int64_t N, int64_t Hv) {
  SchedLayout l{};
  l.chunks = 0;
  l.prefix = ws_align(l.chunks + 4 * static_cast<size_t>(N));
  l.starts = ws_align(l.prefix + 4 * static_cast<size_t>(N + 1));
  l.flags = ws_align(l.starts + 16 * static_cast<size_t>(kMaxSchedCtas));
  l.bytes = ws_align(l.flags + 4 * static_cast<size_t>(N * Hv));
  return l;
}
}  // namespace

// The state pool as rows of Dk f32 ([slots * Hv * Dv][Dk]) in boxes of
// [128 rows][32 columns] with the 128-byte swizzle (one box per TMA copy).
bool make_pool_map(CUtensorMap* m, float* pool, int64_t slots, int64_t Hv) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(slots * Hv * kD)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, pool, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t fused_workspace_bytes(int64_t N, int64_t Hv) {
  if (N <= 0 || Hv <= 0) return 0;
  return sched_layout(N, Hv).bytes;
}

cudaError_t launch_fused(const RecurLaunch& p, void* workspace, size_t workspace_bytes,
                         cudaStream_t s) {
  CUtensorMap tq, tk, tv, ts;
  if (!make_map(&tq, p.q, p.T, p.Hk) || !make_map(&tk, p.k, p.T, p.Hk) ||
      !make_map(&tv, p.v, p.T, p.Hv) || !make_pool_map(&ts, p.pool, p.slots, p.Hv))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(fused_prefill_kernel<false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    FusedSmem::BYTES + 1024);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(fused_prefill_kernel<true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      FusedSmem::BYTES + 1024);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t blocks = static_cast<int64_t>(p.N) * p.Hv;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const int sms = sm_count();
  const SchedLayout l = sched_layout(p.N, p.Hv);
  FusedSched sc{};
  // Ranges pay about 6 % a chunk in bookkeeping, so they are taken where one
  // CTA per chain would leave a wave partly idle: on equal chains, waves
  // ceil(w) against w = chains / SMs, more than 8 % apart.
  const int64_t waves = (blocks + sms - 1) / sms;
  const bool spread = blocks > sms && waves * sms * 100 > blocks * 108;
  if (workspace != nullptr && workspace_bytes >= l.bytes && spread && sms <= kMaxSchedCtas &&
      p.Hv / p.Hk <= sms) {
    // One CTA per SM over the wrap-around schedule.
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    sc.seq_chunks = reinterpret_cast<int32_t*>(ws + l.chunks);
    sc.prefix = reinterpret_cast<int32_t*>(ws + l.prefix);
    sc.starts = reinterpret_cast<int4*>(ws + l.starts);
    sc.flags = reinterpret_cast<unsigned*>(ws + l.flags);
    fused_schedule_kernel<<<1, 1024, 0, s>>>(p, sc, sms);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = FusedSmem::BYTES + 1024;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the flag waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fused_prefill_kernel<true>, tq, tk, tv, ts, p, sc);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  fused_prefill_kernel<false><<<static_cast<unsigned>(blocks), kThreads, FusedSmem::BYTES + 1024, s>>>(
      tq, tk, tv, ts, p, sc);
  note_launch();
  return cudaGetLastError();
}

}  // namespace gdn
