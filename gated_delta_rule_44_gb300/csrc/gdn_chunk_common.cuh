// gdn_chunk_common.cuh -- pieces shared by the two chunked (C = 64) prefill
// implementations: bf16 packing and hi + lo splitting of f32 operands, named
// barriers, bulk copies, and the TMA tensor maps of the q, k, v tiles.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gdn_internal.h"
#include "tcgen05.cuh"

namespace gdn {
namespace chunk {

constexpr int kC = 64;   // chunk length
constexpr int kD = 128;  // Dk = Dv

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Stores 8 floats as bf16 into one 16-byte chunk.
__device__ __forceinline__ void st_bf16x8(void* p, const float* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

// x rounded to nearest with 8 significant bits (Veltkamp's splitting with the
// factor 2^16 + 1), so exactly a bf16 value; x - hi is exact in f32.  Plain
// f32 arithmetic: it runs on the FMA pipe instead of the (quarter-rate)
// conversion unit.  Valid for |x| < FLT_MAX / 65537.
__device__ __forceinline__ float split_hi(float x) {
  const float c = __fmul_rn(x, 65537.0f);
  return __fsub_rn(c, __fsub_rn(c, x));
}

// The bf16 bits of hi (its upper half) and bf16(x - hi) of two values, packed
// as two bf16x2 words: hi + lo carries about 16 significant bits of x.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hw, uint32_t& lw) {
  const float ha = split_hi(a), hb = split_hi(b);
  hw = __byte_perm(__float_as_uint(ha), __float_as_uint(hb), 0x7632);  // upper halves
  lw = pack_bf16x2(__fsub_rn(a, ha), __fsub_rn(b, hb));
}

// hi and lo images of 8 values, each into one 16-byte chunk.
__device__ __forceinline__ void st_split8(void* hi, void* lo, const float* v) {
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int e = 0; e < 8; e += 2) split2(v[e], v[e + 1], hw[e / 2], lw[e / 2]);
  *reinterpret_cast<uint4*>(hi) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4*>(lo) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
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
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also ANDs a predicate over the participating threads.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(mbar)
      : "memory");
}

// Bulk copy shared -> global (one thread), tracked by its bulk async-group.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile(
      "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(
          reinterpret_cast<uint64_t>(dst)),
      "r"(src), "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// Waits until this thread's bulk copies have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// Waits until this thread's bulk copies are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}

// Shared memory rounded up to the 1024-byte alignment of swizzled tiles; the
// pointer keeps the shared address space, so accesses compile to shared ones.
__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  return raw + ((1024u - (umma::smem_u32(raw) & 1023u)) & 1023u);
}

// Sequence and chunk-in-sequence of chunk `gc` in the enumeration of the
// chunks whose index within their sequence lies in [j0, j1) (by sequence,
// then chunk; [0, INT_MAX) enumerates every chunk, so gc is the global chunk
// index), from cu_seqlens (warp 0).  Returns false when gc is past the last
// such chunk or cu_seqlens is malformed.
__device__ inline bool locate_chunk(const int32_t* __restrict__ cu, int N, int T, int gc, int& s_out,
                                    int& j_out, bool& bad, int j0 = 0, int j1 = 0x7fffffff) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  bad = false;
  for (int s0 = 0; s0 < N; s0 += 32) {
    const int s = s0 + lane;
    int nc = 0;
    if (s < N) {
      const int lo = __ldg(cu + s), hi = __ldg(cu + s + 1);
      if (lo < 0 || hi <= lo || hi > T) bad = true;
      const int all = hi > lo ? (hi - lo + kC - 1) / kC : 0;
      nc = max(0, min(all, j1) - j0);
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
      j_out = j0 + gc - base - __shfl_sync(0xffffffffu, excl, src);
      return !bad;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return false;
}

// First global chunk of sequence s (sum of earlier sequences' chunk counts);
// `bad` reports an empty or decreasing earlier range (warp 0).
__device__ inline int chunk_base(const int32_t* __restrict__ cu, int s, bool& bad) {
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

// Upper bound on the chunks of T tokens in N non-empty sequences.
inline int64_t max_chunks(int64_t T, int64_t N) { return T / kC + N; }

// Programmatic dependent launch: a grid launched with the programmatic
// stream-serialisation attribute may start before the grid ahead of it on the
// stream has finished; griddepcontrol.wait blocks until that grid has
// completed and its memory is visible, and launch_dependents lets the next
// such grid start.  Both are no-ops for grids launched the ordinary way.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- host: TMA tensor maps --------------------------------------------------------

// Launches kern with the programmatic stream-serialisation attribute when pdl
// is set (the grid may start while the one ahead of it on the stream runs).
template <typename... Params, typename... Args>
cudaError_t launch_maybe_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  return n;
}



inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
// Rows past `rows` read as zeros.
inline bool make_map(CUtensorMap* m, const void* ptr, int rows, int heads) {
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

}  // namespace chunk
}  // namespace gdn
