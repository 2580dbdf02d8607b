// gdn_internal.h -- launch descriptors shared by the host API (gdn_api.cpp)
// and the kernel translation units.  Everything here is already validated:
// the launchers only choose a configuration and launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// Bits of the per-device status word (see gdn_status.cu).
enum : unsigned {
  kStatusBadIndex = 1u,     // state index outside [-1, slots)
  kStatusBadSeqlens = 2u,   // cu_seqlens not 0..T, empty or decreasing range
  kStatusTimeout = 4u,      // a bounded device wait gave up
};

// Counts one kernel launch (gdn_launch_count()).
void note_launch();

// Device address of the current device's status word (cached per device);
// nullptr if the symbol could not be resolved.
unsigned* status_word();

// Records `msg` as the calling thread's gdn_last_error_message() and returns
// `code` (for sources outside the API translation unit).
int report_error(int code, const char* msg);

struct PrepareLaunch {
  int T, N, Hk, Hv, Dk, Dv, K;
  bool bf16, norm;
  const void* x;
  int64_t x_stride;  // elements
  const float* w;
  const void* a;
  int64_t a_stride;
  const void* b;
  int64_t b_stride;
  const float* A_log;
  const float* dt_bias;
  const int32_t* cu;
  const int32_t* sidx;      // may be null
  const uint8_t* has_init;  // may be null
  float* conv_pool;
  int64_t slots;
  int state_len;                // speculative prepare: conv row length per channel
  const int32_t* num_accepted;  // speculative prepare: [N]
  void* q;
  void* k;
  void* v;
  float* g;
  float* beta;
  unsigned* status;
};
cudaError_t launch_prepare(const PrepareLaunch& p, cudaStream_t s);
// The prepare of a speculative step: sequence s's conv row (slot sidx[s],
// state_len entries per channel) is read at offset num_accepted[s] - 1 and
// shifted by one tap; has_init is ignored.
cudaError_t launch_spec_prepare(const PrepareLaunch& p, cudaStream_t s);

// One token per row (decode) or token-sequential over sequences (recurrent
// prefill) -- the same register-resident row update.
struct RecurLaunch {
  int T, N, Hk, Hv, Dk, Dv;
  bool bf16, norm;
  float scale;
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  float* pool;
  int64_t slots;
  const int32_t* cu;        // null for decode (row b = sequence b)
  const int32_t* sidx;      // may be null; [N, num_cols] for the speculative decode
  const uint8_t* has_init;  // may be null (prefill only)
  const int32_t* num_accepted;  // speculative decode only: [N]
  int num_cols;                 // speculative decode only
  void* out;
  unsigned* status;
  // Gated RMSNorm of the output rows (on when onorm_w != nullptr): out =
  // core / sqrt(mean(core^2) + eps) * w * act(z), core rounded to the
  // activation type first.
  const void* onorm_z;
  int64_t onorm_z_stride;  // elements between token rows of z
  const void* onorm_w;
  float onorm_eps;
  bool onorm_sigmoid;
  bool onorm_in_kernel;  // decode: inside the recurrence kernel where it fits
};
cudaError_t launch_decode(const RecurLaunch& p, cudaStream_t s);
cudaError_t launch_recurrent(const RecurLaunch& p, cudaStream_t s);
// KDA: the recurrent prefill with g [T, Hv, Dk], a log decay per key channel
// (p.norm must be false).
cudaError_t launch_kda(const RecurLaunch& p, cudaStream_t s);
// Speculative multi-token decode: sequence s's initial slot is
// sidx[s * num_cols + num_accepted[s] - 1] and the state after its token j is
// stored into sidx[s * num_cols + j] (negative: skipped); p.norm false.
cudaError_t launch_spec_decode(const RecurLaunch& p, cudaStream_t s);
bool recurrent_supported(int Dk);
// Whether gdn_decode applies the output norm inside the recurrence kernel
// (the row's value-dimension slices, 64 rows each at Dk = 128, fit one CTA
// of at most 4 x 128 threads).
bool decode_norm_in_kernel(int Dk, int Dv);

// Decode in one launch from the packed projections: conv update, SiLU, q/k
// norm, gates and the recurrence (one token per row b; the conv pool and the
// state pool share the slot sidx[b]).
struct PackedDecodeLaunch {
  int B, Hk, Hv, Dk, Dv, K;
  bool bf16, norm;
  float scale;
  const void* x;  // raw (pre-conv) rows: q, k, v channels first
  int64_t x_stride;
  const float* w;
  const void* a;
  int64_t a_stride;
  const void* b;
  int64_t b_stride;
  const float* A_log;
  const float* dt_bias;
  const int32_t* sidx;
  float* conv_pool;  // [slots, C_conv, K-1]
  float* pool;       // [slots, Hv, Dv, Dk]
  int64_t slots;
  void* out;
  unsigned* status;
};
bool packed_decode_supported(int Dk, int Dv, int K);
cudaError_t launch_packed_decode(const PackedDecodeLaunch& p, cudaStream_t s);

// Chunked (C = 64) tensor-core prefill.
struct ChunkedLaunch {
  RecurLaunch r;
  void* workspace;
  size_t workspace_bytes;
};
bool chunked_supported(int Dk, int Dv, bool bf16);

// The chunked form of the KDA recurrence (g [T, Hv, Dk]; p.norm false): two
// launches over a caller workspace of kda_chunked_workspace_bytes().
bool kda_chunked_supported(int Dk, int Dv, bool bf16);
size_t kda_chunked_workspace_bytes(int64_t T, int64_t N, int64_t Hv, int64_t Dk, int64_t Dv);
cudaError_t launch_kda_chunked(const ChunkedLaunch& c, cudaStream_t s);

// The same chunked form in one launch of one CTA per (sequence, value head);
// with a workspace of fused_workspace_bytes() and more chains than SMs, one
// CTA per SM over a wrap-around schedule of the chains' chunks (a small
// schedule launch first).
bool fused_supported(int Dk, int Dv, bool bf16);
size_t fused_workspace_bytes(int64_t N, int64_t Hv);
cudaError_t launch_fused(const RecurLaunch& p, void* workspace, size_t workspace_bytes,
                         cudaStream_t s);

// Gated RMSNorm of the recurrence output.
struct NormLaunch {
  int64_t rows;   // tokens * heads
  int heads, dim;
  bool bf16, sigmoid_gate;
  float eps;
  const void* core;
  const void* z;
  int64_t z_stride;  // elements between token rows of z
  const void* weight;
  void* out;
};
cudaError_t launch_gated_rmsnorm(const NormLaunch& p, cudaStream_t s);
size_t chunked_workspace_bytes(int64_t T, int64_t N, int64_t Hv, int64_t Dk, int64_t Dv);
cudaError_t launch_chunked(const ChunkedLaunch& p, cudaStream_t s);

}  // namespace gdn
