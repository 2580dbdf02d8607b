// gdn_api.cpp -- the C ABI of libgdn: argument validation and dispatch.
//
// Shape and length rules follow [cpu.rs] (ferrum-kernels 0.8.0,
// src/ferrum_kernels/backend/cpu.rs) validate_gated_delta_rule_shape,
// validate_linear_attention_prepare_shape and the cu_seqlens rules of
// recurrent_gated_delta_rule_varlen_f32, with the same message text.  Index
// rules follow [qwen3_5.cpp] (vllm.cpp, src/vllm/model_executor/models/
// qwen3_5.cpp) ValidateGdnStateIndices.  On any error nothing is launched.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

thread_local std::string t_msg;

int fail(int code, std::string m) {
  t_msg = std::move(m);
  return code;
}
int succeed() {
  t_msg.clear();
  return GDN_OK;
}

std::string S(int64_t v) { return std::to_string(v); }

struct LenRule {
  const char* label;
  int64_t actual, expected;
};

template <size_t N>
int check_lengths(const char* prefix, const LenRule (&rules)[N]) {
  for (const auto& r : rules)
    if (r.actual < r.expected)
      return fail(GDN_ERR_SHAPE, std::string(prefix) + " " + r.label + " length " + S(r.actual) +
                                     " < expected " + S(r.expected));
  return GDN_OK;
}

int check_act_dtype(int32_t dt) {
  if (dt != GDN_DTYPE_F32 && dt != GDN_DTYPE_BF16)
    return fail(GDN_ERR_DTYPE, "act_dtype must be GDN_DTYPE_F32 or GDN_DTYPE_BF16, got " + S(dt));
  return GDN_OK;
}

int64_t elem_size(int32_t dt) { return dt == GDN_DTYPE_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int require_ptr(const void* p, const char* label) {
  if (p == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, std::string(label) + " is NULL");
  return GDN_OK;
}

int require_aligned(const void* p, const char* label) {
  if (!aligned16(p))
    return fail(GDN_ERR_INVALID_ARGUMENT, std::string(label) + " must be 16-byte aligned");
  return GDN_OK;
}

// [cpu.rs] validate_gated_delta_rule_shape: dims positive, Hv % Hk == 0.
int check_recurrence_dims(int64_t tokens, int64_t hk, int64_t hv, int64_t dk, int64_t dv) {
  if (tokens <= 0 || hk <= 0 || hv <= 0 || dk <= 0 || dv <= 0)
    return fail(GDN_ERR_SHAPE, "gated_delta_rule shape must be positive, got tokens=" + S(tokens) +
                                   " key_heads=" + S(hk) + " value_heads=" + S(hv) +
                                   " key_dim=" + S(dk) + " value_dim=" + S(dv));
  if (hv % hk != 0)
    return fail(GDN_ERR_SHAPE, "gated_delta_rule value_heads " + S(hv) +
                                   " must be divisible by key_heads " + S(hk));
  return GDN_OK;
}

// [cpu.rs] recurrent_gated_delta_rule_varlen_f32 (and
// linear_attention_prepare_varlen_f32) cu_seqlens rules.  The page prints
// cu.first() / cu.last(), Rust Options, with {:?}: "Some(v)".
int check_cu_host(const int32_t* cu, int64_t n, int64_t total, const char* who) {
  if (cu[0] != 0 || cu[n] != total)
    return fail(GDN_ERR_INVALID_ARGUMENT,
                std::string(who) + " cu_seqlens must start at 0 and end at total_tokens " +
                    S(total) + ", got first=Some(" + S(cu[0]) + ") last=Some(" + S(cu[n]) +
                    ")");
  for (int64_t s = 0; s < n; ++s)
    if (cu[s + 1] <= cu[s])
      return fail(GDN_ERR_INVALID_ARGUMENT, std::string(who) + " sequence " + S(s) +
                                                " has empty or non-monotonic range " +
                                                S(cu[s]) + ".." + S(cu[s + 1]));
  return GDN_OK;
}

// The output-norm option of gdn_decode / gdn_prefill_varlen: the rules of
// gdn_gated_rmsnorm ([cpu.rs] validate_gated_rms_norm_shape) for `tokens` rows
// of Hv * Dv values; fills the launch's norm fields.
int check_out_norm(const gdn_out_norm* n, int64_t tokens, int64_t Hv, int64_t Dv, int32_t act_dtype,
                   gdn::RecurLaunch& p) {
  p.onorm_w = nullptr;
  if (n == nullptr) return GDN_OK;
  const int64_t row = Hv * Dv;
  if (n->z_token_stride < row)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gated_rms_norm z token stride shorter than heads * dim");
  const LenRule rules[] = {
      {"z", n->z_len, (tokens - 1) * n->z_token_stride + row},
      {"weight", n->weight_len, Dv},
  };
  if (int rc = check_lengths("gated_rms_norm", rules)) return rc;
  for (auto pr : {std::make_pair(n->z, "out_norm z"), std::make_pair(n->weight, "out_norm weight")}) {
    if (int rc = require_ptr(pr.first, pr.second)) return rc;
    if (int rc = require_aligned(pr.first, pr.second)) return rc;
  }
  const int64_t es = elem_size(act_dtype), vec = 16 / es;
  if ((n->z_token_stride * es) % 16 != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gated_rms_norm z token stride must be a multiple of 16 bytes");
  if (Dv % vec != 0 || Dv > 128 * vec)
    return fail(GDN_ERR_UNSUPPORTED, "the output norm supports Dv a multiple of " + S(vec) +
                                         " and at most " + S(128 * vec));
  if (!(n->eps >= 0.0f)) return fail(GDN_ERR_INVALID_ARGUMENT, "gated_rms_norm eps must be >= 0");
  p.onorm_z = n->z;
  p.onorm_z_stride = n->z_token_stride;
  p.onorm_w = n->weight;
  p.onorm_eps = n->eps;
  p.onorm_sigmoid = n->sigmoid_gate != 0;
  p.onorm_in_kernel = n->in_kernel != 0;
  return GDN_OK;
}

// The output norm as its own kernel, over the output in place (for the
// prefill forms that do not fuse it).
cudaError_t launch_out_norm_pass(const gdn::RecurLaunch& p, cudaStream_t st) {
  gdn::NormLaunch n{};
  n.rows = (int64_t)p.T * p.Hv;
  n.heads = p.Hv;
  n.dim = p.Dv;
  n.bf16 = p.bf16;
  n.sigmoid_gate = p.onorm_sigmoid;
  n.eps = p.onorm_eps;
  n.core = p.out;
  n.z = p.onorm_z;
  n.z_stride = p.onorm_z_stride;
  n.weight = p.onorm_w;
  n.out = p.out;
  return gdn::launch_gated_rmsnorm(n, st);
}

// [qwen3_5.cpp] ValidateGdnStateIndices: -1 is the only allowed negative, live
// slots in range and distinct (O(n) seen-set).
int check_indices_host(const int32_t* idx, int64_t n, int64_t slots) {
  std::vector<unsigned char> seen(static_cast<size_t>(slots), 0);
  for (int64_t i = 0; i < n; ++i) {
    const int32_t slot = idx[i];
    if (slot < 0) {
      if (slot != -1) return fail(GDN_ERR_INVALID_ARGUMENT, "invalid negative GDN state index");
      continue;
    }
    if (slot >= slots) return fail(GDN_ERR_INVALID_ARGUMENT, "GDN state index out of range");
    if (seen[slot]) return fail(GDN_ERR_INVALID_ARGUMENT, "duplicate live GDN state index");
    seen[slot] = 1;
  }
  return GDN_OK;
}

// [qwen3_5.cpp] spec metadata validation, on the host mirrors: offsets span
// the tokens, a request holds at most num_cols tokens (empty requests are
// allowed, as [cpu_ops.cpp] GdnSpecDecodeKernel skips them), num_accepted in
// [1, num_cols], slots below state_slots; and no live slot is named by two
// requests' rows (their CTAs would race on it).
int check_spec_host(const int32_t* cu, const int32_t* sidx, const int32_t* nat, int64_t n,
                    int64_t cols, int64_t total, int64_t slots) {
  if (cu != nullptr) {
    if (cu[0] != 0 || cu[n] != total)
      return fail(GDN_ERR_INVALID_ARGUMENT, "spec query offsets must span the spec tokens");
    for (int64_t i = 0; i < n; ++i)
      if (cu[i + 1] < cu[i] || cu[i + 1] - cu[i] > cols)
        return fail(GDN_ERR_INVALID_ARGUMENT, "spec request " + S(i) + " has range " +
                                                  S(cu[i]) + ".." + S(cu[i + 1]) +
                                                  ", not 0.." + S(cols) + " tokens");
  }
  if (nat != nullptr)
    for (int64_t i = 0; i < n; ++i)
      if (nat[i] < 1 || nat[i] > cols)
        return fail(GDN_ERR_INVALID_ARGUMENT, "num_accepted_tokens must be in [1, num_spec + 1]");
  if (sidx != nullptr) {
    std::vector<int64_t> owner(static_cast<size_t>(slots), -1);
    for (int64_t i = 0; i < n; ++i)
      for (int64_t c = 0; c < cols; ++c) {
        const int32_t slot = sidx[i * cols + c];
        if (slot < 0) continue;
        if (slot >= slots)
          return fail(GDN_ERR_INVALID_ARGUMENT, "spec GDN state slot out of range");
        if (owner[slot] >= 0 && owner[slot] != i)
          return fail(GDN_ERR_INVALID_ARGUMENT, "spec GDN state slot " + S(slot) +
                                                    " named by two requests");
        owner[slot] = i;
      }
  }
  return GDN_OK;
}

bool fits_i32(int64_t v) { return v >= 0 && v <= INT32_MAX; }

// GDN_DEBUG_CHECKS=1 in the environment (read once): metadata given only in
// device memory is copied to the host and checked as its host mirror would be.
bool debug_checks() {
  static const bool on = [] {
    const char* e = std::getenv("GDN_DEBUG_CHECKS");
    return e != nullptr && std::strcmp(e, "1") == 0;
  }();
  return on;
}

// The host view of n int32 metadata values: the caller's host mirror, else
// (under GDN_DEBUG_CHECKS) a copy of the device array made on the call's
// stream, else nullptr (nothing to check on the host).
int host_view(const int32_t* host, const int32_t* dev, int64_t n, cudaStream_t st,
              std::vector<int32_t>& buf, const int32_t*& out) {
  out = host;
  if (host != nullptr || dev == nullptr || n <= 0 || !debug_checks()) return GDN_OK;
  buf.resize(static_cast<size_t>(n));
  cudaError_t e = cudaMemcpyAsync(buf.data(), dev, static_cast<size_t>(n) * sizeof(int32_t),
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess)
    return fail(GDN_ERR_CUDA, std::string("GDN_DEBUG_CHECKS metadata copy: ") + cudaGetErrorString(e));
  out = buf.data();
  return GDN_OK;
}

}  // namespace

int gdn::report_error(int code, const char* msg) { return fail(code, msg); }

namespace {

int launch_result(cudaError_t e, const char* what) {
  if (e != cudaSuccess)
    return fail(GDN_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return succeed();
}

float resolve_scale(float scale, int64_t dk) {
  return scale < 0.0f ? 1.0f / std::sqrt(static_cast<float>(dk)) : scale;
}

}  // namespace

extern "C" {

int gdn_version(void) { return 100; }

const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE";
    case GDN_ERR_INVALID_ARGUMENT: return "GDN_ERR_INVALID_ARGUMENT";
    case GDN_ERR_DTYPE: return "GDN_ERR_DTYPE";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    case GDN_ERR_DEVICE_CHECK: return "GDN_ERR_DEVICE_CHECK";
    default: return "GDN_ERR_UNKNOWN";
  }
}

const char* gdn_last_error_message(void) { return t_msg.c_str(); }

int gdn_read_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, std::string("sync: ") + cudaGetErrorString(e));
  unsigned* w = gdn::status_word();
  if (w == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
  unsigned v = 0;
  e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(w, 0, sizeof(unsigned));
  if (e != cudaSuccess)
    return fail(GDN_ERR_CUDA, std::string("status read: ") + cudaGetErrorString(e));
  if (v & gdn::kStatusTimeout) return fail(GDN_ERR_TIMEOUT, "a device-side wait timed out");
  if (v & gdn::kStatusBadIndex)
    return fail(GDN_ERR_DEVICE_CHECK, "a kernel saw a state index outside [-1, slots)");
  if (v & gdn::kStatusBadSeqlens)
    return fail(GDN_ERR_DEVICE_CHECK, "a kernel saw malformed cu_seqlens");
  return succeed();
}

namespace {

// The checks gdn_prepare and gdn_spec_prepare share, up to the per-sequence
// metadata; fills *p.  row_len is the conv row length per channel: K-1, or
// the widened row of a speculative step.
int prepare_common(const gdn_prepare_args* a, int64_t row_len, gdn::PrepareLaunch* out) {
  if (int rc = check_act_dtype(a->act_dtype)) return rc;
  // [cpu.rs] validate_linear_attention_prepare_shape
  if (a->T <= 0 || a->Hk <= 0 || a->Hv <= 0 || a->Dk <= 0 || a->Dv <= 0 || a->K <= 0)
    return fail(GDN_ERR_SHAPE, "linear_attention_prepare shape must be positive, got tokens=" +
                                   S(a->T) + " key_heads=" + S(a->Hk) + " value_heads=" +
                                   S(a->Hv) + " key_dim=" + S(a->Dk) + " value_dim=" + S(a->Dv) +
                                   " conv_kernel=" + S(a->K));
  if (a->N <= 0) return fail(GDN_ERR_SHAPE, "linear_attention_prepare_varlen batch must be positive");
  const int64_t qk_total = a->Hk * a->Dk, v_total = a->Hv * a->Dv;
  const int64_t C = 2 * qk_total + v_total;
  const int64_t x_stride = a->mixed_qkv_stride > 0 ? a->mixed_qkv_stride : C;
  const int64_t a_stride = a->a_raw_stride > 0 ? a->a_raw_stride : a->Hv;
  const int64_t b_stride = a->b_raw_stride > 0 ? a->b_raw_stride : a->Hv;
  if (x_stride < C || a_stride < a->Hv || b_stride < a->Hv)
    return fail(GDN_ERR_SHAPE, "linear_attention_prepare row stride shorter than the row");
  const LenRule rules[] = {
      {"mixed_qkv_raw", a->mixed_qkv_len, (a->T - 1) * x_stride + C},
      {"conv_weight", a->conv_weight_len, C * a->K},
      {"a_raw", a->a_raw_len, (a->T - 1) * a_stride + a->Hv},
      {"b_raw", a->b_raw_len, (a->T - 1) * b_stride + a->Hv},
      {"a_log", a->A_log_len, a->Hv},
      {"dt_bias", a->dt_bias_len, a->Hv},
      {"query", a->q_len, a->T * qk_total},
      {"key", a->k_len, a->T * qk_total},
      {"value", a->v_len, a->T * v_total},
      {"g", a->g_len, a->T * a->Hv},
      {"beta", a->beta_len, a->T * a->Hv},
  };
  if (int rc = check_lengths("linear_attention_prepare", rules)) return rc;
  if (a->conv_state_slots <= 0)
    return fail(GDN_ERR_SHAPE, "linear_attention_prepare conv_state must have at least one slot");
  const LenRule pool_rule[] = {{"conv_state", a->conv_state_len, a->conv_state_slots * C * row_len}};
  if (int rc = check_lengths("linear_attention_prepare", pool_rule)) return rc;
  for (auto pr : {std::make_pair((const void*)a->mixed_qkv, "mixed_qkv"),
                  std::make_pair((const void*)a->conv_weight, "conv_weight"),
                  std::make_pair((const void*)a->a_raw, "a_raw"),
                  std::make_pair((const void*)a->b_raw, "b_raw"),
                  std::make_pair((const void*)a->A_log, "A_log"),
                  std::make_pair((const void*)a->dt_bias, "dt_bias"),
                  std::make_pair((const void*)a->cu_seqlens, "cu_seqlens"),
                  std::make_pair((const void*)a->q, "q"), std::make_pair((const void*)a->k, "k"),
                  std::make_pair((const void*)a->v, "v"), std::make_pair((const void*)a->g, "g"),
                  std::make_pair((const void*)a->beta, "beta")})
    if (int rc = require_ptr(pr.first, pr.second)) return rc;
  if (row_len > 0)
    if (int rc = require_ptr(a->conv_state, "conv_state")) return rc;
  // Kernel coverage.
  const int64_t cpt = a->act_dtype == GDN_DTYPE_BF16 ? 8 : 4;  // channels per 16-byte vector
  const bool dk_pow2 = (a->Dk & (a->Dk - 1)) == 0;
  if (a->K > 8 || !dk_pow2 || a->Dk < cpt || a->Dk > 32 * cpt || a->Dv % cpt != 0)
    return fail(GDN_ERR_UNSUPPORTED,
                "gdn_prepare supports K <= 8, Dk a power of two in [" + S(cpt) + ", " +
                    S(32 * cpt) + "] and Dv a multiple of " + S(cpt));
  if (!fits_i32(a->T) || !fits_i32(a->N) || !fits_i32(a->T * C))
    return fail(GDN_ERR_UNSUPPORTED, "gdn_prepare sizes exceed 32-bit token indexing");
  const int64_t es = elem_size(a->act_dtype);
  for (auto pr : {std::make_pair((const void*)a->mixed_qkv, "mixed_qkv"),
                  std::make_pair((const void*)a->q, "q"), std::make_pair((const void*)a->k, "k"),
                  std::make_pair((const void*)a->v, "v")})
    if (int rc = require_aligned(pr.first, pr.second)) return rc;
  if ((x_stride * es) % 16 != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "mixed_qkv row stride must be a multiple of 16 bytes");

  gdn::PrepareLaunch& p = *out;
  p = gdn::PrepareLaunch{};
  p.T = (int)a->T;
  p.N = (int)a->N;
  p.Hk = (int)a->Hk;
  p.Hv = (int)a->Hv;
  p.Dk = (int)a->Dk;
  p.Dv = (int)a->Dv;
  p.K = (int)a->K;
  p.bf16 = a->act_dtype == GDN_DTYPE_BF16;
  p.norm = a->apply_qk_l2norm != 0;
  p.x = a->mixed_qkv;
  p.x_stride = x_stride;
  p.w = a->conv_weight;
  p.a = a->a_raw;
  p.a_stride = a_stride;
  p.b = a->b_raw;
  p.b_stride = b_stride;
  p.A_log = a->A_log;
  p.dt_bias = a->dt_bias;
  p.cu = a->cu_seqlens;
  p.sidx = a->state_indices;
  p.has_init = a->has_initial_state;
  p.conv_pool = a->conv_state;
  p.slots = a->conv_state_slots;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.g = a->g;
  p.beta = a->beta;
  return GDN_OK;
}

}  // namespace

int gdn_prepare(const gdn_prepare_args* a, void* stream) {
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "args is NULL");
  gdn::PrepareLaunch p;
  if (int rc = prepare_common(a, a->K - 1, &p)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<int32_t> cu_buf, idx_buf;
  const int32_t *cuh = nullptr, *idxh = nullptr;
  if (int rc = host_view(a->cu_seqlens_host, a->cu_seqlens, a->N + 1, st, cu_buf, cuh)) return rc;
  if (int rc = host_view(a->state_indices_host, a->state_indices, a->N, st, idx_buf, idxh))
    return rc;
  if (cuh != nullptr)
    if (int rc = check_cu_host(cuh, a->N, a->T, "linear_attention_prepare_varlen")) return rc;
  if (idxh != nullptr)
    if (int rc = check_indices_host(idxh, a->N, a->conv_state_slots)) return rc;
  if (a->state_indices == nullptr && a->N > a->conv_state_slots)
    return fail(GDN_ERR_SHAPE, "linear_attention_prepare conv_state has fewer slots than sequences");
  p.status = gdn::status_word();
  if (p.status == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
  return launch_result(gdn::launch_prepare(p, st), "gdn_prepare");
}

int gdn_spec_prepare(const gdn_spec_prepare_args* sa, void* stream) {
  if (sa == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "args is NULL");
  const gdn_prepare_args* a = &sa->base;
  const int64_t width = a->K - 1, row = sa->conv_state_width, max_q = row - width + 1;
  if (a->K < 2)
    return fail(GDN_ERR_UNSUPPORTED, "gdn_spec_prepare needs conv_kernel >= 2 (a conv tail to carry)");
  if (row < width || max_q < 1)
    return fail(GDN_ERR_SHAPE, "spec conv row of " + S(row) + " entries is shorter than conv_kernel - 1 = " +
                                   S(width));
  if (a->has_initial_state != nullptr)
    return fail(GDN_ERR_INVALID_ARGUMENT, "spec conv update takes no has_initial_state");
  gdn::PrepareLaunch p;
  if (int rc = prepare_common(a, row, &p)) return rc;
  for (auto pr : {std::make_pair((const void*)a->state_indices, "state_indices"),
                  std::make_pair((const void*)sa->num_accepted, "num_accepted")})
    if (int rc = require_ptr(pr.first, pr.second)) return rc;
  if (a->T > a->N * max_q)
    return fail(GDN_ERR_SHAPE, "spec conv update has " + S(a->T) + " tokens, more than requests * "
                               "max_query_len = " + S(a->N * max_q));
  if (row > 16)
    return fail(GDN_ERR_UNSUPPORTED, "gdn_spec_prepare supports conv rows of at most 16 entries");
  // [qwen3_5.cpp] spec metadata rules on the host mirrors: requests of at
  // most max_q tokens, num_accepted in [1, max_q], one conv row per request
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<int32_t> cu_buf, idx_buf, na_buf;
  const int32_t *cuh = nullptr, *idxh = nullptr, *nah = nullptr;
  if (int rc = host_view(a->cu_seqlens_host, a->cu_seqlens, a->N + 1, st, cu_buf, cuh)) return rc;
  if (int rc = host_view(a->state_indices_host, a->state_indices, a->N, st, idx_buf, idxh))
    return rc;
  if (int rc = host_view(sa->num_accepted_host, sa->num_accepted, a->N, st, na_buf, nah)) return rc;
  if (int rc = check_spec_host(cuh, nullptr, nah, a->N, max_q, a->T, a->conv_state_slots))
    return rc;
  if (int rc = check_spec_host(nullptr, idxh, nullptr, a->N, 1, a->T, a->conv_state_slots))
    return rc;
  p.sidx = a->state_indices;
  p.has_init = nullptr;
  p.state_len = (int)row;
  p.num_accepted = sa->num_accepted;
  p.status = gdn::status_word();
  if (p.status == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
  return launch_result(gdn::launch_spec_prepare(p, st), "gdn_spec_prepare");
}

namespace {

// Shared checks of decode and prefill: [cpu.rs] validate_gated_delta_rule_shape
// with the state pool in place of initial/final state.
int check_recurrence(int64_t tokens, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                     int32_t act_dtype, const void* q, int64_t q_len, const void* k,
                     int64_t k_len, const void* v, int64_t v_len, const float* g, int64_t g_len,
                     const float* beta, int64_t beta_len, const float* state,
                     int64_t state_slots, int64_t state_len, const void* out, int64_t out_len) {
  if (int rc = check_act_dtype(act_dtype)) return rc;
  if (int rc = check_recurrence_dims(tokens, Hk, Hv, Dk, Dv)) return rc;
  if (state_slots <= 0) return fail(GDN_ERR_SHAPE, "gated_delta_rule state must have at least one slot");
  const LenRule rules[] = {
      {"query", q_len, tokens * Hk * Dk},
      {"key", k_len, tokens * Hk * Dk},
      {"value", v_len, tokens * Hv * Dv},
      {"g", g_len, tokens * Hv},
      {"beta", beta_len, tokens * Hv},
      {"state", state_len, state_slots * Hv * Dv * Dk},
      {"out", out_len, tokens * Hv * Dv},
  };
  if (int rc = check_lengths("gated_delta_rule", rules)) return rc;
  for (auto pr : {std::make_pair(q, "q"), std::make_pair(k, "k"), std::make_pair(v, "v"),
                  std::make_pair((const void*)g, "g"), std::make_pair((const void*)beta, "beta"),
                  std::make_pair((const void*)state, "state"), std::make_pair(out, "out")})
    if (int rc = require_ptr(pr.first, pr.second)) return rc;
  for (auto pr : {std::make_pair(q, "q"), std::make_pair(k, "k"), std::make_pair(v, "v"),
                  std::make_pair((const void*)state, "state"), std::make_pair(out, "out")})
    if (int rc = require_aligned(pr.first, pr.second)) return rc;
  if (!fits_i32(tokens) || !fits_i32(tokens * Hv * Dv) || !fits_i32(tokens * Hk * Dk))
    return fail(GDN_ERR_UNSUPPORTED, "gated_delta_rule sizes exceed 32-bit token indexing");
  return GDN_OK;
}

}  // namespace

int gdn_packed_decode(const gdn_packed_decode_args* a, void* stream) {
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "args is NULL");
  if (int rc = check_act_dtype(a->act_dtype)) return rc;
  if (a->B <= 0 || a->K <= 0)
    return fail(GDN_ERR_SHAPE, "packed GDN decode shape must be positive, got batch=" + S(a->B) +
                                   " conv_kernel=" + S(a->K));
  if (int rc = check_recurrence_dims(a->B, a->Hk, a->Hv, a->Dk, a->Dv)) return rc;
  const int64_t qk_total = a->Hk * a->Dk, C = 2 * qk_total + a->Hv * a->Dv;
  const int64_t x_stride = a->mixed_qkv_stride > 0 ? a->mixed_qkv_stride : C;
  const int64_t a_stride = a->a_raw_stride > 0 ? a->a_raw_stride : a->Hv;
  const int64_t b_stride = a->b_raw_stride > 0 ? a->b_raw_stride : a->Hv;
  if (x_stride < C || a_stride < a->Hv || b_stride < a->Hv)
    return fail(GDN_ERR_SHAPE, "packed GDN decode row stride shorter than the row");
  if (a->state_slots <= 0) return fail(GDN_ERR_SHAPE, "gated_delta_rule state must have at least one slot");
  const LenRule rules[] = {
      {"mixed_qkv", a->mixed_qkv_len, (a->B - 1) * x_stride + C},
      {"conv_weight", a->conv_weight_len, C * a->K},
      {"a_raw", a->a_raw_len, (a->B - 1) * a_stride + a->Hv},
      {"b_raw", a->b_raw_len, (a->B - 1) * b_stride + a->Hv},
      {"a_log", a->A_log_len, a->Hv},
      {"dt_bias", a->dt_bias_len, a->Hv},
      {"conv_state", a->conv_state_len, a->state_slots * C * (a->K - 1)},
      {"state", a->state_len, a->state_slots * a->Hv * a->Dv * a->Dk},
      {"out", a->out_len, a->B * a->Hv * a->Dv},
  };
  if (int rc = check_lengths("packed_gdn_decode", rules)) return rc;
  for (auto pr : {std::make_pair((const void*)a->mixed_qkv, "mixed_qkv"),
                  std::make_pair((const void*)a->conv_weight, "conv_weight"),
                  std::make_pair((const void*)a->a_raw, "a_raw"),
                  std::make_pair((const void*)a->b_raw, "b_raw"),
                  std::make_pair((const void*)a->A_log, "A_log"),
                  std::make_pair((const void*)a->dt_bias, "dt_bias"),
                  std::make_pair((const void*)a->state_indices, "state_indices"),
                  std::make_pair((const void*)a->conv_state, "conv_state"),
                  std::make_pair((const void*)a->state, "state"),
                  std::make_pair((const void*)a->out, "out")})
    if (int rc = require_ptr(pr.first, pr.second)) return rc;
  if (int rc = require_aligned(a->state, "state")) return rc;
  if (!gdn::packed_decode_supported((int)a->Dk, (int)a->Dv, (int)a->K))
    return fail(GDN_ERR_UNSUPPORTED, "gdn_packed_decode supports Dk in {64, 128}, Dv <= 128 and "
                                     "conv_kernel in [2, 4]");
  if (!fits_i32(a->B * a->Hv * a->Dv) || !fits_i32(C))
    return fail(GDN_ERR_UNSUPPORTED, "packed GDN decode sizes exceed 32-bit indexing");
  {
    std::vector<int32_t> idx_buf;
    const int32_t* idxh = nullptr;
    if (int rc = host_view(a->state_indices_host, a->state_indices, a->B,
                           static_cast<cudaStream_t>(stream), idx_buf, idxh))
      return rc;
    if (idxh != nullptr)
      if (int rc = check_indices_host(idxh, a->B, a->state_slots)) return rc;
  }
  gdn::PackedDecodeLaunch p{};
  p.B = (int)a->B;
  p.Hk = (int)a->Hk;
  p.Hv = (int)a->Hv;
  p.Dk = (int)a->Dk;
  p.Dv = (int)a->Dv;
  p.K = (int)a->K;
  p.bf16 = a->act_dtype == GDN_DTYPE_BF16;
  p.norm = a->apply_qk_l2norm != 0;
  p.scale = resolve_scale(a->scale, a->Dk);
  p.x = a->mixed_qkv;
  p.x_stride = x_stride;
  p.w = a->conv_weight;
  p.a = a->a_raw;
  p.a_stride = a_stride;
  p.b = a->b_raw;
  p.b_stride = b_stride;
  p.A_log = a->A_log;
  p.dt_bias = a->dt_bias;
  p.sidx = a->state_indices;
  p.conv_pool = a->conv_state;
  p.pool = a->state;
  p.slots = a->state_slots;
  p.out = a->out;
  p.status = gdn::status_word();
  if (p.status == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
  return launch_result(gdn::launch_packed_decode(p, static_cast<cudaStream_t>(stream)),
                       "gdn_packed_decode");
}

int gdn_decode(const gdn_decode_args* a, void* stream) {
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "args is NULL");
  if (int rc = check_recurrence(a->B, a->Hk, a->Hv, a->Dk, a->Dv, a->act_dtype, a->q, a->q_len,
                                a->k, a->k_len, a->v, a->v_len, a->g, a->g_len, a->beta,
                                a->beta_len, a->state, a->state_slots, a->state_len, a->out,
                                a->out_len))
    return rc;
  if (!gdn::recurrent_supported((int)a->Dk))
    return fail(GDN_ERR_UNSUPPORTED, "gdn_decode supports Dk in {16, 32, 64, 128, 256}");
  {
    std::vector<int32_t> idx_buf;
    const int32_t* idxh = nullptr;
    if (int rc = host_view(a->state_indices_host, a->state_indices, a->B,
                           static_cast<cudaStream_t>(stream), idx_buf, idxh))
      return rc;
    if (idxh != nullptr)
      if (int rc = check_indices_host(idxh, a->B, a->state_slots)) return rc;
  }
  if (a->state_indices == nullptr && a->B > a->state_slots)
    return fail(GDN_ERR_SHAPE, "gated_delta_rule state has fewer slots than rows");
  gdn::RecurLaunch p{};
  p.T = (int)a->B;
  p.N = (int)a->B;
  p.Hk = (int)a->Hk;
  p.Hv = (int)a->Hv;
  p.Dk = (int)a->Dk;
  p.Dv = (int)a->Dv;
  p.bf16 = a->act_dtype == GDN_DTYPE_BF16;
  p.norm = a->use_qk_l2norm != 0;
  p.scale = resolve_scale(a->scale, a->Dk);
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.g = a->g;
  p.beta = a->beta;
  p.pool = a->state;
  p.slots = a->state_slots;
  p.cu = nullptr;
  p.sidx = a->state_indices;
  p.has_init = nullptr;
  p.out = a->out;
  if (int rc = check_out_norm(a->out_norm, a->B, a->Hv, a->Dv, a->act_dtype, p)) return rc;
  p.status = gdn::status_word();
  if (p.status == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.onorm_w == nullptr || (p.onorm_in_kernel && gdn::decode_norm_in_kernel(p.Dk, p.Dv)))
    return launch_result(gdn::launch_decode(p, st), "gdn_decode");
  // the norm as a second kernel over the output in place
  gdn::RecurLaunch plain = p;
  plain.onorm_w = nullptr;
  if (int rc = launch_result(gdn::launch_decode(plain, st), "gdn_decode")) return rc;
  return launch_result(launch_out_norm_pass(p, st), "gdn_decode(output norm)");
}

int gdn_kda_varlen(const gdn_kda_args* a, void* stream) {
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "args is NULL");
  if (int rc = check_recurrence(a->T, a->Hk, a->Hv, a->Dk, a->Dv, a->act_dtype, a->q, a->q_len,
                                a->k, a->k_len, a->v, a->v_len, a->g, a->g_len, a->beta,
                                a->beta_len, a->state, a->state_slots, a->state_len, a->out,
                                a->out_len))
    return rc;
  if (a->g_len < a->T * a->Hv * a->Dk)
    return fail(GDN_ERR_SHAPE, "kda_gated_delta_rule g length " + S(a->g_len) + " < expected " +
                                   S(a->T * a->Hv * a->Dk));
  if (int rc = require_aligned(a->g, "g")) return rc;
  if (a->N <= 0)
    return fail(GDN_ERR_SHAPE, "kda_gated_delta_rule shape must be positive, got batch=" +
                                   S(a->N) + " total_tokens=" + S(a->T));
  if (require_ptr(a->cu_seqlens, "cu_seqlens")) return GDN_ERR_INVALID_ARGUMENT;
  {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::vector<int32_t> cu_buf, idx_buf;
    const int32_t *cuh = nullptr, *idxh = nullptr;
    if (int rc = host_view(a->cu_seqlens_host, a->cu_seqlens, a->N + 1, st, cu_buf, cuh))
      return rc;
    if (int rc = host_view(a->state_indices_host, a->state_indices, a->N, st, idx_buf, idxh))
      return rc;
    if (cuh != nullptr)
      if (int rc = check_cu_host(cuh, a->N, a->T, "kda_gated_delta_rule")) return rc;
    if (idxh != nullptr)
      if (int rc = check_indices_host(idxh, a->N, a->state_slots)) return rc;
  }
  if (a->state_indices == nullptr && a->N > a->state_slots)
    return fail(GDN_ERR_SHAPE, "kda_gated_delta_rule state has fewer slots than sequences");
  if (!gdn::recurrent_supported((int)a->Dk))
    return fail(GDN_ERR_UNSUPPORTED, "gdn_kda_varlen supports Dk in {16, 32, 64, 128, 256}");
  if (!fits_i32(a->T * a->Hv * a->Dk))
    return fail(GDN_ERR_UNSUPPORTED, "kda_gated_delta_rule sizes exceed 32-bit indexing");
  if (a->algo != GDN_PREFILL_AUTO && a->algo != GDN_PREFILL_CHUNKED &&
      a->algo != GDN_PREFILL_RECURRENT)
    return fail(GDN_ERR_INVALID_ARGUMENT, "unknown or unsupported KDA algo " + S(a->algo));
  const int32_t algo = gdn_kda_resolve_algo(a->T, a->N, a->Dk, a->Dv, a->act_dtype, a->algo);
  if (algo == GDN_PREFILL_CHUNKED) {
    if (!gdn::kda_chunked_supported((int)a->Dk, (int)a->Dv, a->act_dtype == GDN_DTYPE_BF16))
      return fail(GDN_ERR_UNSUPPORTED,
                  "the chunked KDA prefill supports bf16 activations with Dk = Dv = 128");
    const size_t need = gdn::kda_chunked_workspace_bytes(a->T, a->N, a->Hv, a->Dk, a->Dv);
    if (a->workspace == nullptr || a->workspace_bytes < need)
      return fail(GDN_ERR_INVALID_ARGUMENT, "gdn_kda_varlen workspace needs " + S((int64_t)need) +
                                                " bytes, got " + S((int64_t)a->workspace_bytes));
    if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
      return fail(GDN_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  }
  gdn::RecurLaunch p{};
  p.T = (int)a->T;
  p.N = (int)a->N;
  p.Hk = (int)a->Hk;
  p.Hv = (int)a->Hv;
  p.Dk = (int)a->Dk;
  p.Dv = (int)a->Dv;
  p.bf16 = a->act_dtype == GDN_DTYPE_BF16;
  p.norm = false;
  p.scale = resolve_scale(a->scale, a->Dk);
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.g = a->g;
  p.beta = a->beta;
  p.pool = a->state;
  p.slots = a->state_slots;
  p.cu = a->cu_seqlens;
  p.sidx = a->state_indices;
  p.has_init = a->has_initial_state;
  p.out = a->out;
  p.status = gdn::status_word();
  if (p.status == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
  if (algo == GDN_PREFILL_CHUNKED) {
    gdn::ChunkedLaunch c{p, a->workspace, a->workspace_bytes};
    return launch_result(gdn::launch_kda_chunked(c, static_cast<cudaStream_t>(stream)),
                         "gdn_kda_varlen(chunked)");
  }
  return launch_result(gdn::launch_kda(p, static_cast<cudaStream_t>(stream)), "gdn_kda_varlen");
}

int32_t gdn_kda_resolve_algo(int64_t T, int64_t N, int64_t Dk, int64_t Dv, int32_t act_dtype,
                             int32_t algo) {
  if (algo != GDN_PREFILL_AUTO) return algo;
  return T > N && gdn::kda_chunked_supported((int)Dk, (int)Dv, act_dtype == GDN_DTYPE_BF16)
             ? GDN_PREFILL_CHUNKED
             : GDN_PREFILL_RECURRENT;
}

size_t gdn_kda_workspace_bytes(int64_t T, int64_t N, int64_t Hv, int64_t Dk, int64_t Dv,
                               int32_t act_dtype, int32_t algo) {
  if (gdn_kda_resolve_algo(T, N, Dk, Dv, act_dtype, algo) != GDN_PREFILL_CHUNKED) return 0;
  if (T <= 0 || N <= 0 || Hv <= 0) return 0;
  return gdn::kda_chunked_workspace_bytes(T, N, Hv, Dk, Dv);
}

int gdn_spec_decode(const gdn_spec_decode_args* a, void* stream) {
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "args is NULL");
  if (int rc = check_recurrence(a->T, a->Hk, a->Hv, a->Dk, a->Dv, a->act_dtype, a->q, a->q_len,
                                a->k, a->k_len, a->v, a->v_len, a->g, a->g_len, a->beta,
                                a->beta_len, a->state, a->state_slots, a->state_len, a->out,
                                a->out_len))
    return rc;
  if (a->n_reqs <= 0 || a->num_cols < 1)
    return fail(GDN_ERR_SHAPE, "spec GDN decode needs n_reqs >= 1 and num_cols >= 1, got " +
                                   S(a->n_reqs) + " and " + S(a->num_cols));
  if (a->T > a->n_reqs * a->num_cols)
    return fail(GDN_ERR_SHAPE, "spec GDN decode has " + S(a->T) + " tokens, more than n_reqs * "
                               "num_cols = " + S(a->n_reqs * a->num_cols));
  for (auto pr : {std::make_pair((const void*)a->cu_seqlens, "cu_seqlens"),
                  std::make_pair((const void*)a->state_indices, "state_indices"),
                  std::make_pair((const void*)a->num_accepted, "num_accepted")})
    if (int rc = require_ptr(pr.first, pr.second)) return rc;
  {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::vector<int32_t> cu_buf, idx_buf, na_buf;
    const int32_t *cuh = nullptr, *idxh = nullptr, *nah = nullptr;
    if (int rc = host_view(a->cu_seqlens_host, a->cu_seqlens, a->n_reqs + 1, st, cu_buf, cuh))
      return rc;
    if (int rc = host_view(a->state_indices_host, a->state_indices, a->n_reqs * a->num_cols, st,
                           idx_buf, idxh))
      return rc;
    if (int rc = host_view(a->num_accepted_host, a->num_accepted, a->n_reqs, st, na_buf, nah))
      return rc;
    if (int rc = check_spec_host(cuh, idxh, nah, a->n_reqs, a->num_cols, a->T, a->state_slots))
      return rc;
  }
  if (!gdn::recurrent_supported((int)a->Dk))
    return fail(GDN_ERR_UNSUPPORTED, "gdn_spec_decode supports Dk in {16, 32, 64, 128, 256}");
  if (!fits_i32(a->n_reqs * a->num_cols) || !fits_i32(a->T * a->Hv * a->Dv))
    return fail(GDN_ERR_UNSUPPORTED, "spec GDN decode sizes exceed 32-bit indexing");
  gdn::RecurLaunch p{};
  p.T = (int)a->T;
  p.N = (int)a->n_reqs;
  p.Hk = (int)a->Hk;
  p.Hv = (int)a->Hv;
  p.Dk = (int)a->Dk;
  p.Dv = (int)a->Dv;
  p.bf16 = a->act_dtype == GDN_DTYPE_BF16;
  p.norm = false;
  p.scale = resolve_scale(a->scale, a->Dk);
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.g = a->g;
  p.beta = a->beta;
  p.pool = a->state;
  p.slots = a->state_slots;
  p.cu = a->cu_seqlens;
  p.sidx = a->state_indices;
  p.num_accepted = a->num_accepted;
  p.num_cols = (int)a->num_cols;
  p.out = a->out;
  p.status = gdn::status_word();
  if (p.status == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
  return launch_result(gdn::launch_spec_decode(p, static_cast<cudaStream_t>(stream)),
                       "gdn_spec_decode");
}

int gdn_gated_rmsnorm(const gdn_gated_rmsnorm_args* a, void* stream) {
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "args is NULL");
  if (int rc = check_act_dtype(a->act_dtype)) return rc;
  // [cpu.rs] validate_gated_rms_norm_shape
  if (a->tokens <= 0 || a->heads <= 0 || a->dim <= 0)
    return fail(GDN_ERR_SHAPE, "gated_rms_norm shape must be positive, got tokens=" +
                                   S(a->tokens) + " heads=" + S(a->heads) + " dim=" + S(a->dim));
  const int64_t row = a->heads * a->dim, total = a->tokens * row;
  const int64_t z_stride = a->z_token_stride > 0 ? a->z_token_stride : row;
  if (z_stride < row)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gated_rms_norm z token stride shorter than heads * dim");
  const LenRule rules[] = {
      {"core", a->core_len, total},
      {"z", a->z_len, (a->tokens - 1) * z_stride + row},
      {"weight", a->weight_len, a->dim},
      {"out", a->out_len, total},
  };
  if (int rc = check_lengths("gated_rms_norm", rules)) return rc;
  for (auto pr : {std::make_pair(a->core, "core"), std::make_pair(a->z, "z"),
                  std::make_pair(a->weight, "weight"), std::make_pair((const void*)a->out, "out")}) {
    if (int rc = require_ptr(pr.first, pr.second)) return rc;
    if (int rc = require_aligned(pr.first, pr.second)) return rc;
  }
  const int64_t es = elem_size(a->act_dtype), vec = 16 / es;
  if ((z_stride * es) % 16 != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gated_rms_norm z token stride must be a multiple of 16 bytes");
  if (a->dim % vec != 0 || a->dim > 128 * vec)
    return fail(GDN_ERR_UNSUPPORTED, "gdn_gated_rmsnorm supports dim a multiple of " + S(vec) +
                                         " and at most " + S(128 * vec));
  gdn::NormLaunch p{};
  p.rows = total / a->dim;
  p.heads = (int)a->heads;
  p.dim = (int)a->dim;
  p.bf16 = a->act_dtype == GDN_DTYPE_BF16;
  p.sigmoid_gate = a->sigmoid_gate != 0;
  p.eps = a->eps;
  p.core = a->core;
  p.z = a->z;
  p.z_stride = z_stride;
  p.weight = a->weight;
  p.out = a->out;
  return launch_result(gdn::launch_gated_rmsnorm(p, static_cast<cudaStream_t>(stream)),
                       "gdn_gated_rmsnorm");
}

// [qwen3_5.cpp] ValidateGdnAttentionMetadata, the non-speculative part, in
// the page's order and with its messages (without the "qwen3_5: " prefix).
// The causal-conv chunk metadata it also checks has no counterpart here: the
// prepare kernel derives its tiles from cu_seqlens itself.
int gdn_validate_mixed(const gdn_mixed_meta* m) {
  if (m == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "meta is NULL");
  const int64_t nd = m->num_decodes, np = m->num_prefills;
  const int64_t nd_tok = m->num_decode_tokens, np_tok = m->num_prefill_tokens;
  const int64_t nreq = nd + np;
  if (nd < 0 || np < 0 || nd_tok < 0 || np_tok < 0 || m->num_actual_tokens < 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "negative GDN metadata count");
  if (nd_tok != nd)
    return fail(GDN_ERR_INVALID_ARGUMENT, "non-spec decode requires one token per request");
  if (m->num_actual_tokens != nd_tok + np_tok)
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "GDN decode+prefill+spec tokens must equal actual tokens");
  if (nreq == 0) {
    if (m->num_actual_tokens != 0)
      return fail(GDN_ERR_INVALID_ARGUMENT, "GDN tokens require state metadata");
    return succeed();
  }
  if (m->state_indices_host == nullptr)
    return fail(GDN_ERR_INVALID_ARGUMENT, "missing non-spec GDN state indices");
  if (m->state_slots < 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "GDN state cache has invalid slot count");
  const int32_t* idx = m->state_indices_host;
  if (int rc = check_indices_host(idx, nreq, m->state_slots)) return rc;
  if (!m->allow_inert_padding)
    for (int64_t i = 0; i < nreq; ++i)
      if (idx[i] < 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "live GDN state index must be non-negative");
  if (np == 0) return succeed();
  if (m->cu_seqlens_host == nullptr || m->cu_seqlens_prefill_host == nullptr)
    return fail(GDN_ERR_INVALID_ARGUMENT, "incomplete GDN prefill metadata");
  const int32_t* qsl = m->cu_seqlens_host;
  const int32_t* pqsl = m->cu_seqlens_prefill_host;
  const int32_t* pidx = m->prefill_state_indices_host != nullptr
                            ? m->prefill_state_indices_host
                            : idx + nd;
  const uint8_t* init = m->has_initial_state_host;
  const uint8_t* pinit = m->prefill_has_initial_state_host != nullptr
                             ? m->prefill_has_initial_state_host
                             : (init != nullptr ? init + nd : nullptr);
  if (qsl[0] != 0 || qsl[nreq] != nd_tok + np_tok)
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "non-spec GDN query offsets must span the non-spec tokens");
  for (int64_t i = 0; i < nreq; ++i)
    if (qsl[i + 1] <= qsl[i])
      return fail(GDN_ERR_INVALID_ARGUMENT,
                  "non-spec GDN query offsets must be strictly increasing");
  if (qsl[nd] != nd_tok)
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "non-spec GDN decode prefix does not match token count");
  for (int64_t i = 0; i < np; ++i) {
    if (pidx[i] != idx[nd + i])
      return fail(GDN_ERR_INVALID_ARGUMENT, "prefill state indices must match non-spec suffix");
    if (pidx[i] < 0)
      return fail(GDN_ERR_INVALID_ARGUMENT, "prefill GDN state index must be non-negative");
    if (pqsl[i] != qsl[nd + i] - nd_tok)
      return fail(GDN_ERR_INVALID_ARGUMENT,
                  "prefill query offsets must match rebased non-spec suffix");
    const uint8_t a = init != nullptr ? init[nd + i] : 1;
    const uint8_t b = pinit != nullptr ? pinit[i] : 1;
    if ((a != 0) != (b != 0))
      return fail(GDN_ERR_INVALID_ARGUMENT,
                  "prefill initial-state mask must match non-spec suffix");
  }
  if (pqsl[np] != np_tok)
    return fail(GDN_ERR_INVALID_ARGUMENT, "prefill query offsets must span prefill tokens");
  return succeed();
}

// AUTO: the tensor-core forms for bf16 with Dk = Dv = 128, else the recurrent
// one.  The fused form keeps one (sequence, value head) chain per SM and
// prepares its chunks inside it; with fewer chains than SMs the two-launch
// form, which prepares every chunk of every chain in parallel first, is the
// faster of the two.
int32_t gdn_prefill_resolve_algo(int64_t N, int64_t Hv, int64_t Dk, int64_t Dv, int32_t act_dtype,
                                 int32_t algo) {
  if (algo != GDN_PREFILL_AUTO) return algo;
  if (!gdn::fused_supported((int)Dk, (int)Dv, act_dtype == GDN_DTYPE_BF16))
    return GDN_PREFILL_RECURRENT;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 152;
  }
  return N * Hv >= sms ? GDN_PREFILL_FUSED : GDN_PREFILL_CHUNKED;
}

size_t gdn_prefill_workspace_bytes(int64_t T, int64_t N, int64_t Hv, int64_t Dk, int64_t Dv,
                                   int32_t act_dtype, int32_t algo) {
  if (T <= 0 || N <= 0 || Hv <= 0) return 0;
  const int32_t resolved = gdn_prefill_resolve_algo(N, Hv, Dk, Dv, act_dtype, algo);
  if (resolved == GDN_PREFILL_FUSED) return gdn::fused_workspace_bytes(N, Hv);
  if (resolved != GDN_PREFILL_CHUNKED) return 0;
  return gdn::chunked_workspace_bytes(T, N, Hv, Dk, Dv);
}

int gdn_prefill_varlen(const gdn_prefill_args* a, void* stream) {
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "args is NULL");
  if (int rc = check_recurrence(a->T, a->Hk, a->Hv, a->Dk, a->Dv, a->act_dtype, a->q, a->q_len,
                                a->k, a->k_len, a->v, a->v_len, a->g, a->g_len, a->beta,
                                a->beta_len, a->state, a->state_slots, a->state_len, a->out,
                                a->out_len))
    return rc;
  if (a->N <= 0)
    return fail(GDN_ERR_SHAPE, "gated_delta_rule_varlen shape must be positive, got batch=" +
                                   S(a->N) + " total_tokens=" + S(a->T));
  if (require_ptr(a->cu_seqlens, "cu_seqlens")) return GDN_ERR_INVALID_ARGUMENT;
  if (a->algo < GDN_PREFILL_AUTO || a->algo > GDN_PREFILL_FUSED)
    return fail(GDN_ERR_INVALID_ARGUMENT, "unknown prefill algo " + S(a->algo));
  {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::vector<int32_t> cu_buf, idx_buf;
    const int32_t *cuh = nullptr, *idxh = nullptr;
    if (int rc = host_view(a->cu_seqlens_host, a->cu_seqlens, a->N + 1, st, cu_buf, cuh))
      return rc;
    if (int rc = host_view(a->state_indices_host, a->state_indices, a->N, st, idx_buf, idxh))
      return rc;
    if (cuh != nullptr)
      if (int rc = check_cu_host(cuh, a->N, a->T, "gated_delta_rule_varlen")) return rc;
    if (idxh != nullptr)
      if (int rc = check_indices_host(idxh, a->N, a->state_slots)) return rc;
  }
  if (a->state_indices == nullptr && a->N > a->state_slots)
    return fail(GDN_ERR_SHAPE, "gated_delta_rule state has fewer slots than sequences");
  const int32_t algo = gdn_prefill_resolve_algo(a->N, a->Hv, a->Dk, a->Dv, a->act_dtype, a->algo);
  gdn::RecurLaunch p{};
  p.T = (int)a->T;
  p.N = (int)a->N;
  p.Hk = (int)a->Hk;
  p.Hv = (int)a->Hv;
  p.Dk = (int)a->Dk;
  p.Dv = (int)a->Dv;
  p.bf16 = a->act_dtype == GDN_DTYPE_BF16;
  p.norm = a->use_qk_l2norm != 0;
  p.scale = resolve_scale(a->scale, a->Dk);
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.g = a->g;
  p.beta = a->beta;
  p.pool = a->state;
  p.slots = a->state_slots;
  p.cu = a->cu_seqlens;
  p.sidx = a->state_indices;
  p.has_init = a->has_initial_state;
  p.out = a->out;
  if (int rc = check_out_norm(a->out_norm, a->T, a->Hv, a->Dv, a->act_dtype, p)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (algo == GDN_PREFILL_CHUNKED) {
    if (!gdn::chunked_supported((int)a->Dk, (int)a->Dv, p.bf16))
      return fail(GDN_ERR_UNSUPPORTED,
                  "the chunked prefill supports bf16 activations with Dk = Dv = 128");
    const size_t need = gdn::chunked_workspace_bytes(a->T, a->N, a->Hv, a->Dk, a->Dv);
    if (need > 0) {
      if (a->workspace == nullptr || a->workspace_bytes < need)
        return fail(GDN_ERR_INVALID_ARGUMENT, "gdn_prefill_varlen workspace needs " +
                                                  S((int64_t)need) + " bytes, got " +
                                                  S((int64_t)a->workspace_bytes));
      if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
    }
    p.status = gdn::status_word();
    if (p.status == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
    gdn::ChunkedLaunch c{p, a->workspace, a->workspace_bytes};
    if (int rc = launch_result(gdn::launch_chunked(c, st), "gdn_prefill_varlen(chunked)")) return rc;
    if (p.onorm_w == nullptr) return GDN_OK;
    return launch_result(launch_out_norm_pass(p, st), "gdn_prefill_varlen(output norm)");
  }
  if (algo == GDN_PREFILL_FUSED) {
    if (!gdn::fused_supported((int)a->Dk, (int)a->Dv, p.bf16))
      return fail(GDN_ERR_UNSUPPORTED,
                  "the fused chunked prefill supports bf16 activations with Dk = Dv = 128");
    // The workspace is optional here: with gdn_prefill_workspace_bytes() of it
    // the chains are spread over the SMs when they outnumber them.
    if (a->workspace != nullptr && (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
      return fail(GDN_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
    p.status = gdn::status_word();
    if (p.status == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
    if (int rc = launch_result(gdn::launch_fused(p, a->workspace, a->workspace_bytes, st),
                               "gdn_prefill_varlen(fused)"))
      return rc;
    if (p.onorm_w == nullptr) return GDN_OK;
    return launch_result(launch_out_norm_pass(p, st), "gdn_prefill_varlen(output norm)");
  }
  if (!gdn::recurrent_supported((int)a->Dk))
    return fail(GDN_ERR_UNSUPPORTED, "the recurrent prefill supports Dk in {16, 32, 64, 128, 256}");
  p.status = gdn::status_word();
  if (p.status == nullptr) return fail(GDN_ERR_CUDA, "device status word unavailable");
  if (int rc = launch_result(gdn::launch_recurrent(p, st), "gdn_prefill_varlen(recurrent)"))
    return rc;
  if (p.onorm_w == nullptr) return GDN_OK;
  return launch_result(launch_out_norm_pass(p, st), "gdn_prefill_varlen(output norm)");
}

}  // extern "C"
