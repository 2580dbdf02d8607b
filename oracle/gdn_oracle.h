/*
 * gdn_oracle.h -- plain CPU oracle for the gated-delta-rule (GDN) layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists to check the CUDA library
 * against a slow, obviously correct restatement of the method.  Only the test
 * suite, the smoke check and the CPU-baseline leg of the benchmark may load it.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * Sources (page title, then the function on it):
 *   [cpu.rs]       ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs
 *   [cpu_ops.cpp]  vllm.cpp, src/vt/cpu/cpu_ops.cpp
 *   [qwen3_5.cpp]  vllm.cpp, src/vllm/model_executor/models/qwen3_5.cpp
 *
 * Conventions
 *   - Every exported routine comes in an f32 and an f64 instantiation (suffix).
 *     All arithmetic happens in that type; callers widen bf16 inputs exactly.
 *   - Layouts: q,k [T,Hk,Dk]; v,out [T,Hv,Dv]; g,beta [T,Hv];
 *     state pool [slots,Hv,Dv,Dk]; conv-tail pool [slots,C_conv,K-1] oldest
 *     first; mixed_qkv [T, >=C_conv] with row stride x_stride (elements).
 *   - Return value: ORC_OK or an ORC_ERR_* code; msg (if non-NULL) receives the
 *     diagnostic text.
 *
 * Parity pins: every function here is pinned by tests that do not re-type its
 * formula (closed forms, invariants, library routines, brute force); see the
 * module docstrings of tests/test_oracle_*.py.
 */
#ifndef GDN_ORACLE_H_
#define GDN_ORACLE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ORC_OK = 0,
  ORC_ERR_SHAPE = 1,    /* non-positive dims, Hv % Hk != 0, short buffer */
  ORC_ERR_INVALID = 2,  /* bad cu_seqlens, bad state index */
};

/* ---- scalar gate functions, [cpu.rs] sigmoid / silu / softplus ---------- */
float orc_sigmoid_f32(float x);
float orc_silu_f32(float x);
float orc_softplus_f32(float x);
double orc_sigmoid_f64(double x);
double orc_silu_f64(double x);
double orc_softplus_f64(double x);

/* ---- validators ---------------------------------------------------------- */
/* [cpu.rs] validate_gated_delta_rule_shape; lengths are element counts. */
int orc_validate_gated_delta_rule_shape(int64_t query_len, int64_t key_len, int64_t value_len,
                                        int64_t g_len, int64_t beta_len,
                                        int64_t initial_state_len, int64_t out_len,
                                        int64_t final_state_len, int64_t tokens,
                                        int64_t key_heads, int64_t value_heads,
                                        int64_t key_dim, int64_t value_dim, char* msg,
                                        size_t msg_cap);
/* [cpu.rs] validate_linear_attention_prepare_shape. */
int orc_validate_linear_attention_prepare_shape(
    int64_t mixed_qkv_raw_len, int64_t conv_weight_len, int64_t a_raw_len, int64_t b_raw_len,
    int64_t a_log_len, int64_t dt_bias_len, int64_t query_len, int64_t key_len,
    int64_t value_len, int64_t g_len, int64_t beta_len, int64_t tokens, int64_t key_heads,
    int64_t value_heads, int64_t key_dim, int64_t value_dim, int64_t conv_kernel, char* msg,
    size_t msg_cap);
/* [cpu.rs] validate_linear_attention_decode_prepare_shape. */
int orc_validate_linear_attention_decode_prepare_shape(
    int64_t mixed_qkv_raw_len, int64_t conv_weight_len, int64_t conv_state_len,
    int64_t a_raw_len, int64_t b_raw_len, int64_t a_log_len, int64_t dt_bias_len,
    int64_t query_len, int64_t key_len, int64_t value_len, int64_t g_len, int64_t beta_len,
    int64_t next_conv_state_len, int64_t key_heads, int64_t value_heads, int64_t key_dim,
    int64_t value_dim, int64_t conv_kernel, char* msg, size_t msg_cap);
/* Test aid, f64: a first-order bound on how far each output of O2 can move
 * when the stored q, k, v move by at most dq, dk, dv (elementwise, same
 * shapes as q, k, v).  q and k are taken as stored (no in-loop norm); the
 * state pool is only read.  bound [T, Hv, Dv]; state_bound (optional,
 * [slots, Hv, Dv]) bounds every element of each row of each live sequence's
 * final state. */
int orc_gdn_deviation_bound_f64(const double* q, const double* k, const double* v,
                                const double* g, const double* beta, const double* dq,
                                const double* dk, const double* dv, const double* state_pool,
                                int64_t state_slots, const int32_t* state_indices,
                                const uint8_t* has_initial_state, const int32_t* cu_seqlens,
                                int64_t n_seqs, int64_t tokens, int64_t key_heads,
                                int64_t value_heads, int64_t key_dim, int64_t value_dim,
                                double scale, double* bound, double* state_bound,
                                int nthreads);
/* [cpu.rs] recurrent_gated_delta_rule_varlen_f32: cu_seqlens starts at 0, ends
 * at total_tokens, every range non-empty and increasing. */
int orc_validate_cu_seqlens(const int32_t* cu_seqlens, int64_t batch, int64_t total_tokens,
                            char* msg, size_t msg_cap);
/* [cpu.rs] linear_attention_prepare_varlen_f32: the same rules and messages
 * under the label "linear_attention_prepare_varlen". */
int orc_validate_prepare_cu_seqlens(const int32_t* cu_seqlens, int64_t batch,
                                    int64_t total_tokens, char* msg, size_t msg_cap);
/* [qwen3_5.cpp] ValidateGdnStateIndices: -1 is the only negative value, a live
 * slot is < state_slots, no duplicate live slot.  Both the O(n) seen-set pass
 * and (when force_full != 0) the O(n^2) pairwise re-check run. */
int orc_validate_state_indices(const int32_t* indices, int64_t n, int64_t state_slots,
                               int force_full, char* msg, size_t msg_cap);

/* ---- O1: prepare (conv1d + SiLU + split + gates + q/k L2 norm) ------------
 * [cpu.rs] linear_attention_prepare_varlen_f32 and
 * linear_attention_decode_prepare_batch_f32, with the conv tails read from and
 * written back to a slot pool chosen by state_indices (the [cpu_ops.cpp]
 * CausalConv1dUpdateKernel / GdnStateGatherKernel indexing):
 *   state_indices == NULL     -> slot = sequence number
 *   state_indices[s] == -1    -> padded sequence: outputs computed from a zero
 *                                tail, the pool row is neither read nor written
 *   has_initial_state == NULL -> every live sequence starts from its pool tail
 *   has_initial_state[s] == 0 -> zero tail; the new tail is still written
 * nthreads: 0 = hardware concurrency; results do not depend on it. */
#define ORC_PREPARE_PARAMS(R)                                                              \
  const R *mixed_qkv, int64_t x_stride, const R *conv_weight, R *conv_pool,                \
      int64_t conv_slots, const int32_t *state_indices, const uint8_t *has_initial_state, \
      const R *a_raw, int64_t a_stride, const R *b_raw, int64_t b_stride, const R *a_log,  \
      const R *dt_bias, const int32_t *cu_seqlens, int64_t n_seqs, int64_t tokens,         \
      int64_t key_heads, int64_t value_heads, int64_t key_dim, int64_t value_dim,          \
      int64_t conv_kernel, int apply_qk_l2norm, R *query, R *key, R *value, R *g, R *beta, \
      int nthreads
int orc_prepare_varlen_f32(ORC_PREPARE_PARAMS(float));
int orc_prepare_varlen_f64(ORC_PREPARE_PARAMS(double));

/* ---- O8: speculative prepare, [cpu_ops.cpp] CausalConv1dSpecUpdateKernel ----
 * O1 for the draft tokens of a speculative step.  conv_pool is
 * [conv_slots, C_conv, state_len], state_len = (K-1) + (max_q - 1); request i
 * uses row conv_indices[i] (negative: outputs from a zero window, no row
 * written).  With off = num_accepted[i] - 1 the conv window before the first
 * draft is row[off .. off+K-2]; the row becomes row[off+1 .. off+keep] ||
 * drafts, keep = state_len - len.  Split, gates and norm as O1.
 * ORC_ERR_SHAPE for K < 2; ORC_ERR_INVALID for bad cu_seqlens, a request
 * longer than max_q, num_accepted outside [1, max_q] or a slot >= conv_slots. */
int orc_spec_prepare_f32(const float* mixed_qkv, int64_t x_stride, const float* conv_weight,
                         float* conv_pool, int64_t conv_slots, int64_t state_len,
                         const int32_t* conv_indices, const int32_t* num_accepted,
                         const float* a_raw, int64_t a_stride, const float* b_raw,
                         int64_t b_stride, const float* A_log, const float* dt_bias,
                         const int32_t* cu_seqlens, int64_t n_reqs, int64_t tokens,
                         int64_t key_heads, int64_t value_heads, int64_t key_dim,
                         int64_t value_dim, int64_t conv_kernel, int apply_qk_l2norm,
                         float* query, float* key, float* value, float* g, float* beta,
                         int nthreads);
int orc_spec_prepare_f64(const double* mixed_qkv, int64_t x_stride, const double* conv_weight,
                         double* conv_pool, int64_t conv_slots, int64_t state_len,
                         const int32_t* conv_indices, const int32_t* num_accepted,
                         const double* a_raw, int64_t a_stride, const double* b_raw,
                         int64_t b_stride, const double* A_log, const double* dt_bias,
                         const int32_t* cu_seqlens, int64_t n_reqs, int64_t tokens,
                         int64_t key_heads, int64_t value_heads, int64_t key_dim,
                         int64_t value_dim, int64_t conv_kernel, int apply_qk_l2norm,
                         double* query, double* key, double* value, double* g, double* beta,
                         int nthreads);

/* ---- O2: sequential recurrence over varlen sequences ----------------------
 * [cpu.rs] recurrent_gated_delta_rule_varlen_f32 (loop order, q/k norm form,
 * k scaled by k_inv, q by q_inv*scale) on a state pool:
 *   state_indices[s] == -1    -> out rows of sequence s are zero, pool untouched
 *   has_initial_state[s] == 0 -> the recurrence starts from S = 0
 *   the final state of each live sequence is written to its pool slot.
 * items/n_items: optional list of work items (seq*Hv + head) to compute; the
 * out rows of other items are left untouched (NULL = every item). */
#define ORC_RECUR_PARAMS(R)                                                                 \
  const R *query, const R *key, const R *value, const R *g, const R *beta, R *state_pool,   \
      int64_t state_slots, const int32_t *state_indices, const uint8_t *has_initial_state,  \
      const int32_t *cu_seqlens, int64_t n_seqs, int64_t tokens, int64_t key_heads,         \
      int64_t value_heads, int64_t key_dim, int64_t value_dim, R scale, int use_qk_l2norm,  \
      const int32_t *items, int64_t n_items, R *out, int nthreads
int orc_gdn_varlen_f32(ORC_RECUR_PARAMS(float));
int orc_gdn_varlen_f64(ORC_RECUR_PARAMS(double));

/* ---- O7 speculative multi-token decode, [cpu_ops.cpp] GdnSpecDecodeKernel ----
 * Request i owns tokens [cu[i], cu[i+1]) (at most num_cols of them) and row i
 * of state_indices [n_reqs, num_cols].  Its state starts from slot
 * state_indices[i][num_accepted[i] - 1]; after token t the state is stored in
 * slot state_indices[i][t - cu[i]] (a negative slot skips the store).  A
 * negative initial slot zeroes the request's outputs.  q, k used as given;
 * g, beta [T, Hv].  ORC_ERR_INVALID for bad cu_seqlens, num_accepted outside
 * [1, num_cols], requests longer than num_cols, or slots >= state_slots. */
int orc_gdn_spec_decode_f32(const float* query, const float* key, const float* value,
                            const float* g, const float* beta, float* state_pool,
                            int64_t state_slots, const int32_t* cu_seqlens, int64_t n_reqs,
                            int64_t tokens, const int32_t* state_indices, int64_t num_cols,
                            const int32_t* num_accepted, int64_t key_heads, int64_t value_heads,
                            int64_t key_dim, int64_t value_dim, float scale, float* out,
                            int nthreads);
int orc_gdn_spec_decode_f64(const double* query, const double* key, const double* value,
                            const double* g, const double* beta, double* state_pool,
                            int64_t state_slots, const int32_t* cu_seqlens, int64_t n_reqs,
                            int64_t tokens, const int32_t* state_indices, int64_t num_cols,
                            const int32_t* num_accepted, int64_t key_heads, int64_t value_heads,
                            int64_t key_dim, int64_t value_dim, double scale, double* out,
                            int nthreads);

/* ---- O6 KDA: per-key-channel decay, [cpu_ops.cpp] KdaHeadTokenStep /
 * KdaGatedDeltaRuleKernel.  Same contract as orc_gdn_varlen except that g is
 * [T, Hv, Dk] (the log decay of each key channel) and use_qk_l2norm must be 0
 * (q and k are used as given; ORC_ERR_INVALID otherwise). */
int orc_kda_varlen_f32(ORC_RECUR_PARAMS(float));
int orc_kda_varlen_f64(ORC_RECUR_PARAMS(double));

/* ---- O3: decode, one token per row ----------------------------------------
 * [cpu_ops.cpp] GdnDecodeKernel semantics: row b uses pool slot
 * state_indices[b] (NULL -> b) in place; a negative index zeroes out row b and
 * leaves the pool untouched. */
#define ORC_DECODE_PARAMS(R)                                                              \
  const R *query, const R *key, const R *value, const R *g, const R *beta, R *state_pool, \
      int64_t state_slots, const int32_t *state_indices, int64_t batch, int64_t key_heads, \
      int64_t value_heads, int64_t key_dim, int64_t value_dim, R scale, int use_qk_l2norm, \
      R *out, int nthreads
int orc_gdn_decode_f32(ORC_DECODE_PARAMS(float));
int orc_gdn_decode_f64(ORC_DECODE_PARAMS(double));

/* ---- O4: chunked WY/UT form, f64 only (self-check of the algebra) ---------
 * Same contract as orc_gdn_varlen_f64; chunk = tokens per chunk (>= 1). */
int orc_gdn_chunked_f64(const double* query, const double* key, const double* value,
                        const double* g, const double* beta, double* state_pool,
                        int64_t state_slots, const int32_t* state_indices,
                        const uint8_t* has_initial_state, const int32_t* cu_seqlens,
                        int64_t n_seqs, int64_t tokens, int64_t key_heads, int64_t value_heads,
                        int64_t key_dim, int64_t value_dim, double scale, int use_qk_l2norm,
                        int64_t chunk, double* out);

/* ---- O9: chunked form of the KDA recurrence, f64 only (self-check) -------
 * Same contract as orc_kda_varlen_f64 (g [T, Hv, Dk], q and k used as
 * given); chunk = tokens per chunk (>= 1). */
int orc_kda_chunked_f64(const double* query, const double* key, const double* value,
                        const double* g, const double* beta, double* state_pool,
                        int64_t state_slots, const int32_t* state_indices,
                        const uint8_t* has_initial_state, const int32_t* cu_seqlens,
                        int64_t n_seqs, int64_t tokens, int64_t key_heads, int64_t value_heads,
                        int64_t key_dim, int64_t value_dim, double scale, int64_t chunk,
                        double* out);

/* ---- O5 gated RMSNorm of the recurrence output ----------------------------
 * [cpu.rs] gated_rms_norm_f32 / validate_gated_rms_norm_shape, with
 * [cpu_ops.cpp] RmsNormGatedKernel's sigmoid-gate option and strided gate.
 * core, out [tokens, heads, dim] contiguous; z [tokens, heads, dim] with token
 * rows z_stride elements apart (z_stride >= heads * dim); weight [dim].
 * out = core / sqrt(mean(core^2) + eps) * weight * act(z), act = silu, or the
 * sigmoid when sigmoid_gate != 0; one row per (token, head). */
int orc_validate_gated_rms_norm_shape(int64_t core_len, int64_t z_len, int64_t weight_len,
                                      int64_t out_len, int64_t tokens, int64_t heads,
                                      int64_t dim, char* msg, size_t cap);
int orc_gated_rmsnorm_f32(const float* core, const float* z, int64_t z_stride,
                          const float* weight, float* out, int64_t tokens, int64_t heads,
                          int64_t dim, float eps, int sigmoid_gate, int nthreads);
int orc_gated_rmsnorm_f64(const double* core, const double* z, int64_t z_stride,
                          const double* weight, double* out, int64_t tokens, int64_t heads,
                          int64_t dim, double eps, int sigmoid_gate, int nthreads);

#ifdef __cplusplus
}
#endif

#endif /* GDN_ORACLE_H_ */
