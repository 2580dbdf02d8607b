/*
 * gdn.h -- C ABI of libgdn, the gated-delta-rule (GDN) linear-attention layer
 * on GB300 (sm_103a).
 *
 * The layer has two parts, each on a caller-owned CUDA stream:
 *   gdn_prepare         causal depthwise conv1d + SiLU + q/k/v split + q/k L2
 *                       norm + gates g, beta, with the conv tail carried in a
 *                       slot pool
 *   gdn_decode          the state recurrence for one token per sequence
 *   gdn_prefill_varlen  the state recurrence over packed variable-length
 *                       sequences (chunked, tensor-core form)
 * and these variants of them:
 *   gdn_packed_decode   prepare + decode of one token per row in one launch,
 *                       from the packed projections
 *   gdn_prefill_varlen_noalloc   gdn_prefill_varlen on a scratch array inside
 *                       the library's device image
 *   gdn_spec_prepare,   the prepare and the recurrence of a speculative
 *   gdn_spec_decode     multi-token decode step (per-draft state snapshots)
 *   gdn_kda_varlen      the recurrence with one decay per key channel (KDA)
 *   gdn_gated_rmsnorm   the gated RMSNorm applied to the recurrence output
 * and a host-only check of a mixed step's metadata:
 *   gdn_validate_mixed  decode rows first, prefill cu_seqlens rebased
 *
 * Sources (page title, then the function that defines the operation):
 *   [cpu.rs]       ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs
 *   [cpu_ops.cpp]  vllm.cpp, src/vt/cpu/cpu_ops.cpp
 *   [qwen3_5.cpp]  vllm.cpp, src/vllm/model_executor/models/qwen3_5.cpp
 *
 * General rules for every call
 *   - Every pointer is a DEVICE pointer unless its name ends in _host.  The
 *     caller owns every buffer; the library allocates nothing on any call.
 *   - Lengths (*_len) are element counts of the buffers as allocated; a call
 *     fails with GDN_ERR_SHAPE when a buffer is shorter than the shape needs,
 *     with the same message text as [cpu.rs] validate_* ("... {label} length
 *     {actual} < expected {expected}").
 *   - Host-side validation is synchronous; on any error nothing is launched
 *     and no buffer is touched.  Work is asynchronous on `stream` (a
 *     cudaStream_t passed as void*; NULL = the legacy default stream).
 *   - No C++ exception crosses this boundary.  gdn_last_error_message()
 *     returns the calling thread's last diagnostic.
 *   - Errors that only the device can see (a state index outside the pool or a
 *     malformed cu_seqlens when no host mirror was passed) are recorded in a
 *     per-device status word and the offending sequence is skipped;
 *     gdn_read_device_status() returns and clears it.
 *   - GDN_DEBUG_CHECKS=1 in the environment (read once per process): a call
 *     given cu_seqlens, state_indices or num_accepted in device memory only
 *     copies them to the host on its stream, synchronises it, and applies the
 *     host-mirror checks before launching ([qwen3_5.cpp] the fail-closed
 *     validators' optional exhaustive re-check).  Not for use while the
 *     stream is being captured into a graph.
 *   - Layouts (row-major, innermost last):
 *       mixed_qkv [T, >=C_conv], C_conv = 2*Hk*Dk + Hv*Dv, row stride in elements
 *       q, k      [T, Hk, Dk]          v, out [T, Hv, Dv]
 *       g, beta   [T, Hv] f32          a_raw, b_raw [T, >=Hv] (row stride)
 *       state     [slots, Hv, Dv, Dk] f32, the SSM state of one sequence per slot
 *       conv_state[slots, C_conv, K-1] f32, the last K-1 raw inputs, oldest first
 *     Value head h reads key head h / (Hv/Hk)  ([cpu_ops.cpp] GdnTokenStep).
 *   - Alignment: every activation pointer and row stride must give 16-byte
 *     aligned rows (GDN_ERR_INVALID_ARGUMENT otherwise).
 *   - Index rules ([cpu_ops.cpp] GdnDecodeKernel, CausalConv1dUpdateKernel;
 *     [qwen3_5.cpp] ValidateGdnStateIndices):
 *       state_indices == NULL      sequence i uses slot i
 *       state_indices[i] == -1     padding: its outputs are zero (recurrence)
 *                                  and its pool rows are neither read nor written
 *       any other negative, a slot >= slots, or a duplicate live slot is an
 *       error; duplicates are only detected when the _host mirror is passed.
 *       has_initial_state[i] == 0  start from a zero state / zero conv tail; the
 *                                  final state is still written to the slot.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_SHAPE = 1,            /* non-positive dims, Hv % Hk != 0, short buffer */
  GDN_ERR_INVALID_ARGUMENT = 2, /* bad cu_seqlens, bad index, NULL or misaligned pointer */
  GDN_ERR_DTYPE = 3,            /* act_dtype not a gdn_dtype */
  GDN_ERR_UNSUPPORTED = 4,      /* valid, but outside the dims the kernels are built for */
  GDN_ERR_CUDA = 5,             /* a CUDA runtime call failed */
  GDN_ERR_TIMEOUT = 6,          /* a bounded device-side wait ran out */
  GDN_ERR_DEVICE_CHECK = 7      /* a kernel saw a bad index or cu_seqlens */
} gdn_status;

typedef enum gdn_dtype {
  GDN_DTYPE_F32 = 0,
  GDN_DTYPE_BF16 = 1
} gdn_dtype;

/* Which recurrence kernel gdn_prefill_varlen runs. */
typedef enum gdn_prefill_algo {
  GDN_PREFILL_AUTO = 0,      /* a chunked form when supported (bf16, Dk = Dv = 128), else
                                recurrent: see gdn_prefill_resolve_algo */
  GDN_PREFILL_CHUNKED = 1,   /* chunk-64 WY/UT form on tcgen05 tensor cores, two kernels (every
                                chunk's preparation, then a scan; with few chains in pieces of
                                chunk indices chained by programmatic dependent launch) that
                                hand each chunk over through a caller workspace */
  GDN_PREFILL_RECURRENT = 2, /* token-sequential recurrence on CUDA cores */
  GDN_PREFILL_FUSED = 3      /* the chunk-64 form in one launch, a CTA preparing the next
                                chunk while it carries the state: one CTA per (sequence,
                                value head), or, given the optional workspace and more
                                chains than SMs (unless they nearly fill whole waves of
                                one CTA per SM), one CTA per SM over even ranges of the
                                chains' chunks (a short kernel computes the ranges first) */
} gdn_prefill_algo;

/* ---------------------------------------------------------------------------
 * gdn_prepare -- [cpu.rs] linear_attention_prepare_varlen_f32 and
 * linear_attention_decode_prepare_batch_f32; [cpu_ops.cpp]
 * CausalConv1dFwdKernel, CausalConv1dUpdateKernel, GdnPostConvKernel.
 *
 * For each sequence s (tokens cu_seqlens[s] .. cu_seqlens[s+1]-1) and channel c:
 *   y[t,c] = silu( sum_{j<K} conv_weight[c,j] * x~[t - (K-1) + j] )
 * where x~ is the sequence's raw input preceded by its conv tail (zero when
 * has_initial_state[s] == 0).  q = y[:, 0:HkDk], k = y[:, HkDk:2HkDk],
 * v = y[:, 2HkDk:]; when apply_qk_l2norm, q and k are scaled per (token, key
 * head) by 1/sqrt(sum of squares + 1e-6).  Gates per (token, value head):
 *   g = -exp(A_log[h]) * softplus(a_raw + dt_bias[h]),  beta = sigmoid(b_raw)
 * with softplus(x) = x for x > 20.  The conv tail row of the sequence's slot is
 * replaced by the last K-1 raw inputs of tail || x.  A decode batch is N == T
 * with cu_seqlens = 0,1,...,T.  q,k,v are stored in act_dtype (bf16 rounds to
 * nearest even); g, beta in f32.
 * Supported: K in [2, 8]; Dk a power of two in [8, 256] (bf16) or [4, 128]
 * (f32); Dv a multiple of 8 (bf16) or 4 (f32).
 * ------------------------------------------------------------------------- */
typedef struct gdn_prepare_args {
  int64_t T, N;             /* tokens, sequences */
  int64_t Hk, Hv, Dk, Dv;   /* key heads, value heads, key dim, value dim */
  int64_t K;                /* conv width (conv_kernel) */
  int32_t act_dtype;        /* gdn_dtype of mixed_qkv, a_raw, b_raw, q, k, v */
  int32_t apply_qk_l2norm;  /* 1: L2-normalise q and k rows */
  const void* mixed_qkv;    /* [T, mixed_qkv_stride] */
  int64_t mixed_qkv_stride; /* elements per row, >= C_conv; 0 = C_conv */
  int64_t mixed_qkv_len;
  const float* conv_weight; /* [C_conv, K] */
  int64_t conv_weight_len;
  const void* a_raw;        /* [T, a_raw_stride] */
  int64_t a_raw_stride;     /* 0 = Hv */
  int64_t a_raw_len;
  const void* b_raw;        /* [T, b_raw_stride] */
  int64_t b_raw_stride;     /* 0 = Hv */
  int64_t b_raw_len;
  const float* A_log;       /* [Hv] */
  int64_t A_log_len;
  const float* dt_bias;     /* [Hv] */
  int64_t dt_bias_len;
  const int32_t* cu_seqlens;        /* [N+1] */
  const int32_t* state_indices;     /* [N] conv pool slot per sequence, or NULL */
  const uint8_t* has_initial_state; /* [N] or NULL (= all 1) */
  const int32_t* cu_seqlens_host;   /* optional host copy: full validation */
  const int32_t* state_indices_host;/* optional host copy: full validation */
  float* conv_state;        /* [conv_state_slots, C_conv, K-1], updated in place */
  int64_t conv_state_slots;
  int64_t conv_state_len;
  void* q;                  /* [T, Hk, Dk] */
  int64_t q_len;
  void* k;                  /* [T, Hk, Dk] */
  int64_t k_len;
  void* v;                  /* [T, Hv, Dv] */
  int64_t v_len;
  float* g;                 /* [T, Hv] */
  int64_t g_len;
  float* beta;              /* [T, Hv] */
  int64_t beta_len;
} gdn_prepare_args;

int gdn_prepare(const gdn_prepare_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * gdn_out_norm -- an optional gated RMSNorm of the recurrence output, applied
 * where gdn_decode / gdn_prefill_varlen store it: [cpu.rs] gated_rms_norm_f32,
 * [cpu_ops.cpp] RmsNormGatedKernel.  Per (token, value head) row of Dv values
 *   out = core / sqrt(mean_d(core^2) + eps) * weight[d] * act(z[d])
 * where core is the recurrence output rounded to act_dtype (what the unfused
 * pipeline stores and the norm reads back) and act = silu (sigmoid_gate = 0)
 * or sigmoid.  z: token rows of at least Hv * Dv values in act_dtype,
 * z_token_stride elements apart (16-byte aligned rows); weight: [Dv] in
 * act_dtype.  By default the call runs the norm as a second kernel over the
 * output in place (on GB300 that is faster than folding it into the
 * recurrence kernels, whose tails then wait on a row-wide reduction).  With
 * in_kernel = 1 gdn_decode applies it inside the decode kernel when one CTA
 * can hold the whole row (Dv <= 256 at Dk = 64 or 128, Dv <= 128 at Dk = 256,
 * Dv <= 512 at Dk <= 32); the prefill always uses the second kernel.  Same
 * rules as gdn_gated_rmsnorm (lengths, alignment, Dv <= 1024 for bf16).
 * ------------------------------------------------------------------------- */
typedef struct gdn_out_norm {
  const void* z;           /* [tokens, z_token_stride] act_dtype */
  int64_t z_len;
  int64_t z_token_stride;  /* elements between token rows of z (>= Hv * Dv) */
  const void* weight;      /* [Dv] act_dtype */
  int64_t weight_len;
  float eps;
  int32_t sigmoid_gate;    /* 1: sigmoid gate instead of silu */
  int32_t in_kernel;       /* 1: inside the decode kernel where it fits (see above) */
} gdn_out_norm;

/* ---------------------------------------------------------------------------
 * gdn_decode -- [cpu_ops.cpp] GdnDecodeKernel / GdnHeadTokenStep;
 * [cpu.rs] recurrent_gated_delta_rule_batch_f32.
 *
 * Row b is one token of one sequence whose state S = state[state_indices[b],
 * h] ([Dv, Dk]) is updated in place, per value head h:
 *   S *= exp(g);  u = beta * (v - S k);  S += u k^T;  out = S (scale * q)
 * k is not scaled.  scale < 0 selects 1/sqrt(Dk).  When use_qk_l2norm, q and
 * k are first L2-normalised in f32 (eps 1e-6 inside the sqrt).
 * Supported: Dk in {16, 32, 64, 128, 256}; any Dv >= 1.
 * ------------------------------------------------------------------------- */
typedef struct gdn_decode_args {
  int64_t B;                /* rows (sequences), one token each */
  int64_t Hk, Hv, Dk, Dv;
  int32_t act_dtype;        /* gdn_dtype of q, k, v, out */
  int32_t use_qk_l2norm;
  float scale;              /* < 0: 1/sqrt(Dk) */
  const void* q;            /* [B, Hk, Dk] */
  int64_t q_len;
  const void* k;            /* [B, Hk, Dk] */
  int64_t k_len;
  const void* v;            /* [B, Hv, Dv] */
  int64_t v_len;
  const float* g;           /* [B, Hv] */
  int64_t g_len;
  const float* beta;        /* [B, Hv] */
  int64_t beta_len;
  float* state;             /* [state_slots, Hv, Dv, Dk], updated in place */
  int64_t state_slots;
  int64_t state_len;
  const int32_t* state_indices;      /* [B] or NULL (slot = b) */
  const int32_t* state_indices_host; /* optional host copy: full validation */
  void* out;                /* [B, Hv, Dv] */
  int64_t out_len;
  const gdn_out_norm* out_norm;  /* NULL, or the gated RMSNorm applied to out */
} gdn_decode_args;

int gdn_decode(const gdn_decode_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * gdn_prefill_varlen -- [cpu.rs] recurrent_gated_delta_rule_varlen_f32;
 * [cpu_ops.cpp] GdnPrefillKernel.
 *
 * The recurrence of gdn_decode over every token of every sequence in order,
 * starting from the sequence's slot (or zero when has_initial_state[s] == 0),
 * writing out[t] for every token and the final state back to the slot.
 * cu_seqlens must start at 0, end at T, and every range must be non-empty
 * ([cpu.rs] recurrent_gated_delta_rule_varlen_f32).
 * The chunked algorithm splits each sequence into chunks of 64 tokens (the
 * last may be partial; chunks never cross sequences) and needs
 * gdn_prefill_workspace_bytes() bytes of 256-byte aligned device scratch in
 * `workspace`; the fused algorithm takes the same (a few KB) optionally and
 * runs one CTA per chain without it; the recurrent algorithm needs none.
 * ------------------------------------------------------------------------- */
typedef struct gdn_prefill_args {
  int64_t T, N;
  int64_t Hk, Hv, Dk, Dv;
  int32_t act_dtype;        /* gdn_dtype of q, k, v, out */
  int32_t use_qk_l2norm;
  float scale;              /* < 0: 1/sqrt(Dk) */
  int32_t algo;             /* gdn_prefill_algo */
  const void* q;            /* [T, Hk, Dk] */
  int64_t q_len;
  const void* k;
  int64_t k_len;
  const void* v;            /* [T, Hv, Dv] */
  int64_t v_len;
  const float* g;           /* [T, Hv] */
  int64_t g_len;
  const float* beta;
  int64_t beta_len;
  float* state;             /* [state_slots, Hv, Dv, Dk], updated in place */
  int64_t state_slots;
  int64_t state_len;
  const int32_t* cu_seqlens;        /* [N+1] */
  const int32_t* state_indices;     /* [N] or NULL */
  const uint8_t* has_initial_state; /* [N] or NULL (= all 1) */
  const int32_t* cu_seqlens_host;   /* optional host copies: full validation */
  const int32_t* state_indices_host;
  void* out;                /* [T, Hv, Dv] */
  int64_t out_len;
  void* workspace;          /* device scratch, see gdn_prefill_workspace_bytes */
  size_t workspace_bytes;
  const gdn_out_norm* out_norm;  /* NULL, or the gated RMSNorm applied to out */
} gdn_prefill_args;

int gdn_prefill_varlen(const gdn_prefill_args* args, void* stream);

/* gdn_prefill_varlen for callers that cannot allocate device memory (the
 * pages have no counterpart: this is a deployment convenience).  Some callers
 * cannot supply the chunked prefill's scratch buffer: a plug-in inside a host
 * runtime that owns all device memory and gives plug-ins no allocator, or a
 * serving loop that must never call cudaMalloc (it can synchronise the device
 * and can fail under memory pressure).  This call takes the same arguments
 * except that workspace / workspace_bytes are ignored: it uses a fixed 64 MiB
 * scratch array that is part of the library's device image (as the chunked
 * form's workspace, or as the fused form's optional one), and calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   - Limit: sizes whose gdn_prefill_workspace_bytes() exceeds 64 MiB
 *     (67108864 bytes) are rejected with GDN_ERR_INVALID_ARGUMENT before
 *     anything is launched; sizes that need no scratch run as usual.
 *   - Every GPU that loads the array's module holds the 64 MiB until process
 *     exit.  Under CUDA's default lazy module loading that memory is committed
 *     by the first call on each device, which is therefore the set-up step
 *     that can fail (e.g. when the device is out of memory): it returns
 *     GDN_ERR_CUDA with the CUDA error in gdn_last_error_message().
 *   - That first call on each device (with that device current) also looks up
 *     the array's device address once; make it before any stream capture.
 *   - All calls share the one array, and it keeps the last call's contents
 *     (nothing in it needs to start at zero): calls whose GPU work overlaps
 *     (on different streams or from different host threads) race on it. */
int gdn_prefill_varlen_noalloc(const gdn_prefill_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * gdn_packed_decode -- [cpu_ops.cpp] GdnPackedDecodeKernel with the conv
 * update of [cpu_ops.cpp] CausalConv1dUpdateKernel folded in: a decode step in
 * one launch from the packed projections.  The packed layouts of [cpu.rs]
 * linear_attention_prepare_varlen_packed_qkvz_ba_f32 are described with row
 * strides: mixed_qkv rows may carry z after the q, k, v channels
 * (mixed_qkv_stride = C_conv + Hv*Dv), and a merged gate row of b then a
 * gives b_raw = ba, a_raw = ba + Hv, both with stride 2*Hv.
 *
 * For each row b with slot s = state_indices[b] (the conv pool and the state
 * pool share the slot, as their slot counts must match), per conv channel c:
 *   y[c] = silu( sum_{j<K-1} conv_state[s,c,j] w[c,j] + x[b,c] w[c,K-1] )
 * and conv_state[s,c,:] becomes (conv_state[s,c,1:], x[b,c]).  q, k, v split
 * y as gdn_prepare does; q and k are L2-normalised (apply_qk_l2norm) in f32;
 * per value head g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b);
 * then the gated delta rule of gdn_decode on state[s] and out = S (scale q).
 * No intermediate is rounded to act_dtype: only out is stored in it, so the
 * result equals gdn_prepare followed by gdn_decode up to the bf16 rounding of
 * q, k, v that those two calls store.  state_indices[b] = -1 marks a padding
 * row (zero outputs, neither pool touched): a fixed-size batch padded this
 * way can be captured once in a CUDA graph and replayed with new metadata.
 *   - Layout: out [B, Hv, Dv] act_dtype; conv_state [state_slots, C_conv,
 *     K-1] f32; state [state_slots, Hv, Dv, Dk] f32 (16-byte aligned);
 *     conv_weight [C_conv, K] f32; A_log, dt_bias [Hv] f32.
 *   - Errors: GDN_ERR_SHAPE for non-positive sizes, Hv % Hk != 0, short
 *     buffers or strides; GDN_ERR_INVALID_ARGUMENT for NULL pointers, a
 *     misaligned state or failed host-mirror index checks (-1 the only
 *     negative, live slots distinct and in range); GDN_ERR_UNSUPPORTED
 *     outside Dk in {64, 128}, Dv <= 128, K in [2, 4].  Without the host
 *     mirror a bad slot raises the device status word and the row is padded.
 *   - One CTA of 256 threads per (row, key head): it owns the conv channels
 *     of its key head and of that head's value heads.
 * ------------------------------------------------------------------------- */
typedef struct gdn_packed_decode_args {
  int64_t B, Hk, Hv, Dk, Dv, K;  /* rows, heads, dims, conv width */
  int32_t act_dtype;             /* gdn_dtype of mixed_qkv, a_raw, b_raw, out */
  int32_t apply_qk_l2norm;
  float scale;                   /* < 0: 1/sqrt(Dk) */
  const void* mixed_qkv;         /* [B, mixed_qkv_stride] raw (pre-conv) rows */
  int64_t mixed_qkv_stride;      /* 0 = C_conv */
  int64_t mixed_qkv_len;
  const float* conv_weight;      /* [C_conv, K] */
  int64_t conv_weight_len;
  const void* a_raw;             /* [B, a_raw_stride] */
  int64_t a_raw_stride;          /* 0 = Hv */
  int64_t a_raw_len;
  const void* b_raw;             /* [B, b_raw_stride] */
  int64_t b_raw_stride;          /* 0 = Hv */
  int64_t b_raw_len;
  const float* A_log;            /* [Hv] */
  int64_t A_log_len;
  const float* dt_bias;          /* [Hv] */
  int64_t dt_bias_len;
  const int32_t* state_indices;  /* [B], device, required */
  const int32_t* state_indices_host;  /* optional host mirror */
  float* conv_state;             /* [state_slots, C_conv, K-1], updated in place */
  int64_t conv_state_len;
  float* state;                  /* [state_slots, Hv, Dv, Dk], updated in place */
  int64_t state_slots;
  int64_t state_len;
  void* out;                     /* [B, Hv, Dv] */
  int64_t out_len;
} gdn_packed_decode_args;

int gdn_packed_decode(const gdn_packed_decode_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * gdn_kda_varlen -- [cpu_ops.cpp] KdaHeadTokenStep / KdaGatedDeltaRuleKernel:
 * the gated delta rule with one log decay per KEY CHANNEL (KDA).
 *
 * As gdn_prefill_varlen's recurrence, token by token per (sequence, value head),
 * except that g is [T, Hv, Dk] and column d of S decays by exp(g[t, h, d]):
 *   S[:, d] *= exp(g[t,h,d]);  u = beta (v - S k);  S += u k^T;  out = S (scale q)
 * q and k are used as given (no L2 norm).  Decode is the case of N one-token
 * sequences.  State pool, state_indices (-1 = padding), has_initial_state,
 * cu_seqlens and their host mirrors as in gdn_prefill_varlen; g 16-byte
 * aligned.
 * algo (gdn_prefill_algo; see gdn_kda_resolve_algo): RECURRENT runs on CUDA
 * cores, a CTA per (sequence, head, row slice); CHUNKED is the chunk-64 form
 * on tcgen05 tensor cores (bf16, Dk = Dv = 128), two kernels (as
 * GDN_PREFILL_CHUNKED, in pieces when the chains are few) that hand each chunk
 * over through a caller workspace of gdn_kda_workspace_bytes() bytes (256-byte
 * aligned); FUSED is not offered for KDA.
 * Supported: Dk in {16, 32, 64, 128, 256}; any Dv >= 1 (recurrent).
 * Errors as gdn_prefill_varlen (g: "kda_gated_delta_rule g length N <
 * expected T*Hv*Dk").
 * ------------------------------------------------------------------------- */
typedef struct gdn_kda_args {
  int64_t T, N, Hk, Hv, Dk, Dv;
  int32_t act_dtype;        /* gdn_dtype of q, k, v, out */
  float scale;              /* < 0: 1/sqrt(Dk) */
  const void* q;            /* [T, Hk, Dk] */
  int64_t q_len;
  const void* k;            /* [T, Hk, Dk] */
  int64_t k_len;
  const void* v;            /* [T, Hv, Dv] */
  int64_t v_len;
  const float* g;           /* [T, Hv, Dk] log decay per key channel */
  int64_t g_len;
  const float* beta;        /* [T, Hv] */
  int64_t beta_len;
  float* state;             /* [state_slots, Hv, Dv, Dk], updated in place */
  int64_t state_slots;
  int64_t state_len;
  const int32_t* cu_seqlens;         /* [N + 1], device */
  const int32_t* state_indices;      /* [N] or NULL */
  const uint8_t* has_initial_state;  /* [N] or NULL (all 1) */
  const int32_t* cu_seqlens_host;    /* optional host mirrors: full validation */
  const int32_t* state_indices_host;
  void* out;                /* [T, Hv, Dv] */
  int64_t out_len;
  int32_t algo;             /* gdn_prefill_algo: AUTO, CHUNKED or RECURRENT */
  void* workspace;          /* device scratch, see gdn_kda_workspace_bytes */
  size_t workspace_bytes;
} gdn_kda_args;

int gdn_kda_varlen(const gdn_kda_args* args, void* stream);

/* The algorithm gdn_kda_varlen runs for `algo`: AUTO picks CHUNKED when some
 * sequence holds more than one token (T > N) and the chunked form supports the
 * shape (bf16, Dk = Dv = 128), else RECURRENT.  Other values are returned as
 * given. */
int32_t gdn_kda_resolve_algo(int64_t T, int64_t N, int64_t Dk, int64_t Dv, int32_t act_dtype,
                             int32_t algo);

/* Workspace bytes gdn_kda_varlen needs for these sizes and `algo` (0 when the
 * resolved algorithm is the recurrent one): one 113 KB blob per (chunk, value
 * head), for at most T / 64 + N chunks. */
size_t gdn_kda_workspace_bytes(int64_t T, int64_t N, int64_t Hv, int64_t Dk, int64_t Dv,
                               int32_t act_dtype, int32_t algo);

/* ---------------------------------------------------------------------------
 * gdn_spec_prepare -- [cpu_ops.cpp] CausalConv1dSpecUpdateKernel followed by
 * the split, norm and gates of gdn_prepare: the prepare step of a
 * speculative decode (the input of gdn_spec_decode).
 *
 * base holds gdn_prepare's arguments with these changes: N is the number of
 * requests, request i owning the draft tokens cu_seqlens[i] ..
 * cu_seqlens[i+1]-1 (0 to max_q of them); state_indices [N] names each
 * request's conv row (required; negative = none); has_initial_state must be
 * NULL; conv_state is [conv_state_slots, C_conv, conv_state_width] with
 * conv_state_width = (K-1) + (max_q - 1), the widened row of raw inputs.
 * With off = num_accepted[i] - 1, the conv window before the first draft is
 * row[off .. off+K-2], then the drafts themselves:
 *   y[t,c] = silu( sum_{j<K} w[c,j] * (row[off..off+K-2] || x)[t' + j] )
 * for the request's t'-th draft t.  The row then becomes
 * row[off+1 .. off+keep] || drafts (entries past the row read 0),
 * keep = conv_state_width - drafts: shifted by one tap per step, so that the
 * next step's offset picks the window ending at its last accepted token.
 * A negative row: outputs from a zero window, no row written.  An empty
 * request: nothing.
 *   - Host mirrors (base.cu_seqlens_host, base.state_indices_host,
 *     num_accepted_host; optional) validate fully: offsets span 0..T, at most
 *     max_q tokens per request, num_accepted in [1, max_q], rows below
 *     conv_state_slots and distinct.  Without them the kernel raises the
 *     device status word (gdn_read_device_status: GDN_ERR_DEVICE_CHECK) and
 *     skips the request for bad offsets, or computes from a zero window and
 *     writes no row for a bad row index or num_accepted.
 *   - Errors as gdn_prepare, plus GDN_ERR_SHAPE for conv_state_width < K-1
 *     or T > N * max_q, GDN_ERR_INVALID_ARGUMENT for a NULL state_indices or
 *     num_accepted or a non-NULL has_initial_state, and GDN_ERR_UNSUPPORTED
 *     for conv_state_width > 16.
 *   - One CTA per (request, 1024/512-channel block) stages its conv rows in
 *     shared memory, transposed so that each thread reads its channels'
 *     entries as 16-byte vectors.
 * ------------------------------------------------------------------------- */
typedef struct gdn_spec_prepare_args {
  gdn_prepare_args base;
  int64_t conv_state_width;          /* (K-1) + (max_q - 1) */
  const int32_t* num_accepted;       /* [N], device */
  const int32_t* num_accepted_host;  /* optional host mirror */
} gdn_spec_prepare_args;

int gdn_spec_prepare(const gdn_spec_prepare_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * gdn_spec_decode -- [cpu_ops.cpp] GdnSpecDecodeKernel with the metadata rules
 * of [qwen3_5.cpp] (spec metadata validation): speculative multi-token decode.
 *
 * Request i owns the draft tokens [cu_seqlens[i], cu_seqlens[i+1]) (0 to
 * num_cols of them) and row i of state_indices [n_reqs, num_cols].  Its state
 * starts from slot state_indices[i][num_accepted[i] - 1] (the snapshot after
 * the previous step's last accepted token); each token runs the gated delta
 * rule of gdn_prefill_varlen with q, k used as given (no L2 norm):
 *   S *= exp(g);  u = beta (v - S k);  S += u k^T;  out = S (scale q)
 * and the state after token t is stored in slot state_indices[i][t - cu[i]].
 * A negative slot skips that store; a negative initial slot zeroes the
 * request's outputs and writes no slot.  The initial slot is not written
 * back (unless a column names it), so a later step can resume from any
 * snapshot: the snapshot in column j equals the state after running only the
 * first j + 1 draft tokens.
 *   - Layout: q, k [T, Hk, Dk], v [T, Hv, Dv], out [T, Hv, Dv] (act_dtype),
 *     g, beta [T, Hv] f32, state [state_slots, Hv, Dv, Dk] f32, all row-major
 *     and device-resident; cu_seqlens [n_reqs + 1], state_indices
 *     [n_reqs, num_cols], num_accepted [n_reqs] int32 on the device.
 *   - Precondition: no live slot appears in two requests' rows (the optional
 *     host mirrors check it).  Within one row, repeats are allowed.
 *   - Host mirrors (optional, any subset) validate fully before launch:
 *     offsets span 0..T, request lengths in [0, num_cols], num_accepted in
 *     [1, num_cols], slots < state_slots, no slot shared by two requests.
 *     Without them the kernel raises the device status word
 *     (gdn_read_device_status: GDN_ERR_DEVICE_CHECK) and skips the request
 *     (bad offsets), zeroes its outputs (bad num_accepted or initial slot)
 *     or skips the store (bad snapshot slot).
 *   - Errors: GDN_ERR_SHAPE for non-positive sizes, Hv % Hk != 0, short
 *     buffers or T > n_reqs * num_cols; GDN_ERR_INVALID_ARGUMENT for NULL or
 *     misaligned pointers and failed mirror checks ("num_accepted_tokens must
 *     be in [1, num_spec + 1]", "spec GDN state slot out of range", ...);
 *     GDN_ERR_UNSUPPORTED for Dk outside {16, 32, 64, 128, 256}.
 *   - Runs on CUDA cores, one CTA per (request, value head, row slice) holding
 *     its rows in registers across the request's tokens.
 * ------------------------------------------------------------------------- */
typedef struct gdn_spec_decode_args {
  int64_t T, n_reqs, num_cols, Hk, Hv, Dk, Dv;
  int32_t act_dtype;        /* gdn_dtype of q, k, v, out */
  float scale;              /* < 0: 1/sqrt(Dk) */
  const void* q;            /* [T, Hk, Dk] */
  int64_t q_len;
  const void* k;            /* [T, Hk, Dk] */
  int64_t k_len;
  const void* v;            /* [T, Hv, Dv] */
  int64_t v_len;
  const float* g;           /* [T, Hv] */
  int64_t g_len;
  const float* beta;        /* [T, Hv] */
  int64_t beta_len;
  float* state;             /* [state_slots, Hv, Dv, Dk], snapshots written in place */
  int64_t state_slots;
  int64_t state_len;
  const int32_t* cu_seqlens;        /* [n_reqs + 1], device */
  const int32_t* state_indices;     /* [n_reqs, num_cols], device */
  const int32_t* num_accepted;      /* [n_reqs], device */
  const int32_t* cu_seqlens_host;   /* optional host mirrors */
  const int32_t* state_indices_host;
  const int32_t* num_accepted_host;
  void* out;                /* [T, Hv, Dv] */
  int64_t out_len;
} gdn_spec_decode_args;

int gdn_spec_decode(const gdn_spec_decode_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * gdn_gated_rmsnorm -- [cpu.rs] gated_rms_norm_f32 and
 * validate_gated_rms_norm_shape; [cpu_ops.cpp] RmsNormGatedKernel (the
 * sigmoid-gate option, and a gate tensor whose token rows are strided, as a
 * slice of a merged projection).  The step after the recurrence.
 *
 * Per (token t, head h) row of `dim` values:
 *   out[t,h,:] = core[t,h,:] / sqrt(mean_d(core[t,h,d]^2) + eps)
 *                * weight[:] * act(z[t,h,:])
 * act = silu, or the sigmoid when sigmoid_gate != 0.  f32 arithmetic; out is
 * rounded to act_dtype once.
 *
 * core, out [tokens, heads, dim] contiguous; weight [dim]; z [tokens, heads,
 * dim] with token rows z_token_stride elements apart (0 = heads * dim).  All in
 * act_dtype.  Lengths follow cpu.rs (core, z, out >= tokens*heads*dim; z >=
 * (tokens-1)*stride + heads*dim when strided; weight >= dim).  Pointers 16-byte
 * aligned; z_token_stride * element size a multiple of 16 bytes.
 * Supported: dim a multiple of 8 (bf16) or 4 (f32); dim <= 1024 (bf16), 512 (f32).
 * Errors: GDN_ERR_SHAPE (non-positive sizes, short buffers; cpu.rs's texts),
 * GDN_ERR_INVALID_ARGUMENT (NULL or misaligned pointers, bad stride),
 * GDN_ERR_UNSUPPORTED (dim), GDN_ERR_DTYPE; nothing is launched on error.
 * Asynchronous on `stream`; the caller owns every buffer.
 * ------------------------------------------------------------------------- */
typedef struct gdn_gated_rmsnorm_args {
  int64_t tokens, heads, dim;
  int32_t act_dtype;        /* gdn_dtype of core, z, weight, out */
  int32_t sigmoid_gate;     /* 0: silu(z); else sigmoid(z) */
  float eps;
  const void* core;         /* [tokens, heads, dim] */
  int64_t core_len;
  const void* z;            /* [tokens, heads, dim], token rows z_token_stride apart */
  int64_t z_len;
  int64_t z_token_stride;   /* elements; 0 = heads * dim */
  const void* weight;       /* [dim] */
  int64_t weight_len;
  void* out;                /* [tokens, heads, dim] */
  int64_t out_len;
} gdn_gated_rmsnorm_args;

int gdn_gated_rmsnorm(const gdn_gated_rmsnorm_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * gdn_validate_mixed -- [qwen3_5.cpp] ValidateGdnAttentionMetadata (its
 * non-speculative part): the metadata contract of one mixed step, checked on
 * host copies before anything is launched.
 *
 * A mixed step packs num_decodes single-token sequences first, then
 * num_prefills prefill sequences ([qwen3_5.cpp] SubView of the decode prefix
 * and the prefill suffix).  One gdn_prepare runs over all
 * num_actual_tokens tokens, gdn_decode over rows [0, num_decodes) and
 * gdn_prefill_varlen over the rest with cu_seqlens_prefill, which must be the
 * suffix of cu_seqlens rebased to 0.  Rules, in the page's order (messages are
 * the page's, without its "qwen3_5: " prefix):
 *   counts >= 0; num_decode_tokens == num_decodes;
 *   num_actual_tokens == num_decode_tokens + num_prefill_tokens;
 *   state_indices_host follows the index rules of the general section, and
 *   holds no -1 unless allow_inert_padding;
 *   cu_seqlens_host[0] == 0, cu_seqlens_host[nreq] == num_actual_tokens,
 *   strictly increasing, cu_seqlens_host[num_decodes] == num_decode_tokens;
 *   for prefill i: prefill_state_indices_host[i] == state_indices_host[nd+i]
 *   and >= 0, cu_seqlens_prefill_host[i] == cu_seqlens_host[nd+i] - nd_tok,
 *   prefill_has_initial_state_host[i] == has_initial_state_host[nd+i];
 *   cu_seqlens_prefill_host[num_prefills] == num_prefill_tokens.
 * Every pointer is a HOST pointer; the arrays are read, never written.
 * prefill_state_indices_host / prefill_has_initial_state_host may be NULL
 * when the prefill calls take the suffix views of the full arrays (as this
 * library's step helper does); has_initial_state_host NULL means all 1.
 * Returns GDN_OK or GDN_ERR_INVALID_ARGUMENT with the message; launches
 * nothing and needs no GPU.
 * ------------------------------------------------------------------------- */
typedef struct gdn_mixed_meta {
  int64_t num_decodes;                           /* leading single-token sequences */
  int64_t num_prefills;                          /* sequences after them */
  int64_t num_decode_tokens;                     /* tokens of the decode rows */
  int64_t num_prefill_tokens;                    /* tokens of the prefill rows */
  int64_t num_actual_tokens;                     /* T of the step */
  int64_t state_slots;                           /* slots of the state pool */
  int32_t allow_inert_padding;                   /* 1: -1 allowed among decode rows */
  const int32_t* cu_seqlens_host;                /* [nreq + 1] */
  const int32_t* state_indices_host;             /* [nreq] */
  const uint8_t* has_initial_state_host;         /* [nreq] or NULL */
  const int32_t* cu_seqlens_prefill_host;        /* [num_prefills + 1], rebased */
  const int32_t* prefill_state_indices_host;     /* [num_prefills] or NULL */
  const uint8_t* prefill_has_initial_state_host; /* [num_prefills] or NULL */
} gdn_mixed_meta;

int gdn_validate_mixed(const gdn_mixed_meta* meta);

/* Scratch bytes gdn_prefill_varlen needs for these sizes and algorithm (0 for
 * the recurrent algorithm; for the fused one the bytes of its optional
 * workspace).  With GDN_PREFILL_AUTO it depends on
 * the current device too (gdn_prefill_resolve_algo). */
size_t gdn_prefill_workspace_bytes(int64_t T, int64_t N, int64_t Hv, int64_t Dk, int64_t Dv,
                                   int32_t act_dtype, int32_t algo);

/* The algorithm GDN_PREFILL_AUTO resolves to for these sizes on the current
 * device: for bf16 with Dk = Dv = 128 the fused form when there are at least
 * as many (sequence, value head) chains (N * Hv) as SMs, else the two-launch
 * chunked form; the recurrent form otherwise.  Other values of algo are
 * returned as given. */
int32_t gdn_prefill_resolve_algo(int64_t N, int64_t Hv, int64_t Dk, int64_t Dv, int32_t act_dtype,
                                 int32_t algo);

/* Static text for a status code. */
const char* gdn_status_string(int status);

/* The calling thread's last diagnostic ("" after a successful call). */
const char* gdn_last_error_message(void);

/* Synchronises `stream`, then returns (and clears) the current device's
 * status word: GDN_OK, GDN_ERR_DEVICE_CHECK or GDN_ERR_TIMEOUT. */
int gdn_read_device_status(void* stream);

/* Diagnostic of the device-side failure path (the pages have no
 * counterpart): launches one thread that waits, with the same bounded wait
 * every kernel here uses, on an mbarrier that nothing ever arrives on.  After
 * about budget_cycles SM clocks (at most 2e9, about a second) the wait gives
 * up and records GDN_ERR_TIMEOUT in the device status word, as a kernel
 * whose copy or MMA never completed would; nothing else is in flight, and the
 * context stays usable.  Read the result with gdn_read_device_status().
 * Returns GDN_ERR_INVALID_ARGUMENT for a budget outside (0, 2e9]. */
int gdn_check_wait_timeout(long long budget_cycles, void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int gdn_version(void);

/* Number of kernel launches this process has issued through the library
 * (all devices, all threads).  Lets a caller count the kernels a step runs. */
uint64_t gdn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
