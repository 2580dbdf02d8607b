// gdn_oracle.cpp -- plain CPU oracle for the gated-delta-rule (GDN) layer.
//
// TEST INFRASTRUCTURE ONLY: loaded by the test suite, the smoke check and the
// CPU-baseline leg of the benchmark, never by the library's product path.  It
// shares no code with the CUDA library.  Build: g++ -std=c++17 -O2
// -ffp-contract=off -shared -fPIC -pthread (no fused multiply-add, so the f32
// results do not depend on the host's FMA contraction).
//
// Every routine is a token-by-token restatement of the pages' CPU code, in the
// pages' loop order, with a reference to the function it follows:
//   [cpu.rs]       ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs
//   [cpu_ops.cpp]  vllm.cpp, src/vt/cpu/cpu_ops.cpp
//   [qwen3_5.cpp]  vllm.cpp, src/vllm/model_executor/models/qwen3_5.cpp
// The chunked form (orc_gdn_chunked_f64) is not on the pages; it is derived
// from the recurrence and exists only to check that algebra.
//
// Parity pins (tests/test_oracle_*.py) tie each routine to something other than
// itself; see the header for the list.
#include "gdn_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

namespace {

void set_msg(char* msg, size_t cap, const std::string& s) {
  if (msg == nullptr || cap == 0) return;
  std::snprintf(msg, cap, "%s", s.c_str());
}

// Runs body(i) for i in [0, n) on `nthreads` threads (0 = hardware
// concurrency).  Each index is an independent output, so the result is the
// same for every thread count ([cpu_ops.cpp] ForRows: outputs partitioned only).
template <typename F>
void parallel_items(int64_t n, int nthreads, F body) {
  if (nthreads <= 0) {
    unsigned hc = std::thread::hardware_concurrency();
    nthreads = hc == 0 ? 1 : static_cast<int>(hc);
  }
  if (nthreads == 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) body(i);
    return;
  }
  if (nthreads > n) nthreads = static_cast<int>(n);
  std::vector<std::thread> pool;
  const int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    const int64_t lo = t * per, hi = std::min<int64_t>(n, lo + per);
    if (lo >= hi) break;
    pool.emplace_back([=, &body] {
      for (int64_t i = lo; i < hi; ++i) body(i);
    });
  }
  for (auto& th : pool) th.join();
}

// ---- [cpu.rs] sigmoid / silu / softplus -------------------------------------
// sigmoid: two branches so that exp never overflows.
template <typename R>
R sigmoid_(R x) {
  if (x >= R(0)) {
    const R z = std::exp(-x);
    return R(1) / (R(1) + z);
  }
  const R z = std::exp(x);
  return z / (R(1) + z);
}
template <typename R>
R silu_(R x) {
  return x * sigmoid_(x);
}
// softplus: identity above 20, exp below -20, ln(1 + e^x) between.
template <typename R>
R softplus_(R x) {
  if (x > R(20)) return x;
  if (x < R(-20)) return std::exp(x);
  return std::log(R(1) + std::exp(x));
}

// ---- [cpu.rs] recurrent_gated_delta_rule_varlen_f32 cu_seqlens rules -------
// The page formats cu.first() and cu.last(), which are Rust Options, with
// {:?}: a present value prints as "Some(v)".
int check_cu(const int32_t* cu, int64_t batch, int64_t total, char* msg, size_t cap,
             const char* who = "gated_delta_rule_varlen") {
  if (cu == nullptr) {
    set_msg(msg, cap, "cu_seqlens is NULL");
    return ORC_ERR_INVALID;
  }
  if (cu[0] != 0 || static_cast<int64_t>(cu[batch]) != total) {
    set_msg(msg, cap,
            std::string(who) + " cu_seqlens must start at 0 and end at total_tokens " +
                std::to_string(total) + ", got first=Some(" + std::to_string(cu[0]) +
                ") last=Some(" + std::to_string(cu[batch]) + ")");
    return ORC_ERR_INVALID;
  }
  for (int64_t s = 0; s < batch; ++s) {
    if (cu[s + 1] <= cu[s]) {
      set_msg(msg, cap,
              std::string(who) + " sequence " + std::to_string(s) +
                  " has empty or non-monotonic range " + std::to_string(cu[s]) + ".." +
                  std::to_string(cu[s + 1]));
      return ORC_ERR_INVALID;
    }
  }
  return ORC_OK;
}

// Range rule for a pool index ([cpu_ops.cpp] GdnStateGatherKernel range check;
// [qwen3_5.cpp] ValidateGdnStateIndices: -1 is the only allowed negative).
int check_slots(const int32_t* idx, int64_t n, int64_t slots, char* msg, size_t cap) {
  for (int64_t i = 0; i < n; ++i) {
    const int64_t slot = idx != nullptr ? idx[i] : i;
    if (slot == -1) continue;
    if (slot < -1) {
      set_msg(msg, cap, "invalid negative GDN state index");
      return ORC_ERR_INVALID;
    }
    if (slot >= slots) {
      set_msg(msg, cap, "GDN state index out of range");
      return ORC_ERR_INVALID;
    }
  }
  return ORC_OK;
}

template <typename R>
void prepare_gates_norm(const R* a_raw, int64_t a_stride, const R* b_raw, int64_t b_stride,
                        const R* a_log, const R* dt_bias, int64_t tokens, int64_t hk_n,
                        int64_t hv_n, int64_t dk, int apply_norm, R* q, R* k, R* g, R* beta,
                        int nthreads);

// ---- O1: prepare --------------------------------------------------------------
// [cpu.rs] linear_attention_prepare_varlen_f32 per sequence:
//   conv:   acc = sum_j x~[t + j - (K-1)] * w[c, j], x~[i] = x[i] for i >= 0 and
//           the initial tail[(K-1) + i] for i < 0;  y = silu(acc)
//   split:  [0, HkDk) -> q, [HkDk, 2HkDk) -> k, rest -> v
//   gates:  g = -exp(A_log) * softplus(a + dt_bias),  beta = sigmoid(b)
//   tail:   the last K-1 entries of tail || x (oldest first)
//   norm:   q,k *= 1/sqrt(sum sq + 1e-6) per (token, key head)
template <typename R>
int prepare_impl(const R* x, int64_t x_stride, const R* w, R* conv_pool, int64_t conv_slots,
                 const int32_t* sidx, const uint8_t* has_init, const R* a_raw, int64_t a_stride,
                 const R* b_raw, int64_t b_stride, const R* a_log, const R* dt_bias,
                 const int32_t* cu, int64_t n_seqs, int64_t tokens, int64_t hk_n, int64_t hv_n,
                 int64_t dk, int64_t dv, int64_t kw, int apply_norm, R* q, R* k, R* v, R* g,
                 R* beta, int nthreads) {
  if (n_seqs <= 0 || tokens <= 0 || hk_n <= 0 || hv_n <= 0 || dk <= 0 || dv <= 0 || kw <= 0)
    return ORC_ERR_SHAPE;
  if (int rc = check_cu(cu, n_seqs, tokens, nullptr, 0)) return rc;
  if (int rc = check_slots(sidx, n_seqs, conv_slots, nullptr, 0)) return rc;
  const int64_t qk_total = hk_n * dk, v_total = hv_n * dv;
  const int64_t channels = 2 * qk_total + v_total;
  const int64_t width = kw - 1;
  if (x_stride <= 0) x_stride = channels;
  if (a_stride <= 0) a_stride = hv_n;
  if (b_stride <= 0) b_stride = hv_n;

  // Work item = (sequence, channel): it owns its outputs and its tail row.
  parallel_items(n_seqs * channels, nthreads, [&](int64_t item) {
    const int64_t s = item / channels, c = item % channels;
    const int64_t start = cu[s], len = cu[s + 1] - cu[s];
    const int64_t slot = sidx != nullptr ? sidx[s] : s;
    const bool live = slot >= 0;
    const bool init = live && (has_init == nullptr || has_init[s] != 0);
    std::vector<R> old_tail(static_cast<size_t>(width), R(0));
    R* tail_row = live ? conv_pool + (slot * channels + c) * width : nullptr;
    if (init)
      for (int64_t j = 0; j < width; ++j) old_tail[j] = tail_row[j];
    auto tap = [&](int64_t local) -> R {  // x~ at local token index
      return local >= 0 ? x[(start + local) * x_stride + c] : old_tail[width + local];
    };
    for (int64_t lt = 0; lt < len; ++lt) {
      R acc = R(0);
      for (int64_t j = 0; j < kw; ++j) acc += tap(lt + j - width) * w[c * kw + j];
      const R y = silu_(acc);
      const int64_t t = start + lt;
      if (c < qk_total)
        q[t * qk_total + c] = y;
      else if (c < 2 * qk_total)
        k[t * qk_total + (c - qk_total)] = y;
      else
        v[t * v_total + (c - 2 * qk_total)] = y;
    }
    if (live)
      for (int64_t pos = 0; pos < width; ++pos) tail_row[pos] = tap(len + pos - width);
  });

  prepare_gates_norm(a_raw, a_stride, b_raw, b_stride, a_log, dt_bias, tokens, hk_n, hv_n, dk,
                     apply_norm, q, k, g, beta, nthreads);
  return ORC_OK;
}

// The steps of O1 after the conv: gates per (token, value head) and the q/k L2
// norm per (token, key head).
template <typename R>
void prepare_gates_norm(const R* a_raw, int64_t a_stride, const R* b_raw, int64_t b_stride,
                        const R* a_log, const R* dt_bias, int64_t tokens, int64_t hk_n,
                        int64_t hv_n, int64_t dk, int apply_norm, R* q, R* k, R* g, R* beta,
                        int nthreads) {
  parallel_items(tokens, nthreads, [&](int64_t t) {
    for (int64_t h = 0; h < hv_n; ++h) {
      g[t * hv_n + h] = -std::exp(a_log[h]) * softplus_(a_raw[t * a_stride + h] + dt_bias[h]);
      beta[t * hv_n + h] = sigmoid_(b_raw[t * b_stride + h]);
    }
  });

  if (apply_norm) {
    parallel_items(tokens * hk_n, nthreads, [&](int64_t row) {
      const int64_t base = row * dk;
      R q_sum = R(0), k_sum = R(0);
      for (int64_t d = 0; d < dk; ++d) {
        q_sum += q[base + d] * q[base + d];
        k_sum += k[base + d] * k[base + d];
      }
      const R q_inv = R(1) / std::sqrt(q_sum + R(1e-6));
      const R k_inv = R(1) / std::sqrt(k_sum + R(1e-6));
      for (int64_t d = 0; d < dk; ++d) {
        q[base + d] *= q_inv;
        k[base + d] *= k_inv;
      }
    });
  }
}

// ---- O8: speculative prepare ([cpu_ops.cpp] CausalConv1dSpecUpdateKernel) ------
// The conv of O1 for the draft tokens of a speculative step.  Each request's
// conv row holds state_len = (K-1) + (max_q - 1) raw inputs; with
// off = num_accepted - 1 the window before the first draft is row[off ..
// off+K-2] (entries past the row read 0), then the drafts themselves.  The
// row becomes row[off+1 .. off+keep] || drafts, keep = state_len - len: shifted
// by one tap per step, so that the next step's offset picks the window that
// ends at its last accepted token.  Split, gates and norm are O1's.
// A negative slot: outputs from a zero window, no row written; an empty
// request: nothing.
template <typename R>
int spec_prepare_impl(const R* x, int64_t x_stride, const R* w, R* conv_pool, int64_t conv_slots,
                      int64_t state_len, const int32_t* cidx, const int32_t* num_accepted,
                      const R* a_raw, int64_t a_stride, const R* b_raw, int64_t b_stride,
                      const R* a_log, const R* dt_bias, const int32_t* cu, int64_t n_reqs,
                      int64_t tokens, int64_t hk_n, int64_t hv_n, int64_t dk, int64_t dv,
                      int64_t kw, int apply_norm, R* q, R* k, R* v, R* g, R* beta,
                      int nthreads) {
  if (n_reqs <= 0 || tokens <= 0 || hk_n <= 0 || hv_n <= 0 || dk <= 0 || dv <= 0 || kw <= 0)
    return ORC_ERR_SHAPE;
  // K >= 2: with no conv tail (K = 1) a request of max_q tokens would need
  // keep = -1 entries of the old row
  const int64_t width = kw - 1, max_q = state_len - width + 1;
  if (kw < 2 || max_q < 1) return ORC_ERR_SHAPE;
  if (cu[0] != 0 || cu[n_reqs] != tokens) return ORC_ERR_INVALID;
  for (int64_t i = 0; i < n_reqs; ++i) {
    if (cu[i + 1] < cu[i] || cu[i + 1] - cu[i] > max_q) return ORC_ERR_INVALID;
    if (num_accepted[i] < 1 || num_accepted[i] > max_q) return ORC_ERR_INVALID;
    if (cidx[i] >= conv_slots) return ORC_ERR_INVALID;
  }
  const int64_t qk_total = hk_n * dk, v_total = hv_n * dv;
  const int64_t channels = 2 * qk_total + v_total;
  if (x_stride <= 0) x_stride = channels;
  if (a_stride <= 0) a_stride = hv_n;
  if (b_stride <= 0) b_stride = hv_n;

  parallel_items(n_reqs * channels, nthreads, [&](int64_t item) {
    const int64_t i = item / channels, c = item % channels;
    const int64_t lo = cu[i], len = cu[i + 1] - cu[i];
    if (len == 0) return;
    const bool live = cidx[i] >= 0;
    R* row = live ? conv_pool + (cidx[i] * channels + c) * state_len : nullptr;
    const int64_t off = num_accepted[i] - 1;
    auto old_at = [&](int64_t j) -> R { return live && j < state_len ? row[j] : R(0); };
    std::vector<R> stream(static_cast<size_t>(width + len));  // window || drafts
    for (int64_t j = 0; j < width; ++j) stream[j] = old_at(off + j);
    for (int64_t t = 0; t < len; ++t) stream[width + t] = x[(lo + t) * x_stride + c];
    for (int64_t t = 0; t < len; ++t) {
      R acc = R(0);
      for (int64_t j = 0; j < kw; ++j) acc += stream[t + j] * w[c * kw + j];
      const R y = silu_(acc);
      const int64_t tt = lo + t;
      if (c < qk_total)
        q[tt * qk_total + c] = y;
      else if (c < 2 * qk_total)
        k[tt * qk_total + (c - qk_total)] = y;
      else
        v[tt * v_total + (c - 2 * qk_total)] = y;
    }
    if (!live) return;
    const int64_t keep = state_len - len;
    std::vector<R> next(static_cast<size_t>(state_len));
    for (int64_t j = 0; j < keep; ++j) next[j] = old_at(off + 1 + j);
    for (int64_t t = 0; t < len; ++t) next[keep + t] = stream[width + t];
    std::copy(next.begin(), next.end(), row);
  });
  prepare_gates_norm(a_raw, a_stride, b_raw, b_stride, a_log, dt_bias, tokens, hk_n, hv_n, dk,
                     apply_norm, q, k, g, beta, nthreads);
  return ORC_OK;
}

// ---- O2: one (sequence, value head) chain of the recurrence -----------------
// [cpu.rs] recurrent_gated_delta_rule_varlen_f32, inner loops, on one [Dv,Dk]
// state block S (row vd holds S[vd, :]):
//   S *= exp(g);  kv = S k;  delta = (v - kv) * beta;  S += delta k^T;
//   out = S (q * scale)
// with the optional in-loop q/k L2 norm (k scaled by k_inv, q by q_inv*scale).
template <typename R>
void head_chain(const R* q, const R* k, const R* v, const R* g, const R* beta, R* S,
                int64_t t0, int64_t t1, int64_t h, int64_t hk, int64_t hk_n, int64_t hv_n,
                int64_t dk, int64_t dv, R scale, bool use_norm, R* out) {
  for (int64_t t = t0; t < t1; ++t) {
    const R* qt = q + (t * hk_n + hk) * dk;
    const R* kt = k + (t * hk_n + hk) * dk;
    R q_inv = R(1), k_inv = R(1);
    if (use_norm) {
      R q_norm = R(0), k_norm = R(0);
      for (int64_t d = 0; d < dk; ++d) {
        q_norm += qt[d] * qt[d];
        k_norm += kt[d] * kt[d];
      }
      q_inv = R(1) / std::sqrt(q_norm + R(1e-6));
      k_inv = R(1) / std::sqrt(k_norm + R(1e-6));
    }
    const R decay = std::exp(g[t * hv_n + h]);
    const R beta_t = beta[t * hv_n + h];
    for (int64_t vd = 0; vd < dv; ++vd) {
      R* row = S + vd * dk;
      R kv_mem = R(0);
      for (int64_t d = 0; d < dk; ++d) {
        row[d] *= decay;
        kv_mem += row[d] * (kt[d] * k_inv);
      }
      const R delta = (v[(t * hv_n + h) * dv + vd] - kv_mem) * beta_t;
      for (int64_t d = 0; d < dk; ++d) row[d] += delta * (kt[d] * k_inv);
      R acc = R(0);
      for (int64_t d = 0; d < dk; ++d) acc += row[d] * (qt[d] * q_inv * scale);
      out[(t * hv_n + h) * dv + vd] = acc;
    }
  }
}

// The KDA variant of one (sequence, value head) chain, [cpu_ops.cpp]
// KdaHeadTokenStep: the decay is per key channel, g [T, Hv, Dk] (log decay of
// column d of S), and q, k are used as given.  Per token, in the page's order:
// first every row decays and takes its dot with k, then every row gets its
// rank-1 update and its dot with scale * q.
template <typename R>
void kda_head_chain(const R* q, const R* k, const R* v, const R* g, const R* beta, R* S,
                    int64_t t0, int64_t t1, int64_t h, int64_t hk, int64_t hk_n, int64_t hv_n,
                    int64_t dk, int64_t dv, R scale, R* out) {
  std::vector<R> qbuf(dk), kbuf(dk), vbuf(dv), decay(dk);
  for (int64_t t = t0; t < t1; ++t) {
    const R beta_t = beta[t * hv_n + h];
    const R* g_row = g + (t * hv_n + h) * dk;
    for (int64_t d = 0; d < dk; ++d) {
      qbuf[d] = q[(t * hk_n + hk) * dk + d] * scale;
      kbuf[d] = k[(t * hk_n + hk) * dk + d];
      decay[d] = std::exp(g_row[d]);
    }
    for (int64_t vd = 0; vd < dv; ++vd) {
      R* row = S + vd * dk;
      R dot = R(0);
      for (int64_t d = 0; d < dk; ++d) {
        row[d] *= decay[d];
        dot += row[d] * kbuf[d];
      }
      vbuf[vd] = (v[(t * hv_n + h) * dv + vd] - dot) * beta_t;
    }
    for (int64_t vd = 0; vd < dv; ++vd) {
      R* row = S + vd * dk;
      R o = R(0);
      for (int64_t d = 0; d < dk; ++d) {
        row[d] += vbuf[vd] * kbuf[d];
        o += row[d] * qbuf[d];
      }
      out[(t * hv_n + h) * dv + vd] = o;
    }
  }
}

template <typename R>
int varlen_impl(const R* q, const R* k, const R* v, const R* g, const R* beta, R* pool,
                int64_t slots, const int32_t* sidx, const uint8_t* has_init, const int32_t* cu,
                int64_t n_seqs, int64_t tokens, int64_t hk_n, int64_t hv_n, int64_t dk,
                int64_t dv, R scale, int use_norm, const int32_t* items, int64_t n_items, R* out,
                int nthreads, bool kda = false) {
  if (n_seqs <= 0 || tokens <= 0 || hk_n <= 0 || hv_n <= 0 || dk <= 0 || dv <= 0)
    return ORC_ERR_SHAPE;
  if (hv_n % hk_n != 0) return ORC_ERR_SHAPE;
  if (int rc = check_cu(cu, n_seqs, tokens, nullptr, 0)) return rc;
  if (int rc = check_slots(sidx, n_seqs, slots, nullptr, 0)) return rc;
  const int64_t ratio = hv_n / hk_n;  // GQA: value head h reads key head h / ratio
  const int64_t state_len = dv * dk;
  const int64_t total_items = items != nullptr ? n_items : n_seqs * hv_n;
  for (int64_t i = 0; items != nullptr && i < n_items; ++i)
    if (items[i] < 0 || items[i] >= n_seqs * hv_n) return ORC_ERR_INVALID;
  parallel_items(total_items, nthreads, [&](int64_t i) {
    const int64_t item = items != nullptr ? items[i] : i;
    const int64_t s = item / hv_n, h = item % hv_n;
    const int64_t slot = sidx != nullptr ? sidx[s] : s;
    if (slot < 0) {  // padded sequence: zero output, pool untouched
      for (int64_t t = cu[s]; t < cu[s + 1]; ++t)
        for (int64_t d = 0; d < dv; ++d) out[(t * hv_n + h) * dv + d] = R(0);
      return;
    }
    R* S = pool + (slot * hv_n + h) * state_len;
    if (has_init != nullptr && has_init[s] == 0)
      for (int64_t e = 0; e < state_len; ++e) S[e] = R(0);
    if (kda)
      kda_head_chain(q, k, v, g, beta, S, cu[s], cu[s + 1], h, h / ratio, hk_n, hv_n, dk, dv,
                     scale, out);
    else
      head_chain(q, k, v, g, beta, S, cu[s], cu[s + 1], h, h / ratio, hk_n, hv_n, dk, dv,
                 scale, use_norm != 0, out);
  });
  return ORC_OK;
}

// ---- Deviation bound of O2 under moved inputs (test aid, f64) ---------------
// When the stored q, k, v of the recurrence move by at most dq, dk, dv
// (elementwise), how far can each output move, to first order?  O2 is
//   S_t = a S_{t-1} (I - b k k^T) + b v k^T,   o_t = scale S_t q,   a = e^g, b = beta,
// so, to first order in the moves, row c of the state moves by
//   dS_t[c] = a dS_{t-1}[c] (I - b k k^T) + b dv_c k^T - a b (S_{t-1}[c].dk) k^T
//             + b (v_c - a S_{t-1}[c].k) dk^T
// and the output by do_t[c] = scale (dS_t[c].q + S_t[c].dq).  With
// |I - b k k^T|_2 = max(1, |1 - b |k|^2|) this gives the row-norm bound
//   r_t[c] = a r_{t-1}[c] max(1, |1 - b|k|^2|)
//            + b (dv_c |k| + a sum_d |S_{t-1}[c][d]| dk_d |k| + |v_c - a S_{t-1}[c].k| |dk|)
//   |do_t[c]| <= scale (r_t[c] |q| + sum_d |S_t[c][d]| dq_d),
// run alongside the recurrence itself (same loop order as head_chain, no
// in-loop norm).  The state pool is read, not written.  The final r[c] bounds
// every element of row c of the final state (|x_d| <= |x|), written to
// state_bound when it is given.
void deviation_chain(const double* q, const double* k, const double* v, const double* g,
                     const double* beta, const double* dq, const double* dk_, const double* dv_,
                     std::vector<double>& S, int64_t t0, int64_t t1, int64_t h, int64_t hk,
                     int64_t hk_n, int64_t hv_n, int64_t dk, int64_t dv, double scale,
                     double* bound, double* state_bound) {
  std::vector<double> r(dv, 0.0);
  for (int64_t t = t0; t < t1; ++t) {
    const double* qt = q + (t * hk_n + hk) * dk;
    const double* kt = k + (t * hk_n + hk) * dk;
    const double* dqt = dq + (t * hk_n + hk) * dk;
    const double* dkt = dk_ + (t * hk_n + hk) * dk;
    double nq = 0.0, nk = 0.0, ndk = 0.0;
    for (int64_t d = 0; d < dk; ++d) {
      nq += qt[d] * qt[d];
      nk += kt[d] * kt[d];
      ndk += dkt[d] * dkt[d];
    }
    const double a = std::exp(g[t * hv_n + h]), b = beta[t * hv_n + h];
    const double shrink = std::max(1.0, std::fabs(1.0 - b * nk));
    nq = std::sqrt(nq);
    nk = std::sqrt(nk);
    ndk = std::sqrt(ndk);
    for (int64_t c = 0; c < dv; ++c) {
      double* row = S.data() + c * dk;
      double sk = 0.0, kv = 0.0;
      for (int64_t d = 0; d < dk; ++d) {
        sk += std::fabs(row[d]) * dkt[d];
        row[d] *= a;
        kv += row[d] * kt[d];
      }
      const double vc = v[(t * hv_n + h) * dv + c];
      const double delta = (vc - kv) * b;
      double sq = 0.0;
      for (int64_t d = 0; d < dk; ++d) {
        row[d] += delta * kt[d];
        sq += std::fabs(row[d]) * dqt[d];
      }
      r[c] = a * r[c] * shrink +
             b * (dv_[(t * hv_n + h) * dv + c] * nk + a * sk * nk + std::fabs(vc - kv) * ndk);
      bound[(t * hv_n + h) * dv + c] = scale * (r[c] * nq + sq);
    }
  }
  if (state_bound != nullptr)
    for (int64_t c = 0; c < dv; ++c) state_bound[c] = r[c];
}

// ---- O7: speculative multi-token decode ([cpu_ops.cpp] GdnSpecDecodeKernel) --
// Request i owns tokens [cu[i], cu[i+1]) and a row of num_cols pool slots.  Its
// state starts from slot sidx[i][num_accepted[i] - 1] (the snapshot after the
// previous step's last accepted token); after token t the state is stored into
// slot sidx[i][t - cu[i]] (a negative column skips that store).  A negative
// initial slot zeroes the request's outputs and leaves the pool alone.  q, k are used as
// given ([cpu_ops.cpp] GdnHeadTokenStep).
template <typename R>
int spec_decode_impl(const R* q, const R* k, const R* v, const R* g, const R* beta, R* pool,
                     int64_t slots, const int32_t* cu, int64_t n_reqs, int64_t tokens,
                     const int32_t* sidx, int64_t num_cols, const int32_t* num_accepted,
                     int64_t hk_n, int64_t hv_n, int64_t dk, int64_t dv, R scale, R* out,
                     int nthreads) {
  if (n_reqs <= 0 || tokens <= 0 || num_cols <= 0 || hk_n <= 0 || hv_n <= 0 || dk <= 0 ||
      dv <= 0 || hv_n % hk_n != 0)
    return ORC_ERR_SHAPE;
  if (cu[0] != 0 || cu[n_reqs] != tokens) return ORC_ERR_INVALID;
  for (int64_t i = 0; i < n_reqs; ++i) {
    if (cu[i + 1] < cu[i] || cu[i + 1] - cu[i] > num_cols) return ORC_ERR_INVALID;
    if (num_accepted[i] < 1 || num_accepted[i] > num_cols) return ORC_ERR_INVALID;
    for (int64_t c = 0; c < num_cols; ++c)
      if (sidx[i * num_cols + c] >= slots) return ORC_ERR_INVALID;
  }
  const int64_t ratio = hv_n / hk_n, state_len = dv * dk;
  parallel_items(n_reqs * hv_n, nthreads, [&](int64_t item) {
    const int64_t i = item / hv_n, h = item % hv_n;
    const int64_t lo = cu[i], hi = cu[i + 1];
    const int32_t init = sidx[i * num_cols + (num_accepted[i] - 1)];
    if (init < 0) {
      for (int64_t t = lo; t < hi; ++t)
        for (int64_t d = 0; d < dv; ++d) out[(t * hv_n + h) * dv + d] = R(0);
      return;
    }
    if (hi == lo) return;
    std::vector<R> S(pool + (init * hv_n + h) * state_len,
                     pool + (init * hv_n + h) * state_len + state_len);
    for (int64_t t = lo; t < hi; ++t) {
      head_chain(q, k, v, g, beta, S.data(), t, t + 1, h, h / ratio, hk_n, hv_n, dk, dv, scale,
                 false, out);
      const int32_t slot = sidx[i * num_cols + (t - lo)];
      if (slot < 0) continue;
      std::copy(S.begin(), S.end(), pool + (slot * hv_n + h) * state_len);
    }
  });
  return ORC_OK;
}

// ---- O3: decode ([cpu_ops.cpp] GdnDecodeKernel) -----------------------------
template <typename R>
int decode_impl(const R* q, const R* k, const R* v, const R* g, const R* beta, R* pool,
                int64_t slots, const int32_t* sidx, int64_t batch, int64_t hk_n, int64_t hv_n,
                int64_t dk, int64_t dv, R scale, int use_norm, R* out, int nthreads) {
  if (batch <= 0 || hk_n <= 0 || hv_n <= 0 || dk <= 0 || dv <= 0) return ORC_ERR_SHAPE;
  if (hv_n % hk_n != 0) return ORC_ERR_SHAPE;
  if (int rc = check_slots(sidx, batch, slots, nullptr, 0)) return rc;
  const int64_t ratio = hv_n / hk_n;
  parallel_items(batch, nthreads, [&](int64_t b) {
    const int64_t slot = sidx != nullptr ? sidx[b] : b;
    if (slot < 0) {
      for (int64_t e = 0; e < hv_n * dv; ++e) out[b * hv_n * dv + e] = R(0);
      return;
    }
    for (int64_t h = 0; h < hv_n; ++h)
      head_chain(q, k, v, g, beta, pool + (slot * hv_n + h) * dv * dk, b, b + 1, h, h / ratio,
                 hk_n, hv_n, dk, dv, scale, use_norm != 0, out);
  });
  return ORC_OK;
}

// ---- O4: chunked WY/UT form (f64) -------------------------------------------
// Derived from the recurrence.  For a chunk of L tokens with state S0 [Dv,Dk]:
//   gam_i = sum_{t<=i} g_t
//   A_ij  = beta_i exp(gam_i - gam_j) (k_i . k_j)      j < i
//   T     = (I + A)^-1                                  (forward substitution)
//   W     = T diag(beta exp(gam)) K,  Ut = T diag(beta) V,  U = Ut - W S0^T
//   O     = diag(exp(gam)) Qs S0^T + (M o Qs K^T) U,   M_ij = exp(gam_i - gam_j), j <= i
//   S_L   = exp(gam_last) S0 + U^T diag(exp(gam_last - gam)) K
// with Qs = scale * Q.  Every exponent is <= 0.
void chunk_step(const std::vector<double>& Kc, const std::vector<double>& Qc,
                const std::vector<double>& Vc, const std::vector<double>& gc,
                const std::vector<double>& bc, int64_t L, int64_t dk, int64_t dv, double* S,
                std::vector<double>& Oc) {
  std::vector<double> gam(L);
  double run = 0.0;
  for (int64_t i = 0; i < L; ++i) {
    run += gc[i];
    gam[i] = run;
  }
  auto kdot = [&](const std::vector<double>& X, int64_t i, const std::vector<double>& Y,
                  int64_t j) {
    double s = 0.0;
    for (int64_t d = 0; d < dk; ++d) s += X[i * dk + d] * Y[j * dk + d];
    return s;
  };
  std::vector<double> A(L * L, 0.0);
  for (int64_t i = 0; i < L; ++i)
    for (int64_t j = 0; j < i; ++j)
      A[i * L + j] = bc[i] * std::exp(gam[i] - gam[j]) * kdot(Kc, i, Kc, j);
  // T = (I + A)^-1 by forward substitution, column by column.
  std::vector<double> T(L * L, 0.0);
  for (int64_t col = 0; col < L; ++col)
    for (int64_t i = 0; i < L; ++i) {
      double s = (i == col) ? 1.0 : 0.0;
      for (int64_t m = 0; m < i; ++m) s -= A[i * L + m] * T[m * L + col];
      T[i * L + col] = s;
    }
  std::vector<double> W(L * dk, 0.0), U(L * dv, 0.0);
  for (int64_t i = 0; i < L; ++i)
    for (int64_t j = 0; j <= i; ++j) {
      const double tw = T[i * L + j] * bc[j] * std::exp(gam[j]);
      const double tu = T[i * L + j] * bc[j];
      for (int64_t d = 0; d < dk; ++d) W[i * dk + d] += tw * Kc[j * dk + d];
      for (int64_t d = 0; d < dv; ++d) U[i * dv + d] += tu * Vc[j * dv + d];
    }
  for (int64_t i = 0; i < L; ++i)  // U = Ut - W S0^T
    for (int64_t e = 0; e < dv; ++e) {
      double s = 0.0;
      for (int64_t d = 0; d < dk; ++d) s += W[i * dk + d] * S[e * dk + d];
      U[i * dv + e] -= s;
    }
  Oc.assign(L * dv, 0.0);
  for (int64_t i = 0; i < L; ++i) {
    for (int64_t e = 0; e < dv; ++e) {
      double s = 0.0;
      for (int64_t d = 0; d < dk; ++d) s += Qc[i * dk + d] * S[e * dk + d];
      Oc[i * dv + e] = std::exp(gam[i]) * s;
    }
    for (int64_t j = 0; j <= i; ++j) {
      const double p = std::exp(gam[i] - gam[j]) * kdot(Qc, i, Kc, j);
      for (int64_t e = 0; e < dv; ++e) Oc[i * dv + e] += p * U[j * dv + e];
    }
  }
  const double g_last = gam[L - 1];
  for (int64_t e = 0; e < dv; ++e)
    for (int64_t d = 0; d < dk; ++d) {
      double s = std::exp(g_last) * S[e * dk + d];
      for (int64_t j = 0; j < L; ++j)
        s += U[j * dv + e] * std::exp(g_last - gam[j]) * Kc[j * dk + d];
      S[e * dk + d] = s;
    }
}

// ---- O9: chunked form of the KDA recurrence (f64) -----------------------------
// Derived from [cpu_ops.cpp] KdaHeadTokenStep as O4 is from the scalar-decay
// recurrence, with a log decay per key channel d.  For a chunk of L tokens with
// state S0 [Dv,Dk] and gam_i[d] = sum_{t<=i} g_t[d]:
//   A_ij  = beta_i sum_d k_i[d] k_j[d] exp(gam_i[d] - gam_j[d])      j < i
//   T     = (I + A)^-1
//   W_i   = sum_{j<=i} T_ij beta_j (k_j o exp(gam_j)),  Ut_i = sum_{j<=i} T_ij beta_j v_j
//   U     = Ut - W S0^T
//   O_i   = (q_i o exp(gam_i)) S0^T + sum_{j<=i} (sum_d q_i[d] k_j[d] exp(gam_i[d] - gam_j[d])) U_j
//   S_L[:, d] = exp(gam_L[d]) S0[:, d] + sum_j U_j k_j[d] exp(gam_L[d] - gam_j[d])
// with q already scaled.  Every exponent is <= 0: each pair's decay is taken
// as its own difference, never as a product of a growing and a shrinking
// factor.
void kda_chunk_step(const std::vector<double>& Kc, const std::vector<double>& Qc,
                    const std::vector<double>& Vc, const std::vector<double>& Gc,
                    const std::vector<double>& bc, int64_t L, int64_t dk, int64_t dv,
                    double* S, std::vector<double>& Oc) {
  std::vector<double> gam(L * dk);
  for (int64_t d = 0; d < dk; ++d) {
    double run = 0.0;
    for (int64_t i = 0; i < L; ++i) {
      run += Gc[i * dk + d];
      gam[i * dk + d] = run;
    }
  }
  // sum_d X_i[d] Y_j[d] exp(gam_i[d] - gam_j[d])
  auto ddot = [&](const std::vector<double>& X, int64_t i, const std::vector<double>& Y,
                  int64_t j) {
    double s = 0.0;
    for (int64_t d = 0; d < dk; ++d)
      s += X[i * dk + d] * Y[j * dk + d] * std::exp(gam[i * dk + d] - gam[j * dk + d]);
    return s;
  };
  std::vector<double> A(L * L, 0.0);
  for (int64_t i = 0; i < L; ++i)
    for (int64_t j = 0; j < i; ++j) A[i * L + j] = bc[i] * ddot(Kc, i, Kc, j);
  std::vector<double> T(L * L, 0.0);
  for (int64_t col = 0; col < L; ++col)
    for (int64_t i = 0; i < L; ++i) {
      double s = (i == col) ? 1.0 : 0.0;
      for (int64_t m = 0; m < i; ++m) s -= A[i * L + m] * T[m * L + col];
      T[i * L + col] = s;
    }
  std::vector<double> W(L * dk, 0.0), U(L * dv, 0.0);
  for (int64_t i = 0; i < L; ++i)
    for (int64_t j = 0; j <= i; ++j) {
      const double t = T[i * L + j] * bc[j];
      for (int64_t d = 0; d < dk; ++d)
        W[i * dk + d] += t * Kc[j * dk + d] * std::exp(gam[j * dk + d]);
      for (int64_t d = 0; d < dv; ++d) U[i * dv + d] += t * Vc[j * dv + d];
    }
  for (int64_t i = 0; i < L; ++i)  // U = Ut - W S0^T
    for (int64_t e = 0; e < dv; ++e) {
      double s = 0.0;
      for (int64_t d = 0; d < dk; ++d) s += W[i * dk + d] * S[e * dk + d];
      U[i * dv + e] -= s;
    }
  Oc.assign(L * dv, 0.0);
  for (int64_t i = 0; i < L; ++i) {
    for (int64_t e = 0; e < dv; ++e) {
      double s = 0.0;
      for (int64_t d = 0; d < dk; ++d)
        s += Qc[i * dk + d] * std::exp(gam[i * dk + d]) * S[e * dk + d];
      Oc[i * dv + e] = s;
    }
    for (int64_t j = 0; j <= i; ++j) {
      const double pij = ddot(Qc, i, Kc, j);
      for (int64_t e = 0; e < dv; ++e) Oc[i * dv + e] += pij * U[j * dv + e];
    }
  }
  const double* gl = &gam[(L - 1) * dk];
  for (int64_t e = 0; e < dv; ++e)
    for (int64_t d = 0; d < dk; ++d) {
      double s = std::exp(gl[d]) * S[e * dk + d];
      for (int64_t j = 0; j < L; ++j)
        s += U[j * dv + e] * Kc[j * dk + d] * std::exp(gl[d] - gam[j * dk + d]);
      S[e * dk + d] = s;
    }
}

// Gated RMSNorm of the recurrence output, [cpu.rs] gated_rms_norm_f32 (SiLU
// gate) with [cpu_ops.cpp] RmsNormGatedKernel's options: a sigmoid gate and a
// gate tensor [T, H, D] whose token rows are z_stride elements apart.  Per
// (token, head) row of D values:
//   inv = 1 / sqrt(sum_d core^2 / D + eps),  out = core * inv * weight[d] * act(z).
template <typename T>
void gated_rmsnorm_(const T* core, const T* z, int64_t z_stride, const T* weight, T* out,
                    int64_t tokens, int64_t heads, int64_t dim, T eps, bool sigmoid_gate,
                    int nthreads) {
  parallel_items(tokens * heads, nthreads, [&](int64_t row) {
    const T* x = core + row * dim;
    const T* zr = z + (row / heads) * z_stride + (row % heads) * dim;
    T sum_sq = 0;
    for (int64_t d = 0; d < dim; ++d) sum_sq += x[d] * x[d];
    const T inv = T(1) / std::sqrt(sum_sq / static_cast<T>(dim) + eps);
    for (int64_t d = 0; d < dim; ++d) {
      const T act = sigmoid_gate ? sigmoid_(zr[d]) : silu_(zr[d]);
      out[row * dim + d] = x[d] * inv * weight[d] * act;
    }
  });
}

}  // namespace

extern "C" {

float orc_sigmoid_f32(float x) { return sigmoid_(x); }
float orc_silu_f32(float x) { return silu_(x); }
float orc_softplus_f32(float x) { return softplus_(x); }
double orc_sigmoid_f64(double x) { return sigmoid_(x); }
double orc_silu_f64(double x) { return silu_(x); }
double orc_softplus_f64(double x) { return softplus_(x); }

int orc_validate_gated_delta_rule_shape(int64_t query_len, int64_t key_len, int64_t value_len,
                                        int64_t g_len, int64_t beta_len,
                                        int64_t initial_state_len, int64_t out_len,
                                        int64_t final_state_len, int64_t tokens,
                                        int64_t key_heads, int64_t value_heads,
                                        int64_t key_dim, int64_t value_dim, char* msg,
                                        size_t cap) {
  if (tokens <= 0 || key_heads <= 0 || value_heads <= 0 || key_dim <= 0 || value_dim <= 0) {
    set_msg(msg, cap,
            "gated_delta_rule shape must be positive, got tokens=" + std::to_string(tokens) +
                " key_heads=" + std::to_string(key_heads) +
                " value_heads=" + std::to_string(value_heads) +
                " key_dim=" + std::to_string(key_dim) +
                " value_dim=" + std::to_string(value_dim));
    return ORC_ERR_SHAPE;
  }
  if (value_heads % key_heads != 0) {
    set_msg(msg, cap,
            "gated_delta_rule value_heads " + std::to_string(value_heads) +
                " must be divisible by key_heads " + std::to_string(key_heads));
    return ORC_ERR_SHAPE;
  }
  const struct {
    const char* label;
    int64_t actual, expected;
  } rules[] = {
      {"query", query_len, tokens * key_heads * key_dim},
      {"key", key_len, tokens * key_heads * key_dim},
      {"value", value_len, tokens * value_heads * value_dim},
      {"g", g_len, tokens * value_heads},
      {"beta", beta_len, tokens * value_heads},
      {"initial_state", initial_state_len, value_heads * value_dim * key_dim},
      {"out", out_len, tokens * value_heads * value_dim},
      {"final_state", final_state_len, value_heads * value_dim * key_dim},
  };
  for (const auto& r : rules)
    if (r.actual < r.expected) {
      set_msg(msg, cap,
              std::string("gated_delta_rule ") + r.label + " length " +
                  std::to_string(r.actual) + " < expected " + std::to_string(r.expected));
      return ORC_ERR_SHAPE;
    }
  return ORC_OK;
}

int orc_validate_linear_attention_prepare_shape(
    int64_t mixed_len, int64_t conv_weight_len, int64_t a_raw_len, int64_t b_raw_len,
    int64_t a_log_len, int64_t dt_bias_len, int64_t query_len, int64_t key_len,
    int64_t value_len, int64_t g_len, int64_t beta_len, int64_t tokens, int64_t key_heads,
    int64_t value_heads, int64_t key_dim, int64_t value_dim, int64_t conv_kernel, char* msg,
    size_t cap) {
  if (tokens <= 0 || key_heads <= 0 || value_heads <= 0 || key_dim <= 0 || value_dim <= 0 ||
      conv_kernel <= 0) {
    set_msg(msg, cap,
            "linear_attention_prepare shape must be positive, got tokens=" +
                std::to_string(tokens) + " key_heads=" + std::to_string(key_heads) +
                " value_heads=" + std::to_string(value_heads) +
                " key_dim=" + std::to_string(key_dim) +
                " value_dim=" + std::to_string(value_dim) +
                " conv_kernel=" + std::to_string(conv_kernel));
    return ORC_ERR_SHAPE;
  }
  const int64_t qk_total = key_heads * key_dim, v_total = value_heads * value_dim;
  const int64_t channels = 2 * qk_total + v_total;
  const struct {
    const char* label;
    int64_t actual, expected;
  } rules[] = {
      {"mixed_qkv_raw", mixed_len, tokens * channels},
      {"conv_weight", conv_weight_len, channels * conv_kernel},
      {"a_raw", a_raw_len, tokens * value_heads},
      {"b_raw", b_raw_len, tokens * value_heads},
      {"a_log", a_log_len, value_heads},
      {"dt_bias", dt_bias_len, value_heads},
      {"query", query_len, tokens * qk_total},
      {"key", key_len, tokens * qk_total},
      {"value", value_len, tokens * v_total},
      {"g", g_len, tokens * value_heads},
      {"beta", beta_len, tokens * value_heads},
  };
  for (const auto& r : rules)
    if (r.actual < r.expected) {
      set_msg(msg, cap,
              std::string("linear_attention_prepare ") + r.label + " length " +
                  std::to_string(r.actual) + " < expected " + std::to_string(r.expected));
      return ORC_ERR_SHAPE;
    }
  return ORC_OK;
}

int orc_validate_linear_attention_decode_prepare_shape(
    int64_t mixed_len, int64_t conv_weight_len, int64_t conv_state_len, int64_t a_raw_len,
    int64_t b_raw_len, int64_t a_log_len, int64_t dt_bias_len, int64_t query_len,
    int64_t key_len, int64_t value_len, int64_t g_len, int64_t beta_len,
    int64_t next_conv_state_len, int64_t key_heads, int64_t value_heads, int64_t key_dim,
    int64_t value_dim, int64_t conv_kernel, char* msg, size_t cap) {
  if (key_heads <= 0 || value_heads <= 0 || key_dim <= 0 || value_dim <= 0 ||
      conv_kernel <= 0) {
    set_msg(msg, cap,
            "linear_attention_decode_prepare shape must be positive, got key_heads=" +
                std::to_string(key_heads) + " value_heads=" + std::to_string(value_heads) +
                " key_dim=" + std::to_string(key_dim) +
                " value_dim=" + std::to_string(value_dim) +
                " conv_kernel=" + std::to_string(conv_kernel));
    return ORC_ERR_SHAPE;
  }
  const int64_t qk_total = key_heads * key_dim, v_total = value_heads * value_dim;
  const int64_t channels = 2 * qk_total + v_total;
  const int64_t tail = channels * (conv_kernel - 1);
  const struct {
    const char* label;
    int64_t actual, expected;
  } rules[] = {
      {"mixed_qkv_raw", mixed_len, channels},
      {"conv_weight", conv_weight_len, channels * conv_kernel},
      {"conv_state", conv_state_len, tail},
      {"a_raw", a_raw_len, value_heads},
      {"b_raw", b_raw_len, value_heads},
      {"a_log", a_log_len, value_heads},
      {"dt_bias", dt_bias_len, value_heads},
      {"query", query_len, qk_total},
      {"key", key_len, qk_total},
      {"value", value_len, v_total},
      {"g", g_len, value_heads},
      {"beta", beta_len, value_heads},
      {"next_conv_state", next_conv_state_len, tail},
  };
  for (const auto& r : rules)
    if (r.actual < r.expected) {
      set_msg(msg, cap,
              std::string("linear_attention_decode_prepare ") + r.label + " length " +
                  std::to_string(r.actual) + " < expected " + std::to_string(r.expected));
      return ORC_ERR_SHAPE;
    }
  return ORC_OK;
}

int orc_validate_cu_seqlens(const int32_t* cu, int64_t batch, int64_t total, char* msg,
                            size_t cap) {
  if (batch <= 0 || total <= 0) {
    set_msg(msg, cap, "gated_delta_rule_varlen shape must be positive");
    return ORC_ERR_SHAPE;
  }
  return check_cu(cu, batch, total, msg, cap);
}

// [cpu.rs] linear_attention_prepare_varlen_f32: the same cu_seqlens rules
// under the prepare's label.
int orc_validate_prepare_cu_seqlens(const int32_t* cu, int64_t batch, int64_t total, char* msg,
                                    size_t cap) {
  if (batch <= 0 || total <= 0) {
    set_msg(msg, cap, "linear_attention_prepare_varlen shape must be positive");
    return ORC_ERR_SHAPE;
  }
  return check_cu(cu, batch, total, msg, cap, "linear_attention_prepare_varlen");
}

int orc_validate_state_indices(const int32_t* indices, int64_t n, int64_t slots,
                               int force_full, char* msg, size_t cap) {
  if (slots < 0) {
    set_msg(msg, cap, "GDN state cache has invalid slot count");
    return ORC_ERR_INVALID;
  }
  std::vector<unsigned char> seen(static_cast<size_t>(slots), 0);
  for (int64_t i = 0; i < n; ++i) {
    const int32_t slot = indices[i];
    if (slot < 0) {
      if (slot != -1) {
        set_msg(msg, cap, "invalid negative GDN state index");
        return ORC_ERR_INVALID;
      }
      continue;
    }
    if (slot >= slots) {
      set_msg(msg, cap, "GDN state index out of range");
      return ORC_ERR_INVALID;
    }
    if (seen[slot]) {
      set_msg(msg, cap, "duplicate live GDN state index");
      return ORC_ERR_INVALID;
    }
    seen[slot] = 1;
  }
  if (force_full) {
    for (int64_t i = 0; i < n; ++i) {
      if (indices[i] < 0) continue;
      for (int64_t j = 0; j < i; ++j)
        if (indices[j] == indices[i]) {
          set_msg(msg, cap, "duplicate live GDN state index");
          return ORC_ERR_INVALID;
        }
    }
  }
  return ORC_OK;
}

#define ORC_SPEC_PREP_PARAMS(R)                                                             \
  const R *mixed_qkv, int64_t x_stride, const R *conv_weight, R *conv_pool,                 \
      int64_t conv_slots, int64_t state_len, const int32_t *conv_indices,                   \
      const int32_t *num_accepted, const R *a_raw, int64_t a_stride, const R *b_raw,        \
      int64_t b_stride, const R *A_log, const R *dt_bias, const int32_t *cu_seqlens,        \
      int64_t n_reqs, int64_t tokens, int64_t key_heads, int64_t value_heads,               \
      int64_t key_dim, int64_t value_dim, int64_t conv_kernel, int apply_qk_l2norm,         \
      R *query, R *key, R *value, R *g, R *beta, int nthreads
#define ORC_SPEC_PREP_ARGS                                                                  \
  mixed_qkv, x_stride, conv_weight, conv_pool, conv_slots, state_len, conv_indices,         \
      num_accepted, a_raw, a_stride, b_raw, b_stride, A_log, dt_bias, cu_seqlens, n_reqs,   \
      tokens, key_heads, value_heads, key_dim, value_dim, conv_kernel, apply_qk_l2norm,     \
      query, key, value, g, beta, nthreads
int orc_spec_prepare_f32(ORC_SPEC_PREP_PARAMS(float)) {
  return spec_prepare_impl<float>(ORC_SPEC_PREP_ARGS);
}
int orc_spec_prepare_f64(ORC_SPEC_PREP_PARAMS(double)) {
  return spec_prepare_impl<double>(ORC_SPEC_PREP_ARGS);
}

int orc_prepare_varlen_f32(ORC_PREPARE_PARAMS(float)) {
  return prepare_impl<float>(mixed_qkv, x_stride, conv_weight, conv_pool, conv_slots,
                             state_indices, has_initial_state, a_raw, a_stride, b_raw, b_stride,
                             a_log, dt_bias, cu_seqlens, n_seqs, tokens, key_heads, value_heads,
                             key_dim, value_dim, conv_kernel, apply_qk_l2norm, query, key, value,
                             g, beta, nthreads);
}
int orc_prepare_varlen_f64(ORC_PREPARE_PARAMS(double)) {
  return prepare_impl<double>(mixed_qkv, x_stride, conv_weight, conv_pool, conv_slots,
                              state_indices, has_initial_state, a_raw, a_stride, b_raw, b_stride,
                              a_log, dt_bias, cu_seqlens, n_seqs, tokens, key_heads,
                              value_heads, key_dim, value_dim, conv_kernel, apply_qk_l2norm,
                              query, key, value, g, beta, nthreads);
}

int orc_gdn_varlen_f32(ORC_RECUR_PARAMS(float)) {
  return varlen_impl<float>(query, key, value, g, beta, state_pool, state_slots, state_indices,
                            has_initial_state, cu_seqlens, n_seqs, tokens, key_heads,
                            value_heads, key_dim, value_dim, scale, use_qk_l2norm, items,
                            n_items, out, nthreads);
}
int orc_gdn_varlen_f64(ORC_RECUR_PARAMS(double)) {
  return varlen_impl<double>(query, key, value, g, beta, state_pool, state_slots, state_indices,
                             has_initial_state, cu_seqlens, n_seqs, tokens, key_heads,
                             value_heads, key_dim, value_dim, scale, use_qk_l2norm, items,
                             n_items, out, nthreads);
}

int orc_gdn_deviation_bound_f64(const double* q, const double* k, const double* v,
                                const double* g, const double* beta, const double* dq,
                                const double* dk, const double* dv, const double* state_pool,
                                int64_t state_slots, const int32_t* state_indices,
                                const uint8_t* has_initial_state, const int32_t* cu_seqlens,
                                int64_t n_seqs, int64_t tokens, int64_t key_heads,
                                int64_t value_heads, int64_t key_dim, int64_t value_dim,
                                double scale, double* bound, double* state_bound,
                                int nthreads) {
  if (n_seqs <= 0 || tokens <= 0 || key_heads <= 0 || value_heads <= 0 || key_dim <= 0 ||
      value_dim <= 0 || value_heads % key_heads != 0)
    return ORC_ERR_SHAPE;
  if (int rc = check_cu(cu_seqlens, n_seqs, tokens, nullptr, 0)) return rc;
  if (int rc = check_slots(state_indices, n_seqs, state_slots, nullptr, 0)) return rc;
  const int64_t ratio = value_heads / key_heads, state_len = value_dim * key_dim;
  parallel_items(n_seqs * value_heads, nthreads, [&](int64_t item) {
    const int64_t s = item / value_heads, h = item % value_heads;
    const int64_t slot = state_indices != nullptr ? state_indices[s] : s;
    if (slot < 0) {  // padded: outputs are zeros on both sides
      for (int64_t t = cu_seqlens[s]; t < cu_seqlens[s + 1]; ++t)
        for (int64_t c = 0; c < value_dim; ++c) bound[(t * value_heads + h) * value_dim + c] = 0.0;
      return;
    }
    std::vector<double> S(state_len, 0.0);
    if (has_initial_state == nullptr || has_initial_state[s] != 0)
      for (int64_t e = 0; e < state_len; ++e)
        S[e] = state_pool[(slot * value_heads + h) * state_len + e];
    deviation_chain(q, k, v, g, beta, dq, dk, dv, S, cu_seqlens[s], cu_seqlens[s + 1], h,
                    h / ratio, key_heads, value_heads, key_dim, value_dim, scale, bound,
                    state_bound != nullptr
                        ? state_bound + (slot * value_heads + h) * value_dim
                        : nullptr);
  });
  return ORC_OK;
}

int orc_kda_varlen_f32(ORC_RECUR_PARAMS(float)) {
  if (use_qk_l2norm != 0) return ORC_ERR_INVALID;  // KDA uses q, k as given
  return varlen_impl<float>(query, key, value, g, beta, state_pool, state_slots, state_indices,
                            has_initial_state, cu_seqlens, n_seqs, tokens, key_heads,
                            value_heads, key_dim, value_dim, scale, 0, items, n_items, out,
                            nthreads, true);
}
int orc_kda_varlen_f64(ORC_RECUR_PARAMS(double)) {
  if (use_qk_l2norm != 0) return ORC_ERR_INVALID;
  return varlen_impl<double>(query, key, value, g, beta, state_pool, state_slots, state_indices,
                             has_initial_state, cu_seqlens, n_seqs, tokens, key_heads,
                             value_heads, key_dim, value_dim, scale, 0, items, n_items, out,
                             nthreads, true);
}

#define ORC_SPEC_PARAMS(R)                                                                  \
  const R *query, const R *key, const R *value, const R *g, const R *beta, R *state_pool,   \
      int64_t state_slots, const int32_t *cu_seqlens, int64_t n_reqs, int64_t tokens,       \
      const int32_t *state_indices, int64_t num_cols, const int32_t *num_accepted,          \
      int64_t key_heads, int64_t value_heads, int64_t key_dim, int64_t value_dim, R scale,  \
      R *out, int nthreads
int orc_gdn_spec_decode_f32(ORC_SPEC_PARAMS(float)) {
  return spec_decode_impl<float>(query, key, value, g, beta, state_pool, state_slots, cu_seqlens,
                                 n_reqs, tokens, state_indices, num_cols, num_accepted,
                                 key_heads, value_heads, key_dim, value_dim, scale, out,
                                 nthreads);
}
int orc_gdn_spec_decode_f64(ORC_SPEC_PARAMS(double)) {
  return spec_decode_impl<double>(query, key, value, g, beta, state_pool, state_slots,
                                  cu_seqlens, n_reqs, tokens, state_indices, num_cols,
                                  num_accepted, key_heads, value_heads, key_dim, value_dim,
                                  scale, out, nthreads);
}

int orc_gdn_decode_f32(ORC_DECODE_PARAMS(float)) {
  return decode_impl<float>(query, key, value, g, beta, state_pool, state_slots, state_indices,
                            batch, key_heads, value_heads, key_dim, value_dim, scale,
                            use_qk_l2norm, out, nthreads);
}
int orc_gdn_decode_f64(ORC_DECODE_PARAMS(double)) {
  return decode_impl<double>(query, key, value, g, beta, state_pool, state_slots, state_indices,
                             batch, key_heads, value_heads, key_dim, value_dim, scale,
                             use_qk_l2norm, out, nthreads);
}

int orc_gdn_chunked_f64(const double* q, const double* k, const double* v, const double* g,
                        const double* beta, double* pool, int64_t slots, const int32_t* sidx,
                        const uint8_t* has_init, const int32_t* cu, int64_t n_seqs,
                        int64_t tokens, int64_t hk_n, int64_t hv_n, int64_t dk, int64_t dv,
                        double scale, int use_norm, int64_t chunk, double* out) {
  if (n_seqs <= 0 || tokens <= 0 || hk_n <= 0 || hv_n <= 0 || dk <= 0 || dv <= 0 || chunk <= 0)
    return ORC_ERR_SHAPE;
  if (hv_n % hk_n != 0) return ORC_ERR_SHAPE;
  if (int rc = check_cu(cu, n_seqs, tokens, nullptr, 0)) return rc;
  if (int rc = check_slots(sidx, n_seqs, slots, nullptr, 0)) return rc;
  const int64_t ratio = hv_n / hk_n;
  for (int64_t s = 0; s < n_seqs; ++s)
    for (int64_t h = 0; h < hv_n; ++h) {
      const int64_t slot = sidx != nullptr ? sidx[s] : s;
      if (slot < 0) {
        for (int64_t t = cu[s]; t < cu[s + 1]; ++t)
          for (int64_t d = 0; d < dv; ++d) out[(t * hv_n + h) * dv + d] = 0.0;
        continue;
      }
      double* S = pool + (slot * hv_n + h) * dv * dk;
      if (has_init != nullptr && has_init[s] == 0)
        for (int64_t e = 0; e < dv * dk; ++e) S[e] = 0.0;
      const int64_t hk = h / ratio;
      for (int64_t c0 = cu[s]; c0 < cu[s + 1]; c0 += chunk) {
        const int64_t L = std::min<int64_t>(chunk, cu[s + 1] - c0);
        std::vector<double> Kc(L * dk), Qc(L * dk), Vc(L * dv), gc(L), bc(L), Oc;
        for (int64_t i = 0; i < L; ++i) {
          const int64_t t = c0 + i;
          const double* qt = q + (t * hk_n + hk) * dk;
          const double* kt = k + (t * hk_n + hk) * dk;
          double qi = 1.0, ki = 1.0;
          if (use_norm) {
            double qn = 0.0, kn = 0.0;
            for (int64_t d = 0; d < dk; ++d) {
              qn += qt[d] * qt[d];
              kn += kt[d] * kt[d];
            }
            qi = 1.0 / std::sqrt(qn + 1e-6);
            ki = 1.0 / std::sqrt(kn + 1e-6);
          }
          for (int64_t d = 0; d < dk; ++d) {
            Kc[i * dk + d] = kt[d] * ki;
            Qc[i * dk + d] = qt[d] * qi * scale;
          }
          for (int64_t d = 0; d < dv; ++d) Vc[i * dv + d] = v[(t * hv_n + h) * dv + d];
          gc[i] = g[t * hv_n + h];
          bc[i] = beta[t * hv_n + h];
        }
        chunk_step(Kc, Qc, Vc, gc, bc, L, dk, dv, S, Oc);
        for (int64_t i = 0; i < L; ++i)
          for (int64_t d = 0; d < dv; ++d) out[((c0 + i) * hv_n + h) * dv + d] = Oc[i * dv + d];
      }
    }
  return ORC_OK;
}

int orc_kda_chunked_f64(const double* q, const double* k, const double* v, const double* g,
                        const double* beta, double* pool, int64_t slots, const int32_t* sidx,
                        const uint8_t* has_init, const int32_t* cu, int64_t n_seqs,
                        int64_t tokens, int64_t hk_n, int64_t hv_n, int64_t dk, int64_t dv,
                        double scale, int64_t chunk, double* out) {
  if (n_seqs <= 0 || tokens <= 0 || hk_n <= 0 || hv_n <= 0 || dk <= 0 || dv <= 0 || chunk <= 0)
    return ORC_ERR_SHAPE;
  if (hv_n % hk_n != 0) return ORC_ERR_SHAPE;
  if (int rc = check_cu(cu, n_seqs, tokens, nullptr, 0)) return rc;
  if (int rc = check_slots(sidx, n_seqs, slots, nullptr, 0)) return rc;
  const int64_t ratio = hv_n / hk_n;
  for (int64_t s = 0; s < n_seqs; ++s)
    for (int64_t h = 0; h < hv_n; ++h) {
      const int64_t slot = sidx != nullptr ? sidx[s] : s;
      if (slot < 0) {
        for (int64_t t = cu[s]; t < cu[s + 1]; ++t)
          for (int64_t d = 0; d < dv; ++d) out[(t * hv_n + h) * dv + d] = 0.0;
        continue;
      }
      double* S = pool + (slot * hv_n + h) * dv * dk;
      if (has_init != nullptr && has_init[s] == 0)
        for (int64_t e = 0; e < dv * dk; ++e) S[e] = 0.0;
      const int64_t hk = h / ratio;
      for (int64_t c0 = cu[s]; c0 < cu[s + 1]; c0 += chunk) {
        const int64_t L = std::min<int64_t>(chunk, cu[s + 1] - c0);
        std::vector<double> Kc(L * dk), Qc(L * dk), Vc(L * dv), Gc(L * dk), bc(L), Oc;
        for (int64_t i = 0; i < L; ++i) {
          const int64_t t = c0 + i;
          for (int64_t d = 0; d < dk; ++d) {
            Kc[i * dk + d] = k[(t * hk_n + hk) * dk + d];
            Qc[i * dk + d] = q[(t * hk_n + hk) * dk + d] * scale;
            Gc[i * dk + d] = g[(t * hv_n + h) * dk + d];
          }
          for (int64_t d = 0; d < dv; ++d) Vc[i * dv + d] = v[(t * hv_n + h) * dv + d];
          bc[i] = beta[t * hv_n + h];
        }
        kda_chunk_step(Kc, Qc, Vc, Gc, bc, L, dk, dv, S, Oc);
        for (int64_t i = 0; i < L; ++i)
          for (int64_t d = 0; d < dv; ++d) out[((c0 + i) * hv_n + h) * dv + d] = Oc[i * dv + d];
      }
    }
  return ORC_OK;
}

int orc_validate_gated_rms_norm_shape(int64_t core_len, int64_t z_len, int64_t weight_len,
                                      int64_t out_len, int64_t tokens, int64_t heads,
                                      int64_t dim, char* msg, size_t cap) {
  if (tokens <= 0 || heads <= 0 || dim <= 0) {
    set_msg(msg, cap,
            "gated_rms_norm shape must be positive, got tokens=" + std::to_string(tokens) +
                " heads=" + std::to_string(heads) + " dim=" + std::to_string(dim));
    return ORC_ERR_SHAPE;
  }
  const int64_t expected = tokens * heads * dim;
  const struct {
    const char* label;
    int64_t actual, expected;
  } rules[] = {{"core", core_len, expected},
               {"z", z_len, expected},
               {"weight", weight_len, dim},
               {"out", out_len, expected}};
  for (const auto& r : rules)
    if (r.actual < r.expected) {
      set_msg(msg, cap,
              std::string("gated_rms_norm ") + r.label + " length " + std::to_string(r.actual) +
                  " < expected " + std::to_string(r.expected));
      return ORC_ERR_SHAPE;
    }
  return ORC_OK;
}

#define ORC_GRN_PARAMS(T)                                                                   \
  const T *core, const T *z, int64_t z_stride, const T *weight, T *out, int64_t tokens,    \
      int64_t heads, int64_t dim, T eps, int sigmoid_gate, int nthreads
int orc_gated_rmsnorm_f32(ORC_GRN_PARAMS(float)) {
  gated_rmsnorm_<float>(core, z, z_stride, weight, out, tokens, heads, dim, eps,
                        sigmoid_gate != 0, nthreads);
  return ORC_OK;
}
int orc_gated_rmsnorm_f64(ORC_GRN_PARAMS(double)) {
  gated_rmsnorm_<double>(core, z, z_stride, weight, out, tokens, heads, dim, eps,
                         sigmoid_gate != 0, nthreads);
  return ORC_OK;
}

}  // extern "C"
