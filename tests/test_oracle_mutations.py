"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of oracle/gdn_oracle.cpp (on
the CPU), builds it with the oracle's flags, routes the oracle wrapper to that
build and checks that the named pin now fails.  The mistakes are the kinds a
restatement of the pages could make: a dropped or misplaced decay, a flipped
sign, a swapped operand, a wrong GQA index, reversed conv taps, a wrong tail
window, eps outside the sqrt, a wrong sigmoid branch or softplus threshold, a
dropped factor in the chunked form, a gated norm over the sum instead of the
mean, swapped gates or unstrided gate rows, a KDA decay taken from one channel
or applied after the dot, a speculative decode that starts from the wrong
column, stores each snapshot one column late or loses the state at a -1 column, a
speculative conv window read one tap late, a conv row shifted by the
request length instead of one tap, a chunked KDA form without its decay in W.
"""
import os

import numpy as np
import pytest

import oracle
import test_oracle_gated_norm as N
import test_oracle_kda as KD
import test_oracle_gates as G
import test_oracle_prepare as P
import test_oracle_recurrence as R
import test_oracle_spec_decode as SD
import test_oracle_spec_prepare as SP

MUTATIONS = [
    ("decay_after_dot",
     "        row[d] *= decay;\n        kv_mem += row[d] * (kt[d] * k_inv);",
     "        kv_mem += row[d] * (kt[d] * k_inv);\n        row[d] *= decay;",
     [R.test_matches_householder_form]),
    ("delta_sign",
     "(v[(t * hv_n + h) * dv + vd] - kv_mem) * beta_t",
     "(kv_mem - v[(t * hv_n + h) * dv + vd]) * beta_t",
     [R.test_matches_householder_form, R.test_exact_overwrite_with_orthonormal_keys]),
    ("k_instead_of_q_in_output",
     "acc += row[d] * (qt[d] * q_inv * scale)",
     "acc += row[d] * (kt[d] * q_inv * scale)",
     [R.test_matches_householder_form]),
    ("gqa_modulo",
     "      head_chain(q, k, v, g, beta, S, cu[s], cu[s + 1], h, h / ratio,",
     "      head_chain(q, k, v, g, beta, S, cu[s], cu[s + 1], h, h % hk_n,",
     [R.test_gqa_mapping]),
    ("conv_taps_reversed",
     "acc += tap(lt + j - width) * w[c * kw + j];",
     "acc += tap(lt + j - width) * w[c * kw + (kw - 1 - j)];",
     [P.test_conv_matches_numpy_convolve, P.test_impulse_response_reverses_taps]),
    ("tail_window",
     "tail_row[pos] = tap(len + pos - width);",
     "tail_row[pos] = tap(pos - width);",
     [P.test_new_tail_is_last_inputs]),
    ("norm_eps_outside_sqrt",
     "const R q_inv = R(1) / std::sqrt(q_sum + R(1e-6));",
     "const R q_inv = R(1) / (std::sqrt(q_sum) + R(1e-6));",
     [P.test_l2_norm_closed_form]),
    ("sigmoid_negative_branch",
     "  return z / (R(1) + z);",
     "  return R(1) / (R(1) + z);",
     [G.test_sigmoid_matches_expit]),
    ("softplus_threshold",
     "if (x > R(20)) return x;",
     "if (x > R(2)) return x;",
     [G.test_softplus_matches_logaddexp]),
    ("gated_norm_sum_not_mean",
     "std::sqrt(sum_sq / static_cast<T>(dim) + eps)",
     "std::sqrt(sum_sq + eps)",
     [lambda: N.test_unit_rms_without_eps(False)]),
    ("gated_norm_eps_outside_sqrt",
     "std::sqrt(sum_sq / static_cast<T>(dim) + eps)",
     "(std::sqrt(sum_sq / static_cast<T>(dim)) + eps)",
     [N.test_constant_row_closed_form]),
    ("gated_norm_gates_swapped",
     "sigmoid_gate ? sigmoid_(zr[d]) : silu_(zr[d])",
     "sigmoid_gate ? silu_(zr[d]) : sigmoid_(zr[d])",
     [N.test_constant_row_closed_form]),
    ("gated_norm_gate_rows_unstrided",
     "z + (row / heads) * z_stride + (row % heads) * dim",
     "z + row * dim",
     [N.test_strided_gate_rows]),
    ("kda_decay_of_channel_0",
     "decay[d] = std::exp(g_row[d]);",
     "decay[d] = std::exp(g_row[0]);",
     [KD.test_key_channel_permutation]),
    ("kda_decay_after_dot",
     "        row[d] *= decay[d];\n        dot += row[d] * kbuf[d];",
     "        dot += row[d] * kbuf[d];\n        row[d] *= decay[d];",
     [lambda: KD.test_uniform_channel_decay_is_gdn(np.float64)]),
    ("spec_initial_column_off_by_one",
     "const int32_t init = sidx[i * num_cols + (num_accepted[i] - 1)];",
     "const int32_t init = sidx[i * num_cols + (num_accepted[i] % num_cols)];",
     [SD.test_initial_slot_is_column_of_last_accepted]),
    ("spec_snapshot_one_column_late",
     "const int32_t slot = sidx[i * num_cols + (t - lo)];",
     "const int32_t slot = sidx[i * num_cols + (t - lo + 1) % num_cols];",
     [SD.test_brute_force_tiny]),
    ("spec_null_column_resets_state",
     "      if (slot < 0) continue;\n      std::copy(",
     "      if (slot < 0) { std::fill(S.begin(), S.end(), R(0)); continue; }\n      std::copy(",
     [SD.test_null_initial_slot_and_null_columns]),
    ("spec_conv_window_one_tap_late",
     "for (int64_t j = 0; j < width; ++j) stream[j] = old_at(off + j);",
     "for (int64_t j = 0; j < width; ++j) stream[j] = old_at(off + 1 + j);",
     [lambda: SP.test_outputs_are_the_convolution_of_the_accepted_history(4)]),
    ("spec_conv_row_shift_by_len",
     "for (int64_t j = 0; j < keep; ++j) next[j] = old_at(off + 1 + j);",
     "for (int64_t j = 0; j < keep; ++j) next[j] = old_at(off + len + j);",
     [lambda: SP.test_outputs_are_the_convolution_of_the_accepted_history(4)]),
    ("kda_chunked_drops_decay_in_W",
     "W[i * dk + d] += t * Kc[j * dk + d] * std::exp(gam[j * dk + d]);",
     "W[i * dk + d] += t * Kc[j * dk + d];",
     [lambda: KD.test_chunked_form_equals_recurrence(16, False)]),
    ("chunked_drops_decay_in_W",
     "const double tw = T[i * L + j] * bc[j] * std::exp(gam[j]);",
     "const double tw = T[i * L + j] * bc[j];",
     [lambda: R.test_chunked_equals_sequential(65, 16)]),
]


@pytest.fixture(scope="module")
def variants(tmp_path_factory):
    src = oracle.source_text()
    built = {}
    for name, old, new, _ in MUTATIONS:
        assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
        d = tmp_path_factory.mktemp(name)
        built[name] = oracle.build_variant(src.replace(old, new), str(d))
    return built


def test_unmutated_copy_passes(tmp_path):
    path = oracle.build_variant(oracle.source_text(), str(tmp_path))
    with oracle.using_library(path):
        R.test_matches_householder_form()
        P.test_conv_matches_numpy_convolve()
        G.test_sigmoid_matches_expit()


@pytest.mark.parametrize("case", range(len(MUTATIONS)), ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(case, variants):
    name, _, _, pins = MUTATIONS[case]
    with oracle.using_library(variants[name]):
        for pin in pins:
            with pytest.raises(AssertionError):
                pin()
