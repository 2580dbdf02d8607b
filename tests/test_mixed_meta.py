"""The mixed-step metadata contract, checked on the host before any launch.

[qwen3_5.cpp] (vllm.cpp, src/vllm/model_executor/models/qwen3_5.cpp)
ValidateGdnAttentionMetadata fixes how one packed step is split: the decode
rows come first and hold one token each, the prefill sequences follow, and the
prefill call's cu_seqlens is the suffix of the full cu_seqlens rebased to 0
(SubView of the prefill rows).  The C ABI's gdn_validate_mixed applies those
rules, with the page's messages; each case below breaks one rule and expects
the page's message for it.  Nothing here needs a GPU: the validator is host
code and raises before any launch.
"""
import pytest
import torch

from gated_delta_rule_44_gb300 import binding as B
from gated_delta_rule_44_gb300 import layer


def meta(**over):
    # 3 decodes (slots 5, -1, 2), then prefills of 4 and 6 tokens (slots 0, 7)
    m = dict(num_decodes=3, num_prefills=2, num_actual_tokens=13, state_slots=8,
             cu_seqlens_host=torch.tensor([0, 1, 2, 3, 7, 13], dtype=torch.int32),
             state_indices_host=torch.tensor([5, -1, 2, 0, 7], dtype=torch.int32),
             has_initial_state_host=torch.tensor([1, 1, 1, 0, 1], dtype=torch.uint8),
             cu_seqlens_prefill_host=torch.tensor([0, 4, 10], dtype=torch.int32))
    m.update(over)
    return m


def rejects(msg, **over):
    with pytest.raises(B.GdnError) as ei:
        B.gdn_validate_mixed(**meta(**over))
    assert ei.value.code == B.GDN_ERR_INVALID_ARGUMENT
    assert ei.value.msg == msg


def test_valid_step_passes():
    B.gdn_validate_mixed(**meta())
    # decode-only and prefill-only steps
    B.gdn_validate_mixed(**meta(num_prefills=0, num_actual_tokens=3, cu_seqlens_prefill_host=None,
                                cu_seqlens_host=torch.tensor([0, 1, 2, 3], dtype=torch.int32),
                                state_indices_host=torch.tensor([5, -1, 2], dtype=torch.int32),
                                has_initial_state_host=None))
    B.gdn_validate_mixed(**meta(num_decodes=0, num_actual_tokens=10,
                                cu_seqlens_host=torch.tensor([0, 4, 10], dtype=torch.int32),
                                state_indices_host=torch.tensor([0, 7], dtype=torch.int32),
                                has_initial_state_host=torch.tensor([0, 1], dtype=torch.uint8)))
    # the prefill-only arrays given explicitly, equal to the suffixes
    B.gdn_validate_mixed(**meta(prefill_state_indices_host=torch.tensor([0, 7], dtype=torch.int32),
                                prefill_has_initial_state_host=torch.tensor([0, 1],
                                                                            dtype=torch.uint8)))


def test_wrong_rebase_is_rejected():
    # the prefill offsets left un-rebased (still counting the 3 decode tokens)
    rejects("prefill query offsets must match rebased non-spec suffix",
            cu_seqlens_prefill_host=torch.tensor([3, 7, 13], dtype=torch.int32))
    # rebased by the wrong amount
    rejects("prefill query offsets must match rebased non-spec suffix",
            cu_seqlens_prefill_host=torch.tensor([0, 5, 10], dtype=torch.int32))


def test_prefill_offsets_must_span_prefill_tokens():
    rejects("prefill query offsets must span prefill tokens",
            cu_seqlens_prefill_host=torch.tensor([0, 4, 9], dtype=torch.int32))


def test_decode_rows_are_single_token_and_first():
    # a 2-token "decode" row: the decode prefix no longer ends at token 3
    rejects("non-spec GDN decode prefix does not match token count",
            cu_seqlens_host=torch.tensor([0, 1, 3, 4, 7, 13], dtype=torch.int32),
            cu_seqlens_prefill_host=torch.tensor([0, 3, 9], dtype=torch.int32),
            num_actual_tokens=13)
    rejects("non-spec decode requires one token per request", num_decode_tokens=4,
            num_prefill_tokens=9)


def test_token_counts_must_add_up():
    rejects("GDN decode+prefill+spec tokens must equal actual tokens", num_prefill_tokens=9)
    rejects("negative GDN metadata count", num_prefills=-1)
    rejects("GDN tokens require state metadata", num_decodes=0, num_prefills=0,
            num_actual_tokens=4, num_prefill_tokens=4)


def test_offsets_span_and_increase():
    rejects("non-spec GDN query offsets must span the non-spec tokens",
            cu_seqlens_host=torch.tensor([0, 1, 2, 3, 7, 12], dtype=torch.int32))
    rejects("non-spec GDN query offsets must be strictly increasing",
            cu_seqlens_host=torch.tensor([0, 1, 1, 3, 7, 13], dtype=torch.int32))


def test_index_rules():
    rejects("prefill state indices must match non-spec suffix",
            prefill_state_indices_host=torch.tensor([0, 6], dtype=torch.int32))
    rejects("prefill GDN state index must be non-negative",
            state_indices_host=torch.tensor([5, -1, 2, -1, 7], dtype=torch.int32))
    rejects("duplicate live GDN state index",
            state_indices_host=torch.tensor([5, -1, 2, 5, 7], dtype=torch.int32))
    rejects("GDN state index out of range",
            state_indices_host=torch.tensor([5, -1, 2, 0, 8], dtype=torch.int32))
    rejects("live GDN state index must be non-negative", allow_inert_padding=False)
    rejects("missing non-spec GDN state indices", state_indices_host=None)
    rejects("incomplete GDN prefill metadata", cu_seqlens_prefill_host=None)


def test_initial_state_mask_must_match_suffix():
    rejects("prefill initial-state mask must match non-spec suffix",
            prefill_has_initial_state_host=torch.tensor([1, 1], dtype=torch.uint8))


def test_step_helper_rejects_a_wrong_rebase_before_launching():
    """GdnStep.run checks the host copies first: with a mis-rebased prefill
    cu_seqlens it raises the page's message and launches nothing (here the
    buffers are CPU tensors, so any launch would fail differently)."""
    m = meta()
    step = layer.GdnStep(13, 5, 3, 1, 2, 128, 128, 4, torch.bfloat16, "cpu")
    before = B.gdn_launch_count()
    dummy = torch.zeros(1)
    with pytest.raises(B.GdnError) as ei:
        step.run(dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                 torch.zeros(8, 2, 128, 128), dummy, dummy,
                 cu_seqlens_host=m["cu_seqlens_host"],
                 state_indices_host=m["state_indices_host"],
                 has_initial_state_host=m["has_initial_state_host"],
                 cu_seqlens_prefill_host=torch.tensor([3, 7, 13], dtype=torch.int32))
    assert ei.value.msg == "prefill query offsets must match rebased non-spec suffix"
    assert B.gdn_launch_count() == before
    with pytest.raises(B.GdnError) as ei:
        step.run(dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                 torch.zeros(8, 2, 128, 128), dummy, dummy,
                 cu_seqlens_host=m["cu_seqlens_host"], state_indices_host=m["state_indices_host"])
    assert ei.value.msg == "incomplete GDN prefill metadata"
