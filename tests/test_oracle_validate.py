"""Pins of the oracle's validators against the texts and rules the pages print.

Shape rules and message formats: [cpu.rs] (ferrum-kernels 0.8.0,
src/ferrum_kernels/backend/cpu.rs) validate_gated_delta_rule_shape,
validate_linear_attention_prepare_shape,
validate_linear_attention_decode_prepare_shape and the cu_seqlens checks of
recurrent_gated_delta_rule_varlen_f32; the expected texts live in
tests/golden/validate_messages.txt, formatted from those format strings.
Index rules: [qwen3_5.cpp] (vllm.cpp, src/vllm/model_executor/models/
qwen3_5.cpp) ValidateGdnStateIndices (-1 the only negative, live slot in
range, no duplicate live slot; the O(n^2) re-check agrees with the seen-set).
"""
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def golden():
    out = {}
    with open(os.path.join(HERE, "golden", "validate_messages.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split("|", 1)
            out[k.strip()] = v.strip()
    return out


G = golden()


def gdr(**over):
    # tokens=2, Hk=1, Hv=2, Dk=3, Dv=2: q,k 6; v 8; g,beta 4; state 12; out 8
    a = dict(query=6, key=6, value=8, g=4, beta=4, init=12, out=8, final=12, T=2, Hk=1, Hv=2,
             Dk=3, Dv=2)
    a.update(over)
    return oracle.validate_gated_delta_rule_shape(a["query"], a["key"], a["value"], a["g"],
                                                  a["beta"], a["init"], a["out"], a["final"],
                                                  a["T"], a["Hk"], a["Hv"], a["Dk"], a["Dv"])


def test_gdr_ok():
    assert gdr() == (0, "")


@pytest.mark.parametrize("case,over", [
    ("gdr_query_short", dict(query=5)),
    ("gdr_beta_short", dict(beta=3)),
    ("gdr_final_short", dict(final=11)),
    ("gdr_not_positive", dict(T=0)),
    ("gdr_gqa", dict(Hk=2, Hv=3)),
])
def test_gdr_messages(case, over):
    rc, msg = gdr(**over)
    assert rc == oracle.ORC_ERR_SHAPE
    assert msg == G[case]


def test_gdr_first_failing_label_wins():
    # lengths are checked in the printed order: query before key before value
    rc, msg = gdr(query=0, key=0)
    assert msg.startswith("gated_delta_rule query ")


def prep(**over):
    # T=1, Hk=1, Hv=1, Dk=1, Dv=1 -> C=3; K=... channel counts
    a = dict(mixed=3, w=6, a=1, b=1, alog=1, dt=1, q=1, k=1, v=1, g=1, beta=1, T=1, Hk=1, Hv=1,
             Dk=1, Dv=1, K=2)
    a.update(over)
    return oracle.validate_linear_attention_prepare_shape(
        a["mixed"], a["w"], a["a"], a["b"], a["alog"], a["dt"], a["q"], a["k"], a["v"], a["g"],
        a["beta"], a["T"], a["Hk"], a["Hv"], a["Dk"], a["Dv"], a["K"])


def test_prepare_messages():
    assert prep() == (0, "")
    rc, msg = prep(Hk=2, mixed=5, w=9, q=2, k=2, K=2)
    # C = 2*2 + 1 = 5 channels, K = 2 -> conv_weight needs 10
    assert rc == oracle.ORC_ERR_SHAPE and msg == G["prep_conv_weight_short"]
    rc, msg = prep(K=0)
    assert msg == G["prep_not_positive"]


def test_prepare_does_not_check_gqa():
    # the prepare validator never checks Hv % Hk (the pages' rule set)
    rc, _ = prep(Hk=2, Hv=3, mixed=2 * 2 + 3, w=(2 * 2 + 3) * 2, a=3, b=3, alog=3, dt=3, q=2, k=2,
                 v=3, g=3, beta=3)
    assert rc == 0


def test_decode_prepare_message():
    # C = 2*1*1 + 1*2 = 4 channels, K = 3 -> conv tails need 4*2 = 8
    rc, msg = oracle.validate_linear_attention_decode_prepare_shape(
        4, 12, 8, 1, 1, 1, 1, 1, 1, 2, 1, 1, 7, 1, 1, 1, 2, 3)
    assert rc == oracle.ORC_ERR_SHAPE and msg == G["dprep_next_conv_state_short"]


def test_cu_seqlens_messages():
    rc, msg = oracle.validate_cu_seqlens([0, 2, 4], 2, 5)
    assert rc == oracle.ORC_ERR_INVALID and msg == G["cu_bounds"]
    rc, msg = oracle.validate_cu_seqlens([0, 2, 2, 5], 3, 5)
    assert rc == oracle.ORC_ERR_INVALID and msg == G["cu_empty"]
    assert oracle.validate_cu_seqlens([0, 1, 5], 2, 5) == (0, "")
    rc, _ = oracle.validate_cu_seqlens([0, 3, 2, 5], 3, 5)
    assert rc == oracle.ORC_ERR_INVALID


def test_prepare_cu_seqlens_messages():
    rc, msg = oracle.validate_prepare_cu_seqlens([1, 3, 7], 2, 7)
    assert rc == oracle.ORC_ERR_INVALID and msg == G["prep_cu_bounds"]
    rc, msg = oracle.validate_prepare_cu_seqlens([0, 0, 7], 2, 7)
    assert rc == oracle.ORC_ERR_INVALID and msg == G["prep_cu_empty"]
    assert oracle.validate_prepare_cu_seqlens([0, 3, 7], 2, 7) == (0, "")


@pytest.mark.parametrize("idx,slots,ok,frag", [
    ([0, 1, 2], 3, True, ""),
    ([-1, 2, -1, 0], 3, True, ""),
    ([0, -2], 3, False, "invalid negative"),
    ([0, 3], 3, False, "out of range"),
    ([1, 0, 1], 3, False, "duplicate live"),
    ([], 0, True, ""),
])
def test_state_indices(idx, slots, ok, frag):
    for full in (False, True):
        rc, msg = oracle.validate_state_indices(np.array(idx, np.int32), slots, force_full=full)
        assert (rc == 0) == ok
        assert frag in msg


def test_state_indices_full_recheck_agrees():
    rng = np.random.default_rng(0)
    for _ in range(200):
        n = int(rng.integers(1, 12))
        idx = rng.integers(-1, 8, size=n).astype(np.int32)
        a = oracle.validate_state_indices(idx, 8, force_full=False)[0]
        b = oracle.validate_state_indices(idx, 8, force_full=True)[0]
        live = idx[idx >= 0]
        assert a == b == (0 if len(set(live.tolist())) == len(live) else oracle.ORC_ERR_INVALID)
