"""The C-ABI library builds, loads and exports every symbol include/gdn.h
declares; host-side validation answers through the ABI with the documented
codes and the [cpu.rs] (ferrum-kernels 0.8.0, src/ferrum_kernels/backend/
cpu.rs) message texts.  No test here launches a kernel: every call fails
validation (or, on a machine without a GPU, at the device lookup) before any
launch, and the fake device addresses are never dereferenced on the host.
"""
import ctypes
import os
import re

import numpy as np
import pytest

from gated_delta_rule_44_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x100000  # a 16-byte aligned address never dereferenced by host code


def header_functions():
    with open(os.path.join(ROOT, "include", "gdn.h")) as fh:
        text = fh.read()
    return sorted(set(re.findall(r"^(?:const\s+)?[A-Za-z_0-9]+\s*\*?\s*(gdn_[a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_boundary():
    fns = header_functions()
    for name in ("gdn_prepare", "gdn_decode", "gdn_prefill_varlen", "gdn_prefill_workspace_bytes",
                 "gdn_status_string", "gdn_last_error_message", "gdn_read_device_status"):
        assert name in fns


def test_library_exports_every_declared_symbol():
    L = B.lib()
    for name in header_functions():
        assert hasattr(L, name), name
    assert set(B.EXPORTED) <= set(header_functions())


def test_status_strings():
    L = B.lib()
    for code, name in ((0, "GDN_OK"), (1, "GDN_ERR_SHAPE"), (2, "GDN_ERR_INVALID_ARGUMENT"),
                       (3, "GDN_ERR_DTYPE"), (4, "GDN_ERR_UNSUPPORTED"), (5, "GDN_ERR_CUDA"),
                       (6, "GDN_ERR_TIMEOUT"), (7, "GDN_ERR_DEVICE_CHECK")):
        assert L.gdn_status_string(code).decode() == name
    assert B.gdn_version() >= 100


def decode_args(B_=2, Hk=1, Hv=2, Dk=128, Dv=64, **over):
    a = dict(B=B_, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act_dtype=B.GDN_DTYPE_BF16, use_qk_l2norm=0,
             scale=-1.0, q=FAKE, q_len=B_ * Hk * Dk, k=FAKE, k_len=B_ * Hk * Dk, v=FAKE,
             v_len=B_ * Hv * Dv, g=FAKE, g_len=B_ * Hv, beta=FAKE, beta_len=B_ * Hv, state=FAKE,
             state_slots=4, state_len=4 * Hv * Dv * Dk, state_indices=None,
             state_indices_host=None, out=FAKE, out_len=B_ * Hv * Dv)
    a.update(over)
    return B.gdn_decode_args(**a)


def call_decode(args):
    L = B.lib()
    rc = L.gdn_decode(ctypes.byref(args), None)
    return rc, L.gdn_last_error_message().decode()


def test_decode_shape_messages():
    rc, msg = call_decode(decode_args(q_len=2 * 128 - 1))
    assert rc == B.GDN_ERR_SHAPE and msg == "gated_delta_rule query length 255 < expected 256"
    rc, msg = call_decode(decode_args(Hk=2, Hv=3, q_len=10**9, k_len=10**9))
    assert rc == B.GDN_ERR_SHAPE
    assert msg == "gated_delta_rule value_heads 3 must be divisible by key_heads 2"
    rc, msg = call_decode(decode_args(B_=0))
    assert rc == B.GDN_ERR_SHAPE and msg.startswith("gated_delta_rule shape must be positive")
    rc, msg = call_decode(decode_args(state_len=4 * 2 * 64 * 128 - 1))
    assert rc == B.GDN_ERR_SHAPE and "state length" in msg


def test_decode_other_rejections():
    assert call_decode(decode_args(act_dtype=7))[0] == B.GDN_ERR_DTYPE
    assert call_decode(decode_args(q=None))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_decode(decode_args(q=FAKE + 2))[0] == B.GDN_ERR_INVALID_ARGUMENT
    rc, msg = call_decode(decode_args(Dk=48, q_len=96, k_len=96, state_len=4 * 2 * 64 * 48))
    assert rc == B.GDN_ERR_UNSUPPORTED
    idx = (ctypes.c_int32 * 2)(1, 1)
    rc, msg = call_decode(decode_args(state_indices=FAKE, state_indices_host=ctypes.addressof(idx)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and msg == "duplicate live GDN state index"
    idx = (ctypes.c_int32 * 2)(-2, 1)
    rc, msg = call_decode(decode_args(state_indices=FAKE, state_indices_host=ctypes.addressof(idx)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and msg == "invalid negative GDN state index"
    idx = (ctypes.c_int32 * 2)(0, 4)
    rc, msg = call_decode(decode_args(state_indices=FAKE, state_indices_host=ctypes.addressof(idx)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and msg == "GDN state index out of range"


def prefill_args(T=10, N=2, Hk=1, Hv=2, Dk=128, Dv=128, **over):
    a = dict(T=T, N=N, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act_dtype=B.GDN_DTYPE_BF16, use_qk_l2norm=0,
             scale=-1.0, algo=B.GDN_PREFILL_RECURRENT, q=FAKE, q_len=T * Hk * Dk, k=FAKE,
             k_len=T * Hk * Dk, v=FAKE, v_len=T * Hv * Dv, g=FAKE, g_len=T * Hv, beta=FAKE,
             beta_len=T * Hv, state=FAKE, state_slots=N, state_len=N * Hv * Dv * Dk,
             cu_seqlens=FAKE, state_indices=None, has_initial_state=None, cu_seqlens_host=None,
             state_indices_host=None, out=FAKE, out_len=T * Hv * Dv, workspace=None,
             workspace_bytes=0)
    a.update(over)
    return B.gdn_prefill_args(**a)


def call_prefill(args):
    L = B.lib()
    rc = L.gdn_prefill_varlen(ctypes.byref(args), None)
    return rc, L.gdn_last_error_message().decode()


def test_prefill_cu_seqlens_messages():
    cu = (ctypes.c_int32 * 3)(0, 4, 9)
    rc, msg = call_prefill(prefill_args(cu_seqlens_host=ctypes.addressof(cu)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT
    assert msg == ("gated_delta_rule_varlen cu_seqlens must start at 0 and end at total_tokens 10,"
                   " got first=Some(0) last=Some(9)")
    cu = (ctypes.c_int32 * 3)(0, 0, 10)
    rc, msg = call_prefill(prefill_args(cu_seqlens_host=ctypes.addressof(cu)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT
    assert msg == "gated_delta_rule_varlen sequence 0 has empty or non-monotonic range 0..0"
    assert call_prefill(prefill_args(algo=9))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_prefill(prefill_args(cu_seqlens=None))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_prefill(prefill_args(N=0))[0] == B.GDN_ERR_SHAPE


def test_prefill_workspace_rules():
    # many chains: the fused form; few: the two-launch chunked form (no GPU
    # here: the SM count defaults to 152)
    assert B.gdn_prefill_resolve_algo(4, 64, 128, 128, B.GDN_DTYPE_BF16) == B.GDN_PREFILL_FUSED
    assert B.gdn_prefill_resolve_algo(1, 32, 128, 128, B.GDN_DTYPE_BF16) == B.GDN_PREFILL_CHUNKED
    assert B.gdn_prefill_resolve_algo(4, 64, 32, 32, B.GDN_DTYPE_F32) == \
        B.GDN_PREFILL_RECURRENT
    assert B.gdn_prefill_resolve_algo(1, 32, 128, 128, B.GDN_DTYPE_BF16,
                                      B.GDN_PREFILL_FUSED) == B.GDN_PREFILL_FUSED
    assert B.gdn_prefill_workspace_bytes(100, 2, 4, 32, 32, B.GDN_DTYPE_F32) == 0
    # the fused form's optional workspace: per-sequence chunk counts and
    # prefix, 1024 per-CTA starts, a flag per chain, each 256-byte aligned;
    # a misaligned one is rejected; an unknown algorithm is rejected
    a256 = lambda x: (x + 255) // 256 * 256
    assert B.gdn_prefill_workspace_bytes(8192, 4, 64, 128, 128, B.GDN_DTYPE_BF16) == \
        a256(4 * 4) + a256(4 * 5) + 16 * 1024 + a256(4 * 4 * 64)
    rc, msg = call_prefill(prefill_args(algo=B.GDN_PREFILL_FUSED, workspace=FAKE + 16,
                                        workspace_bytes=1 << 20))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and "256-byte aligned" in msg
    assert B.gdn_prefill_workspace_bytes(4096, 1, 32, 128, 128, B.GDN_DTYPE_BF16) > 0
    assert call_prefill(prefill_args(algo=4))[0] == B.GDN_ERR_INVALID_ARGUMENT
    rc, msg = call_prefill(prefill_args(Dk=64, Dv=64, algo=B.GDN_PREFILL_FUSED))
    assert rc == B.GDN_ERR_UNSUPPORTED and "fused" in msg
    need = B.gdn_prefill_workspace_bytes(4096, 1, 32, 128, 128, B.GDN_DTYPE_BF16,
                                         B.GDN_PREFILL_CHUNKED)
    if need > 0:
        rc, msg = call_prefill(prefill_args(algo=B.GDN_PREFILL_CHUNKED, workspace=None))
        assert rc == B.GDN_ERR_INVALID_ARGUMENT and "workspace needs" in msg


def prepare_args(T=3, N=1, Hk=1, Hv=1, Dk=8, Dv=8, K=4, **over):
    C = 2 * Hk * Dk + Hv * Dv
    a = dict(T=T, N=N, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K, act_dtype=B.GDN_DTYPE_BF16,
             apply_qk_l2norm=1, mixed_qkv=FAKE, mixed_qkv_stride=0, mixed_qkv_len=T * C,
             conv_weight=FAKE, conv_weight_len=C * K, a_raw=FAKE, a_raw_stride=0,
             a_raw_len=T * Hv, b_raw=FAKE, b_raw_stride=0, b_raw_len=T * Hv, A_log=FAKE,
             A_log_len=Hv, dt_bias=FAKE, dt_bias_len=Hv, cu_seqlens=FAKE, state_indices=None,
             has_initial_state=None, cu_seqlens_host=None, state_indices_host=None,
             conv_state=FAKE, conv_state_slots=N, conv_state_len=N * C * (K - 1), q=FAKE,
             q_len=T * Hk * Dk, k=FAKE, k_len=T * Hk * Dk, v=FAKE, v_len=T * Hv * Dv, g=FAKE,
             g_len=T * Hv, beta=FAKE, beta_len=T * Hv)
    a.update(over)
    return B.gdn_prepare_args(**a)


def call_prepare(args):
    L = B.lib()
    rc = L.gdn_prepare(ctypes.byref(args), None)
    return rc, L.gdn_last_error_message().decode()


def test_prepare_messages():
    rc, msg = call_prepare(prepare_args(conv_weight_len=95))
    assert rc == B.GDN_ERR_SHAPE
    assert msg == "linear_attention_prepare conv_weight length 95 < expected 96"
    rc, msg = call_prepare(prepare_args(K=0))
    assert rc == B.GDN_ERR_SHAPE and msg.endswith("conv_kernel=0")
    rc, msg = call_prepare(prepare_args(mixed_qkv_stride=20, mixed_qkv_len=10**6))
    assert rc == B.GDN_ERR_SHAPE  # stride shorter than a row of 24 channels
    rc, msg = call_prepare(prepare_args(K=9, conv_weight_len=10**6, conv_state_len=10**6))
    assert rc == B.GDN_ERR_UNSUPPORTED
    rc, msg = call_prepare(prepare_args(Dk=12, q_len=10**6, k_len=10**6, mixed_qkv_len=10**6,
                                        conv_weight_len=10**6, conv_state_len=10**6))
    assert rc == B.GDN_ERR_UNSUPPORTED
    rc, msg = call_prepare(prepare_args(mixed_qkv_stride=28, mixed_qkv_len=10**6))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT  # 28 bf16 = 56 bytes: rows not 16-byte aligned
    rc, msg = call_prepare(prepare_args(act_dtype=5))
    assert rc == B.GDN_ERR_DTYPE


def test_prepare_cu_seqlens_messages():
    """The prepare's host-mirror cu_seqlens rules carry the label of [cpu.rs]
    linear_attention_prepare_varlen_f32 and print the bounds in Rust's Option
    Debug form, as the page's format string does."""
    cu = (ctypes.c_int32 * 3)(1, 2, 7)
    rc, msg = call_prepare(prepare_args(T=7, N=2, cu_seqlens_host=ctypes.addressof(cu)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT
    assert msg == ("linear_attention_prepare_varlen cu_seqlens must start at 0 and end at"
                   " total_tokens 7, got first=Some(1) last=Some(7)")
    cu = (ctypes.c_int32 * 3)(0, 0, 7)
    rc, msg = call_prepare(prepare_args(T=7, N=2, cu_seqlens_host=ctypes.addressof(cu)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT
    assert msg == "linear_attention_prepare_varlen sequence 0 has empty or non-monotonic range 0..0"


def test_valid_call_without_gpu_stops_before_launch():
    import torch
    if torch.cuda.is_available():
        pytest.skip("this machine has a GPU")
    rc, msg = call_decode(decode_args())
    assert rc == B.GDN_ERR_CUDA


def norm_args(T=3, H=2, D=128, **over):
    a = dict(tokens=T, heads=H, dim=D, act_dtype=B.GDN_DTYPE_BF16, sigmoid_gate=0, eps=1e-6,
             core=FAKE, core_len=T * H * D, z=FAKE, z_len=T * H * D, z_token_stride=0,
             weight=FAKE, weight_len=D, out=FAKE, out_len=T * H * D)
    a.update(over)
    return B.gdn_gated_rmsnorm_args(**a)


def call_norm(args):
    L = B.lib()
    rc = L.gdn_gated_rmsnorm(ctypes.byref(args), None)
    return rc, L.gdn_last_error_message().decode()


def test_gated_rmsnorm_shape_messages():
    # [cpu.rs] validate_gated_rms_norm_shape texts
    rc, msg = call_norm(norm_args(T=0))
    assert rc == B.GDN_ERR_SHAPE
    assert msg == "gated_rms_norm shape must be positive, got tokens=0 heads=2 dim=128"
    for field, label, n, expected in (("core_len", "core", 767, 768), ("z_len", "z", 700, 768),
                                      ("weight_len", "weight", 127, 128),
                                      ("out_len", "out", 1, 768)):
        rc, msg = call_norm(norm_args(**{field: n}))
        assert rc == B.GDN_ERR_SHAPE
        assert msg == f"gated_rms_norm {label} length {n} < expected {expected}"


def test_gated_rmsnorm_other_rejections():
    assert call_norm(norm_args(act_dtype=9))[0] == B.GDN_ERR_DTYPE
    assert call_norm(norm_args(core=None))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_norm(norm_args(z=FAKE + 4))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_norm(norm_args(z_token_stride=100))[0] == B.GDN_ERR_INVALID_ARGUMENT  # < H*D
    assert call_norm(norm_args(z_token_stride=260, z_len=10**6))[0] == B.GDN_ERR_INVALID_ARGUMENT
    rc, msg = call_norm(norm_args(D=12, core_len=72, z_len=72, weight_len=12, out_len=72))
    assert rc == B.GDN_ERR_UNSUPPORTED and "multiple of 8" in msg
    big = 2048
    rc, _ = call_norm(norm_args(D=big, core_len=6 * big, z_len=6 * big, weight_len=big,
                                out_len=6 * big))
    assert rc == B.GDN_ERR_UNSUPPORTED


def kda_args(T=4, N=2, Hk=1, Hv=2, Dk=128, Dv=64, **over):
    a = dict(T=T, N=N, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act_dtype=B.GDN_DTYPE_BF16, scale=-1.0,
             q=FAKE, q_len=T * Hk * Dk, k=FAKE, k_len=T * Hk * Dk, v=FAKE, v_len=T * Hv * Dv,
             g=FAKE, g_len=T * Hv * Dk, beta=FAKE, beta_len=T * Hv, state=FAKE, state_slots=4,
             state_len=4 * Hv * Dv * Dk, cu_seqlens=FAKE, state_indices=None,
             has_initial_state=None, cu_seqlens_host=None, state_indices_host=None, out=FAKE,
             out_len=T * Hv * Dv)
    a.update(over)
    return B.gdn_kda_args(**a)


def call_kda(args):
    L = B.lib()
    rc = L.gdn_kda_varlen(ctypes.byref(args), None)
    return rc, L.gdn_last_error_message().decode()


def test_kda_rejections():
    rc, msg = call_kda(kda_args(g_len=4 * 2 * 128 - 1))
    assert rc == B.GDN_ERR_SHAPE and msg == "kda_gated_delta_rule g length 1023 < expected 1024"
    rc, msg = call_kda(kda_args(q_len=10))
    assert rc == B.GDN_ERR_SHAPE and msg == "gated_delta_rule query length 10 < expected 512"
    assert call_kda(kda_args(g=FAKE + 4))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_kda(kda_args(N=0))[0] == B.GDN_ERR_SHAPE
    assert call_kda(kda_args(cu_seqlens=None))[0] == B.GDN_ERR_INVALID_ARGUMENT
    rc, _ = call_kda(kda_args(Dk=48, q_len=10**6, k_len=10**6, g_len=10**6, state_len=10**8))
    assert rc == B.GDN_ERR_UNSUPPORTED
    cu = (ctypes.c_int32 * 3)(0, 4, 4)  # empty second sequence
    rc, msg = call_kda(kda_args(cu_seqlens_host=ctypes.cast(cu, ctypes.c_void_p).value))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and "empty or non-monotonic" in msg


def test_kda_algo_rules():
    """AUTO takes the chunked tensor-core form for bf16 with Dk = Dv = 128 when
    some sequence holds more than one token; it needs a caller workspace of one
    blob per (chunk, value head)."""
    R = B.gdn_kda_resolve_algo
    assert R(100, 2, 128, 128) == B.GDN_PREFILL_CHUNKED
    assert R(2, 2, 128, 128) == B.GDN_PREFILL_RECURRENT            # one token each
    assert R(100, 2, 128, 64) == B.GDN_PREFILL_RECURRENT
    assert R(100, 2, 128, 128, B.GDN_DTYPE_F32) == B.GDN_PREFILL_RECURRENT
    assert R(100, 2, 128, 128, algo=B.GDN_PREFILL_RECURRENT) == B.GDN_PREFILL_RECURRENT
    blob = B.gdn_kda_workspace_bytes(64, 1, 1, 128, 128) // (64 // 64 + 1)
    assert blob == 113 * 1024
    assert B.gdn_kda_workspace_bytes(4096, 3, 32, 128, 128) == (4096 // 64 + 3) * 32 * blob
    assert B.gdn_kda_workspace_bytes(100, 2, 4, 128, 64) == 0
    big = dict(T=130, N=2, Dv=128, v_len=130 * 2 * 128, out_len=130 * 2 * 128,
               q_len=130 * 128, k_len=130 * 128, g_len=130 * 2 * 128, beta_len=260,
               state_len=4 * 2 * 128 * 128)
    rc, msg = call_kda(kda_args(**big))
    need = B.gdn_kda_workspace_bytes(130, 2, 2, 128, 128)
    assert rc == B.GDN_ERR_INVALID_ARGUMENT
    assert msg == f"gdn_kda_varlen workspace needs {need} bytes, got 0"
    rc, _ = call_kda(kda_args(**big, workspace=FAKE, workspace_bytes=need - 1))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT
    rc, msg = call_kda(kda_args(**big, workspace=FAKE + 16, workspace_bytes=need))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and msg == "workspace must be 256-byte aligned"
    rc, msg = call_kda(kda_args(**big, algo=B.GDN_PREFILL_FUSED))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and "KDA algo 3" in msg
    rc, msg = call_kda(kda_args(algo=B.GDN_PREFILL_CHUNKED))                # Dv = 64
    assert rc == B.GDN_ERR_UNSUPPORTED and "Dk = Dv = 128" in msg


def spec_args(T=5, n_reqs=2, num_cols=3, Hk=1, Hv=2, Dk=128, Dv=64, **over):
    a = dict(T=T, n_reqs=n_reqs, num_cols=num_cols, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv,
             act_dtype=B.GDN_DTYPE_BF16, scale=-1.0, q=FAKE, q_len=T * Hk * Dk, k=FAKE,
             k_len=T * Hk * Dk, v=FAKE, v_len=T * Hv * Dv, g=FAKE, g_len=T * Hv, beta=FAKE,
             beta_len=T * Hv, state=FAKE, state_slots=8, state_len=8 * Hv * Dv * Dk,
             cu_seqlens=FAKE, state_indices=FAKE, num_accepted=FAKE, cu_seqlens_host=None,
             state_indices_host=None, num_accepted_host=None, out=FAKE, out_len=T * Hv * Dv)
    a.update(over)
    return B.gdn_spec_decode_args(**a)


def call_spec(args):
    L = B.lib()
    rc = L.gdn_spec_decode(ctypes.byref(args), None)
    return rc, L.gdn_last_error_message().decode()


def _host(*vals):
    arr = (ctypes.c_int32 * len(vals))(*vals)
    _host.keep.append(arr)
    return ctypes.cast(arr, ctypes.c_void_p).value


_host.keep = []


def test_spec_decode_rejections():
    assert call_spec(spec_args(n_reqs=0))[0] == B.GDN_ERR_SHAPE
    assert call_spec(spec_args(num_cols=0))[0] == B.GDN_ERR_SHAPE
    rc, msg = call_spec(spec_args(T=7))  # 7 tokens > 2 requests x 3 columns
    assert rc == B.GDN_ERR_SHAPE and "more than n_reqs * num_cols" in msg
    assert call_spec(spec_args(num_accepted=None))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_spec(spec_args(state_indices=None))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_spec(spec_args(g_len=9))[0] == B.GDN_ERR_SHAPE
    rc, _ = call_spec(spec_args(Dk=48, q_len=10**6, k_len=10**6, state_len=10**8))
    assert rc == B.GDN_ERR_UNSUPPORTED
    # host mirrors: [qwen3_5.cpp] spec metadata rules
    rc, msg = call_spec(spec_args(cu_seqlens_host=_host(0, 2, 4)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and msg == "spec query offsets must span the spec tokens"
    rc, msg = call_spec(spec_args(cu_seqlens_host=_host(0, 1, 5)))  # request 1: 4 > 3 tokens
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and "not 0..3 tokens" in msg
    rc, msg = call_spec(spec_args(num_accepted_host=_host(1, 4)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT
    assert msg == "num_accepted_tokens must be in [1, num_spec + 1]"
    assert call_spec(spec_args(num_accepted_host=_host(0, 1)))[0] == B.GDN_ERR_INVALID_ARGUMENT
    rc, msg = call_spec(spec_args(state_indices_host=_host(0, 1, 2, 3, 4, 8)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and msg == "spec GDN state slot out of range"
    rc, msg = call_spec(spec_args(state_indices_host=_host(0, 1, 2, 3, 2, -1)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and "named by two requests" in msg


def spec_prepare_args(T=6, N=2, max_q=3, K=4, width=None, **over):
    C = 2 * 1 * 8 + 1 * 8
    width = (K - 1) + (max_q - 1) if width is None else width
    base = dict(T=T, N=N, K=K, state_indices=FAKE, conv_state_slots=4,
                conv_state_len=4 * C * width)
    base.update({k: v for k, v in over.items() if k in dict(B.gdn_prepare_args._fields_)})
    a = B.gdn_spec_prepare_args(base=prepare_args(**base), conv_state_width=width,
                                num_accepted=over.get("num_accepted", FAKE),
                                num_accepted_host=over.get("num_accepted_host"))
    return a


def call_spec_prepare(args):
    L = B.lib()
    rc = L.gdn_spec_prepare(ctypes.byref(args), None)
    return rc, L.gdn_last_error_message().decode()


def test_spec_prepare_rejections():
    rc, msg = call_spec_prepare(spec_prepare_args(width=2))   # shorter than K-1 = 3
    assert rc == B.GDN_ERR_SHAPE and "shorter than conv_kernel - 1" in msg
    rc, msg = call_spec_prepare(spec_prepare_args(K=1, width=2, conv_weight_len=24))
    assert rc == B.GDN_ERR_UNSUPPORTED
    rc, msg = call_spec_prepare(spec_prepare_args(has_initial_state=FAKE))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and "has_initial_state" in msg
    assert call_spec_prepare(spec_prepare_args(state_indices=None))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_spec_prepare(spec_prepare_args(num_accepted=None))[0] == B.GDN_ERR_INVALID_ARGUMENT
    rc, msg = call_spec_prepare(spec_prepare_args(T=7))   # 7 > 2 requests x max_q 3
    assert rc == B.GDN_ERR_SHAPE and "more than requests * max_query_len" in msg
    rc, _ = call_spec_prepare(spec_prepare_args(max_q=15, conv_state_len=10**6))
    assert rc == B.GDN_ERR_UNSUPPORTED                    # a row of 17 entries
    rc, msg = call_spec_prepare(spec_prepare_args(conv_state_len=10))
    assert rc == B.GDN_ERR_SHAPE and "conv_state length 10" in msg
    # host mirrors
    rc, msg = call_spec_prepare(spec_prepare_args(cu_seqlens_host=_host(0, 4, 6)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and "not 0..3 tokens" in msg
    rc, msg = call_spec_prepare(spec_prepare_args(num_accepted_host=_host(1, 4)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT
    assert msg == "num_accepted_tokens must be in [1, num_spec + 1]"
    rc, msg = call_spec_prepare(spec_prepare_args(state_indices_host=_host(1, 1)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and "named by two requests" in msg
    rc, msg = call_spec_prepare(spec_prepare_args(state_indices_host=_host(0, 4)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and msg == "spec GDN state slot out of range"


def packed_args(Bn=4, Hk=1, Hv=2, Dk=64, Dv=64, K=4, **over):
    C = 2 * Hk * Dk + Hv * Dv
    a = dict(B=Bn, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K, act_dtype=B.GDN_DTYPE_BF16,
             apply_qk_l2norm=1, scale=-1.0, mixed_qkv=FAKE, mixed_qkv_stride=0,
             mixed_qkv_len=Bn * C, conv_weight=FAKE, conv_weight_len=C * K, a_raw=FAKE,
             a_raw_stride=0, a_raw_len=Bn * Hv, b_raw=FAKE, b_raw_stride=0, b_raw_len=Bn * Hv,
             A_log=FAKE, A_log_len=Hv, dt_bias=FAKE, dt_bias_len=Hv, state_indices=FAKE,
             state_indices_host=None, conv_state=FAKE, conv_state_len=8 * C * (K - 1),
             state=FAKE, state_slots=8, state_len=8 * Hv * Dv * Dk, out=FAKE,
             out_len=Bn * Hv * Dv)
    a.update(over)
    return B.gdn_packed_decode_args(**a)


def call_packed(args):
    L = B.lib()
    rc = L.gdn_packed_decode(ctypes.byref(args), None)
    return rc, L.gdn_last_error_message().decode()


def test_packed_decode_rejections():
    assert call_packed(packed_args(Bn=0))[0] == B.GDN_ERR_SHAPE
    assert call_packed(packed_args(Hk=2, Hv=3))[0] == B.GDN_ERR_SHAPE   # Hv % Hk != 0
    rc, msg = call_packed(packed_args(conv_state_len=5))
    assert rc == B.GDN_ERR_SHAPE and msg.startswith("packed_gdn_decode conv_state length 5")
    rc, msg = call_packed(packed_args(mixed_qkv_stride=100))
    assert rc == B.GDN_ERR_SHAPE and "row stride shorter" in msg
    assert call_packed(packed_args(state_indices=None))[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert call_packed(packed_args(state=FAKE + 4))[0] == B.GDN_ERR_INVALID_ARGUMENT
    rc, msg = call_packed(packed_args(Dk=32, mixed_qkv_len=10**6, conv_weight_len=10**6,
                                      conv_state_len=10**7, state_len=10**8))
    assert rc == B.GDN_ERR_UNSUPPORTED and "Dk in {64, 128}" in msg
    assert call_packed(packed_args(K=5, conv_weight_len=10**6,
                                   conv_state_len=10**7))[0] == B.GDN_ERR_UNSUPPORTED
    rc, msg = call_packed(packed_args(state_indices_host=_host(0, 1, 1, -1)))
    assert rc == B.GDN_ERR_INVALID_ARGUMENT and msg == "duplicate live GDN state index"


def out_norm(T, Hv, Dv, **over):
    n = dict(z=FAKE, z_len=T * Hv * Dv, z_token_stride=Hv * Dv, weight=FAKE, weight_len=Dv,
             eps=1e-6, sigmoid_gate=0)
    n.update(over)
    return B.gdn_out_norm(**n)


def test_out_norm_option_rejections():
    """The output-norm option of gdn_decode / gdn_prefill_varlen follows the
    gated_rms_norm rules ([cpu.rs] validate_gated_rms_norm_shape) for the
    call's output rows."""
    def dec(**over):
        n = out_norm(2, 2, 64, **over)
        return call_decode(decode_args(out_norm=ctypes.pointer(n)))

    rc, msg = dec(z_len=2 * 2 * 64 - 1)
    assert rc == B.GDN_ERR_SHAPE and msg == "gated_rms_norm z length 255 < expected 256"
    rc, msg = dec(weight_len=63)
    assert rc == B.GDN_ERR_SHAPE and msg == "gated_rms_norm weight length 63 < expected 64"
    assert dec(z_token_stride=100)[0] == B.GDN_ERR_INVALID_ARGUMENT       # < Hv * Dv
    assert dec(z_token_stride=132, z_len=10**6)[0] == B.GDN_ERR_INVALID_ARGUMENT  # 264 B rows
    assert dec(z=None)[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert dec(weight=FAKE + 2)[0] == B.GDN_ERR_INVALID_ARGUMENT
    assert dec(eps=-1.0)[0] == B.GDN_ERR_INVALID_ARGUMENT
    n = out_norm(2, 2, 12)
    rc, msg = call_decode(decode_args(Dv=12, v_len=48, out_len=48, state_len=4 * 2 * 12 * 128,
                                      out_norm=ctypes.pointer(n)))
    assert rc == B.GDN_ERR_UNSUPPORTED and "multiple of 8" in msg
    # the prefill: z rows for every token
    n = out_norm(10, 2, 128, z_len=9 * 256 + 255)
    rc, msg = call_prefill(prefill_args(out_norm=ctypes.pointer(n)))
    assert rc == B.GDN_ERR_SHAPE and msg == "gated_rms_norm z length 2559 < expected 2560"


def test_out_norm_valid_call_without_gpu_stops_before_launch():
    import torch
    if torch.cuda.is_available():
        pytest.skip("this machine has a GPU")
    n = out_norm(2, 2, 64, z_token_stride=136, z_len=136 + 128)
    assert call_decode(decode_args(out_norm=ctypes.pointer(n)))[0] == B.GDN_ERR_CUDA
