"""Thin ctypes binding of libgdn (include/gdn.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions take torch tensors (device memory and streams come from
PyTorch) and raise ``GdnError`` on a non-zero status.  There is no fallback:
if the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading
from typing import Optional

import torch

from . import build as _build

GDN_OK = 0
GDN_ERR_SHAPE = 1
GDN_ERR_INVALID_ARGUMENT = 2
GDN_ERR_DTYPE = 3
GDN_ERR_UNSUPPORTED = 4
GDN_ERR_CUDA = 5
GDN_ERR_TIMEOUT = 6
GDN_ERR_DEVICE_CHECK = 7

GDN_DTYPE_F32 = 0
GDN_DTYPE_BF16 = 1

GDN_PREFILL_AUTO = 0
GDN_PREFILL_CHUNKED = 1
GDN_PREFILL_RECURRENT = 2
GDN_PREFILL_FUSED = 3

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_vp = ctypes.c_void_p
_f32 = ctypes.c_float


class gdn_prepare_args(ctypes.Structure):
    _fields_ = [("T", _i64), ("N", _i64), ("Hk", _i64), ("Hv", _i64), ("Dk", _i64), ("Dv", _i64),
                ("K", _i64), ("act_dtype", _i32), ("apply_qk_l2norm", _i32),
                ("mixed_qkv", _vp), ("mixed_qkv_stride", _i64), ("mixed_qkv_len", _i64),
                ("conv_weight", _vp), ("conv_weight_len", _i64),
                ("a_raw", _vp), ("a_raw_stride", _i64), ("a_raw_len", _i64),
                ("b_raw", _vp), ("b_raw_stride", _i64), ("b_raw_len", _i64),
                ("A_log", _vp), ("A_log_len", _i64), ("dt_bias", _vp), ("dt_bias_len", _i64),
                ("cu_seqlens", _vp), ("state_indices", _vp), ("has_initial_state", _vp),
                ("cu_seqlens_host", _vp), ("state_indices_host", _vp),
                ("conv_state", _vp), ("conv_state_slots", _i64), ("conv_state_len", _i64),
                ("q", _vp), ("q_len", _i64), ("k", _vp), ("k_len", _i64), ("v", _vp),
                ("v_len", _i64), ("g", _vp), ("g_len", _i64), ("beta", _vp),
                ("beta_len", _i64)]


class gdn_packed_decode_args(ctypes.Structure):
    _fields_ = [("B", _i64), ("Hk", _i64), ("Hv", _i64), ("Dk", _i64), ("Dv", _i64), ("K", _i64),
                ("act_dtype", _i32), ("apply_qk_l2norm", _i32), ("scale", _f32),
                ("mixed_qkv", _vp), ("mixed_qkv_stride", _i64), ("mixed_qkv_len", _i64),
                ("conv_weight", _vp), ("conv_weight_len", _i64),
                ("a_raw", _vp), ("a_raw_stride", _i64), ("a_raw_len", _i64),
                ("b_raw", _vp), ("b_raw_stride", _i64), ("b_raw_len", _i64),
                ("A_log", _vp), ("A_log_len", _i64), ("dt_bias", _vp), ("dt_bias_len", _i64),
                ("state_indices", _vp), ("state_indices_host", _vp),
                ("conv_state", _vp), ("conv_state_len", _i64),
                ("state", _vp), ("state_slots", _i64), ("state_len", _i64),
                ("out", _vp), ("out_len", _i64)]


class gdn_spec_prepare_args(ctypes.Structure):
    _fields_ = [("base", gdn_prepare_args), ("conv_state_width", _i64), ("num_accepted", _vp),
                ("num_accepted_host", _vp)]


class gdn_out_norm(ctypes.Structure):
    _fields_ = [("z", _vp), ("z_len", _i64), ("z_token_stride", _i64), ("weight", _vp),
                ("weight_len", _i64), ("eps", _f32), ("sigmoid_gate", _i32), ("in_kernel", _i32)]


class gdn_decode_args(ctypes.Structure):
    _fields_ = [("B", _i64), ("Hk", _i64), ("Hv", _i64), ("Dk", _i64), ("Dv", _i64),
                ("act_dtype", _i32), ("use_qk_l2norm", _i32), ("scale", _f32),
                ("q", _vp), ("q_len", _i64), ("k", _vp), ("k_len", _i64), ("v", _vp),
                ("v_len", _i64), ("g", _vp), ("g_len", _i64), ("beta", _vp), ("beta_len", _i64),
                ("state", _vp), ("state_slots", _i64), ("state_len", _i64),
                ("state_indices", _vp), ("state_indices_host", _vp),
                ("out", _vp), ("out_len", _i64), ("out_norm", ctypes.POINTER(gdn_out_norm))]


class gdn_prefill_args(ctypes.Structure):
    _fields_ = [("T", _i64), ("N", _i64), ("Hk", _i64), ("Hv", _i64), ("Dk", _i64), ("Dv", _i64),
                ("act_dtype", _i32), ("use_qk_l2norm", _i32), ("scale", _f32), ("algo", _i32),
                ("q", _vp), ("q_len", _i64), ("k", _vp), ("k_len", _i64), ("v", _vp),
                ("v_len", _i64), ("g", _vp), ("g_len", _i64), ("beta", _vp), ("beta_len", _i64),
                ("state", _vp), ("state_slots", _i64), ("state_len", _i64),
                ("cu_seqlens", _vp), ("state_indices", _vp), ("has_initial_state", _vp),
                ("cu_seqlens_host", _vp), ("state_indices_host", _vp),
                ("out", _vp), ("out_len", _i64), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t),
                ("out_norm", ctypes.POINTER(gdn_out_norm))]


class gdn_kda_args(ctypes.Structure):
    _fields_ = [("T", _i64), ("N", _i64), ("Hk", _i64), ("Hv", _i64), ("Dk", _i64), ("Dv", _i64),
                ("act_dtype", _i32), ("scale", _f32),
                ("q", _vp), ("q_len", _i64), ("k", _vp), ("k_len", _i64), ("v", _vp),
                ("v_len", _i64), ("g", _vp), ("g_len", _i64), ("beta", _vp), ("beta_len", _i64),
                ("state", _vp), ("state_slots", _i64), ("state_len", _i64),
                ("cu_seqlens", _vp), ("state_indices", _vp), ("has_initial_state", _vp),
                ("cu_seqlens_host", _vp), ("state_indices_host", _vp),
                ("out", _vp), ("out_len", _i64), ("algo", _i32), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t)]


class gdn_spec_decode_args(ctypes.Structure):
    _fields_ = [("T", _i64), ("n_reqs", _i64), ("num_cols", _i64), ("Hk", _i64), ("Hv", _i64),
                ("Dk", _i64), ("Dv", _i64), ("act_dtype", _i32), ("scale", _f32),
                ("q", _vp), ("q_len", _i64), ("k", _vp), ("k_len", _i64), ("v", _vp),
                ("v_len", _i64), ("g", _vp), ("g_len", _i64), ("beta", _vp), ("beta_len", _i64),
                ("state", _vp), ("state_slots", _i64), ("state_len", _i64),
                ("cu_seqlens", _vp), ("state_indices", _vp), ("num_accepted", _vp),
                ("cu_seqlens_host", _vp), ("state_indices_host", _vp), ("num_accepted_host", _vp),
                ("out", _vp), ("out_len", _i64)]


class gdn_gated_rmsnorm_args(ctypes.Structure):
    _fields_ = [("tokens", _i64), ("heads", _i64), ("dim", _i64), ("act_dtype", _i32),
                ("sigmoid_gate", _i32), ("eps", _f32), ("core", _vp), ("core_len", _i64),
                ("z", _vp), ("z_len", _i64), ("z_token_stride", _i64), ("weight", _vp),
                ("weight_len", _i64), ("out", _vp), ("out_len", _i64)]


class gdn_mixed_meta(ctypes.Structure):
    _fields_ = [("num_decodes", _i64), ("num_prefills", _i64), ("num_decode_tokens", _i64),
                ("num_prefill_tokens", _i64), ("num_actual_tokens", _i64), ("state_slots", _i64),
                ("allow_inert_padding", _i32), ("cu_seqlens_host", _vp),
                ("state_indices_host", _vp), ("has_initial_state_host", _vp),
                ("cu_seqlens_prefill_host", _vp), ("prefill_state_indices_host", _vp),
                ("prefill_has_initial_state_host", _vp)]


EXPORTED = ("gdn_prepare", "gdn_decode", "gdn_prefill_varlen", "gdn_kda_varlen",
            "gdn_spec_prepare", "gdn_spec_decode", "gdn_packed_decode", "gdn_gated_rmsnorm",
            "gdn_prefill_workspace_bytes",
            "gdn_prefill_resolve_algo", "gdn_kda_resolve_algo", "gdn_kda_workspace_bytes",
            "gdn_status_string", "gdn_last_error_message",
            "gdn_read_device_status", "gdn_version", "gdn_launch_count", "gdn_validate_mixed",
            "gdn_check_wait_timeout")


class GdnError(RuntimeError):
    def __init__(self, code: int, name: str, msg: str):
        super().__init__(f"{name}: {msg}")
        self.code = code
        self.status = name
        self.msg = msg


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Build (if stale) and load libgdn.so; raises if that is impossible."""
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(_build.build_library())
            for name in ("gdn_prepare", "gdn_decode", "gdn_prefill_varlen", "gdn_kda_varlen",
                         "gdn_spec_prepare", "gdn_spec_decode", "gdn_packed_decode", "gdn_gated_rmsnorm",
                         "gdn_read_device_status", "gdn_version", "gdn_validate_mixed"):
                getattr(L, name).restype = ctypes.c_int
            L.gdn_prepare.argtypes = [ctypes.POINTER(gdn_prepare_args), _vp]
            L.gdn_decode.argtypes = [ctypes.POINTER(gdn_decode_args), _vp]
            L.gdn_prefill_varlen.argtypes = [ctypes.POINTER(gdn_prefill_args), _vp]
            L.gdn_gated_rmsnorm.argtypes = [ctypes.POINTER(gdn_gated_rmsnorm_args), _vp]
            L.gdn_kda_varlen.argtypes = [ctypes.POINTER(gdn_kda_args), _vp]
            L.gdn_spec_decode.argtypes = [ctypes.POINTER(gdn_spec_decode_args), _vp]
            L.gdn_spec_prepare.argtypes = [ctypes.POINTER(gdn_spec_prepare_args), _vp]
            L.gdn_packed_decode.argtypes = [ctypes.POINTER(gdn_packed_decode_args), _vp]
            L.gdn_read_device_status.argtypes = [_vp]
            L.gdn_validate_mixed.argtypes = [ctypes.POINTER(gdn_mixed_meta)]
            L.gdn_check_wait_timeout.restype = ctypes.c_int
            L.gdn_check_wait_timeout.argtypes = [ctypes.c_longlong, _vp]
            L.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
            L.gdn_prefill_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64, _i64, _i32, _i32]
            L.gdn_prefill_resolve_algo.restype = _i32
            L.gdn_prefill_resolve_algo.argtypes = [_i64, _i64, _i64, _i64, _i32, _i32]
            L.gdn_kda_resolve_algo.restype = _i32
            L.gdn_kda_resolve_algo.argtypes = [_i64, _i64, _i64, _i64, _i32, _i32]
            L.gdn_kda_workspace_bytes.restype = ctypes.c_size_t
            L.gdn_kda_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64, _i64, _i32, _i32]
            L.gdn_status_string.restype = ctypes.c_char_p
            L.gdn_status_string.argtypes = [ctypes.c_int]
            L.gdn_last_error_message.restype = ctypes.c_char_p
            L.gdn_last_error_message.argtypes = []
            L.gdn_launch_count.restype = ctypes.c_uint64
            L.gdn_launch_count.argtypes = []
            _lib = L
        return _lib


def _check(rc: int) -> None:
    if rc != GDN_OK:
        L = lib()
        raise GdnError(rc, L.gdn_status_string(rc).decode(), L.gdn_last_error_message().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDN_DTYPE_BF16
    if t.dtype == torch.float32:
        return GDN_DTYPE_F32
    raise GdnError(GDN_ERR_DTYPE, "GDN_ERR_DTYPE", f"unsupported activation dtype {t.dtype}")


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _n(t: Optional[torch.Tensor]) -> int:
    """Elements reachable from the tensor's first element (its allocation length)."""
    if t is None:
        return 0
    if t.numel() == 0:
        return 0
    return int(sum((s - 1) * st for s, st in zip(t.shape, t.stride())) + 1)


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _host_i32(t: Optional[torch.Tensor]):
    if t is None:
        return None, None
    h = t.detach().to("cpu", torch.int32).contiguous()
    return h, h.data_ptr()


def _prepare_args(mixed_qkv, conv_weight, a_raw, b_raw, A_log, dt_bias, cu_seqlens, conv_state,
                  q, k, v, g, beta, Hk, Hv, Dk, Dv, K, state_indices, has_initial_state,
                  cu_seqlens_host, state_indices_host, apply_qk_l2norm):
    """gdn_prepare_args of the call, and the host mirrors it points to (kept
    alive by the caller)."""
    T = mixed_qkv.shape[0]
    N = cu_seqlens.numel() - 1
    cuh, cuh_p = _host_i32(cu_seqlens_host)
    sih, sih_p = _host_i32(state_indices_host)
    a = gdn_prepare_args(
        T=T, N=N, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K, act_dtype=_dt(mixed_qkv),
        apply_qk_l2norm=int(apply_qk_l2norm),
        mixed_qkv=_p(mixed_qkv), mixed_qkv_stride=mixed_qkv.stride(0), mixed_qkv_len=_n(mixed_qkv),
        conv_weight=_p(conv_weight), conv_weight_len=_n(conv_weight),
        a_raw=_p(a_raw), a_raw_stride=a_raw.stride(0), a_raw_len=_n(a_raw),
        b_raw=_p(b_raw), b_raw_stride=b_raw.stride(0), b_raw_len=_n(b_raw),
        A_log=_p(A_log), A_log_len=_n(A_log), dt_bias=_p(dt_bias), dt_bias_len=_n(dt_bias),
        cu_seqlens=_p(cu_seqlens), state_indices=_p(state_indices),
        has_initial_state=_p(has_initial_state), cu_seqlens_host=cuh_p,
        state_indices_host=sih_p, conv_state=_p(conv_state),
        conv_state_slots=conv_state.shape[0] if conv_state is not None else 0,
        conv_state_len=_n(conv_state), q=_p(q), q_len=_n(q), k=_p(k), k_len=_n(k), v=_p(v),
        v_len=_n(v), g=_p(g), g_len=_n(g), beta=_p(beta), beta_len=_n(beta))
    return a, (cuh, sih)


def gdn_prepare(mixed_qkv, conv_weight, a_raw, b_raw, A_log, dt_bias, cu_seqlens, conv_state,
                q, k, v, g, beta, *, Hk, Hv, Dk, Dv, K, state_indices=None,
                has_initial_state=None, cu_seqlens_host=None, state_indices_host=None,
                apply_qk_l2norm=True, stream=None) -> None:
    """include/gdn.h gdn_prepare; outputs q, k, v, g, beta are written, the
    conv_state pool is updated in place."""
    a, keep = _prepare_args(mixed_qkv, conv_weight, a_raw, b_raw, A_log, dt_bias, cu_seqlens,
                            conv_state, q, k, v, g, beta, Hk, Hv, Dk, Dv, K, state_indices,
                            has_initial_state, cu_seqlens_host, state_indices_host,
                            apply_qk_l2norm)
    _check(lib().gdn_prepare(ctypes.byref(a), _stream(stream)))


def gdn_spec_prepare(mixed_qkv, conv_weight, a_raw, b_raw, A_log, dt_bias, cu_seqlens,
                     conv_state, conv_indices, num_accepted, q, k, v, g, beta, *, Hk, Hv, Dk, Dv,
                     K, cu_seqlens_host=None, conv_indices_host=None, num_accepted_host=None,
                     apply_qk_l2norm=True, stream=None) -> None:
    """include/gdn.h gdn_spec_prepare; conv_state [slots, C_conv, width] with
    width = (K-1) + (max_q-1), updated in place; conv_indices, num_accepted
    [requests] int32."""
    base, keep = _prepare_args(mixed_qkv, conv_weight, a_raw, b_raw, A_log, dt_bias, cu_seqlens,
                               conv_state, q, k, v, g, beta, Hk, Hv, Dk, Dv, K, conv_indices,
                               None, cu_seqlens_host, conv_indices_host, apply_qk_l2norm)
    nah, nah_p = _host_i32(num_accepted_host)
    a = gdn_spec_prepare_args(base=base, conv_state_width=conv_state.shape[2],
                              num_accepted=_p(num_accepted), num_accepted_host=nah_p)
    _check(lib().gdn_spec_prepare(ctypes.byref(a), _stream(stream)))


def gdn_packed_decode(mixed_qkv, conv_weight, a_raw, b_raw, A_log, dt_bias, state_indices,
                      conv_state, state, out, *, Hk, Hv, Dk, Dv, K, scale=-1.0,
                      apply_qk_l2norm=True, state_indices_host=None, stream=None) -> None:
    """include/gdn.h gdn_packed_decode.  mixed_qkv [B, >= C_conv] raw rows
    (row stride taken from the tensor, so a [B, C_conv + Hv*Dv] qkvz tensor
    works as is); a_raw, b_raw [B, >= Hv] views (see packed_ba_views);
    conv_state and state are updated in place."""
    B_ = mixed_qkv.shape[0]
    sih, sih_p = _host_i32(state_indices_host)
    a = gdn_packed_decode_args(
        B=B_, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K, act_dtype=_dt(mixed_qkv),
        apply_qk_l2norm=int(apply_qk_l2norm), scale=float(scale),
        mixed_qkv=_p(mixed_qkv), mixed_qkv_stride=mixed_qkv.stride(0), mixed_qkv_len=_n(mixed_qkv),
        conv_weight=_p(conv_weight), conv_weight_len=_n(conv_weight),
        a_raw=_p(a_raw), a_raw_stride=a_raw.stride(0), a_raw_len=_n(a_raw),
        b_raw=_p(b_raw), b_raw_stride=b_raw.stride(0), b_raw_len=_n(b_raw),
        A_log=_p(A_log), A_log_len=_n(A_log), dt_bias=_p(dt_bias), dt_bias_len=_n(dt_bias),
        state_indices=_p(state_indices), state_indices_host=sih_p,
        conv_state=_p(conv_state), conv_state_len=_n(conv_state), state=_p(state),
        state_slots=state.shape[0], state_len=_n(state), out=_p(out), out_len=_n(out))
    _check(lib().gdn_packed_decode(ctypes.byref(a), _stream(stream)))


def packed_ba_views(ba: torch.Tensor, Hv: int):
    """(a_raw, b_raw) views of a merged gate tensor [T, 2*Hv] whose rows hold
    b then a ([cpu.rs] linear_attention_prepare_varlen_packed_qkvz_ba_f32)."""
    return ba[:, Hv:2 * Hv], ba[:, :Hv]


def _out_norm(norm_z, norm_weight, norm_eps, norm_sigmoid, tokens, Hv, Dv, in_kernel=False):
    """The gdn_out_norm option: None, or (struct, pointer) with z's row stride
    taken from the tensor (a [T, Hv, Dv] gate or a [T, >= Hv*Dv] slice)."""
    if norm_weight is None:
        return None, None
    zs = norm_z.stride(0)
    n = gdn_out_norm(z=_p(norm_z), z_len=max(tokens - 1, 0) * zs + Hv * Dv, z_token_stride=zs,
                     weight=_p(norm_weight), weight_len=_n(norm_weight), eps=float(norm_eps),
                     sigmoid_gate=int(bool(norm_sigmoid)), in_kernel=int(bool(in_kernel)))
    return n, ctypes.pointer(n)


def gdn_decode(q, k, v, g, beta, state, out, *, scale=-1.0, state_indices=None,
               state_indices_host=None, use_qk_l2norm=False, norm_z=None, norm_weight=None,
               norm_eps=1e-6, norm_sigmoid=False, norm_in_kernel=False, stream=None) -> None:
    """include/gdn.h gdn_decode; `state` [slots,Hv,Dv,Dk] f32 updated in place.
    With norm_weight (and norm_z) the gated RMSNorm is applied to `out`."""
    B, Hk, Dk = q.shape
    _, Hv, Dv = v.shape
    sih, sih_p = _host_i32(state_indices_host)
    nrm, nrm_p = _out_norm(norm_z, norm_weight, norm_eps, norm_sigmoid, B, Hv, Dv, norm_in_kernel)
    a = gdn_decode_args(
        B=B, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act_dtype=_dt(q), use_qk_l2norm=int(use_qk_l2norm),
        scale=float(scale), q=_p(q), q_len=_n(q), k=_p(k), k_len=_n(k), v=_p(v), v_len=_n(v),
        g=_p(g), g_len=_n(g), beta=_p(beta), beta_len=_n(beta), state=_p(state),
        state_slots=state.shape[0], state_len=_n(state), state_indices=_p(state_indices),
        state_indices_host=sih_p, out=_p(out), out_len=_n(out), out_norm=nrm_p)
    _check(lib().gdn_decode(ctypes.byref(a), _stream(stream)))


def gdn_kda_resolve_algo(T, N, Dk, Dv, act_dtype=GDN_DTYPE_BF16, algo=GDN_PREFILL_AUTO) -> int:
    return int(lib().gdn_kda_resolve_algo(T, N, Dk, Dv, act_dtype, algo))


def gdn_kda_workspace_bytes(T, N, Hv, Dk, Dv, act_dtype=GDN_DTYPE_BF16,
                            algo=GDN_PREFILL_AUTO) -> int:
    return int(lib().gdn_kda_workspace_bytes(T, N, Hv, Dk, Dv, act_dtype, algo))


def gdn_kda_varlen(q, k, v, g, beta, state, cu_seqlens, out, *, scale=-1.0, state_indices=None,
                   has_initial_state=None, cu_seqlens_host=None, state_indices_host=None,
                   algo=GDN_PREFILL_AUTO, workspace=None, stream=None) -> None:
    """include/gdn.h gdn_kda_varlen; g [T, Hv, Dk] f32; `state` updated in place.
    `workspace`: a uint8 device tensor of at least gdn_kda_workspace_bytes()
    bytes; when None and the resolved algorithm needs one, one is allocated
    here for the call."""
    T, Hk, Dk = q.shape
    _, Hv, Dv = v.shape
    N = cu_seqlens.numel() - 1
    cuh, cuh_p = _host_i32(cu_seqlens_host)
    sih, sih_p = _host_i32(state_indices_host)
    if workspace is None:
        nbytes = gdn_kda_workspace_bytes(T, N, Hv, Dk, Dv, _dt(q), algo)
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    a = gdn_kda_args(
        T=T, N=N, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act_dtype=_dt(q), scale=float(scale),
        q=_p(q), q_len=_n(q), k=_p(k), k_len=_n(k), v=_p(v), v_len=_n(v), g=_p(g), g_len=_n(g),
        beta=_p(beta), beta_len=_n(beta), state=_p(state), state_slots=state.shape[0],
        state_len=_n(state), cu_seqlens=_p(cu_seqlens), state_indices=_p(state_indices),
        has_initial_state=_p(has_initial_state), cu_seqlens_host=cuh_p,
        state_indices_host=sih_p, out=_p(out), out_len=_n(out), algo=int(algo),
        workspace=_p(workspace),
        workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size())
    _check(lib().gdn_kda_varlen(ctypes.byref(a), _stream(stream)))


def gdn_spec_decode(q, k, v, g, beta, state, cu_seqlens, state_indices, num_accepted, out, *,
                    scale=-1.0, cu_seqlens_host=None, state_indices_host=None,
                    num_accepted_host=None, stream=None) -> None:
    """include/gdn.h gdn_spec_decode; state_indices [n_reqs, num_cols] int32;
    the snapshots are written into `state` in place."""
    T, Hk, Dk = q.shape
    _, Hv, Dv = v.shape
    n_reqs, num_cols = state_indices.shape
    cuh, cuh_p = _host_i32(cu_seqlens_host)
    sih, sih_p = _host_i32(state_indices_host)
    nah, nah_p = _host_i32(num_accepted_host)
    a = gdn_spec_decode_args(
        T=T, n_reqs=n_reqs, num_cols=num_cols, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act_dtype=_dt(q),
        scale=float(scale), q=_p(q), q_len=_n(q), k=_p(k), k_len=_n(k), v=_p(v), v_len=_n(v),
        g=_p(g), g_len=_n(g), beta=_p(beta), beta_len=_n(beta), state=_p(state),
        state_slots=state.shape[0], state_len=_n(state), cu_seqlens=_p(cu_seqlens),
        state_indices=_p(state_indices), num_accepted=_p(num_accepted), cu_seqlens_host=cuh_p,
        state_indices_host=sih_p, num_accepted_host=nah_p, out=_p(out), out_len=_n(out))
    _check(lib().gdn_spec_decode(ctypes.byref(a), _stream(stream)))


def gdn_gated_rmsnorm(core, z, weight, out, *, eps=1e-6, sigmoid_gate=False, stream=None) -> None:
    """include/gdn.h gdn_gated_rmsnorm.  core, out [T, H, D]; weight [D]; z
    [T, H, D] or a [T, >= H*D] tensor whose rows are the gate's token rows
    (e.g. a slice of a merged projection), row stride taken from it."""
    T, H, D = core.shape
    z_stride = z.stride(0)
    a = gdn_gated_rmsnorm_args(
        tokens=T, heads=H, dim=D, act_dtype=_dt(core), sigmoid_gate=int(bool(sigmoid_gate)),
        eps=float(eps), core=_p(core), core_len=_n(core), z=_p(z),
        z_len=(T - 1) * z_stride + H * D, z_token_stride=z_stride, weight=_p(weight),
        weight_len=_n(weight), out=_p(out), out_len=_n(out))
    _check(lib().gdn_gated_rmsnorm(ctypes.byref(a), _stream(stream)))


def gdn_prefill_workspace_bytes(T, N, Hv, Dk, Dv, act_dtype=GDN_DTYPE_BF16,
                                algo=GDN_PREFILL_AUTO) -> int:
    return int(lib().gdn_prefill_workspace_bytes(T, N, Hv, Dk, Dv, act_dtype, algo))


def gdn_prefill_resolve_algo(N, Hv, Dk, Dv, act_dtype=GDN_DTYPE_BF16,
                             algo=GDN_PREFILL_AUTO) -> int:
    return int(lib().gdn_prefill_resolve_algo(N, Hv, Dk, Dv, act_dtype, algo))


def gdn_prefill_varlen(q, k, v, g, beta, state, cu_seqlens, out, *, scale=-1.0,
                       state_indices=None, has_initial_state=None, cu_seqlens_host=None,
                       state_indices_host=None, use_qk_l2norm=False, algo=GDN_PREFILL_AUTO,
                       workspace=None, norm_z=None, norm_weight=None, norm_eps=1e-6,
                       norm_sigmoid=False, stream=None) -> None:
    """include/gdn.h gdn_prefill_varlen; `state` updated in place.  `workspace`
    is a uint8 device tensor of at least gdn_prefill_workspace_bytes() bytes.
    With norm_weight (and norm_z) the gated RMSNorm is applied to `out`."""
    T, Hk, Dk = q.shape
    _, Hv, Dv = v.shape
    N = cu_seqlens.numel() - 1
    cuh, cuh_p = _host_i32(cu_seqlens_host)
    sih, sih_p = _host_i32(state_indices_host)
    nrm, nrm_p = _out_norm(norm_z, norm_weight, norm_eps, norm_sigmoid, T, Hv, Dv)
    a = gdn_prefill_args(
        T=T, N=N, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, act_dtype=_dt(q), use_qk_l2norm=int(use_qk_l2norm),
        scale=float(scale), algo=int(algo), q=_p(q), q_len=_n(q), k=_p(k), k_len=_n(k),
        v=_p(v), v_len=_n(v), g=_p(g), g_len=_n(g), beta=_p(beta), beta_len=_n(beta),
        state=_p(state), state_slots=state.shape[0], state_len=_n(state),
        cu_seqlens=_p(cu_seqlens), state_indices=_p(state_indices),
        has_initial_state=_p(has_initial_state), cu_seqlens_host=cuh_p,
        state_indices_host=sih_p, out=_p(out), out_len=_n(out), workspace=_p(workspace),
        workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
        out_norm=nrm_p)
    _check(lib().gdn_prefill_varlen(ctypes.byref(a), _stream(stream)))


def _host_u8(t: Optional[torch.Tensor]):
    if t is None:
        return None, None
    h = t.detach().to("cpu", torch.uint8).contiguous()
    return h, h.data_ptr()


def gdn_validate_mixed(*, num_decodes, num_prefills, num_actual_tokens, state_slots,
                       cu_seqlens_host, state_indices_host, cu_seqlens_prefill_host,
                       has_initial_state_host=None, prefill_state_indices_host=None,
                       prefill_has_initial_state_host=None, num_decode_tokens=None,
                       num_prefill_tokens=None, allow_inert_padding=True) -> None:
    """include/gdn.h gdn_validate_mixed on host copies of a mixed step's
    metadata (tensors on any device; they are copied to the host).  Raises
    GdnError on the first broken rule; launches nothing."""
    nd_tok = num_decodes if num_decode_tokens is None else num_decode_tokens
    np_tok = (num_actual_tokens - nd_tok) if num_prefill_tokens is None else num_prefill_tokens
    cu, cu_p = _host_i32(cu_seqlens_host)
    si, si_p = _host_i32(state_indices_host)
    hi, hi_p = _host_u8(has_initial_state_host)
    cp, cp_p = _host_i32(cu_seqlens_prefill_host)
    ps, ps_p = _host_i32(prefill_state_indices_host)
    ph, ph_p = _host_u8(prefill_has_initial_state_host)
    nreq = num_decodes + num_prefills
    for name, t, n in (("cu_seqlens", cu, nreq + 1), ("state_indices", si, nreq),
                       ("has_initial_state", hi, nreq), ("cu_seqlens_prefill", cp, num_prefills + 1),
                       ("prefill_state_indices", ps, num_prefills),
                       ("prefill_has_initial_state", ph, num_prefills)):
        if t is not None and t.numel() < n:
            raise GdnError(GDN_ERR_SHAPE, "GDN_ERR_SHAPE",
                           f"{name} holds {t.numel()} entries, the step needs {n}")
    m = gdn_mixed_meta(num_decodes=num_decodes, num_prefills=num_prefills,
                       num_decode_tokens=nd_tok, num_prefill_tokens=np_tok,
                       num_actual_tokens=num_actual_tokens, state_slots=state_slots,
                       allow_inert_padding=int(bool(allow_inert_padding)),
                       cu_seqlens_host=cu_p, state_indices_host=si_p, has_initial_state_host=hi_p,
                       cu_seqlens_prefill_host=cp_p, prefill_state_indices_host=ps_p,
                       prefill_has_initial_state_host=ph_p)
    _check(lib().gdn_validate_mixed(ctypes.byref(m)))


def gdn_read_device_status(stream=None) -> None:
    """Synchronises the stream and raises GdnError if a kernel flagged an error."""
    _check(lib().gdn_read_device_status(_stream(stream)))


def gdn_check_wait_timeout(budget_cycles: int, stream=None) -> None:
    """include/gdn.h gdn_check_wait_timeout: one bounded device wait that runs
    out on purpose; gdn_read_device_status then raises GDN_ERR_TIMEOUT."""
    _check(lib().gdn_check_wait_timeout(int(budget_cycles), _stream(stream)))


def gdn_version() -> int:
    return int(lib().gdn_version())


def gdn_launch_count() -> int:
    """Kernel launches issued through the library by this process so far."""
    return int(lib().gdn_launch_count())
