"""Plain CPU oracle for the gated-delta-rule (GDN) layer -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``gdn_oracle.cpp`` (a slow,
token-by-token C++ restatement of the pages' CPU code, built with
``-ffp-contract=off``) through ``ctypes``.  It shares no code with the CUDA
library and never calls it.

Sources:
  [cpu.rs]       ferrum-kernels 0.8.0, src/ferrum_kernels/backend/cpu.rs
  [cpu_ops.cpp]  vllm.cpp, src/vt/cpu/cpu_ops.cpp
  [qwen3_5.cpp]  vllm.cpp, src/vllm/model_executor/models/qwen3_5.cpp

Arrays are numpy; ``dtype`` selects the f32 or f64 instantiation.  Pools
(``state_pool``, ``conv_pool``) are updated IN PLACE, exactly like the library
calls they check; pass a copy when the original must survive.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_HDR = os.path.join(_HERE, "gdn_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_ERR_SHAPE, ORC_ERR_INVALID = 0, 1, 2


class OracleError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"oracle error {code}: {msg}")
        self.code = code
        self.msg = msg


def build(force: bool = False) -> str:
    """Compile the oracle shared library (g++, C++17, -O2, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-Wall", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
        return _lib


class using_library:
    """Context manager that routes every oracle call to another build of the
    oracle source (used by the mutation tests, which compile a copy with one
    planted mistake)."""

    def __init__(self, path: str):
        self.path = path
        self.prev = None

    def __enter__(self):
        global _lib
        L = ctypes.CDLL(self.path)
        _declare(L)
        with _lock:
            self.prev = _lib
            _lib = L
        return L

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.prev
        return False


def build_variant(src_text: str, out_dir: str) -> str:
    """Compiles `src_text` (a modified copy of gdn_oracle.cpp) with the same
    flags into out_dir; returns the library path."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "gdn_oracle.cpp")
    with open(src, "w") as fh:
        fh.write(src_text)
    with open(_HDR) as fh:
        hdr = fh.read()
    with open(os.path.join(out_dir, "gdn_oracle.h"), "w") as fh:
        fh.write(hdr)
    lib_path = os.path.join(out_dir, "libgdn_oracle_variant.so")
    subprocess.run(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", "-o", lib_path, src], check=True)
    return lib_path


def source_text() -> str:
    with open(_SRC) as fh:
        return fh.read()


_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def _declare(L):
    for suf, ct in (("f32", ctypes.c_float), ("f64", ctypes.c_double)):
        for name in ("sigmoid", "silu", "softplus"):
            fn = getattr(L, f"orc_{name}_{suf}")
            fn.restype = ct
            fn.argtypes = [ct]
        fn = getattr(L, f"orc_prepare_varlen_{suf}")
        fn.restype = ctypes.c_int
        fn.argtypes = ([_vp, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _vp, _vp, _vp]
                       + [_i64] * 7 + [ctypes.c_int] + [_vp] * 5 + [ctypes.c_int])
        fn = getattr(L, f"orc_gdn_varlen_{suf}")
        fn.restype = ctypes.c_int
        fn.argtypes = ([_vp] * 6 + [_i64, _vp, _vp, _vp] + [_i64] * 6 + [ct, ctypes.c_int, _vp,
                       _i64, _vp, ctypes.c_int])
        fn = getattr(L, f"orc_spec_prepare_{suf}")
        fn.restype = ctypes.c_int
        fn.argtypes = ([_vp, _i64, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _vp, _vp,
                        _vp] + [_i64] * 7 + [ctypes.c_int] + [_vp] * 5 + [ctypes.c_int])
        fn = getattr(L, f"orc_gdn_spec_decode_{suf}")
        fn.restype = ctypes.c_int
        fn.argtypes = ([_vp] * 6 + [_i64, _vp, _i64, _i64, _vp, _i64, _vp] + [_i64] * 4
                       + [ct, _vp, ctypes.c_int])
        fn = getattr(L, f"orc_kda_varlen_{suf}")
        fn.restype = ctypes.c_int
        fn.argtypes = ([_vp] * 6 + [_i64, _vp, _vp, _vp] + [_i64] * 6 + [ct, ctypes.c_int, _vp,
                       _i64, _vp, ctypes.c_int])
        fn = getattr(L, f"orc_gdn_decode_{suf}")
        fn.restype = ctypes.c_int
        fn.argtypes = ([_vp] * 6 + [_i64, _vp] + [_i64] * 5 + [ct, ctypes.c_int, _vp,
                       ctypes.c_int])
    L.orc_gdn_chunked_f64.restype = ctypes.c_int
    L.orc_gdn_chunked_f64.argtypes = ([_vp] * 6 + [_i64, _vp, _vp, _vp] + [_i64] * 6
                                      + [ctypes.c_double, ctypes.c_int, _i64, _vp])
    L.orc_kda_chunked_f64.restype = ctypes.c_int
    L.orc_kda_chunked_f64.argtypes = ([_vp] * 6 + [_i64, _vp, _vp, _vp] + [_i64] * 6
                                      + [ctypes.c_double, _i64, _vp])
    L.orc_validate_gated_delta_rule_shape.restype = ctypes.c_int
    L.orc_validate_gated_delta_rule_shape.argtypes = [_i64] * 13 + [ctypes.c_char_p,
                                                                    ctypes.c_size_t]
    L.orc_validate_linear_attention_prepare_shape.restype = ctypes.c_int
    L.orc_validate_linear_attention_prepare_shape.argtypes = [_i64] * 17 + [ctypes.c_char_p,
                                                                            ctypes.c_size_t]
    L.orc_validate_linear_attention_decode_prepare_shape.restype = ctypes.c_int
    L.orc_validate_linear_attention_decode_prepare_shape.argtypes = (
        [_i64] * 18 + [ctypes.c_char_p, ctypes.c_size_t])
    L.orc_gdn_deviation_bound_f64.restype = ctypes.c_int
    L.orc_gdn_deviation_bound_f64.argtypes = ([_vp] * 9 + [_i64, _vp, _vp, _vp] + [_i64] * 6
                                              + [ctypes.c_double, _vp, _vp, ctypes.c_int])
    L.orc_validate_cu_seqlens.restype = ctypes.c_int
    L.orc_validate_cu_seqlens.argtypes = [_vp, _i64, _i64, ctypes.c_char_p, ctypes.c_size_t]
    L.orc_validate_prepare_cu_seqlens.restype = ctypes.c_int
    L.orc_validate_prepare_cu_seqlens.argtypes = [_vp, _i64, _i64, ctypes.c_char_p,
                                                  ctypes.c_size_t]
    for suf, ct in (("f32", ctypes.c_float), ("f64", ctypes.c_double)):
        fn = getattr(L, f"orc_gated_rmsnorm_{suf}")
        fn.restype = ctypes.c_int
        fn.argtypes = [_vp, _vp, _i64, _vp, _vp, _i64, _i64, _i64, ct, ctypes.c_int, ctypes.c_int]
    L.orc_validate_gated_rms_norm_shape.restype = ctypes.c_int
    L.orc_validate_gated_rms_norm_shape.argtypes = [_i64] * 7 + [ctypes.c_char_p, ctypes.c_size_t]
    L.orc_validate_state_indices.restype = ctypes.c_int
    L.orc_validate_state_indices.argtypes = [_vp, _i64, _i64, ctypes.c_int, ctypes.c_char_p,
                                             ctypes.c_size_t]


def _suffix(dtype) -> str:
    dt = np.dtype(dtype)
    if dt == np.float32:
        return "f32"
    if dt == np.float64:
        return "f64"
    raise TypeError(f"oracle supports float32/float64, got {dt}")


def _arr(a, dtype, name):
    """Contiguous view/copy of `a` as `dtype` (never a view into caller data
    unless it already matches)."""
    if a is None:
        return None
    x = np.ascontiguousarray(a, dtype=dtype)
    return x


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _inplace(a, dtype, name):
    if not (isinstance(a, np.ndarray) and a.dtype == np.dtype(dtype) and a.flags.c_contiguous):
        raise TypeError(f"{name} must be a C-contiguous numpy array of {np.dtype(dtype)} "
                        "(it is updated in place)")
    return a


def _check(rc: int, what: str):
    if rc != ORC_OK:
        raise OracleError(rc, what)


# ---- scalar gate functions ----------------------------------------------------

def sigmoid(x: float, dtype=np.float64) -> float:
    return getattr(_load(), f"orc_sigmoid_{_suffix(dtype)}")(x)


def silu(x: float, dtype=np.float64) -> float:
    return getattr(_load(), f"orc_silu_{_suffix(dtype)}")(x)


def softplus(x: float, dtype=np.float64) -> float:
    return getattr(_load(), f"orc_softplus_{_suffix(dtype)}")(x)


# ---- validators (return (code, message)) ---------------------------------------

def _msgbuf():
    return ctypes.create_string_buffer(512)


def validate_gated_delta_rule_shape(*lens_and_dims):
    b = _msgbuf()
    rc = _load().orc_validate_gated_delta_rule_shape(*[int(v) for v in lens_and_dims], b, 512)
    return rc, b.value.decode()


def validate_linear_attention_prepare_shape(*lens_and_dims):
    b = _msgbuf()
    rc = _load().orc_validate_linear_attention_prepare_shape(*[int(v) for v in lens_and_dims],
                                                             b, 512)
    return rc, b.value.decode()


def validate_linear_attention_decode_prepare_shape(*lens_and_dims):
    b = _msgbuf()
    rc = _load().orc_validate_linear_attention_decode_prepare_shape(
        *[int(v) for v in lens_and_dims], b, 512)
    return rc, b.value.decode()


def validate_cu_seqlens(cu, batch, total):
    c = np.ascontiguousarray(cu, dtype=np.int32)
    b = _msgbuf()
    rc = _load().orc_validate_cu_seqlens(_ptr(c), int(batch), int(total), b, 512)
    return rc, b.value.decode()


def validate_prepare_cu_seqlens(cu, batch, total):
    c = np.ascontiguousarray(cu, dtype=np.int32)
    b = _msgbuf()
    rc = _load().orc_validate_prepare_cu_seqlens(_ptr(c), int(batch), int(total), b, 512)
    return rc, b.value.decode()


def validate_state_indices(indices, state_slots, force_full=False):
    c = np.ascontiguousarray(indices, dtype=np.int32)
    b = _msgbuf()
    rc = _load().orc_validate_state_indices(_ptr(c), c.size, int(state_slots), int(force_full),
                                            b, 512)
    return rc, b.value.decode()


# ---- O1 prepare ----------------------------------------------------------------

def prepare_varlen(mixed_qkv, conv_weight, conv_pool, a_raw, b_raw, A_log, dt_bias, cu_seqlens,
                   Hk, Hv, Dk, Dv, K, state_indices=None, has_initial_state=None,
                   apply_qk_l2norm=True, dtype=np.float32, nthreads=0):
    """O1.  mixed_qkv [T, C_conv]; conv_pool [slots, C_conv, K-1] (in place).

    Returns dict(q [T,Hk,Dk], k, v [T,Hv,Dv], g [T,Hv], beta [T,Hv])."""
    sfx = _suffix(dtype)
    x = _arr(mixed_qkv, dtype, "mixed_qkv")
    T = x.shape[0]
    x_stride = x.shape[1]
    w = _arr(conv_weight, dtype, "conv_weight")
    pool = _inplace(conv_pool, dtype, "conv_pool")
    a = _arr(a_raw, dtype, "a_raw").reshape(T, -1)
    b = _arr(b_raw, dtype, "b_raw").reshape(T, -1)
    al = _arr(A_log, dtype, "A_log")
    dtb = _arr(dt_bias, dtype, "dt_bias")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    N = cu.size - 1
    si = None if state_indices is None else np.ascontiguousarray(state_indices, dtype=np.int32)
    hi = None if has_initial_state is None else np.ascontiguousarray(has_initial_state,
                                                                     dtype=np.uint8)
    q = np.empty((T, Hk, Dk), dtype)
    k = np.empty((T, Hk, Dk), dtype)
    v = np.empty((T, Hv, Dv), dtype)
    g = np.empty((T, Hv), dtype)
    beta = np.empty((T, Hv), dtype)
    slots = pool.shape[0]
    rc = getattr(_load(), f"orc_prepare_varlen_{sfx}")(
        _ptr(x), x_stride, _ptr(w), _ptr(pool), slots, _ptr(si), _ptr(hi), _ptr(a), a.shape[1],
        _ptr(b), b.shape[1], _ptr(al), _ptr(dtb), _ptr(cu), N, T, Hk, Hv, Dk, Dv, K,
        int(apply_qk_l2norm), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), int(nthreads))
    _check(rc, "prepare_varlen")
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def spec_prepare(mixed_qkv, conv_weight, conv_pool, a_raw, b_raw, A_log, dt_bias, cu_seqlens,
                 conv_indices, num_accepted, Hk, Hv, Dk, Dv, K, apply_qk_l2norm=True,
                 dtype=np.float32, nthreads=0):
    """O8.  mixed_qkv [T, C_conv]; conv_pool [slots, C_conv, state_len] (in
    place); conv_indices, num_accepted [n_reqs].

    Returns dict(q [T,Hk,Dk], k, v [T,Hv,Dv], g [T,Hv], beta [T,Hv])."""
    sfx = _suffix(dtype)
    x = _arr(mixed_qkv, dtype, "mixed_qkv")
    T = x.shape[0]
    w = _arr(conv_weight, dtype, "conv_weight")
    pool = _inplace(conv_pool, dtype, "conv_pool")
    a = _arr(a_raw, dtype, "a_raw").reshape(T, -1)
    b = _arr(b_raw, dtype, "b_raw").reshape(T, -1)
    al = _arr(A_log, dtype, "A_log")
    dtb = _arr(dt_bias, dtype, "dt_bias")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    ci = np.ascontiguousarray(conv_indices, dtype=np.int32)
    na = np.ascontiguousarray(num_accepted, dtype=np.int32)
    q = np.empty((T, Hk, Dk), dtype)
    k = np.empty((T, Hk, Dk), dtype)
    v = np.empty((T, Hv, Dv), dtype)
    g = np.empty((T, Hv), dtype)
    beta = np.empty((T, Hv), dtype)
    rc = getattr(_load(), f"orc_spec_prepare_{sfx}")(
        _ptr(x), x.shape[1], _ptr(w), _ptr(pool), pool.shape[0], pool.shape[2], _ptr(ci),
        _ptr(na), _ptr(a), a.shape[1], _ptr(b), b.shape[1], _ptr(al), _ptr(dtb), _ptr(cu),
        cu.size - 1, T, Hk, Hv, Dk, Dv, K, int(apply_qk_l2norm), _ptr(q), _ptr(k), _ptr(v),
        _ptr(g), _ptr(beta), int(nthreads))
    _check(rc, "spec_prepare")
    return dict(q=q, k=k, v=v, g=g, beta=beta)


# ---- O2 / O3 / O4 recurrence ------------------------------------------------------

def _recur_inputs(q, k, v, g, beta, dtype):
    q = _arr(q, dtype, "q")
    k = _arr(k, dtype, "k")
    v = _arr(v, dtype, "v")
    g = _arr(g, dtype, "g")
    beta = _arr(beta, dtype, "beta")
    T, Hk, Dk = q.shape
    _, Hv, Dv = v.shape
    return q, k, v, g, beta, T, Hk, Dk, Hv, Dv


def gdn_deviation_bound(q, k, v, g, beta, dq, dk, dv, state_pool, cu_seqlens, scale,
                        state_indices=None, has_initial_state=None, nthreads=0,
                        with_state=False):
    """Test aid: a first-order bound [T, Hv, Dv] on how far each output of O2
    moves when the stored q, k, v move by at most dq, dk, dv (f64; the state
    pool is only read).  With with_state, also a bound [slots, Hv, Dv] on every
    element of each row of the live sequences' final states (0 elsewhere)."""
    q, k, v, g, beta, T, Hk, Dk, Hv, Dv = _recur_inputs(q, k, v, g, beta, np.float64)
    dq = _arr(dq, np.float64, "dq")
    dk = _arr(dk, np.float64, "dk")
    dv = _arr(dv, np.float64, "dv")
    pool = np.ascontiguousarray(state_pool, dtype=np.float64)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    si = None if state_indices is None else np.ascontiguousarray(state_indices, dtype=np.int32)
    hi = None if has_initial_state is None else np.ascontiguousarray(has_initial_state,
                                                                     dtype=np.uint8)
    bound = np.zeros((T, Hv, Dv), np.float64)
    sbound = np.zeros((pool.shape[0], Hv, Dv), np.float64) if with_state else None
    rc = _load().orc_gdn_deviation_bound_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(pool), pool.shape[0], _ptr(si), _ptr(hi), _ptr(cu), cu.size - 1, T, Hk, Hv, Dk, Dv,
        float(scale), _ptr(bound), _ptr(sbound), int(nthreads))
    _check(rc, "gdn_deviation_bound")
    return (bound, sbound) if with_state else bound


def gdn_varlen(q, k, v, g, beta, state_pool, cu_seqlens, scale, state_indices=None,
               has_initial_state=None, use_qk_l2norm=False, items=None, out=None,
               dtype=np.float32, nthreads=0):
    """O2.  q,k [T,Hk,Dk]; v [T,Hv,Dv]; g,beta [T,Hv]; state_pool [slots,Hv,Dv,Dk]
    updated in place.  Returns out [T,Hv,Dv] (only `items` rows written if given)."""
    sfx = _suffix(dtype)
    q, k, v, g, beta, T, Hk, Dk, Hv, Dv = _recur_inputs(q, k, v, g, beta, dtype)
    pool = _inplace(state_pool, dtype, "state_pool")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    si = None if state_indices is None else np.ascontiguousarray(state_indices, dtype=np.int32)
    hi = None if has_initial_state is None else np.ascontiguousarray(has_initial_state,
                                                                     dtype=np.uint8)
    it = None if items is None else np.ascontiguousarray(items, dtype=np.int32)
    if out is None:
        out = np.zeros((T, Hv, Dv), dtype)
    out = _inplace(out, dtype, "out")
    rc = getattr(_load(), f"orc_gdn_varlen_{sfx}")(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(pool), pool.shape[0], _ptr(si),
        _ptr(hi), _ptr(cu), cu.size - 1, T, Hk, Hv, Dk, Dv, float(scale), int(use_qk_l2norm),
        _ptr(it), 0 if it is None else it.size, _ptr(out), int(nthreads))
    _check(rc, "gdn_varlen")
    return out


def gdn_spec_decode(q, k, v, g, beta, state_pool, cu_seqlens, state_indices, num_accepted,
                    scale, out=None, dtype=np.float32, nthreads=0):
    """O7.  state_indices [n_reqs, num_cols] (int32), num_accepted [n_reqs];
    state_pool [slots, Hv, Dv, Dk] updated in place (the snapshots).  Returns
    out [T, Hv, Dv]."""
    sfx = _suffix(dtype)
    q, k, v, g, beta, T, Hk, Dk, Hv, Dv = _recur_inputs(q, k, v, g, beta, dtype)
    pool = _inplace(state_pool, dtype, "state_pool")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    si = np.ascontiguousarray(state_indices, dtype=np.int32)
    na = np.ascontiguousarray(num_accepted, dtype=np.int32)
    if out is None:
        out = np.zeros((T, Hv, Dv), dtype)
    out = _inplace(out, dtype, "out")
    rc = getattr(_load(), f"orc_gdn_spec_decode_{sfx}")(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(pool), pool.shape[0], _ptr(cu),
        cu.size - 1, T, _ptr(si), si.shape[1], _ptr(na), Hk, Hv, Dk, Dv, float(scale),
        _ptr(out), int(nthreads))
    _check(rc, "gdn_spec_decode")
    return out


def kda_varlen(q, k, v, g, beta, state_pool, cu_seqlens, scale, state_indices=None,
               has_initial_state=None, items=None, out=None, dtype=np.float32, nthreads=0):
    """O6, the KDA recurrence.  As gdn_varlen, but g [T,Hv,Dk] is a log decay per
    key channel and q, k are used as given (no L2 norm)."""
    sfx = _suffix(dtype)
    q, k, v, g, beta, T, Hk, Dk, Hv, Dv = _recur_inputs(q, k, v, g, beta, dtype)
    if g.shape != (T, Hv, Dk):
        raise ValueError(f"KDA g must be [T, Hv, Dk] = {(T, Hv, Dk)}, got {g.shape}")
    pool = _inplace(state_pool, dtype, "state_pool")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    si = None if state_indices is None else np.ascontiguousarray(state_indices, dtype=np.int32)
    hi = None if has_initial_state is None else np.ascontiguousarray(has_initial_state,
                                                                     dtype=np.uint8)
    it = None if items is None else np.ascontiguousarray(items, dtype=np.int32)
    if out is None:
        out = np.zeros((T, Hv, Dv), dtype)
    out = _inplace(out, dtype, "out")
    rc = getattr(_load(), f"orc_kda_varlen_{sfx}")(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(pool), pool.shape[0], _ptr(si),
        _ptr(hi), _ptr(cu), cu.size - 1, T, Hk, Hv, Dk, Dv, float(scale), 0,
        _ptr(it), 0 if it is None else it.size, _ptr(out), int(nthreads))
    _check(rc, "kda_varlen")
    return out


def gdn_decode(q, k, v, g, beta, state_pool, scale, state_indices=None, use_qk_l2norm=False,
               dtype=np.float32, nthreads=0):
    """O3.  One token per row b; pool slot state_indices[b] updated in place."""
    sfx = _suffix(dtype)
    q, k, v, g, beta, B, Hk, Dk, Hv, Dv = _recur_inputs(q, k, v, g, beta, dtype)
    pool = _inplace(state_pool, dtype, "state_pool")
    si = None if state_indices is None else np.ascontiguousarray(state_indices, dtype=np.int32)
    out = np.empty((B, Hv, Dv), dtype)
    rc = getattr(_load(), f"orc_gdn_decode_{sfx}")(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(pool), pool.shape[0], _ptr(si), B,
        Hk, Hv, Dk, Dv, float(scale), int(use_qk_l2norm), _ptr(out), int(nthreads))
    _check(rc, "gdn_decode")
    return out


def gdn_chunked_f64(q, k, v, g, beta, state_pool, cu_seqlens, scale, chunk,
                    state_indices=None, has_initial_state=None, use_qk_l2norm=False):
    """O4 (f64 only): the chunked WY/UT form; same contract as gdn_varlen."""
    q, k, v, g, beta, T, Hk, Dk, Hv, Dv = _recur_inputs(q, k, v, g, beta, np.float64)
    pool = _inplace(state_pool, np.float64, "state_pool")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    si = None if state_indices is None else np.ascontiguousarray(state_indices, dtype=np.int32)
    hi = None if has_initial_state is None else np.ascontiguousarray(has_initial_state,
                                                                     dtype=np.uint8)
    out = np.zeros((T, Hv, Dv), np.float64)
    rc = _load().orc_gdn_chunked_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(pool), pool.shape[0], _ptr(si),
        _ptr(hi), _ptr(cu), cu.size - 1, T, Hk, Hv, Dk, Dv, float(scale), int(use_qk_l2norm),
        int(chunk), _ptr(out))
    _check(rc, "gdn_chunked_f64")
    return out


def kda_chunked_f64(q, k, v, g, beta, state_pool, cu_seqlens, scale, chunk,
                    state_indices=None, has_initial_state=None):
    """O9 (f64 only): the chunked form of the KDA recurrence; same contract as
    kda_varlen (g [T, Hv, Dk])."""
    q, k, v, g, beta, T, Hk, Dk, Hv, Dv = _recur_inputs(q, k, v, g, beta, np.float64)
    pool = _inplace(state_pool, np.float64, "state_pool")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    si = None if state_indices is None else np.ascontiguousarray(state_indices, dtype=np.int32)
    hi = None if has_initial_state is None else np.ascontiguousarray(has_initial_state,
                                                                     dtype=np.uint8)
    out = np.zeros((T, Hv, Dv), np.float64)
    rc = _load().orc_kda_chunked_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(pool), pool.shape[0], _ptr(si),
        _ptr(hi), _ptr(cu), cu.size - 1, T, Hk, Hv, Dk, Dv, float(scale), int(chunk), _ptr(out))
    _check(rc, "kda_chunked_f64")
    return out


def num_threads_default() -> int:
    return os.cpu_count() or 1


# ---- O5 gated RMSNorm -------------------------------------------------------------

def validate_gated_rms_norm_shape(core_len, z_len, weight_len, out_len, tokens, heads, dim):
    b = _msgbuf()
    rc = _load().orc_validate_gated_rms_norm_shape(int(core_len), int(z_len), int(weight_len),
                                                    int(out_len), int(tokens), int(heads),
                                                    int(dim), b, 512)
    return rc, b.value.decode()


def gated_rmsnorm(core, z, weight, eps, sigmoid_gate=False, dtype=np.float64, nthreads=0):
    """out [T, H, D] = core / sqrt(mean_d core^2 + eps) * weight * act(z) per (token, head).
    core [T, H, D]; z [T, H, D] or [T, >= H*D] (token rows of the gate, as a
    merged projection's slice: the first H*D entries of each row are used)."""
    dt = np.dtype(dtype)
    core = _arr(core, dt, "core")
    T, H, D = core.shape
    z = _arr(z, dt, "z")
    z2 = z.reshape(T, -1)
    if z2.shape[1] < H * D:
        raise ValueError("z rows shorter than heads * dim")
    w = _arr(weight, dt, "weight")
    out = np.empty_like(core)
    rc, msg = validate_gated_rms_norm_shape(core.size, T * H * D, w.size, out.size, T, H, D)
    if rc != ORC_OK:
        raise OracleError(rc, msg)
    fn = getattr(_load(), f"orc_gated_rmsnorm_{_suffix(dt)}")
    _check(fn(_ptr(core), _ptr(z2), z2.shape[1], _ptr(w), _ptr(out), T, H, D, eps,
              int(bool(sigmoid_gate)), int(nthreads)), "gated_rmsnorm")
    return out
