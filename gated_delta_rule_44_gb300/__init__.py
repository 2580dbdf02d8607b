"""GB300-native gated-delta-rule (GDN) linear-attention layer.

The compute path is libgdn (C ABI in include/gdn.h; CUDA kernels for sm_103a
under csrc/).  This package holds its thin ctypes binding, the build step, a
mixed-step helper and the seeded synthetic workloads.  The library is loaded
on first use; there is no CPU fallback.
"""
from .binding import (GDN_DTYPE_BF16, GDN_DTYPE_F32, GDN_PREFILL_AUTO, GDN_PREFILL_CHUNKED,
                      GDN_PREFILL_FUSED, GDN_PREFILL_RECURRENT, GdnError, gdn_decode, gdn_prefill_resolve_algo,
                      gdn_prefill_varlen, gdn_prefill_workspace_bytes, gdn_prepare,
                      gdn_read_device_status, gdn_version, lib)
from .layer import GdnStep, mixed_step

__all__ = [
    "GDN_DTYPE_BF16", "GDN_DTYPE_F32", "GDN_PREFILL_AUTO", "GDN_PREFILL_CHUNKED",
    "GDN_PREFILL_FUSED", "GDN_PREFILL_RECURRENT", "GdnError", "GdnStep", "gdn_decode", "gdn_prefill_resolve_algo",
    "gdn_prefill_varlen", "gdn_prefill_workspace_bytes", "gdn_prepare", "gdn_read_device_status",
    "gdn_version", "lib", "mixed_step",
]
