"""Exact tiled attention (forward and backward) for one GB300 (sm_103a).

The compute path is the shared library built from ``csrc/`` (``libattn.so``):
hand-written tcgen05/TMA kernels behind a C ABI (``include/attn.h``).  This
package only marshals arguments into that library; it has no CPU fallback.

``synth`` (seeded input generation) imports without the library.  The binding
functions load the library on first use and raise if it is missing.
"""
from __future__ import annotations

__all__ = ["attn_fwd", "attn_fwd_raw", "attn_fwd_fp8", "attn_fwd_fp8_raw", "attn_fwd_fp4p", "attn_fwd_fp4p_raw", "attn_fwd_host", "attn_fwd_host_raw", "fwd_host_workspace_bytes", "attn_fwd_fp8_host", "attn_fwd_fp8_host_raw", "fp8_host_workspace_bytes", "attn_fwd_fp4p_host", "attn_fwd_fp4p_host_raw", "fp4p_host_workspace_bytes", "attn_status_string", "load_library", "AttnError",
           "attn_fwd_partial", "attn_fwd_partial_raw", "attn_merge", "attn_merge_raw",
           "attn_fwd_splitkv", "attn_fwd_splitkv_raw", "splitkv_workspace_bytes",
           "attn_bwd", "attn_bwd_raw", "bwd_workspace_bytes", "attn_bwd_host", "bwd_host_workspace_bytes",
           "check_device_errors", "set_wait_timeout_ns", "selftest_wait_timeout", "measure_exp2_rates", "eval_exp2",
           "diag_tmem_row_max", "diag_fwd_schedule", "diag_force_fwd_order", "diag_set_pair_tail",
           "ORDER_HEADS", "ORDER_ZIGZAG", "ORDER_GROUPS"]


def __getattr__(name):
    if name in __all__:
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
