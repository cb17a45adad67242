"""ctypes binding of libattn.so (argument marshalling only).

Every step of the attention computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or the device is not sm_103,
the calls raise AttnError.
"""
from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

ATTN_OK = 0
ATTN_BF16 = 0
# attn_status codes (include/attn.h)
ATTN_ERR_NULL = -1
ATTN_ERR_DIMS = -2
ATTN_ERR_UNSUPPORTED_HEADDIM = -3
ATTN_ERR_DTYPE = -4
ATTN_ERR_ALIGN = -5
ATTN_ERR_OVERFLOW = -6
ATTN_ERR_LAUNCH = -7
ATTN_ERR_TIMEOUT = -8
ATTN_ERR_ARCH = -9
ATTN_ERR_SCALE = -10
ATTN_ERR_CUDA = -11
ATTN_ERR_SCRATCH = -12
ATTN_ERR_WORKSPACE = -13

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {attn_status_string(status)} ({status})" if what else attn_status_string(status))


def load_library():
    """Loads libattn.so (built by exact_tiled_attention_16_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m exact_tiled_attention_16_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp]
    lib.attn_fwd.restype = ci
    lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp]
    lib.attn_fwd_fp8.restype = ci
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp, ctypes.c_size_t, vp]
    lib.attn_fwd_host.restype = ci
    lib.attn_fwd_host_workspace_bytes.argtypes = [ci, ci, ci, ci]
    lib.attn_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_fwd_fp8_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp, ctypes.c_size_t,
                                      vp]
    lib.attn_fwd_fp8_host.restype = ci
    lib.attn_fwd_fp8_host_workspace_bytes.argtypes = [ci, ci, ci, ci]
    lib.attn_fwd_fp8_host_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_fwd_fp4p_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp,
                                       ctypes.c_size_t, vp]
    lib.attn_fwd_fp4p_host.restype = ci
    lib.attn_fwd_fp4p_host_workspace_bytes.argtypes = [ci, ci, ci, ci]
    lib.attn_fwd_fp4p_host_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_fwd_fp4p.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp]
    lib.attn_fwd_fp4p.restype = ci
    lib.attn_fwd_partial.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, cf, vp]
    lib.attn_fwd_partial.restype = ci
    lib.attn_merge.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ci, vp, vp, ci, ci, ci, ci, ci, vp]
    lib.attn_merge.restype = ci
    lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp, ctypes.c_size_t, vp]
    lib.attn_fwd_splitkv.restype = ci
    lib.attn_splitkv_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
    lib.attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp, ctypes.c_size_t, vp]
    lib.attn_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp, ctypes.c_size_t,
                                  vp]
    lib.attn_bwd_host.restype = ci
    lib.attn_bwd_host_workspace_bytes.argtypes = [ci, ci, ci, ci]
    lib.attn_bwd_host_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_bwd.restype = ci
    lib.attn_bwd_workspace_bytes.argtypes = [ci, ci, ci]
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_status_string.argtypes = [ci]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_check_device_errors.argtypes = [vp, ctypes.POINTER(ci)]
    lib.attn_check_device_errors.restype = ci
    lib.attn_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
    lib.attn_set_wait_timeout_ns.restype = ci
    lib.attn_selftest_wait_timeout.argtypes = [vp]
    lib.attn_selftest_wait_timeout.restype = ci
    lib.attn_measure_exp2_rates.argtypes = [ctypes.POINTER(cf), ctypes.POINTER(cf), vp]
    lib.attn_measure_exp2_rates.restype = ci
    lib.attn_eval_exp2.argtypes = [vp, vp, vp, ctypes.c_longlong, vp]
    lib.attn_eval_exp2.restype = ci
    lib.attn_diag_tmem_row_max.argtypes = [vp, vp, vp, vp, vp]
    lib.attn_diag_tmem_row_max.restype = ci
    lib.attn_diag_fwd_schedule.argtypes = [ci, ci, ci, ci, ci, ci, ctypes.c_longlong, ci, ci, vp, vp,
                                           ctypes.c_longlong]
    lib.attn_diag_fwd_schedule.restype = ci
    lib.attn_diag_force_fwd_order.argtypes = [ci, ci]
    lib.attn_diag_force_fwd_order.restype = ci
    lib.attn_diag_set_pair_tail.argtypes = [ci]
    lib.attn_diag_set_pair_tail.restype = ci
    _lib = lib
    return lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def attn_fwd_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int, causal: bool,
                 scale: float, stream: int, dtype: int = ATTN_BF16) -> int:
    """Direct call with device pointers; returns the attn_status."""
    return load_library().attn_fwd(q or None, k or None, v or None, o or None, lse or None, B, H, N, d,
                                   1 if causal else 0, float(scale), dtype, stream or None)


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None,
             want_lse: bool = True, stream=None):
    """Exact attention forward for torch CUDA tensors q, k, v [B,H,N,d] bf16.

    Returns (o, lse); o is bf16 [B,H,N,d], lse float32 [B,H,N] (None if
    want_lse is False and no lse buffer was given).  Output buffers may be passed
    in to avoid allocation.  Asynchronous on `stream` (default: torch's current
    stream)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [B,H,N,d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same shape [B,H,N,d]")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    rc = attn_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                      lse.data_ptr() if lse is not None else 0, B, H, N, d, causal, scale,
                      _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return o, lse


def attn_fwd_fp8_raw(q8: int, k8: int, v8: int, q_scale: int, k_scale: int, v_scale: int, o: int, lse: int,
                     B: int, H: int, N: int, d: int, causal: bool, scale: float, stream: int) -> int:
    """Direct call of the block-scaled FP8 entry point with device pointers."""
    return load_library().attn_fwd_fp8(q8 or None, k8 or None, v8 or None, q_scale or None, k_scale or None,
                                       v_scale or None, o or None, lse or None, B, H, N, d,
                                       1 if causal else 0, float(scale), stream or None)


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool = False, scale: float | None = None,
                 o=None, lse=None, want_lse: bool = True, stream=None):
    """Block-scaled FP8 attention forward for torch CUDA tensors.

    q8, k8, v8: e4m3 codes [B,H,N,d] (torch.uint8 or torch.float8_e4m3fn);
    *_scale: float32 [B,H,ceil(N/128)].  Returns (o bf16 [B,H,N,d], lse)."""
    import torch
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if t.element_size() != 1 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous CUDA e4m3 (1-byte) tensor [B,H,N,d]")
    B, H, N, d = q8.shape
    T = (N + 127) // 128
    for name, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, H, T):
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor [B,H,ceil(N/128)]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    rc = attn_fwd_fp8_raw(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), q_scale.data_ptr(), k_scale.data_ptr(),
                          v_scale.data_ptr(), o.data_ptr(), lse.data_ptr() if lse is not None else 0,
                          B, H, N, d, causal, scale, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp8")
    return o, lse


def fwd_host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().attn_fwd_host_workspace_bytes(B, H, N, d))


def fp8_host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().attn_fwd_fp8_host_workspace_bytes(B, H, N, d))


def attn_fwd_fp8_host_raw(q8: int, k8: int, v8: int, q_scale: int, k_scale: int, v_scale: int, o: int, lse: int,
                          B: int, H: int, N: int, d: int, causal: bool, scale: float, workspace: int,
                          workspace_bytes: int, stream: int) -> int:
    return load_library().attn_fwd_fp8_host(q8 or None, k8 or None, v8 or None, q_scale or None, k_scale or None,
                                            v_scale or None, o or None, lse or None, B, H, N, d,
                                            1 if causal else 0, float(scale), workspace or None,
                                            int(workspace_bytes), stream or None)


def attn_fwd_fp8_host(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool = False, scale: float | None = None,
                      o=None, lse=None, want_lse: bool = True, workspace=None, stream=None):
    """attn_fwd_fp8 on HOST tensors (page-locked for full speed): e4m3 codes
    q8, k8, v8 [B,H,N,d] (1-byte dtype) and float32 block scales [B,H,ceil(N/128)];
    transfers and kernels are pipelined by the library.  Returns host (o bf16,
    lse), valid once `stream` (default: torch's current stream) has completed.  The
    device workspace is allocated with torch when not given."""
    import torch
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if t.element_size() != 1 or t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous host e4m3 (1-byte) tensor [B,H,N,d]")
    if k8.shape != q8.shape or v8.shape != q8.shape:
        raise ValueError("q8, k8 and v8 must have the same shape [B,H,N,d]")
    B, H, N, d = q8.shape
    T = (N + 127) // 128
    for name, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        if t.dtype != torch.float32 or t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, H, T):
            raise ValueError(f"{name} must be a contiguous host float32 tensor [B,H,ceil(N/128)]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = q8.is_pinned()
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, pin_memory=pin)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    need = fp8_host_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = attn_fwd_fp8_host_raw(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), q_scale.data_ptr(), k_scale.data_ptr(),
                               v_scale.data_ptr(), o.data_ptr(), lse.data_ptr() if lse is not None else 0,
                               B, H, N, d, causal, scale, workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp8_host")
    return o, lse


def attn_fwd_host_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int, causal: bool,
                      scale: float, workspace: int, workspace_bytes: int, stream: int) -> int:
    return load_library().attn_fwd_host(q or None, k or None, v or None, o or None, lse or None, B, H, N, d,
                                        1 if causal else 0, float(scale), workspace or None, int(workspace_bytes),
                                        stream or None)


def attn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None,
                  want_lse: bool = True, workspace=None, stream=None):
    """attn_fwd on HOST tensors q, k, v [B,H,N,d] bf16 (page-locked for full
    speed); transfers and kernels are pipelined by the library.  Returns host
    (o, lse), valid once `stream` (default: torch's current stream) has
    completed.  The device workspace is allocated with torch when not given."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous host bf16 tensor [B,H,N,d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same shape [B,H,N,d]")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = q.is_pinned()
    if o is None:
        o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    need = fwd_host_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = attn_fwd_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr() if lse is not None else 0, B, H, N, d, causal, scale,
                           workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                           _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")
    return o, lse


def fp4p_host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().attn_fwd_fp4p_host_workspace_bytes(B, H, N, d))


def attn_fwd_fp4p_host_raw(q8: int, k8: int, vt4: int, q_scale: int, k_scale: int, vt_scale: int, o: int, lse: int,
                           B: int, H: int, N: int, d: int, causal: bool, scale: float, workspace: int,
                           workspace_bytes: int, stream: int) -> int:
    return load_library().attn_fwd_fp4p_host(q8 or None, k8 or None, vt4 or None, q_scale or None, k_scale or None,
                                             vt_scale or None, o or None, lse or None, B, H, N, d,
                                             1 if causal else 0, float(scale), workspace or None,
                                             int(workspace_bytes), stream or None)


def attn_fwd_fp4p_host(q8, k8, vt4, q_scale, k_scale, vt_scale, causal: bool = False, scale: float | None = None,
                       o=None, lse=None, want_lse: bool = True, workspace=None, stream=None):
    """attn_fwd_fp4p on HOST tensors (page-locked for full speed), in its layouts;
    transfers and kernels are pipelined by the library.  Returns host (o bf16,
    lse), valid once `stream` (default: torch's current stream) has completed."""
    import torch
    for name, t, dt in (("q8", q8, torch.uint8), ("k8", k8, torch.uint8), ("vt4", vt4, torch.uint8),
                        ("q_scale", q_scale, torch.float32), ("k_scale", k_scale, torch.float32),
                        ("vt_scale", vt_scale, torch.uint8)):
        if t.dtype != dt or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host {dt} tensor")
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or vt4.shape != (B, H, d, N // 2) or vt_scale.shape != (B, H, d, N // 32):
        raise ValueError("shapes: q8, k8 [B,H,N,d]; vt4 [B,H,d,N/2]; vt_scale [B,H,d,N/32]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = q8.is_pinned()
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, pin_memory=pin)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    need = fp4p_host_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = attn_fwd_fp4p_host_raw(q8.data_ptr(), k8.data_ptr(), vt4.data_ptr(), q_scale.data_ptr(),
                                k_scale.data_ptr(), vt_scale.data_ptr(), o.data_ptr(),
                                lse.data_ptr() if lse is not None else 0, B, H, N, d, causal, scale,
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp4p_host")
    return o, lse


def attn_fwd_fp4p_raw(q8: int, k8: int, vt4: int, q_scale: int, k_scale: int, vt_scale: int, o: int, lse: int,
                      B: int, H: int, N: int, d: int, causal: bool, scale: float, stream: int) -> int:
    return load_library().attn_fwd_fp4p(q8 or None, k8 or None, vt4 or None, q_scale or None, k_scale or None,
                                        vt_scale or None, o or None, lse or None, B, H, N, d, 1 if causal else 0,
                                        float(scale), stream or None)


def attn_fwd_fp4p(q8, k8, vt4, q_scale, k_scale, vt_scale, causal: bool = False, scale: float | None = None,
                  o=None, lse=None, want_lse: bool = True, stream=None):
    """Direct-P FP4 attention forward.  q8, k8: uint8 e4m3 codes [B,H,N,d] with
    fp32 block scales [B,H,N/128]; vt4: uint8 MXFP4 codes of V^T [B,H,d,N/2];
    vt_scale: uint8 E8M0 scales [B,H,d,N/32].  Returns (o bf16, lse fp32)."""
    import torch
    for name, t, dt in (("q8", q8, torch.uint8), ("k8", k8, torch.uint8), ("vt4", vt4, torch.uint8),
                        ("q_scale", q_scale, torch.float32), ("k_scale", k_scale, torch.float32),
                        ("vt_scale", vt_scale, torch.uint8)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or vt4.shape != (B, H, d, N // 2) or vt_scale.shape != (B, H, d, N // 32):
        raise ValueError("shapes: q8, k8 [B,H,N,d]; vt4 [B,H,d,N/2]; vt_scale [B,H,d,N/32]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    rc = attn_fwd_fp4p_raw(q8.data_ptr(), k8.data_ptr(), vt4.data_ptr(), q_scale.data_ptr(), k_scale.data_ptr(),
                           vt_scale.data_ptr(), o.data_ptr(), lse.data_ptr() if lse is not None else 0, B, H, N, d,
                           causal, scale, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp4p")
    return o, lse


def _check_bf16(*named):
    import torch
    for name, t in named:
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [B,H,N,d]")


def attn_fwd_partial_raw(q: int, k: int, v: int, o_part: int, lse_part: int, B: int, H: int, Nq: int, Nk: int,
                         d: int, causal: bool, q_offset: int, k_offset: int, scale: float, stream: int) -> int:
    return load_library().attn_fwd_partial(q or None, k or None, v or None, o_part or None, lse_part or None,
                                           B, H, Nq, Nk, d, 1 if causal else 0, q_offset, k_offset,
                                           float(scale), stream or None)


def attn_fwd_partial(q, k, v, causal: bool = False, q_offset: int = 0, k_offset: int = 0,
                     scale: float | None = None, o_part=None, lse_part=None, stream=None):
    """Attention of q [B,H,Nq,d] against one K/V shard [B,H,Nk,d] (bf16, CUDA).

    Returns (o_part float32 [B,H,Nq,d], lse_part float32 [B,H,Nq]): the shard's
    partial result, O normalised by the shard's own sum; rows without a visible
    key get O = 0 and lse = -inf."""
    import torch
    _check_bf16(("q", q), ("k", k), ("v", v))
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != d:
        raise ValueError("k and v must be [B,H,Nk,d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o_part is None:
        o_part = torch.empty((B, H, Nq, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    rc = attn_fwd_partial_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(),
                              B, H, Nq, Nk, d, causal, q_offset, k_offset, scale, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_partial")
    return o_part, lse_part


def attn_merge_raw(o_parts, lse_parts, o: int, lse: int, out_fp32: bool, B: int, H: int, N: int, d: int,
                   stream: int) -> int:
    n = len(o_parts)
    arr_o = (ctypes.c_void_p * max(1, n))(*[x or None for x in o_parts])
    arr_l = (ctypes.c_void_p * max(1, n))(*[x or None for x in lse_parts])
    return load_library().attn_merge(arr_o, arr_l, n, o or None, lse or None, 1 if out_fp32 else 0,
                                     B, H, N, d, stream or None)


def attn_merge(parts, out=None, lse=None, out_fp32: bool = False, stream=None):
    """Exact merge of partial results [(o_s float32 [B,H,N,d], lse_s float32 [B,H,N]), ...].

    Returns (o, lse); o is bf16 unless out_fp32.  `out`/`lse` may be the first
    partial's tensors (in-place running merge, out_fp32=True)."""
    import torch
    o0, l0 = parts[0]
    B, H, N, d = o0.shape
    for o_s, l_s in parts:
        if o_s.dtype != torch.float32 or l_s.dtype != torch.float32 or o_s.shape != o0.shape \
                or l_s.shape != l0.shape or not o_s.is_contiguous() or not l_s.is_contiguous():
            raise ValueError("partials must be contiguous float32 [B,H,N,d] and [B,H,N]")
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=o0.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=o0.device)
    rc = attn_merge_raw([o.data_ptr() for o, _ in parts], [l.data_ptr() for _, l in parts], out.data_ptr(),
                        lse.data_ptr(), out_fp32, B, H, N, d, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_merge")
    return out, lse


def splitkv_workspace_bytes(B: int, H: int, Nq: int, d: int, num_splits: int) -> int:
    return int(load_library().attn_splitkv_workspace_bytes(B, H, Nq, d, num_splits))


def attn_fwd_splitkv_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Nq: int, Nk: int, d: int,
                         causal: bool, scale: float, num_splits: int, workspace: int, workspace_bytes: int,
                         stream: int) -> int:
    return load_library().attn_fwd_splitkv(q or None, k or None, v or None, o or None, lse or None, B, H, Nq, Nk,
                                           d, 1 if causal else 0, float(scale), num_splits, workspace or None,
                                           int(workspace_bytes), stream or None)


def attn_fwd_splitkv(q, k, v, num_splits: int, causal: bool = False, scale: float | None = None, o=None,
                     lse=None, want_lse: bool = True, workspace=None, stream=None):
    """Split-K/V attention: q [B,H,Nq,d], k/v [B,H,Nk,d] bf16 CUDA tensors.

    Under the causal mask the queries are the last Nq of the Nk positions.  The
    scratch workspace (a CUDA tensor of at least splitkv_workspace_bytes bytes)
    is allocated with torch when not given."""
    import torch
    _check_bf16(("q", q), ("k", k), ("v", v))
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    need = splitkv_workspace_bytes(B, H, Nq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = attn_fwd_splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr() if lse is not None else 0, B, H, Nq, Nk, d, causal, scale,
                              num_splits, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_splitkv")
    return o, lse


def bwd_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(load_library().attn_bwd_workspace_bytes(B, H, N))


def attn_bwd_raw(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int, B: int, H: int,
                 N: int, d: int, causal: bool, scale: float, workspace: int, workspace_bytes: int,
                 stream: int) -> int:
    return load_library().attn_bwd(q or None, k or None, v or None, o or None, dout or None, lse or None,
                                   dq or None, dk or None, dv or None, B, H, N, d, 1 if causal else 0,
                                   float(scale), workspace or None, int(workspace_bytes), stream or None)


def attn_bwd(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None, dq=None, dk=None,
             dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attn_fwd for bf16 CUDA tensors [B,H,N,d].

    o and lse are attn_fwd's outputs for the same q, k, v, causal flag and scale;
    dout is the gradient of o.  The workspace (a CUDA tensor of at least
    bwd_workspace_bytes bytes) is allocated with torch when not given."""
    import torch
    _check_bf16(("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout))
    if any(t.shape != q.shape for t in (k, v, o, dout)):
        raise ValueError("q, k, v, o and dout must have the same shape [B,H,N,d]")
    B, H, N, d = q.shape
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be a contiguous CUDA float32 tensor [B,H,N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    need = bwd_workspace_bytes(B, H, N)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = attn_bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, causal, scale,
                      workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def bwd_host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().attn_bwd_host_workspace_bytes(B, H, N, d))


def attn_bwd_host(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None, dq=None, dk=None,
                  dv=None, workspace=None, stream=None):
    """attn_bwd on HOST tensors (bf16 [B,H,N,d], lse float32 [B,H,N]; page-locked
    for full speed); transfers and kernels are pipelined by the library.  Returns
    host (dq, dk, dv), valid once `stream` (default: torch's current stream) has
    completed."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous host bf16 tensor [B,H,N,d]")
    if any(t.shape != q.shape for t in (k, v, o, dout)):
        raise ValueError("q, k, v, o and dout must have the same shape [B,H,N,d]")
    B, H, N, d = q.shape
    if lse.dtype != torch.float32 or lse.is_cuda or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be a contiguous host float32 tensor [B,H,N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = q.is_pinned()
    dq = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if dq is None else dq
    dk = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if dk is None else dk
    dv = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if dv is None else dv
    need = bwd_host_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = load_library().attn_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                                      lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                      1 if causal else 0, float(scale), workspace.data_ptr(),
                                      workspace.numel() * workspace.element_size(), _stream_handle(stream) or None)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_host")
    return dq, dk, dv


def check_device_errors(stream=None):
    """Synchronises the stream and returns (status, where) of the device error word."""
    where = ctypes.c_int(0)
    rc = load_library().attn_check_device_errors(_stream_handle(stream) or None, ctypes.byref(where))
    return rc, where.value


def set_wait_timeout_ns(ns: int) -> int:
    return load_library().attn_set_wait_timeout_ns(int(ns))


def selftest_wait_timeout(stream=None) -> int:
    return load_library().attn_selftest_wait_timeout(_stream_handle(stream) or None)


def measure_exp2_rates(stream=None):
    """(ex2 per SM clock per SM on the special-function unit, FMA-pipe polynomial
    exponentials per SM clock per SM), measured on the current device."""
    a, b = ctypes.c_float(0.0), ctypes.c_float(0.0)
    rc = load_library().attn_measure_exp2_rates(ctypes.byref(a), ctypes.byref(b), _stream_handle(stream) or None)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_measure_exp2_rates")
    return float(a.value), float(b.value)


def eval_exp2(x, stream=None):
    """(y_poly, y_sfu) for a CUDA float32 tensor x: the FMA-pipe polynomial
    exponential and ex2.approx, evaluated by the library's device code."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 tensor")
    y_poly = torch.empty_like(x)
    y_sfu = torch.empty_like(x)
    rc = load_library().attn_eval_exp2(x.data_ptr(), y_poly.data_ptr(), y_sfu.data_ptr(), x.numel(),
                                       _stream_handle(stream) or None)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_eval_exp2")
    return y_poly, y_sfu


def diag_tmem_row_max(x, stream=None):
    """(vals, row_max, block_max) for a contiguous CUDA float32 tensor x of shape
    (128, 128): the tile passed through tensor memory and loaded back with the
    loads-with-maximum the forward kernel uses (the row's, and each 32-column
    group's)."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous() or tuple(x.shape) != (128, 128):
        raise ValueError("x must be a contiguous CUDA float32 tensor of shape (128, 128)")
    vals = torch.empty_like(x)
    row_max = torch.empty(128, dtype=torch.float32, device=x.device)
    block_max = torch.empty((128, 4), dtype=torch.float32, device=x.device)
    rc = load_library().attn_diag_tmem_row_max(x.data_ptr(), vals.data_ptr(), row_max.data_ptr(),
                                               block_max.data_ptr(), _stream_handle(stream) or None)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_diag_tmem_row_max")
    return vals, row_max, block_max


ORDER_HEADS, ORDER_ZIGZAG, ORDER_GROUPS = 0, 1, 2


def diag_fwd_schedule(BH, Nq, Nk, causal, d=128, num_sms=152, q_offset=0, k_offset=0, kv_key_bytes=None,
                      table_ok=True, fp8=False):
    """The forward kernel's unit schedule for a launch shape (host only, no GPU):
    (info, seq) with info = {order, group_heads, grid, rounds, makespan, table,
    pair_tail} and seq an int32 array [grid, rounds] of unit ids (-3 - unit: the
    odd CTA of a split pair-tail unit, -2: skipped iteration, -1: done).
    table_ok: a BF16 attn_fwd launch (True) or another entry point; fp8: an
    attn_fwd_fp8 launch (K/V bytes per key 2 d unless given)."""
    import numpy as np
    kv = (2 * d if fp8 else 4 * d) if kv_key_bytes is None else kv_key_bytes
    kind = 2 if fp8 else (1 if table_ok else 0)
    lib = load_library()
    info = (ctypes.c_int * 7)()
    args = (BH, Nq, Nk, int(bool(causal)), q_offset, k_offset, kv, kind, num_sms)
    rc = lib.attn_diag_fwd_schedule(*args, ctypes.cast(info, ctypes.c_void_p), None, 0)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_diag_fwd_schedule")
    grid, rounds = info[2], info[3]
    seq = np.empty((grid, rounds), dtype=np.int32)
    rc = lib.attn_diag_fwd_schedule(*args, ctypes.cast(info, ctypes.c_void_p), seq.ctypes.data, seq.size)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_diag_fwd_schedule")
    keys = ("order", "group_heads", "grid", "rounds", "makespan", "table", "pair_tail")
    return dict(zip(keys, list(info))), seq


def diag_force_fwd_order(order=-1, group_heads=0):
    """Force the unit order of later unsplit causal forward launches (order -1:
    the library's own choice again)."""
    rc = load_library().attn_diag_force_fwd_order(order, group_heads)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_diag_force_fwd_order")


def diag_set_pair_tail(enable=True):
    """Enable or disable the split of the last, partly filled round over CTA pairs
    for later launches of this process."""
    load_library().attn_diag_set_pair_tail(1 if enable else 0)
