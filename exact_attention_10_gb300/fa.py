"""ctypes binding of include/fa.h (argument marshalling only).

Every compute step runs in the CUDA library; if it is missing this module
raises instead of falling back to anything else.  torch is used for device
memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

FA_BF16, FA_FP16 = 0, 1
FA_BWD_DETERMINISTIC = 1
STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_VALUE", 2: "FA_ERR_MISALIGNED", 3: "FA_ERR_UNSUPPORTED_DEVICE",
          4: "FA_ERR_CUDA", 5: "FA_ERR_DEVICE_TIMEOUT", 6: "FA_ERR_NO_ALLOC_LIMIT"}
EXPORTS = ("fa_bwd", "fa_bwd_band", "fa_bwd_ex", "fa_fwd", "fa_fwd_band", "fa_fwd_ex", "fa_fwd_noalloc", "fa_fwd_qkv", "fa_sync_status",
           "fa_status_string")
SCHEDULES = {"auto": 0, "whole_tiles": 1, "balanced": 2}

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)})")


def load(path: str = LIB_PATH):
    """Load the CUDA library (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"CUDA library not built: {path} is missing (run exact_attention_10_gb300.build)")
    lib = ctypes.CDLL(path)
    vp, c_int = ctypes.c_void_p, ctypes.c_int
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, ctypes.c_float, c_int, vp]
    lib.fa_fwd.restype = c_int
    lib.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, ctypes.c_float, c_int, c_int, vp]
    lib.fa_fwd_ex.restype = c_int
    lib.fa_fwd_noalloc.argtypes = lib.fa_fwd_ex.argtypes
    lib.fa_fwd_noalloc.restype = c_int
    lib.fa_fwd_qkv.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, ctypes.c_float, c_int,
                               c_int, vp]
    lib.fa_fwd_qkv.restype = c_int
    lib.fa_fwd_band.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, c_int, ctypes.c_float,
                                c_int, c_int, vp]
    lib.fa_fwd_band.restype = c_int
    lib.fa_bwd.argtypes = [vp] * 9 + [c_int] * 5 + [ctypes.c_float, c_int, vp]
    lib.fa_bwd.restype = c_int
    lib.fa_bwd_band.argtypes = [vp] * 9 + [c_int] * 7 + [ctypes.c_float, c_int, vp]
    lib.fa_bwd_band.restype = c_int
    lib.fa_bwd_ex.argtypes = [vp] * 9 + [c_int] * 7 + [ctypes.c_float, c_int, ctypes.c_uint, vp]
    lib.fa_bwd_ex.restype = c_int
    lib.fa_sync_status.argtypes = [vp]
    lib.fa_sync_status.restype = c_int
    lib.fa_status_string.argtypes = [c_int]
    lib.fa_status_string.restype = ctypes.c_char_p
    if path == LIB_PATH:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().fa_status_string(int(status)).decode()
    except OSError:
        return "library not loaded"


def fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int, N: int, D: int,
            causal: int, scale: float, dtype: int, stream: int = 0, schedule: int | None = None) -> int:
    """Call fa_fwd (or fa_fwd_ex with a schedule code) with raw integer
    pointers; returns the status code unchanged."""
    if schedule is None:
        return load().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, D, causal, scale, dtype, stream)
    return load().fa_fwd_ex(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, D, causal, scale, dtype, schedule, stream)


def sync_status(stream: int = 0) -> int:
    return load().fa_sync_status(stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float16:
        return FA_FP16
    raise TypeError(f"fa_fwd takes bfloat16 or float16 tensors, got {t.dtype}")


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None,
            schedule: str = "auto", window: tuple[int, int] | None = None):
    """Attention forward on CUDA tensors q [B, H, Nq, D], k and v [B, H, Nkv, D];
    returns (O [B, H, Nq, D], LSE [B, H, Nq]).  With Nq != Nkv the causal mask
    is aligned bottom-right (fa_fwd_qkv).  ``window = (left, right)`` masks
    with a band instead (fa_fwd_band; a negative bound is unbounded; causal
    is ignored then).

    ``out`` / ``lse`` may be given to write into existing buffers.
    ``schedule`` is "auto", "whole_tiles" or "balanced" (fa_schedule).
    Raises FAError on any non-OK status.  Asynchronous on ``stream``
    (default: the current torch stream).
    """
    import torch
    if q.dim() != 4 or k.shape != v.shape or k.dim() != 4 or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q must be [B, H, Nq, D] and k, v [B, H, Nkv, D]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    code = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    B, H, N, D = q.shape
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    if schedule not in SCHEDULES:
        raise ValueError(f"schedule must be one of {sorted(SCHEDULES)}")
    Nkv = k.shape[2]
    if window is not None:
        rc = load().fa_fwd_band(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, Nkv,
                                D, int(window[0]), int(window[1]), float(scale), code, SCHEDULES[schedule], st)
    elif Nkv == N:
        rc = fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, D,
                     int(bool(causal)), float(scale), code, st, SCHEDULES[schedule])
    else:
        rc = load().fa_fwd_qkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, Nkv,
                               D, int(bool(causal)), float(scale), code, SCHEDULES[schedule], st)
    if rc != 0:
        raise FAError(rc, "fa_fwd")
    return out, lse


def backward(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
             stream=None, window: tuple[int, int] | None = None, deterministic: bool = False):
    """Attention backward on CUDA tensors: q, o, do [B, H, Nq, D], k, v
    [B, H, Nkv, D] and lse [B, H, Nq] as ``forward`` returned them (same
    causal / window); returns (dQ, dK, dV).  Square unmasked or causal calls
    go to fa_bwd; a window, or Nq != Nkv (bottom-right causal), to fa_bwd_band;
    ``deterministic`` (dQ by the second pass, the same bits on every call) to
    fa_bwd_ex with FA_BWD_DETERMINISTIC.

    ``dq`` / ``dk`` / ``dv`` may be given to write into existing buffers.
    Raises FAError on any non-OK status.  Asynchronous on ``stream``
    (default: the current torch stream).
    """
    import torch
    if (q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or o.shape != q.shape or do.shape != q.shape
            or lse.shape != q.shape[:3] or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]):
        raise ValueError("q, o, do must be [B, H, Nq, D], k, v [B, H, Nkv, D] and lse [B, H, Nq]")
    if not all(x.is_contiguous() for x in (q, k, v, o, do, lse)):
        raise ValueError("inputs must be contiguous")
    code = _dtype_code(q)
    if any(x.dtype != q.dtype for x in (k, v, o, do)) or lse.dtype != torch.float32:
        raise TypeError("q, k, v, o, do must share a dtype; lse must be float32")
    B, H, N, D = q.shape
    Nkv = k.shape[2]
    if scale is None:
        scale = D ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
            dk.data_ptr(), dv.data_ptr())
    if deterministic:
        left, right = window if window is not None else (-1, 0 if causal else -1)
        rc = load().fa_bwd_ex(*ptrs, B, H, N, Nkv, D, int(left), int(right), float(scale), code, FA_BWD_DETERMINISTIC, st)
    elif window is None and Nkv == N:
        rc = load().fa_bwd(*ptrs, B, H, N, D, int(bool(causal)), float(scale), code, st)
    else:
        left, right = window if window is not None else (-1, 0 if causal else -1)
        rc = load().fa_bwd_band(*ptrs, B, H, N, Nkv, D, int(left), int(right), float(scale), code, st)
    if rc != 0:
        raise FAError(rc, "fa_bwd")
    return dq, dk, dv
