"""fp64 CPU oracle for the FlashAttention-2 forward pass (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The CUDA library never does, and
this package imports nothing from the library: the two share only the seeded
input generators in ``exact_attention_10_gb300.inputs``, which hold none of the
method's arithmetic.

The arithmetic lives in ``attn_ref.c`` (plain C99 + OpenMP, fp64); this module
only marshals arrays into it.  See that file's header for the definition it
follows and the pages it cites.  Every function returns float64 results that
are not rounded to the input dtype.

Parity pins: every function here is pinned in ``tests/test_oracle_pins.py``
against closed forms, invariants, an independent library (PyTorch's fp64 CPU
scaled-dot-product attention) and a figure printed on the pages.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build as _build, LIB_PATH

_DTYPE_CODE = {"bf16": 0, "fp16": 1, "f64": 2}
_lib = None


def _load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    so = path or LIB_PATH
    if path is None and not os.path.exists(so):
        _build()
    lib = ctypes.CDLL(so)
    c_long_p = ctypes.POINTER(ctypes.c_long)
    c_double_p = ctypes.POINTER(ctypes.c_double)
    lib.attn_ref_num_threads.restype = ctypes.c_int
    lib.attn_ref_decode.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_long, c_double_p]
    lib.attn_ref_decode.restype = None
    lib.attn_ref_forward.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_long, ctypes.c_long,
                                                            ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                                            c_double_p, c_double_p]
    lib.attn_ref_forward.restype = ctypes.c_int
    lib.attn_ref_forward_qkv.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_long, ctypes.c_long,
                                                                ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                                                ctypes.c_double, c_double_p, c_double_p]
    lib.attn_ref_forward_qkv.restype = ctypes.c_int
    lib.attn_ref_forward_band.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] + [ctypes.c_long] * 6 + [
        ctypes.c_double, c_double_p, c_double_p]
    lib.attn_ref_forward_band.restype = ctypes.c_int
    lib.attn_ref_backward_band.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] + [ctypes.c_long] * 6 + [
        ctypes.c_double] + [c_double_p] * 4
    lib.attn_ref_backward_band.restype = ctypes.c_int
    lib.attn_ref_rows.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_long, ctypes.c_long,
                                                         ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                                         c_long_p, c_long_p, ctypes.c_long, c_double_p, c_double_p]
    lib.attn_ref_rows.restype = ctypes.c_int
    lib.attn_ref_probs.argtypes = [c_double_p, c_double_p, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                   ctypes.c_double, c_double_p]
    lib.attn_ref_probs.restype = None
    lib.attn_ref_tiled.argtypes = [c_double_p] * 3 + [ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                                      ctypes.c_double, ctypes.c_long, ctypes.c_long,
                                                      c_double_p, c_double_p]
    lib.attn_ref_tiled.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _as_input(x):
    """Return (contiguous numpy array, dtype name) for a torch tensor or numpy array.

    bf16 / fp16 tensors are passed as their raw 16-bit patterns; the C side
    decodes them exactly.  float64 is passed as is.  Anything else is refused.
    """
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), "bf16"
        if x.dtype == torch.float16:
            return x.view(torch.int16).numpy().view(np.uint16), "fp16"
        if x.dtype == torch.float64:
            return x.numpy(), "f64"
        raise TypeError(f"oracle input dtype {x.dtype} not supported (bf16, fp16, float64)")
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, "f64"
    raise TypeError(f"oracle input dtype {x.dtype} not supported")


def _ptr(a: np.ndarray, ctype=ctypes.c_void_p):
    if ctype is ctypes.c_void_p:
        return a.ctypes.data_as(ctypes.c_void_p)
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _scale_as_double(scale: float) -> float:
    # The library receives the scale as a float32; the oracle uses that exact value.
    return float(np.float32(scale))


def num_threads(lib=None) -> int:
    return (lib or _load()).attn_ref_num_threads()


def decode(bits: np.ndarray, dtype: str, lib=None) -> np.ndarray:
    """Decode uint16 bf16/fp16 bit patterns to float64 (exactly)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.size, dtype=np.float64)
    (lib or _load()).attn_ref_decode(_ptr(bits), _DTYPE_CODE[dtype], bits.size, _ptr(out, ctypes.c_double))
    return out.reshape(bits.shape)


def forward(q, k, v, causal: bool, scale: float, lib=None):
    """Exact attention of [..., N, D] inputs.  Returns (O float64 [..., N, D], LSE float64 [..., N])."""
    qa, dt = _as_input(q)
    ka, dtk = _as_input(k)
    va, dtv = _as_input(v)
    if not (dt == dtk == dtv):
        raise TypeError("q, k, v must share a dtype")
    if not (qa.shape == ka.shape == va.shape) or qa.ndim < 2:
        raise ValueError("q, k, v must share one [..., N, D] shape")
    N, D = qa.shape[-2], qa.shape[-1]
    BH = int(np.prod(qa.shape[:-2])) if qa.ndim > 2 else 1
    O = np.empty(qa.shape, dtype=np.float64)
    L = np.empty(qa.shape[:-1], dtype=np.float64)
    rc = (lib or _load()).attn_ref_forward(_ptr(qa), _ptr(ka), _ptr(va), _DTYPE_CODE[dt], BH, N, D,
                                           int(bool(causal)), _scale_as_double(scale),
                                           _ptr(O, ctypes.c_double), _ptr(L, ctypes.c_double))
    if rc != 0:
        raise MemoryError("oracle forward failed to allocate scratch")
    return O, L


def forward_qkv(q, k, v, causal: bool, scale: float, lib=None):
    """Exact attention of Nq queries [..., Nq, D] against Nkv keys and values
    [..., Nkv, D], causal mask aligned bottom-right (query i sees keys
    j <= i + Nkv - Nq; a query that sees none gets O = 0, LSE = -inf).
    Returns (O float64 [..., Nq, D], LSE float64 [..., Nq])."""
    qa, dt = _as_input(q)
    ka, dtk = _as_input(k)
    va, dtv = _as_input(v)
    if not (dt == dtk == dtv):
        raise TypeError("q, k, v must share a dtype")
    if ka.shape != va.shape or qa.ndim < 2 or qa.shape[:-2] != ka.shape[:-2] or qa.shape[-1] != ka.shape[-1]:
        raise ValueError("q [..., Nq, D] and k, v [..., Nkv, D] must agree")
    Nq, Nkv, D = qa.shape[-2], ka.shape[-2], qa.shape[-1]
    BH = int(np.prod(qa.shape[:-2])) if qa.ndim > 2 else 1
    O = np.empty(qa.shape, dtype=np.float64)
    L = np.empty(qa.shape[:-1], dtype=np.float64)
    rc = (lib or _load()).attn_ref_forward_qkv(_ptr(qa), _ptr(ka), _ptr(va), _DTYPE_CODE[dt], BH, Nq, Nkv, D,
                                               int(bool(causal)), _scale_as_double(scale),
                                               _ptr(O, ctypes.c_double), _ptr(L, ctypes.c_double))
    if rc != 0:
        raise MemoryError("oracle forward failed to allocate scratch")
    return O, L


def forward_band(q, k, v, left: int, right: int, scale: float, lib=None):
    """Exact attention of [..., Nq, D] queries against [..., Nkv, D] keys under
    a band mask: query i sees keys j in [i' - left, i' + right], i' = i + Nkv
    - Nq; a negative bound is unbounded.  A row whose band holds no key gets
    O = 0, LSE = -inf.  Returns (O float64 [..., Nq, D], LSE float64 [..., Nq])."""
    qa, dt = _as_input(q)
    ka, dtk = _as_input(k)
    va, dtv = _as_input(v)
    if not (dt == dtk == dtv):
        raise TypeError("q, k, v must share a dtype")
    if ka.shape != va.shape or qa.ndim < 2 or qa.shape[:-2] != ka.shape[:-2] or qa.shape[-1] != ka.shape[-1]:
        raise ValueError("q [..., Nq, D] and k, v [..., Nkv, D] must agree")
    Nq, Nkv, D = qa.shape[-2], ka.shape[-2], qa.shape[-1]
    BH = int(np.prod(qa.shape[:-2])) if qa.ndim > 2 else 1
    O = np.empty(qa.shape, dtype=np.float64)
    L = np.empty(qa.shape[:-1], dtype=np.float64)
    rc = (lib or _load()).attn_ref_forward_band(_ptr(qa), _ptr(ka), _ptr(va), _DTYPE_CODE[dt], BH, Nq, Nkv, D,
                                                int(left), int(right), _scale_as_double(scale),
                                                _ptr(O, ctypes.c_double), _ptr(L, ctypes.c_double))
    if rc != 0:
        raise MemoryError("oracle forward failed to allocate scratch")
    return O, L


def backward_band(q, k, v, do, left: int, right: int, scale: float, with_delta: bool = False, lib=None):
    """Gradients of the band-masked attention of ``forward_band`` for the
    upstream gradient ``do`` (shape of O): returns float64 (dQ, dK, dV), and
    delta = rowsum(P * dP) [..., Nq] as a fourth item if ``with_delta``."""
    qa, dt = _as_input(q)
    ka, dtk = _as_input(k)
    va, dtv = _as_input(v)
    da, dtd = _as_input(do)
    if not (dt == dtk == dtv == dtd):
        raise TypeError("q, k, v, do must share a dtype")
    if (ka.shape != va.shape or da.shape != qa.shape or qa.ndim < 2 or qa.shape[:-2] != ka.shape[:-2]
            or qa.shape[-1] != ka.shape[-1]):
        raise ValueError("q, do [..., Nq, D] and k, v [..., Nkv, D] must agree")
    Nq, Nkv, D = qa.shape[-2], ka.shape[-2], qa.shape[-1]
    BH = int(np.prod(qa.shape[:-2])) if qa.ndim > 2 else 1
    dQ = np.empty(qa.shape, dtype=np.float64)
    dK = np.empty(ka.shape, dtype=np.float64)
    dV = np.empty(ka.shape, dtype=np.float64)
    delta = np.empty(qa.shape[:-1], dtype=np.float64)
    rc = (lib or _load()).attn_ref_backward_band(_ptr(qa), _ptr(ka), _ptr(va), _ptr(da), _DTYPE_CODE[dt], BH, Nq,
                                                 Nkv, D, int(left), int(right), _scale_as_double(scale),
                                                 _ptr(dQ, ctypes.c_double), _ptr(dK, ctypes.c_double),
                                                 _ptr(dV, ctypes.c_double), _ptr(delta, ctypes.c_double))
    if rc != 0:
        raise MemoryError("oracle backward failed to allocate scratch")
    return (dQ, dK, dV, delta) if with_delta else (dQ, dK, dV)


def backward(q, k, v, do, causal: bool, scale: float, lib=None):
    """Gradients (dQ, dK, dV) of the square attention of ``forward``
    (bottom-right causal when Nq != Nkv): the band (unbounded, 0) or none."""
    return backward_band(q, k, v, do, -1, 0 if causal else -1, scale, lib=lib)


def rows(q, k, v, causal: bool, scale: float, bh_idx, row_idx, lib=None):
    """Selected rows of the exact attention.

    ``bh_idx`` indexes the flattened leading dims (batch*head), ``row_idx`` the
    query row; ``bh_idx`` must be non-decreasing.  Returns (O [n, D], LSE [n]).
    """
    qa, dt = _as_input(q)
    ka, _ = _as_input(k)
    va, _ = _as_input(v)
    N, D = qa.shape[-2], qa.shape[-1]
    BH = int(np.prod(qa.shape[:-2])) if qa.ndim > 2 else 1
    bh = np.ascontiguousarray(bh_idx, dtype=np.int64)
    ri = np.ascontiguousarray(row_idx, dtype=np.int64)
    if bh.shape != ri.shape or bh.ndim != 1:
        raise ValueError("bh_idx and row_idx must be 1-D of equal length")
    O = np.empty((bh.size, D), dtype=np.float64)
    L = np.empty(bh.size, dtype=np.float64)
    rc = (lib or _load()).attn_ref_rows(_ptr(qa), _ptr(ka), _ptr(va), _DTYPE_CODE[dt], BH, N, D,
                                        int(bool(causal)), _scale_as_double(scale),
                                        _ptr(bh, ctypes.c_long), _ptr(ri, ctypes.c_long), bh.size,
                                        _ptr(O, ctypes.c_double), _ptr(L, ctypes.c_double))
    if rc == -2:
        raise ValueError("bad row index, or bh_idx not non-decreasing")
    if rc != 0:
        raise MemoryError("oracle rows failed to allocate scratch")
    return O, L


def probs(q, k, causal: bool, scale: float, lib=None) -> np.ndarray:
    """Explicit softmax(S) of one [N, D] head given as float64 arrays.  Returns [N, N]."""
    qa = np.ascontiguousarray(q, dtype=np.float64)
    ka = np.ascontiguousarray(k, dtype=np.float64)
    N, D = qa.shape
    P = np.empty((N, N), dtype=np.float64)
    (lib or _load()).attn_ref_probs(_ptr(qa, ctypes.c_double), _ptr(ka, ctypes.c_double), N, D,
                                    int(bool(causal)), _scale_as_double(scale), _ptr(P, ctypes.c_double))
    return P


def tiled(q, k, v, causal: bool, scale: float, BM: int, BN: int, lib=None):
    """The tiled online-softmax recurrence in fp64 on float64 [..., N, D] inputs."""
    qa = np.ascontiguousarray(q, dtype=np.float64)
    ka = np.ascontiguousarray(k, dtype=np.float64)
    va = np.ascontiguousarray(v, dtype=np.float64)
    N, D = qa.shape[-2], qa.shape[-1]
    BH = int(np.prod(qa.shape[:-2])) if qa.ndim > 2 else 1
    O = np.empty(qa.shape, dtype=np.float64)
    L = np.empty(qa.shape[:-1], dtype=np.float64)
    rc = (lib or _load()).attn_ref_tiled(_ptr(qa, ctypes.c_double), _ptr(ka, ctypes.c_double),
                                         _ptr(va, ctypes.c_double), BH, N, D, int(bool(causal)),
                                         _scale_as_double(scale), BM, BN, _ptr(O, ctypes.c_double),
                                         _ptr(L, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle tiled recurrence failed")
    return O, L
