"""ctypes binding of the C ABI in ``include/sa.h`` (argument marshalling only).

Every step of the attention runs in the CUDA library; this module passes
pointers, sizes and the current CUDA stream.  It raises ``SaError`` for any
non-OK status and ``RuntimeError`` if the compiled library is missing -- there
is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_CUDA, SA_ERR_TIMEOUT, SA_ERR_NO_MEMORY = range(6)
SA_BF16, SA_FP32, SA_TF32 = 0, 1, 2
SA_PV_AUTO, SA_PV_SINGLE, SA_PV_SPLIT = 0, 1, 2
SA_MAX_GLOBALS = 256
STAGES = ("gather", "band", "global_rows", "merge")

STATUS_NAMES = {0: "SA_OK", 1: "SA_ERR_INVALID_ARG", 2: "SA_ERR_UNSUPPORTED", 3: "SA_ERR_CUDA",
                4: "SA_ERR_TIMEOUT", 5: "SA_ERR_NO_MEMORY"}

# Every function include/sa.h declares, with its ctypes signature.
_VP, _I, _F, _I32P, _I64P = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p


class _Profile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64 * 4), ("ms", ctypes.c_double * 4)]


SIGNATURES = {
    "sa_forward": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I32P, _I32P, _I, _F, _I, _VP]),
    "sa_forward_lse": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I32P, _I32P, _I, _F,
                            _I, _VP]),
    "sa_count_pairs": (_I, [_I, _I, _I32P, _I, _I32P, _I, _I64P, _I64P]),
    "sa_last_error": (ctypes.c_char_p, []),
    "sa_sync_status": (_I, [_VP]),
    "sa_check_stalled_wait": (_I, [ctypes.c_uint32, _VP]),
    "sa_profile_begin": (_I, []),
    "sa_profile_end": (_I, [ctypes.POINTER(_Profile)]),
    "sa_version": (ctypes.c_char_p, []),
    "sa_forward_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I32P, _I32P, _I,
                                _F, _I, _VP]),
    "sa_forward_chunked": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _VP]),
    "sa_count_pairs_chunked": (_I, [_I, _I, _I, _I64P]),
    "sa_forward_gather": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I,
                               _VP]),
    "sa_forward_global_proj": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I,
                                    _I32P, _I32P, _I, _F, _I, _VP]),
    "sa_forward_host": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I32P, _I32P, _I, _F,
                             _I, _I]),
    "sa_set_pv_mode": (_I, [_I]),
    "sa_get_pv_mode": (_I, []),
    "sa_uses_split_p": (_I, [_I, _I, _I, _I32P, _I, _I32P, _I, _I, _I, _F]),
}
SA_NOALLOC_SCRATCH_BYTES = 8 << 20


class SaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIBPATH


def load(path: Optional[str] = None):
    """Load the compiled library (build it first with ``build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


# the SA_DEBUG build's test entry point (include/sa_debug.h)
DEBUG_SIGNATURES = {
    "sa_debug_check_band_items": (_I, [_VP, _I, _VP, _I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
}

_lib_debug = None


def library_path_debug() -> str:
    return _build.LIBPATH_DEBUG


def load_debug():
    """Load the SA_DEBUG build (build it first with ``build.build(debug=True)``):
    the same entry points with device-side range checks of every work
    description, plus ``sa_debug_check_band_items``.  It is loaded beside the
    release library, not in its place."""
    global _lib_debug
    if _lib_debug is not None:
        return _lib_debug
    p = library_path_debug()
    if not os.path.exists(p):
        raise RuntimeError(f"SA_DEBUG library not built: {p} is missing (run build.build(debug=True))")
    lib = ctypes.CDLL(p)
    for name, (res, args) in {**SIGNATURES, **DEBUG_SIGNATURES}.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib_debug = lib
    return lib


def _check(status: int):
    if status != SA_OK:
        raise SaError(status, load().sa_last_error().decode(errors="replace"))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32).reshape(-1))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None or a.size == 0 else a.ctypes.data_as(ctypes.c_void_p)


def count_pairs(N: int, window: int, dilation: Sequence[int] | None, H: int,
                globals_: Sequence[int] = ()):
    """(per_head int64[H], total) -- exact in-mask pair counts (host only)."""
    dil = None if dilation is None else _i32(dilation)
    g = _i32(globals_)
    per = np.zeros(H, dtype=np.int64)
    tot = ctypes.c_int64(0)
    _check(load().sa_count_pairs(int(N), int(window), _ptr(dil), int(H), _ptr(g), int(g.size),
                                 _ptr(per), ctypes.byref(tot)))
    return per, int(tot.value)


def forward(q, k, v, window: int, dilation: Sequence[int] | None = None,
            globals_: Sequence[int] = (), scale: Optional[float] = None, out=None,
            lse=None, stream=None, tf32: bool = False):
    """out = sparse attention of torch CUDA tensors q, k, v ([B, H, N, D]).

    ``lse``: None, or a float32 CUDA tensor [B, H, N] to receive log-sum-exp.
    ``tf32``: for float32 tensors, run the products on the tensor cores in tf32
    (SA_TF32, D = 64) instead of fp32 on the CUDA cores (SA_FP32).
    Runs on ``stream`` (default: torch's current stream); returns ``out``.
    """
    import torch

    if q.dtype == torch.bfloat16:
        dt = SA_BF16
    elif q.dtype == torch.float32:
        dt = SA_TF32 if tf32 else SA_FP32
    else:
        raise TypeError(f"unsupported dtype {q.dtype} (bfloat16 or float32)")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or t.shape != q.shape:
            raise ValueError("q, k, v must be contiguous CUDA tensors of one shape and dtype")
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    B, H, N, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    dil = None if dilation is None else _i32(dilation)
    if dil is not None and dil.size != H:
        raise ValueError("dilation needs one entry per head")
    g = _i32(globals_)
    sc = float(scale if scale is not None else 1.0 / math.sqrt(D))
    h_stream = ctypes.c_void_p(stream.cuda_stream)
    with torch.cuda.device(q.device):
        if lse is None:
            st = load().sa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   B, H, N, D, int(window), _ptr(dil), _ptr(g), int(g.size),
                                   sc, dt, h_stream)
        else:
            st = load().sa_forward_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       lse.data_ptr(), B, H, N, D, int(window), _ptr(dil),
                                       _ptr(g), int(g.size), sc, dt, h_stream)
    _check(st)
    return out


def forward_host(q, k, v, window: int, dilation: Sequence[int] | None = None,
                 globals_: Sequence[int] = (), scale: Optional[float] = None, out=None,
                 lse=None, tf32: bool = False, heads_per_group: int = 0, device=None):
    """``forward`` on host (CPU) torch tensors: sa_forward_host copies them to
    ``device`` (default: the current CUDA device), runs the attention and
    copies ``out`` (and ``lse``, a float32 CPU tensor [B, H, N]) back, with the
    copies of one group of heads overlapping the computation of another.
    Pinned tensors (``.pin_memory()``) let the copies overlap.  Synchronous;
    returns ``out``.
    """
    import torch

    if q.dtype == torch.bfloat16:
        dt = SA_BF16
    elif q.dtype == torch.float32:
        dt = SA_TF32 if tf32 else SA_FP32
    else:
        raise TypeError(f"unsupported dtype {q.dtype} (bfloat16 or float32)")
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or t.shape != q.shape:
            raise ValueError("q, k, v must be contiguous CPU tensors of one shape and dtype")
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    B, H, N, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if out.is_cuda or not out.is_contiguous() or out.dtype != q.dtype or out.shape != q.shape:
        raise ValueError("out must be a contiguous CPU tensor like q")
    if lse is not None and (lse.is_cuda or not lse.is_contiguous() or lse.dtype != torch.float32
                            or tuple(lse.shape) != (B, H, N)):
        raise ValueError("lse must be a contiguous float32 CPU tensor [B, H, N]")
    dil = None if dilation is None else _i32(dilation)
    if dil is not None and dil.size != H:
        raise ValueError("dilation needs one entry per head")
    g = _i32(globals_)
    sc = float(scale if scale is not None else 1.0 / math.sqrt(D))
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = load().sa_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    None if lse is None else lse.data_ptr(), B, H, N, D,
                                    int(window), _ptr(dil), _ptr(g), int(g.size), sc, dt,
                                    int(heads_per_group))
    _check(st)
    return out


def forward_global_proj(q, k, v, q_global, k_global, v_global, window: int,
                        dilation: Sequence[int] | None = None, globals_: Sequence[int] = (),
                        scale: Optional[float] = None, out=None, lse=None, stream=None):
    """Like ``forward``, with separate projections for the global attention
    (sa_forward_global_proj): a global row scores ``q_global . k_global`` over
    every key and averages ``v_global``; the other rows use q, k, v.  All six
    inputs are contiguous CUDA tensors of one shape and dtype."""
    import torch

    dt = SA_BF16 if q.dtype == torch.bfloat16 else SA_FP32 if q.dtype == torch.float32 else None
    if dt is None:
        raise TypeError(f"unsupported dtype {q.dtype} (bfloat16 or float32)")
    for t in (q, k, v, q_global, k_global, v_global):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or t.shape != q.shape:
            raise ValueError("q, k, v and the global projections must be contiguous CUDA "
                             "tensors of one shape and dtype")
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    B, H, N, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    dil = None if dilation is None else _i32(dilation)
    if dil is not None and dil.size != H:
        raise ValueError("dilation needs one entry per head")
    g = _i32(globals_)
    sc = float(scale if scale is not None else 1.0 / math.sqrt(D))
    with torch.cuda.device(q.device):
        st = load().sa_forward_global_proj(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), q_global.data_ptr(), k_global.data_ptr(),
            v_global.data_ptr(), out.data_ptr(), None if lse is None else lse.data_ptr(), B, H,
            N, D, int(window), _ptr(dil), _ptr(g), int(g.size), sc, dt,
            ctypes.c_void_p(stream.cuda_stream))
    _check(st)
    return out


def forward_gather(q, k, v, idx, scale: Optional[float] = None, out=None, lse=None,
                   stream=None):
    """Attention of each query row over the keys its list names
    (sa_forward_gather).  q: [B, H, Nq, D]; k, v: [B, H, Nk, D] (CUDA,
    bfloat16 or float32, contiguous); idx: int32 CUDA tensor [B, H, Nq, K]
    (entries outside [0, Nk) are padding).  Returns ``out`` [B, H, Nq, D]."""
    import torch

    dt = SA_BF16 if q.dtype == torch.bfloat16 else SA_FP32 if q.dtype == torch.float32 else None
    if dt is None:
        raise TypeError(f"unsupported dtype {q.dtype} (bfloat16 or float32)")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or t.dim() != 4:
            raise ValueError("q, k, v must be contiguous 4-d CUDA tensors of one dtype")
    B, H, Nq, D = q.shape
    if k.shape != v.shape or k.shape[:2] != (B, H) or k.shape[3] != D:
        raise ValueError("k and v must be [B, H, Nk, D] with q's B, H and D")
    Nk = k.shape[2]
    if (idx.dtype != torch.int32 or not idx.is_cuda or not idx.is_contiguous()
            or idx.dim() != 4 or tuple(idx.shape[:3]) != (B, H, Nq)):
        raise ValueError("idx must be a contiguous int32 CUDA tensor [B, H, Nq, K]")
    K = idx.shape[3]
    if out is None:
        out = torch.empty_like(q)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sc = float(scale if scale is not None else 1.0 / math.sqrt(D))
    with torch.cuda.device(q.device):
        st = load().sa_forward_gather(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), idx.data_ptr() if K else None,
            out.data_ptr(), None if lse is None else lse.data_ptr(), B, H, Nq, Nk, D, K, sc, dt,
            ctypes.c_void_p(stream.cuda_stream))
    _check(st)
    return out


def count_pairs_chunked(N: int, n_memory: int, chunk: int) -> int:
    """Exact in-mask pair count of one head of the chunked pattern (host only)."""
    per = ctypes.c_int64(0)
    _check(load().sa_count_pairs_chunked(int(N), int(n_memory), int(chunk), ctypes.byref(per)))
    return int(per.value)


def forward_chunked(q, k, v, n_memory: int, chunk: int, scale: Optional[float] = None,
                    out=None, lse=None, stream=None):
    """GMAT chunked attention with ``n_memory`` memory tokens at the front of the
    sequence and ``chunk``-long chunks after them (sa_forward_chunked); torch
    CUDA tensors [B, H, N, D], bfloat16 or float32.  Returns ``out``."""
    import torch

    dt = SA_BF16 if q.dtype == torch.bfloat16 else SA_FP32 if q.dtype == torch.float32 else None
    if dt is None:
        raise TypeError(f"unsupported dtype {q.dtype} (bfloat16 or float32)")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or t.shape != q.shape:
            raise ValueError("q, k, v must be contiguous CUDA tensors of one shape and dtype")
    B, H, N, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sc = float(scale if scale is not None else 1.0 / math.sqrt(D))
    with torch.cuda.device(q.device):
        st = load().sa_forward_chunked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       None if lse is None else lse.data_ptr(), B, H, N, D,
                                       int(n_memory), int(chunk), sc, dt,
                                       ctypes.c_void_p(stream.cuda_stream))
    _check(st)
    return out


def forward_noalloc(q, k, v, window: int, dilation: Sequence[int] | None = None,
                    globals_: Sequence[int] = (), scale: Optional[float] = None, out=None,
                    lse=None, stream=None):
    """Like ``forward``, through sa_forward_noalloc: the library allocates no
    device memory and uses its static scratch array instead (see include/sa.h)."""
    import torch

    dt = SA_BF16 if q.dtype == torch.bfloat16 else SA_FP32 if q.dtype == torch.float32 else None
    if dt is None:
        raise TypeError(f"unsupported dtype {q.dtype} (bfloat16 or float32)")
    B, H, N, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    dil = None if dilation is None else _i32(dilation)
    g = _i32(globals_)
    sc = float(scale if scale is not None else 1.0 / math.sqrt(D))
    with torch.cuda.device(q.device):
        st = load().sa_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       None if lse is None else lse.data_ptr(), B, H, N, D,
                                       int(window), _ptr(dil), _ptr(g), int(g.size), sc, dt,
                                       ctypes.c_void_p(stream.cuda_stream))
    _check(st)
    return out


def sync_status(stream=None):
    import torch
    s = stream or torch.cuda.current_stream()
    _check(load().sa_sync_status(ctypes.c_void_p(s.cuda_stream)))


def check_stalled_wait(limit_us: int = 20000, stream=None):
    """Enqueue the failure-detection check (sa_check_stalled_wait): a kernel
    whose wait is never satisfied gives up after ``limit_us`` microseconds; the
    next ``sync_status`` raises SaError(SA_ERR_TIMEOUT)."""
    import torch
    s = stream or torch.cuda.current_stream()
    _check(load().sa_check_stalled_wait(int(limit_us), ctypes.c_void_p(s.cuda_stream)))


def profile_begin():
    _check(load().sa_profile_begin())


def profile_end() -> dict:
    prof = _Profile()
    _check(load().sa_profile_end(ctypes.byref(prof)))
    return {name: {"launches": int(prof.launches[i]), "ms": float(prof.ms[i])}
            for i, name in enumerate(STAGES)}


def set_pv_mode(mode: int):
    """Precision of the P V product on the bf16 tensor-core path
    (sa_set_pv_mode): SA_PV_AUTO, SA_PV_SINGLE or SA_PV_SPLIT."""
    _check(load().sa_set_pv_mode(int(mode)))


def get_pv_mode() -> int:
    return int(load().sa_get_pv_mode())


def uses_split_p(N: int, D: int, window: int, dilation: Sequence[int] | None, H: int,
                 globals_: Sequence[int] = (), chunk: int = 0, n_memory: int = 0,
                 scale: Optional[float] = None) -> bool:
    """Whether a bf16 call of this shape and scale splits P (sa_uses_split_p)."""
    dil = None if dilation is None else _i32(dilation)
    g = _i32(globals_)
    sc = float(scale if scale is not None else 1.0 / math.sqrt(D))
    return bool(load().sa_uses_split_p(int(N), int(D), int(window), _ptr(dil), int(H), _ptr(g),
                                       int(g.size), int(chunk), int(n_memory), sc))


def version() -> str:
    return load().sa_version().decode()
