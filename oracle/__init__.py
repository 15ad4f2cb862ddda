"""fp64 CPU oracle for banded + global sparse attention (forward pass).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product library never
loads it, and it shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain C, double precision, one explicit
mask row per query); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  Input arrays may be float32, float64, or uint16 holding
raw bfloat16 bit patterns (read exactly: bf16 -> double is lossless).

Pins that tie it to the pages and to mathematics, not to itself, are in
``tests/test_oracle.py``; every function here is pinned there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIBPATH = os.path.join(_HERE, "_build", "liboracle.so")

PATTERN_LONGFORMER = 0
PATTERN_GMAT_BAND = 1
PATTERN_GMAT_CHUNK = 2

_DTYPE_CODE = {np.dtype(np.uint16): 0, np.dtype(np.float32): 1, np.dtype(np.float64): 2}

_lock = threading.Lock()


def compile_library(source: str = SOURCE, out: str = LIBPATH) -> str:
    """Compile ``source`` into a shared library at ``out`` with gcc."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", source, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Build the default oracle library if missing or older than its source."""
    with _lock:
        if force or not os.path.exists(LIBPATH) or \
                os.path.getmtime(LIBPATH) < os.path.getmtime(SOURCE):
            compile_library()
    return LIBPATH


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """Handle on one compiled oracle library (the default one, or a test mutant)."""

    def __init__(self, libpath: str | None = None):
        self.libpath = libpath or build()
        lib = ctypes.CDLL(self.libpath)
        i32p = ctypes.c_void_p
        lib.oracle_global_set.argtypes = [i32p, ctypes.c_int, ctypes.c_int, i32p]
        lib.oracle_global_set.restype = ctypes.c_int
        lib.oracle_mask_longformer.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               i32p, ctypes.c_int, ctypes.c_void_p]
        lib.oracle_mask_longformer.restype = None
        lib.oracle_mask_gmat.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p]
        lib.oracle_mask_gmat.restype = None
        lib.oracle_count_pairs_longformer.argtypes = [
            ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, i32p, ctypes.c_int,
            ctypes.c_int, ctypes.c_void_p]
        lib.oracle_count_pairs_longformer.restype = ctypes.c_int
        lib.oracle_count_pairs_gmat.argtypes = [ctypes.c_int] * 6
        lib.oracle_count_pairs_gmat.restype = ctypes.c_int64
        common = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5
        tail = [ctypes.c_double, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int]
        lib.oracle_forward_longformer.argtypes = common + [
            ctypes.c_int, i32p, i32p, ctypes.c_int] + tail
        lib.oracle_forward_longformer.restype = ctypes.c_int
        lib.oracle_forward_gmat.argtypes = common + [ctypes.c_int] * 4 + tail
        lib.oracle_forward_longformer_global_proj.argtypes = [
            ctypes.c_void_p] * 6 + [ctypes.c_int] * 6 + [i32p, i32p, ctypes.c_int] + tail
        lib.oracle_forward_longformer_global_proj.restype = ctypes.c_int
        lib.oracle_forward_gmat.restype = ctypes.c_int
        lib.oracle_forward_gather.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 7 + tail
        lib.oracle_forward_gather.restype = ctypes.c_int
        self.lib = lib

    # -- global set --------------------------------------------------------
    def global_set(self, idx, N: int) -> np.ndarray:
        """Sorted unique global positions; ValueError if one is outside [0, N)."""
        idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32).reshape(-1))
        out = np.zeros(max(1, idx.size), dtype=np.int32)
        n = self.lib.oracle_global_set(_ptr(idx), int(idx.size), int(N), _ptr(out))
        if n < 0:
            raise ValueError("global index outside [0, N)")
        return out[:n].copy()

    # -- masks (small N) ---------------------------------------------------
    def mask_longformer(self, N: int, window: int, dilation: int = 1, globals_=()) -> np.ndarray:
        g = self.global_set(globals_, N)
        m = np.zeros((N, N), dtype=np.uint8)
        self.lib.oracle_mask_longformer(int(N), int(window), int(dilation), _ptr(g),
                                        int(g.size), _ptr(m))
        return m.astype(bool)

    def mask_gmat(self, N: int, M: int, window: int = 0, chunk: int | None = None) -> np.ndarray:
        pattern = PATTERN_GMAT_BAND if chunk is None else PATTERN_GMAT_CHUNK
        m = np.zeros((N, N), dtype=np.uint8)
        self.lib.oracle_mask_gmat(pattern, int(N), int(M), int(window), int(chunk or 1), _ptr(m))
        return m.astype(bool)

    # -- pair counts ---------------------------------------------------------
    def count_pairs_longformer(self, N: int, window: int, dilation, globals_=(),
                               threads: int | None = None) -> np.ndarray:
        """Per-head in-mask pair counts (int64), by materialising every mask row."""
        dil = np.ascontiguousarray(np.asarray(dilation, dtype=np.int32).reshape(-1))
        g = self.global_set(globals_, N)
        out = np.zeros(dil.size, dtype=np.int64)
        rc = self.lib.oracle_count_pairs_longformer(
            int(N), int(window), _ptr(dil), int(dil.size), _ptr(g), int(g.size),
            int(threads or default_threads()), _ptr(out))
        if rc:
            raise MemoryError("oracle count failed")
        return out

    def count_pairs_gmat(self, N: int, M: int, window: int = 0, chunk: int | None = None,
                         threads: int | None = None) -> int:
        pattern = PATTERN_GMAT_BAND if chunk is None else PATTERN_GMAT_CHUNK
        return int(self.lib.oracle_count_pairs_gmat(pattern, int(N), int(M), int(window),
                                                    int(chunk or 1),
                                                    int(threads or default_threads())))

    # -- forward -------------------------------------------------------------
    @staticmethod
    def _inputs(*tensors):
        arrs = [np.ascontiguousarray(a) for a in tensors]
        dt = arrs[0].dtype
        if any(a.dtype != dt for a in arrs) or dt not in _DTYPE_CODE:
            raise TypeError("q, k, v (and global projections) must share one dtype: "
                            "uint16 (bf16 bits), float32 or float64")
        if arrs[0].ndim != 4 or any(a.shape != arrs[0].shape for a in arrs):
            raise ValueError("q, k, v (and global projections) must be [B, H, N, D] of one shape")
        return arrs, _DTYPE_CODE[dt]

    @staticmethod
    def _rows(rows, total):
        if rows is None:
            return None, total
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        if r.size and (r.min() < 0 or r.max() >= total):
            raise ValueError("row index out of range")
        return r, int(r.size)

    def forward_longformer(self, q, k, v, window: int, dilation=None, globals_=(),
                           scale: float | None = None, rows=None, threads: int | None = None,
                           want_lse: bool = True, global_proj=None):
        """Masked-softmax attention in fp64.

        q, k, v: [B, H, N, D].  dilation: per-head list (None = all 1).
        rows: optional flattened row ids ((b*H + h)*N + i); None = every row.
        global_proj: optional (qg, kg, vg) of q's shape and dtype -- separate
        global projections: a global row then scores qg . kg over every key and
        averages vg; the other rows use q, k, v throughout.
        Returns (out [B,H,N,D] or [n_rows,D], lse [B,H,N] or [n_rows]) as float64.
        """
        if global_proj is not None:
            (q, k, v, qg, kg, vg), code = self._inputs(q, k, v, *global_proj)
        else:
            (q, k, v), code = self._inputs(q, k, v)
        B, H, N, D = q.shape
        dil = np.ones(H, dtype=np.int32) if dilation is None else \
            np.ascontiguousarray(np.asarray(dilation, dtype=np.int32).reshape(-1))
        if dil.size != H:
            raise ValueError("dilation must have one entry per head")
        g = self.global_set(globals_, N)
        sc = float(scale if scale is not None else 1.0 / np.sqrt(D))
        r, n = self._rows(rows, B * H * N)
        out = np.empty((n, D), dtype=np.float64)
        lse = np.empty(n, dtype=np.float64) if want_lse else None
        if global_proj is not None:
            rc = self.lib.oracle_forward_longformer_global_proj(
                _ptr(q), _ptr(k), _ptr(v), _ptr(qg), _ptr(kg), _ptr(vg), code, B, H, N, D,
                int(window), _ptr(dil), _ptr(g), int(g.size), sc, _ptr(r), int(n), _ptr(out),
                _ptr(lse), int(threads or default_threads()))
        else:
            rc = self.lib.oracle_forward_longformer(
                _ptr(q), _ptr(k), _ptr(v), code, B, H, N, D, int(window), _ptr(dil), _ptr(g),
                int(g.size), sc, _ptr(r), int(n), _ptr(out), _ptr(lse),
                int(threads or default_threads()))
        if rc:
            raise MemoryError("oracle forward failed")
        if rows is None:
            out = out.reshape(B, H, N, D)
            lse = None if lse is None else lse.reshape(B, H, N)
        return out, lse

    def forward_gmat(self, q, k, v, M: int, window: int = 0, chunk: int | None = None,
                     scale: float | None = None, rows=None, threads: int | None = None,
                     want_lse: bool = True):
        """GMAT attention over the concatenated [memory; main] sequence, fp64.

        Positions [0, M) are memory tokens.  chunk=None: band of half-width
        window//2 among main tokens; chunk=C: C-long chunks among main tokens.
        """
        (q, k, v), code = self._inputs(q, k, v)
        B, H, N, D = q.shape
        pattern = PATTERN_GMAT_BAND if chunk is None else PATTERN_GMAT_CHUNK
        sc = float(scale if scale is not None else 1.0 / np.sqrt(D))
        r, n = self._rows(rows, B * H * N)
        out = np.empty((n, D), dtype=np.float64)
        lse = np.empty(n, dtype=np.float64) if want_lse else None
        rc = self.lib.oracle_forward_gmat(
            _ptr(q), _ptr(k), _ptr(v), code, B, H, N, D, pattern, int(M), int(window),
            int(chunk or 1), sc, _ptr(r), int(n), _ptr(out), _ptr(lse),
            int(threads or default_threads()))
        if rc:
            raise MemoryError("oracle forward failed")
        if rows is None:
            out = out.reshape(B, H, N, D)
            lse = None if lse is None else lse.reshape(B, H, N)
        return out, lse


    def forward_gather(self, q, k, v, idx, scale: float | None = None, rows=None,
                       threads: int | None = None, want_lse: bool = True):
        """Attention over per-query key lists, fp64 (Unlimiformer, sections 2.2-2.3).

        q: [B, H, Nq, D]; k, v: [B, H, Nk, D] (one dtype); idx: int32
        [B, H, Nq, K], row i of head (b, h) scoring the keys it lists; entries
        outside [0, Nk) are padding, a repeated entry counts once per listing.
        Returns (out [B,H,Nq,D] or [n_rows,D], lse [B,H,Nq] or [n_rows]); a row
        with no valid entry gives 0 and -inf.
        """
        arrs = [np.ascontiguousarray(a) for a in (q, k, v)]
        code = _DTYPE_CODE.get(arrs[0].dtype)
        if code is None or any(a.dtype != arrs[0].dtype for a in arrs):
            raise TypeError("q, k, v must share one dtype: uint16 (bf16 bits), float32 or float64")
        q, k, v = arrs
        if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape or q.shape[:2] != k.shape[:2] \
                or q.shape[3] != k.shape[3]:
            raise ValueError("q must be [B, H, Nq, D] and k, v [B, H, Nk, D]")
        B, H, Nq, D = q.shape
        Nk = k.shape[2]
        idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
        if idx.ndim != 4 or idx.shape[:3] != (B, H, Nq):
            raise ValueError("idx must be [B, H, Nq, K]")
        K = idx.shape[3]
        sc = float(scale if scale is not None else 1.0 / np.sqrt(D))
        r, n = self._rows(rows, B * H * Nq)
        out = np.empty((n, D), dtype=np.float64)
        lse = np.empty(n, dtype=np.float64) if want_lse else None
        rc = self.lib.oracle_forward_gather(
            _ptr(q), _ptr(k), _ptr(v), _ptr(idx), code, B, H, Nq, Nk, D, K, sc, _ptr(r),
            int(n), _ptr(out), _ptr(lse), int(threads or default_threads()))
        if rc:
            raise MemoryError("oracle forward failed")
        if rows is None:
            out = out.reshape(B, H, Nq, D)
            lse = None if lse is None else lse.reshape(B, H, Nq)
        return out, lse


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
