"""Seeded synthetic inputs for banded + global sparse attention.

This module only draws numbers and describes workload shapes; it holds none of
the attention arithmetic.  Both the CUDA path's tests/benchmark and the fp64
oracle take their inputs from here, so the two sides see identical bits.

Recipe (the pages fix no data; these are the workload shapes the method is
described on):
  * q, k, v are i.i.d. standard normal, drawn as float32 from
    ``numpy.random.default_rng(1000 + c)`` in the order q, k, v, each of shape
    [B, H, N, D], for workload number c (1..5).
  * bf16 workloads round those float32 values to bfloat16 (round to nearest,
    ties to even); the float32 workload keeps them as drawn.
  * the scattered-globals workload draws its 32 global positions with
    ``default_rng(2000 + c).choice(N, 32, replace=False)`` and sorts them.
  * scale = 1/sqrt(D).

Attention over per-query key lists (the retrieval form: each query attends to
the top-k keys a kNN index returned) has its own recipe, since the pages give
no datastore and no index: q [B, H, Nq, D] and k, v [B, H, Nk, D] are drawn as
above from ``default_rng(3000 + seed)``; each query's list holds K positions
drawn uniformly from [0, Nk) by the same generator, sorted ascending, with every
draw that repeats an earlier one turned into padding (-1) -- distinct keys, as
a top-k list has, and slightly ragged lists.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    number: int
    name: str
    B: int
    H: int
    N: int
    D: int
    window: int
    dilation: tuple          # per head
    globals_: tuple          # positions (sorted, unique)
    dtype: str               # "fp32" or "bf16"
    memory: int = 0          # GMAT memory tokens prefixed (0 = plain Longformer form)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def describe(self) -> str:
        dil = sorted(set(self.dilation))
        g = self.globals_
        if len(g) and list(g) == list(range(g[0], g[0] + len(g))):
            gs = f"{{{g[0]}..{g[-1]}}}" if len(g) > 1 else f"{{{g[0]}}}"
        else:
            gs = f"{len(g)} seeded"
        return (f"{self.name}: B={self.B} H={self.H} N={self.N} D={self.D} "
                f"window={self.window} dilation={dil} globals={gs} {self.dtype}")


def _seeded_globals(number: int, N: int, count: int) -> tuple:
    rng = np.random.default_rng(2000 + number)
    return tuple(int(x) for x in np.sort(rng.choice(N, count, replace=False)))


def workloads() -> dict:
    """The five workload shapes, keyed by number 1..5."""
    return {
        1: Workload(1, "tiny Longformer mask", 1, 2, 1024, 64, 512, (1, 1), (0,), "fp32"),
        2: Workload(2, "Longformer-base shape", 1, 12, 4096, 64, 512, (1,) * 12, (0,), "bf16"),
        3: Workload(3, "GMAT memory prefix", 2, 12, 64 + 8192, 64, 256, (1,) * 12,
                    tuple(range(64)), "bf16", memory=64),
        4: Workload(4, "dilated + scattered globals", 2, 12, 16384, 64, 512,
                    (1,) * 6 + (2,) * 6, _seeded_globals(4, 16384, 32), "bf16"),
        5: Workload(5, "long context", 1, 16, 131072, 128, 1024, (1,) * 16,
                    tuple(range(64)), "bf16"),
    }


def workload(number: int) -> Workload:
    return workloads()[number]


def custom(B: int, H: int, N: int, D: int, window: int, dilation: Sequence[int] | int = 1,
           globals_: Sequence[int] = (), dtype: str = "bf16", number: int = 0,
           name: str = "custom", memory: int = 0) -> Workload:
    if isinstance(dilation, int):
        dilation = (dilation,) * H
    return Workload(number, name, B, H, N, D, window, tuple(int(d) for d in dilation),
                    tuple(sorted(set(int(g) for g in globals_))), dtype, memory)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).reshape(-1)
    out = np.empty(u.shape, dtype=np.uint16)
    step = 1 << 20
    for s in range(0, u.size, step):
        uc = u[s:s + step]
        r = uc >> np.uint32(16)
        r &= np.uint32(1)
        r += np.uint32(0x7FFF)
        r += uc
        r >>= np.uint32(16)
        out[s:s + step] = r
    return out.reshape(np.shape(x))


def bf16_bits_to_float32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def draw_qkv(w: Workload, seed: Optional[int] = None):
    """(q, k, v) as numpy arrays: uint16 bf16 bits for bf16 workloads, float32 otherwise."""
    rng = np.random.default_rng(1000 + w.number if seed is None else seed)
    shape = (w.B, w.H, w.N, w.D)
    out = []
    for _ in range(3):
        x = rng.standard_normal(shape, dtype=np.float32)
        out.append(bf16_bits(x) if w.dtype == "bf16" else x)
    return tuple(out)


@dataclasses.dataclass(frozen=True)
class GatherWorkload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    D: int
    K: int          # list length per query
    dtype: str      # "fp32" or "bf16"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} H={self.H} Nq={self.Nq} Nk={self.Nk} D={self.D} "
                f"K={self.K} {self.dtype}")


def gather_workload() -> GatherWorkload:
    """Retrieval attention at long-context scale: 4096 queries per head, each
    attending to 1024 of a 131072-key datastore (the top-k width the
    Unlimiformer page uses is the model's context window)."""
    return GatherWorkload("retrieval attention", 1, 16, 4096, 131072, 128, 1024, "bf16")


def draw_gather(w: GatherWorkload, seed: int = 0):
    """(q, k, v, idx): q, k, v as in draw_qkv (uint16 bf16 bits or float32),
    idx int32 [B, H, Nq, K] (see the module docstring)."""
    rng = np.random.default_rng(3000 + seed)
    arrs = []
    for shape in ((w.B, w.H, w.Nq, w.D), (w.B, w.H, w.Nk, w.D), (w.B, w.H, w.Nk, w.D)):
        x = rng.standard_normal(shape, dtype=np.float32)
        arrs.append(bf16_bits(x) if w.dtype == "bf16" else x)
    idx = np.sort(rng.integers(0, w.Nk, size=(w.B, w.H, w.Nq, w.K), dtype=np.int32), axis=-1)
    if w.K > 1:
        rep = np.zeros(idx.shape, dtype=bool)
        rep[..., 1:] = idx[..., 1:] == idx[..., :-1]
        idx[rep] = -1
    return tuple(arrs) + (idx,)
