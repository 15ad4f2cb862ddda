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
