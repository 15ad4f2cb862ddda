"""sa_forward_noalloc: the entry point for callers that cannot allocate device
memory (it takes all scratch from the library's static device array).

Checked through the C ABI against the fp64 oracle, twice in a row each (the
static array keeps the previous call's contents, so the second call must not
depend on them), within the tolerance of the parity tests:
|gpu - oracle| <= 2e-3 + 1e-2 |oracle| per element, and the log-sum-exp within
1e-3 (1 + |oracle|).  Small problems are compared on every row; the
131072-long sequence (16 heads, 64 globals: its global-row pass fits the array
only after several halvings of its key-chunk count) on sampled rows, which the
oracle computes one by one.  The file is named to be collected last.
"""
import ctypes
import zlib

import numpy as np
import pytest

from sparse_long_context_banded_gb300 import build, inputs, sa

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
LSE_TOL = 1e-3

CASES = [
    # B, H, N, D, window, dilation, globals, dtype, rows compared (None: all)
    (1, 3, 3000, 64, 256, [1, 2, 3], [0, 5, 2999], "bf16", None),
    (2, 2, 1024, 128, 512, [1, 1], [0], "fp32", None),
    (1, 2, 777, 128, 100, [2, 1], [], "bf16", None),
    (1, 16, 131072, 128, 1024, [1] * 16, list(range(64)), "bf16", 1200),
]


def _draw(case):
    B, H, N, D, window, dil, G, dtype, _ = case
    w = inputs.custom(B, H, N, D, window, dilation=dil, globals_=G, dtype=dtype, number=0)
    return w, inputs.draw_qkv(w, seed=zlib.crc32(repr(case[:8]).encode()) % (1 << 30))


def _device(a, torch):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def _rows(w, n_random):
    """Tile seams, the tail, global rows and seeded random rows of every head."""
    rng = np.random.default_rng(w.N)
    rows = set()
    for bh in range(w.B * w.H):
        for i in (0, 1, 63, 64, 127, 128, 4095, w.N // 2, w.N - 129, w.N - 1):
            rows.add(bh * w.N + i)
    for bh in (0, w.B * w.H - 1):
        for g in w.globals_[:4] + w.globals_[-4:]:
            rows.add(bh * w.N + g)
    rows.update(int(x) for x in rng.integers(0, w.B * w.H * w.N, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}N{c[2]}D{c[3]}{c[7]}")
def test_noalloc_matches_oracle_twice(case, oracle):
    import torch
    build.build()
    B, H, N, D, window, dil, G, dtype, n_rows = case
    w, (q, k, v) = _draw(case)
    rows = None if n_rows is None else _rows(w, n_rows)
    ref, ref_lse = oracle.forward_longformer(q, k, v, window, dil, G, scale=w.scale, rows=rows)
    tq, tk, tv = (_device(a, torch) for a in (q, k, v))
    for call in range(2):
        lse = torch.full((B, H, N), float("nan"), device="cuda")
        out = torch.full_like(tq, float("nan"))
        sa.forward_noalloc(tq, tk, tv, window, dil, G, scale=w.scale, out=out, lse=lse)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        got_lse = lse.cpu().numpy().astype(np.float64)
        if rows is not None:
            got = got.reshape(-1, D)[rows]
            got_lse = got_lse.reshape(-1)[rows]
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        err = np.abs(got - ref)
        bound = ATOL + RTOL * np.abs(ref)
        assert (err <= bound).all(), f"call {call}: max excess {(err - bound).max()}"
        lse_err = np.abs(got_lse - ref_lse)
        assert (lse_err <= LSE_TOL * (1 + np.abs(ref_lse))).all(), f"call {call}: lse differs"


def test_noalloc_does_not_grow_device_memory():
    import torch
    case = CASES[0]
    w, (q, k, v) = _draw(case)
    tq, tk, tv = (_device(a, torch) for a in (q, k, v))
    out = torch.empty_like(tq)
    sa.forward_noalloc(tq, tk, tv, w.window, w.dilation, w.globals_, out=out)  # first call: set-up
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        sa.forward_noalloc(tq, tk, tv, w.window, w.dilation, w.globals_, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    lib = sa.load()
    fake = 0x10000  # never dereferenced: the size check comes first
    g = np.arange(64, dtype=np.int32)
    st = lib.sa_forward_noalloc(fake, fake, fake, fake, None, 64, 16, 131072, 128, 1024, None,
                                g.ctypes.data_as(ctypes.c_void_p), 64, 0.088, sa.SA_BF16, None)
    assert st == sa.SA_ERR_UNSUPPORTED
    msg = lib.sa_last_error().decode()
    assert "static scratch" in msg and str(sa.SA_NOALLOC_SCRATCH_BYTES) in msg
