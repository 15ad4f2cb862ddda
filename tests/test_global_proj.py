"""Longformer global attention with separate projections (Ultralytics glossary
"Longformer", section "How the Longformer attention works": the global
attention has query, key and value projections of its own).

CPU: argument validation of sa_forward_global_proj before any GPU use.  GPU
(marked): the CUDA path against the fp64 oracle's
forward_longformer(global_proj=...), every row, the bf16 tensor-core path and
the fp32 CUDA-core path; tolerance as in test_parity_gpu (|gpu - oracle| <=
2e-3 + 1e-2 |oracle|).  Passing q, k, v themselves as the global projections
must give sa_forward's result bit for bit.
"""
import ctypes

import numpy as np
import pytest

from sparse_long_context_banded_gb300 import build, inputs, sa

FAKE = 0x10000  # aligned, non-null; validation fails before any use


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sa.load()


def _call(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, qg=FAKE, kg=FAKE, vg=FAKE, out=FAKE, lse=None, B=1, H=1,
             N=64, D=64, window=8, g=[0], scale=0.125, dtype=sa.SA_BF16)
    a.update(kw)
    g = None if a["g"] is None else np.asarray(a["g"], dtype=np.int32)
    return lib.sa_forward_global_proj(
        a["q"], a["k"], a["v"], a["qg"], a["kg"], a["vg"], a["out"], a["lse"], a["B"], a["H"],
        a["N"], a["D"], a["window"], None,
        None if g is None else g.ctypes.data_as(ctypes.c_void_p), 0 if g is None else int(g.size),
        a["scale"], a["dtype"], None)


@pytest.mark.parametrize("kw", [dict(qg=None), dict(kg=None), dict(vg=None), dict(kg=FAKE + 4),
                                dict(vg=FAKE + 2), dict(q=None), dict(N=0), dict(g=[64]),
                                dict(window=-2)],
                         ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_rejects_bad_arguments(lib, kw):
    assert _call(lib, **kw) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_last_error()


GPU_CASES = [
    # B, H, N, D, window, dilation, globals, dtype
    (1, 2, 1000, 64, 256, [1, 1], [0], "bf16"),
    (1, 2, 777, 128, 300, [1, 2], [5, 700, 5], "bf16"),
    (1, 3, 640, 64, 128, [1, 2, 3], [639], "bf16"),          # global at N-1, dilation
    (2, 1, 515, 128, 200, [2], [0, 1, 514], "fp32"),
    (1, 2, 4096, 128, 1024, [1, 1], list(range(64)), "bf16"),
    (1, 1, 2050, 64, 600, [4], list(range(0, 2050, 97)), "bf16"),
    (1, 1, 200, 64, 0, [1], list(range(200)), "bf16"),       # every position global
    (1, 2, 300, 64, 40, [1, 1], [], "bf16"),                 # no globals: projections unread
    (1, 1, 1, 128, 0, [1], [0], "fp32"),
]


def _draw(case, seed):
    B, H, N, D, _, _, _, dtype = case
    w = inputs.custom(B, H, N, D, 0, dtype=dtype, number=0)
    return inputs.draw_qkv(w, seed=seed) + inputs.draw_qkv(w, seed=seed + 1)


@pytest.mark.gpu
@pytest.mark.parametrize("case", GPU_CASES, ids=lambda c: "B{}H{}N{}D{}w{}d{}g{}{}".format(
    c[0], c[1], c[2], c[3], c[4], max(c[5]), len(c[6]), c[7]))
def test_global_proj_matches_oracle(oracle, case):
    import torch

    from test_parity_gpu import assert_close, assert_lse_close, to_device

    B, H, N, D, window, dil, G, dtype = case
    arrays = _draw(case, 9000 + N + len(G))
    ref, ref_lse = oracle.forward_longformer(*arrays[:3], window, dil, G,
                                             global_proj=arrays[3:])
    t = [to_device(a, torch) for a in arrays]
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    out = sa.forward_global_proj(*t, window, dil, G, lse=lse)
    sa.sync_status()
    got = out.float().cpu().numpy().astype(np.float64)
    assert_close(got, ref, f"global projections {case}")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, f"global projections {case}")


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_same_projections_equal_plain_forward(dtype):
    import torch

    from test_parity_gpu import to_device

    case = (1, 2, 1500, 128, 384, [1, 2], [0, 3, 1499], dtype)
    q, k, v = (to_device(a, torch) for a in _draw(case, 77)[:3])
    plain = sa.forward(q, k, v, 384, [1, 2], [0, 3, 1499])
    same = sa.forward_global_proj(q, k, v, q, k, v, 384, [1, 2], [0, 3, 1499])
    sa.sync_status()
    assert torch.equal(plain, same)
