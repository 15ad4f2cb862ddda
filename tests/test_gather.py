"""Attention over per-query key lists ("Unlimiformer", sections 2.2-2.3: each
query attends only to the keys its retrieval returned).

CPU: argument validation of sa_forward_gather before any GPU use.  GPU (marked):
the CUDA kernel against the fp64 oracle's forward_gather -- every row of small
cases (ragged lists, padding, out-of-range entries, repeats, empty rows, list
lengths that are not a multiple of the 32-key group, bf16 and fp32, D 64 and
128), and sampled rows of the 131072-key retrieval workload.  Tolerance as in
test_parity_gpu: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| per element,
log-sum-exp within 1e-3 (1 + |oracle|); rows with no valid entry must give
exactly 0 and -inf.
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
    a = dict(q=FAKE, k=FAKE, v=FAKE, idx=FAKE, out=FAKE, lse=None, B=1, H=1, Nq=8, Nk=16,
             D=64, K=4, scale=0.125, dtype=sa.SA_BF16)
    a.update(kw)
    return lib.sa_forward_gather(a["q"], a["k"], a["v"], a["idx"], a["out"], a["lse"], a["B"],
                                 a["H"], a["Nq"], a["Nk"], a["D"], a["K"], a["scale"],
                                 a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), sa.SA_ERR_INVALID_ARG), (dict(out=None), sa.SA_ERR_INVALID_ARG),
    (dict(idx=None), sa.SA_ERR_INVALID_ARG), (dict(K=-1), sa.SA_ERR_INVALID_ARG),
    (dict(Nq=0), sa.SA_ERR_INVALID_ARG), (dict(Nk=0), sa.SA_ERR_INVALID_ARG),
    (dict(B=0), sa.SA_ERR_INVALID_ARG), (dict(k=FAKE + 8), sa.SA_ERR_INVALID_ARG),
    (dict(idx=FAKE + 2), sa.SA_ERR_INVALID_ARG), (dict(scale=float("inf")), sa.SA_ERR_INVALID_ARG),
    (dict(dtype=5), sa.SA_ERR_INVALID_ARG), (dict(D=96), sa.SA_ERR_UNSUPPORTED),
], ids=lambda x: str(x))
def test_rejects_bad_arguments(lib, kw, status):
    assert _call(lib, **kw) == status
    assert lib.sa_last_error()


def test_generator_lists_are_distinct_and_in_range():
    w = inputs.GatherWorkload("t", 1, 2, 40, 300, 64, 100, "bf16")
    q, k, v, idx = inputs.draw_gather(w, 3)
    assert idx.dtype == np.int32 and idx.shape == (1, 2, 40, 100)
    valid = idx[idx >= 0]
    assert valid.max() < 300 and (idx >= -1).all()
    for row in idx.reshape(-1, 100):
        r = row[row >= 0]
        assert np.unique(r).size == r.size
    assert 0 < (idx < 0).mean() < 0.3


GPU_CASES = [
    # B, H, Nq, Nk, D, K, dtype
    (1, 2, 100, 500, 128, 64, "bf16"),
    (2, 1, 77, 1000, 64, 37, "bf16"),      # K not a multiple of 32
    (1, 3, 50, 64, 64, 64, "bf16"),         # lists hold most of the keys
    (1, 1, 33, 4000, 128, 300, "bf16"),
    (1, 2, 65, 700, 128, 1, "bf16"),        # one key per row
    (1, 2, 100, 500, 128, 64, "fp32"),
    (2, 2, 31, 129, 64, 45, "fp32"),
]


def _gpu_run(q, k, v, idx, scale):
    import torch

    from test_parity_gpu import to_device

    tq, tk, tv = (to_device(a, torch) for a in (q, k, v))
    ti = torch.from_numpy(np.ascontiguousarray(idx)).cuda()
    B, H, Nq, _ = q.shape
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    out = sa.forward_gather(tq, tk, tv, ti, scale=scale, lse=lse)
    sa.sync_status()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _check(got, got_lse, ref, ref_lse, what):
    from test_parity_gpu import assert_close, assert_lse_close

    empty = np.isneginf(ref_lse)
    assert (got[empty] == 0).all() and np.isneginf(got_lse[empty]).all(), what
    assert_close(got[~empty], ref[~empty], what)
    assert_lse_close(got_lse[~empty], ref_lse[~empty], what)


@pytest.mark.gpu
@pytest.mark.parametrize("case", GPU_CASES, ids=lambda c: "B{}H{}Nq{}Nk{}D{}K{}{}".format(*c))
def test_gather_matches_oracle(oracle, case):
    B, H, Nq, Nk, D, K, dtype = case
    w = inputs.GatherWorkload("case", B, H, Nq, Nk, D, K, dtype)
    q, k, v, idx = inputs.draw_gather(w, seed=Nq + Nk + K)
    rng = np.random.default_rng(K)
    idx[rng.random(idx.shape) < 0.05] = Nk + 7   # out-of-range entries are padding too
    idx[0, 0, 1] = -1                             # a row with no valid entry
    if K >= 3:
        idx[0, 0, 2, :3] = idx[0, 0, 2, 0] if idx[0, 0, 2, 0] >= 0 else 5  # a repeated key
    ref, ref_lse = oracle.forward_gather(q, k, v, idx, scale=w.scale)
    got, got_lse = _gpu_run(q, k, v, idx, w.scale)
    _check(got, got_lse, ref, ref_lse, str(case))


@pytest.mark.gpu
def test_gather_empty_lists():
    import torch

    w = inputs.GatherWorkload("empty", 1, 1, 5, 20, 64, 3, "bf16")
    q, k, v, idx = inputs.draw_gather(w, 1)
    idx[:] = -1
    got, got_lse = _gpu_run(q, k, v, idx, w.scale)
    assert (got == 0).all() and np.isneginf(got_lse).all()
    # K = 0: no list at all
    tq = torch.zeros((1, 1, 5, 64), dtype=torch.bfloat16, device="cuda")
    tk = torch.zeros((1, 1, 20, 64), dtype=torch.bfloat16, device="cuda")
    ti = torch.zeros((1, 1, 5, 0), dtype=torch.int32, device="cuda")
    out = sa.forward_gather(tq, tk, tk, ti)
    sa.sync_status()
    assert (out.float() == 0).all()


@pytest.mark.gpu
def test_gather_retrieval_workload_sampled(oracle):
    """The 131072-key retrieval workload at full size, compared on sampled rows
    (the first and last rows of every head and seeded random rows)."""
    w = inputs.gather_workload()
    q, k, v, idx = inputs.draw_gather(w)
    got, got_lse = _gpu_run(q, k, v, idx, w.scale)
    n = w.B * w.H * w.Nq
    rng = np.random.default_rng(5)
    rows = set(rng.integers(0, n, size=600).tolist())
    for bh in range(w.B * w.H):
        rows |= {bh * w.Nq, bh * w.Nq + w.Nq - 1}
    rows = np.array(sorted(rows), dtype=np.int64)
    ref, ref_lse = oracle.forward_gather(q, k, v, idx, scale=w.scale, rows=rows)
    _check(got.reshape(-1, w.D)[rows], got_lse.reshape(-1)[rows], ref, ref_lse, w.describe())
