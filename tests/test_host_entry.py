"""sa_forward_host: host buffers in, host buffers out, through the C ABI.

GPU (marked): the outputs and log-sum-exp against the fp64 oracle at the
parity tolerance (|gpu - oracle| <= 2e-3 + 1e-2 |oracle|; lse 1e-3 (1 + |oracle|)),
on every row of small problems, for every way of cutting the (b, h) slices into
groups (one head, two heads, a whole batch element, two batch elements, the
library's choice), with pinned and with pageable host memory; and on sampled
rows of the 131072-token workload with the library's grouping (sixteen groups of
one head), the configuration the end-to-end bench line times.  The result
must not depend on the grouping: band rows are computed by the same tiles
whichever group holds them.
"""
import numpy as np
import pytest

from sparse_long_context_banded_gb300 import inputs, sa

from test_parity_gpu import assert_close, assert_lse_close, sample_rows, workload_inputs

pytestmark = pytest.mark.gpu


def host(a, torch, pin):
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 \
        else torch.from_numpy(a)
    return t.pin_memory() if pin else t.clone()


def run_host(q, k, v, window, dilation, globals_, scale=None, heads_per_group=0, pin=True):
    import torch
    hq, hk, hv = (host(a, torch, pin) for a in (q, k, v))
    B, H, N, D = q.shape
    out = torch.empty_like(hq)
    if pin:
        out = out.pin_memory()
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32)
    sa.forward_host(hq, hk, hv, window, dilation, globals_, scale=scale, out=out, lse=lse,
                    heads_per_group=heads_per_group)
    return out.float().numpy().astype(np.float64), lse.numpy().astype(np.float64)


CASES = [
    # B, H, N, D, window, dilation, globals, dtype
    (2, 3, 700, 64, 100, [1, 2, 3], [0, 5, 699], "bf16"),
    (3, 2, 515, 128, 200, [2, 1], list(range(64)), "bf16"),
    (2, 2, 300, 64, 64, [1, 1], [7], "fp32"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}D{}-{}".format(*c[:4], c[7]))
@pytest.mark.parametrize("heads_per_group", [0, 1, 2, 3, 7])
def test_host_entry_every_row(case, heads_per_group, oracle):
    B, H, N, D, window, dil, G, dtype = case
    w = inputs.custom(B, H, N, D, window, dilation=dil, globals_=G, dtype=dtype)
    q, k, v = inputs.draw_qkv(w, seed=41)
    got, got_lse = run_host(q, k, v, window, dil, G, heads_per_group=heads_per_group)
    ref, ref_lse = oracle.forward_longformer(q, k, v, window, dil, G, scale=D ** -0.5)
    what = f"host entry {case} heads_per_group={heads_per_group}"
    assert_close(got, ref, what)
    assert_lse_close(got_lse, ref_lse, what)


EDGE_CASES = [
    # B, H, N, D, window, dilation, globals, dtype, tf32
    (1, 1, 1, 64, 16, [1], [0], "bf16", False),          # one row, one head
    (1, 1, 129, 128, 0, [1], [], "bf16", False),         # no window, no globals
    (1, 2, 700, 64, 128, [1, 2], [0, 699], "fp32", True),  # fp32 inputs on the tensor cores (tf32)
]


@pytest.mark.parametrize("case", EDGE_CASES, ids=lambda c: "B{}H{}N{}D{}-{}{}".format(
    *c[:4], c[7], "-tf32" if c[8] else ""))
def test_host_entry_edge_cases(case, oracle):
    import torch
    B, H, N, D, window, dil, G, dtype, tf32 = case
    w = inputs.custom(B, H, N, D, window, dilation=dil, globals_=G, dtype=dtype)
    q, k, v = inputs.draw_qkv(w, seed=44)
    hq, hk, hv = (host(a, torch, True) for a in (q, k, v))
    out = sa.forward_host(hq, hk, hv, window, dil, G, tf32=tf32)  # no lse
    ref, _ = oracle.forward_longformer(q, k, v, window, dil, G, scale=D ** -0.5, want_lse=False)
    assert_close(out.float().numpy().astype(np.float64), ref, f"host entry {case}")


def test_host_entry_pageable_matches_pinned():
    B, H, N, D = 2, 4, 1200, 64
    w = inputs.custom(B, H, N, D, 256, dilation=[1, 2, 1, 3], globals_=[0, 600], dtype="bf16")
    q, k, v = inputs.draw_qkv(w, seed=42)
    a, a_lse = run_host(q, k, v, 256, w.dilation, w.globals_, heads_per_group=1, pin=True)
    b, b_lse = run_host(q, k, v, 256, w.dilation, w.globals_, heads_per_group=1, pin=False)
    assert np.array_equal(a, b) and np.array_equal(a_lse, b_lse)


def test_host_entry_grouping_leaves_band_rows_unchanged():
    """Band rows (not global) are bitwise the same whatever the grouping."""
    B, H, N, D = 1, 4, 2000, 128
    G = [3, 1500]
    w = inputs.custom(B, H, N, D, 300, dilation=[1, 1, 2, 2], globals_=G, dtype="bf16")
    q, k, v = inputs.draw_qkv(w, seed=43)
    outs = [run_host(q, k, v, 300, w.dilation, G, heads_per_group=g)[0] for g in (1, 2, 4)]
    band = np.setdiff1d(np.arange(N), G)
    for o in outs[1:]:
        assert np.array_equal(o[:, :, band], outs[0][:, :, band])


def test_host_entry_rejects_device_tensors():
    import torch
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        sa.forward_host(q, q, q, 8)
    h = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sa.forward_host(h, h, h, 8, out=q)


def test_host_entry_long_context_sampled(oracle):
    """The 131072-token workload through the host entry, as the end-to-end
    bench line runs it (pinned inputs, the library's grouping)."""
    w, (q, k, v) = workload_inputs(5)
    got, got_lse = run_host(q, k, v, w.window, w.dilation, w.globals_, scale=w.scale)
    rows = sample_rows(w, np.random.default_rng(55), 600)
    ref, ref_lse = oracle.forward_longformer(q, k, v, w.window, w.dilation, w.globals_,
                                             scale=w.scale, rows=rows)
    assert_close(got.reshape(-1, w.D)[rows], ref, "host entry " + w.describe())
    assert_lse_close(got_lse.reshape(-1)[rows], ref_lse, "host entry " + w.describe())
