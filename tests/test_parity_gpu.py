"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerance (per output element): |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|, for
bf16 and fp32 inputs alike.  Log-sum-exp: |gpu - oracle| <= 1e-3 * (1 + |oracle|).
Small problems are compared on every row; the five workload shapes at full size
are compared on sampled rows (all tile seams, the ragged tail, global rows and
seeded random rows), which the oracle computes one by one.
"""
import zlib

import numpy as np
import pytest

from sparse_long_context_banded_gb300 import inputs, sa

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
LSE_TOL = 1e-3


def to_device(a, torch):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def run_gpu(q, k, v, window, dilation, globals_, scale=None, tf32=False):
    import torch
    tq, tk, tv = (to_device(a, torch) for a in (q, k, v))
    B, H, N, D = q.shape
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    out = sa.forward(tq, tk, tv, window, dilation, globals_, scale=scale, lse=lse, tf32=tf32)
    sa.sync_status()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def assert_close(got, ref, what):
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any() or not np.isfinite(got).all():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at "
                             f"{idx}: got {got[idx]!r} ref {ref[idx]!r}")


def assert_lse_close(got, ref, what):
    err = np.abs(got - ref)
    bound = LSE_TOL * (1 + np.abs(ref))
    if (err > bound).any() or not np.isfinite(got).all():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what} lse: worst at {i}: got {got[i]} ref {ref[i]}")


def make(B, H, N, D, dtype, seed):
    w = inputs.custom(B, H, N, D, 0, dtype=dtype, number=0)
    return inputs.draw_qkv(w, seed=seed)


SMALL_CASES = [
    # B, H, N, D, window, dilation, globals, dtype
    (1, 2, 1000, 64, 256, [1, 1], [0], "bf16"),
    (1, 2, 777, 128, 300, [1, 2], [5, 700, 5], "bf16"),
    (2, 1, 129, 64, 0, [1], [], "bf16"),
    (1, 1, 1, 64, 16, [1], [0], "bf16"),
    (1, 1, 1, 128, 0, [1], [], "fp32"),
    (1, 2, 300, 64, 1000, [1, 1], [], "bf16"),          # window >= 2N: dense
    (1, 1, 200, 64, 0, [1], list(range(200)), "bf16"),  # every position global
    (1, 3, 640, 64, 128, [1, 2, 3], [639], "bf16"),     # global at N-1, dilation
    (1, 2, 500, 64, 512, [3, 7], [1, 2, 3], "bf16"),    # d*h >= N
    (1, 2, 1024, 64, 512, [1, 1], [0], "fp32"),
    (2, 2, 515, 128, 200, [2, 1], [0, 1, 514], "fp32"),
    (1, 2, 4096, 128, 1024, [1, 1], list(range(64)), "bf16"),
    (1, 1, 2050, 64, 600, [4], list(range(0, 2050, 97)), "bf16"),
    (1, 2, 1500, 64, 255, [1, 2], [3, 1499], "bf16"),    # odd window: half width 127
    (1, 2, 2000, 128, 511, [1, 3], [7, 100, 1999], "bf16"),
    # bands narrower than a 64-key sub-tile: whole sub-tiles masked for some rows
    (1, 2, 1111, 128, 100, [1, 3], [17], "bf16"),
    (1, 1, 4500, 64, 62, [2], [], "bf16"),
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: "B{}H{}N{}D{}w{}d{}g{}{}".format(
    c[0], c[1], c[2], c[3], c[4], max(c[5]), len(c[6]), c[7]))
def test_small_full(case, oracle):
    B, H, N, D, window, dil, G, dtype = case
    q, k, v = make(B, H, N, D, dtype, seed=zlib.crc32(repr(case).encode()))
    got, got_lse = run_gpu(q, k, v, window, dil, G)
    ref, ref_lse = oracle.forward_longformer(q, k, v, window, dil, G)
    assert_close(got, ref, str(case))
    assert_lse_close(got_lse, ref_lse, str(case))


# A scale several times 1/sqrt(D) makes each row's softmax peak on a few keys,
# where single bf16 weights in the P V product no longer average out (as for
# rows with few keys): the automatic choice splits P into two bf16 parts for
# |scale| sqrt(D) > 1.25, and the bf16 path meets the tolerance there too.
SCALE_CASES = [
    (1, 1, 640, 64, 128, [1], [5], "bf16", 0.6),                 # large positive scale
    (1, 2, 1000, 128, 256, [1, 2], [0, 999], "bf16", 0.5),
    (1, 1, 700, 64, 300, [1], [3], "bf16", -1.0),
    (1, 1, 2000, 128, 1024, [1], list(range(64)), "bf16", 0.3),
    # B, H, N, D, window, dilation, globals, dtype, scale
    (1, 2, 1000, 128, 256, [1, 2], [0, 999], "bf16", -0.0883),   # negative scale
    (1, 1, 700, 64, 300, [1], [3], "bf16", -0.125),
    (1, 1, 700, 64, 300, [1], [3], "fp32", -1.0),
    (1, 2, 515, 64, 200, [1, 1], [0], "fp32", -0.125),
    (1, 1, 640, 128, 128, [1], [0, 1], "bf16", 0.0),             # zero scale: plain averages
    (1, 1, 640, 64, 128, [1], [0, 1], "fp32", 0.0),
    (1, 1, 640, 64, 128, [1], [5], "bf16", 0.2),
    (1, 1, 640, 64, 128, [1], [5], "fp32", 0.6),                 # large positive scale
]


@pytest.mark.parametrize("case", SCALE_CASES, ids=lambda c: "N{}D{}s{}{}".format(
    c[2], c[3], c[8], c[7]))
def test_scale_sign_and_size(case, oracle):
    B, H, N, D, window, dil, G, dtype, scale = case
    q, k, v = make(B, H, N, D, dtype, seed=zlib.crc32(repr(case).encode()))
    got, got_lse = run_gpu(q, k, v, window, dil, G, scale)
    ref, ref_lse = oracle.forward_longformer(q, k, v, window, dil, G, scale=scale)
    assert_close(got, ref, str(case))
    assert_lse_close(got_lse, ref_lse, str(case))


# fp32 inputs with tf32 products on the tensor cores (SA_TF32, D = 64): the
# fp32 cases above at the workloads' scale 1/sqrt(D), every row.
TF32_CASES = [
    (1, 2, 1024, 64, 512, [1, 1], [0]),               # the tiny Longformer-mask shape
    (1, 2, 777, 64, 300, [1, 2], [5, 700, 5]),
    (2, 1, 129, 64, 0, [1], []),
    (1, 1, 1, 64, 16, [1], [0]),
    (1, 3, 640, 64, 128, [1, 2, 3], [639]),
    (1, 1, 200, 64, 0, [1], list(range(200))),        # every position global
    (1, 2, 300, 64, 1000, [1, 1], []),                # dense
    (1, 1, 2050, 64, 600, [4], list(range(0, 2050, 97))),
]


@pytest.mark.parametrize("case", TF32_CASES, ids=lambda c: "B{}H{}N{}w{}d{}g{}".format(
    c[0], c[1], c[2], c[4], max(c[5]), len(c[6])))
def test_tf32_full(case, oracle):
    B, H, N, D, window, dil, G = case
    q, k, v = make(B, H, N, D, "fp32", seed=zlib.crc32(repr(case).encode()))
    got, got_lse = run_gpu(q, k, v, window, dil, G, tf32=True)
    ref, ref_lse = oracle.forward_longformer(q, k, v, window, dil, G)
    assert_close(got, ref, "tf32 " + str(case))
    assert_lse_close(got_lse, ref_lse, "tf32 " + str(case))


# Both precisions of the P V product on the bf16 tensor-core path, whatever
# the automatic choice would be: single bf16 P (the workloads' setting) and P
# split into two bf16 parts.  The global sets cover every layout of the
# global-row work: none; up to 64 rows (packed twice into a query tile, one
# copy per key half); 65-128 rows (one query tile, the CTA's two tiles taking
# alternate key tiles); more than 128 (two query tiles over the same keys).
PV_CASES = [
    # B, H, N, D, window, dilation, globals (a count: scattered; a list), dtype
    (1, 2, 900, 64, 128, [1, 3], [], "bf16"),
    (1, 2, 2000, 128, 512, [1, 1], list(range(64)), "bf16"),
    (1, 1, 4096, 128, 1024, [1], [0], "bf16"),
    (1, 2, 1500, 64, 256, [1, 2], list(range(100)), "bf16"),
    (1, 1, 1300, 128, 300, [1], 90, "bf16"),
    (1, 1, 3000, 64, 200, [2], 150, "bf16"),
    (2, 1, 333, 128, 64, [1], 7, "bf16"),
]


@pytest.mark.parametrize("mode", ["single", "split"])
@pytest.mark.parametrize("case", PV_CASES, ids=lambda c: "B{}H{}N{}D{}w{}d{}g{}".format(
    c[0], c[1], c[2], c[3], c[4], max(c[5]), c[6] if isinstance(c[6], int) else len(c[6])))
def test_pv_modes(case, mode, oracle):
    B, H, N, D, window, dil, G, dtype = case
    if isinstance(G, int):
        G = sorted(np.random.default_rng(N + G).choice(N, G, replace=False).tolist())
    q, k, v = make(B, H, N, D, dtype, seed=zlib.crc32(repr(case).encode()))
    sa.set_pv_mode(sa.SA_PV_SINGLE if mode == "single" else sa.SA_PV_SPLIT)
    try:
        got, got_lse = run_gpu(q, k, v, window, dil, G)
    finally:
        sa.set_pv_mode(sa.SA_PV_AUTO)
    ref, ref_lse = oracle.forward_longformer(q, k, v, window, dil, G)
    assert_close(got, ref, f"{mode} {case}")
    assert_lse_close(got_lse, ref_lse, f"{mode} {case}")


def test_split_p_error_smaller_on_sharp_rows(oracle):
    """On a sharp softmax, splitting P brings the bf16 output error down to the
    bf16 rounding of the output itself."""
    q, k, v = make(1, 1, 640, 64, "bf16", seed=77)
    errs = {}
    for mode in (sa.SA_PV_SINGLE, sa.SA_PV_SPLIT):
        sa.set_pv_mode(mode)
        try:
            got, _ = run_gpu(q, k, v, 128, [1], [5], 0.6)
        finally:
            sa.set_pv_mode(sa.SA_PV_AUTO)
        ref, _ = oracle.forward_longformer(q, k, v, 128, [1], [5], scale=0.6, want_lse=False)
        errs[mode] = np.abs(got - ref) / (1e-3 + np.abs(ref))
    assert errs[sa.SA_PV_SPLIT].max() < errs[sa.SA_PV_SINGLE].max()
    assert errs[sa.SA_PV_SPLIT].max() < 1.0 / 128  # within an output rounding (2^-8) and a bit


def test_tf32_rejects_d128():
    import torch
    q = torch.zeros((1, 1, 64, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(sa.SaError) as e:
        sa.forward(q, q, q, 16, tf32=True)
    assert e.value.status == sa.SA_ERR_UNSUPPORTED


# The largest global set (SA_MAX_GLOBALS = 256): four 64-key global tiles per
# band item and two 128-row query tiles per global-row item, with and without
# dilation, scattered and contiguous.
MAX_GLOBAL_CASES = [
    (1, 2, 3000, 128, 256, [1, 2], "scattered", "bf16"),
    (1, 1, 2049, 64, 512, [1], "prefix", "bf16"),
    (1, 1, 1500, 64, 100, [3], "scattered", "fp32"),
]


@pytest.mark.parametrize("case", MAX_GLOBAL_CASES, ids=lambda c: "N{}D{}d{}{}{}".format(
    c[2], c[3], max(c[5]), c[6], c[7]))
def test_max_globals(case, oracle):
    B, H, N, D, window, dil, kind, dtype = case
    rng = np.random.default_rng(N)
    G = (sorted(rng.choice(N, sa.SA_MAX_GLOBALS, replace=False).tolist()) if kind == "scattered"
         else list(range(sa.SA_MAX_GLOBALS)))
    q, k, v = make(B, H, N, D, dtype, seed=zlib.crc32(repr(case).encode()))
    got, got_lse = run_gpu(q, k, v, window, dil, G)
    ref, ref_lse = oracle.forward_longformer(q, k, v, window, dil, G)
    assert_close(got, ref, str(case))
    assert_lse_close(got_lse, ref_lse, str(case))


def test_too_many_globals_rejected():
    import torch
    q = torch.zeros((1, 1, 300, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa.SaError) as e:
        sa.forward(q, q, q, 16, None, list(range(sa.SA_MAX_GLOBALS + 1)))
    assert e.value.status == sa.SA_ERR_UNSUPPORTED


def sample_rows(w, rng, n_random):
    """Flattened row ids covering tile seams, the tail, globals and random rows."""
    rows = set()
    N = w.N
    seams = [0, 1, 63, 64, 127, 128, 129, 255, 256, 257, N // 2, N - 129, N - 128, N - 2, N - 1]
    for bh in range(w.B * w.H):
        for i in seams:
            if 0 <= i < N:
                rows.add(bh * N + i)
    G = list(w.globals_)
    for bh in sorted(set([0, w.B * w.H - 1])):
        for g in (G if len(G) <= 32 else G[:4] + G[-4:]):
            rows.add(bh * N + g)
    for x in rng.integers(0, w.B * w.H * N, size=n_random):
        rows.add(int(x))
    return np.array(sorted(rows), dtype=np.int64)


_cache = {}


def workload_inputs(number):
    if number not in _cache:
        _cache.clear()
        w = inputs.workload(number)
        _cache[number] = (w, inputs.draw_qkv(w))
    return _cache[number]


def test_tiny_workload_tf32(oracle):
    """The fp32 tiny Longformer-mask workload through the tf32 tensor-core path,
    every row."""
    w, (q, k, v) = workload_inputs(1)
    got, got_lse = run_gpu(q, k, v, w.window, w.dilation, w.globals_, w.scale, tf32=True)
    ref, ref_lse = oracle.forward_longformer(q, k, v, w.window, w.dilation, w.globals_,
                                             scale=w.scale)
    assert_close(got, ref, "tf32 " + w.describe())
    assert_lse_close(got_lse, ref_lse, "tf32 " + w.describe())


@pytest.mark.parametrize("number", [1, 2, 3, 4, 5])
def test_workload_sampled(number, oracle):
    w, (q, k, v) = workload_inputs(number)
    got, got_lse = run_gpu(q, k, v, w.window, w.dilation, w.globals_, w.scale)
    rng = np.random.default_rng(number)
    rows = sample_rows(w, rng, 3000 if number < 5 else 1500)
    ref, ref_lse = oracle.forward_longformer(q, k, v, w.window, w.dilation, w.globals_,
                                             scale=w.scale, rows=rows)
    assert_close(got.reshape(-1, w.D)[rows], ref, w.describe())
    assert_lse_close(got_lse.reshape(-1)[rows], ref_lse, w.describe())
    assert np.isfinite(got).all()


def test_memory_prefix_matches_gmat_oracle(oracle):
    """The memory-prefix workload run as globals {0..M-1} equals the GMAT
    pattern evaluated literally (memory prefix + main-sequence band)."""
    w, (q, k, v) = workload_inputs(3)
    got, _ = run_gpu(q, k, v, w.window, w.dilation, w.globals_, w.scale)
    rows = sample_rows(w, np.random.default_rng(33), 1000)
    ref, _ = oracle.forward_gmat(q, k, v, w.memory, window=w.window, scale=w.scale, rows=rows,
                                 want_lse=False)
    assert_close(got.reshape(-1, w.D)[rows], ref, "GMAT memory prefix")


def test_deterministic_and_stream_ordered():
    import torch
    q, k, v = make(1, 2, 3000, 64, "bf16", seed=5)
    tq, tk, tv = (to_device(a, torch) for a in (q, k, v))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = sa.forward(tq, tk, tv, 256, None, [0, 17])
        b = sa.forward(tq, tk, tv, 256, None, [0, 17])
    s.synchronize()
    sa.sync_status(s)
    assert torch.equal(a, b)


def test_profile_counts_launches():
    import torch
    q, k, v = make(1, 1, 512, 64, "bf16", seed=6)
    tq, tk, tv = (to_device(a, torch) for a in (q, k, v))
    # scattered globals: gather, then band tiles and global rows in one
    # tensor-core launch, then the merge
    sa.profile_begin()
    for _ in range(3):
        sa.forward(tq, tk, tv, 64, None, [3, 100])
    prof = sa.profile_end()
    assert [prof[s]["launches"] for s in sa.STAGES] == [3, 3, 0, 3]
    assert all(prof[s]["ms"] > 0 for s in ("gather", "band", "merge"))
    # contiguous globals: read in place, nothing gathered
    sa.profile_begin()
    for _ in range(3):
        sa.forward(tq, tk, tv, 64, None, [3, 4, 5])
    prof = sa.profile_end()
    assert [prof[s]["launches"] for s in sa.STAGES] == [0, 3, 0, 3]
    sa.profile_begin()
    sa.forward(tq, tk, tv, 64, None, [])
    prof = sa.profile_end()
    assert [prof[s]["launches"] for s in sa.STAGES] == [0, 1, 0, 0]
    # more residue classes than one launch addresses (dilation 17: 17 classes):
    # two band launches and the global rows in a launch of their own
    sa.profile_begin()
    sa.forward(tq, tk, tv, 64, [17], [3, 4, 5])
    prof = sa.profile_end()
    assert [prof[s]["launches"] for s in sa.STAGES] == [0, 2, 1, 1]
    # fp32 on the CUDA cores: four kernels
    q32 = tq.float()
    sa.profile_begin()
    sa.forward(q32, q32, q32, 64, None, [3, 100])
    prof = sa.profile_end()
    assert [prof[s]["launches"] for s in sa.STAGES] == [1, 1, 1, 1]


def test_concurrent_threads_and_streams():
    """Two host threads, each on a stream of its own, call the library at the
    same time with different problem shapes (different schedules, scratch from
    the same pool); every result equals the same call made alone."""
    import threading

    import torch
    problems = [
        (make(1, 2, 3000, 64, "bf16", seed=11), 256, [1, 2], [0, 17, 2999]),
        (make(1, 2, 2304, 128, "bf16", seed=12), 1024, [1, 1], list(range(64))),
    ]
    dev = [[to_device(a, torch) for a in qkv] for qkv, _, _, _ in problems]
    alone = []
    for (qkv, window, dil, G), (tq, tk, tv) in zip(problems, dev):
        alone.append(sa.forward(tq, tk, tv, window, dil, G))
    torch.cuda.synchronize()
    sa.sync_status()
    results = [[], []]
    errors = []

    def worker(i):
        try:
            (qkv, window, dil, G), (tq, tk, tv) = problems[i], dev[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(20):
                    results[i].append(sa.forward(tq, tk, tv, window, dil, G))
            s.synchronize()
            sa.sync_status(s)
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        assert len(results[i]) == 20
        for r in results[i]:
            assert torch.equal(r, alone[i])


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_cuda_graph_capture_and_replay():
    """A call captured into a CUDA graph (after one call of the same shape
    outside capture, which builds the schedule) replays with new input values
    and gives exactly what an eager call gives; a first call under capture is
    refused before anything is enqueued."""
    import torch
    B, H, N, D, window, dil, G = 1, 2, 2304, 128, 1024, [1, 1], list(range(64))
    q0, k0, v0 = make(B, H, N, D, "bf16", seed=21)
    tq, tk, tv = (to_device(a, torch) for a in (q0, k0, v0))
    out = torch.empty_like(tq)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    sa.forward(tq, tk, tv, window, dil, G, out=out, lse=lse)  # builds the schedule
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        sa.forward(tq, tk, tv, window, dil, G, out=out, lse=lse, stream=s)  # warm on this stream
        s.synchronize()
        with torch.cuda.graph(graph, stream=s):
            sa.forward(tq, tk, tv, window, dil, G, out=out, lse=lse, stream=s)
    torch.cuda.synchronize()
    for seed in (22, 23):
        q1, k1, v1 = make(B, H, N, D, "bf16", seed=seed)
        for dst, src in zip((tq, tk, tv), (q1, k1, v1)):
            dst.copy_(to_device(src, torch))
        graph.replay()
        torch.cuda.synchronize()
        sa.sync_status()
        got, got_lse = out.clone(), lse.clone()
        ref_lse = torch.empty_like(lse)
        ref = sa.forward(tq, tk, tv, window, dil, G, lse=ref_lse)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
        assert torch.equal(got_lse, ref_lse)
    # a shape never run outside capture: refused, nothing captured
    small = torch.zeros((1, 2, 1000, D), dtype=torch.bfloat16, device="cuda")
    small_out = torch.empty_like(small)
    g2 = torch.cuda.CUDAGraph()
    status = None
    with torch.cuda.stream(s):
        with torch.cuda.graph(g2, stream=s):
            try:
                sa.forward(small, small, small, 333, dil, [5], out=small_out, stream=s)
            except sa.SaError as e:
                status = e.status
    assert status == sa.SA_ERR_INVALID_ARG
