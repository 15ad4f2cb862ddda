"""The C-ABI library on the host: it loads, exports what include/*.h declares,
counts pairs exactly, and rejects bad arguments before touching a GPU."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

from oracle_pins import closed_form_counts
from sparse_long_context_banded_gb300 import build, inputs, sa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sa.load()


def declared_functions(debug=False):
    """Functions declared in include/sa.h (the release library's ABI), or in
    include/sa_debug.h (the SA_DEBUG build's test entry point)."""
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "sa_debug.h" if debug else "sa.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(sa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "sa_forward" in names and "sa_count_pairs" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in sa.SIGNATURES, f"{n} has no binding"


def test_headers_are_covered():
    """Every header in include/ is one of the two checked above and below."""
    assert sorted(os.path.basename(h) for h in glob.glob(os.path.join(ROOT, "include", "*.h"))) == \
        ["sa.h", "sa_debug.h"]


def test_debug_build_exports_every_declared_symbol():
    build.build(debug=True)
    dbg = sa.load_debug()
    names = declared_functions(debug=True)
    assert names == ["sa_debug_check_band_items"]
    for n in names + declared_functions():
        assert hasattr(dbg, n), n
        assert n in sa.SIGNATURES or n in sa.DEBUG_SIGNATURES, f"{n} has no binding"
    rel = sa.load()
    assert not hasattr(rel, "sa_debug_check_band_items")


def test_version(lib):
    assert "sm_103a" in sa.version()


@pytest.mark.parametrize("number", [1, 2, 3, 4, 5])
def test_count_pairs_bit_exact(lib, number, oracle):
    w = inputs.workload(number)
    per, total = sa.count_pairs(w.N, w.window, w.dilation, w.H, w.globals_)
    ref = [closed_form_counts(w.N, w.window, d, w.globals_) for d in w.dilation]
    assert per.tolist() == ref
    assert total == sum(ref)
    if number <= 4:
        assert per.tolist() == oracle.count_pairs_longformer(
            w.N, w.window, w.dilation, w.globals_).tolist()
    expected = {1: 922108, 2: 24517608, 3: 75396096 // 2, 5: 2412698624}
    if number in expected:
        assert total == expected[number]


def test_count_pairs_page_example(lib):
    got = [sa.count_pairs(n, 512, None, 1, [0])[1] for n in (1024, 2048, 4096)]
    assert got == [461054, 988414, 2043134]
    assert [f"{x / 1e6:.1f}" for x in got] == ["0.5", "1.0", "2.0"]


def test_count_pairs_random_cases(lib, oracle):
    rng = np.random.default_rng(3)
    for _ in range(60):
        N = int(rng.integers(1, 300))
        w = int(rng.integers(0, 2 * N + 2))
        H = int(rng.integers(1, 4))
        dil = [int(x) for x in rng.integers(1, 6, size=H)]
        G = [int(x) for x in rng.integers(0, N, size=int(rng.integers(0, 6)))]
        per, total = sa.count_pairs(N, w, dil, H, G)
        ref = oracle.count_pairs_longformer(N, w, dil, G)
        assert per.tolist() == ref.tolist(), (N, w, dil, G)


def test_count_pairs_duplicates_are_a_set(lib):
    a = sa.count_pairs(500, 40, [2], 1, [7, 7, 100, 7])
    b = sa.count_pairs(500, 40, [2], 1, [100, 7])
    assert a[1] == b[1]


def _status(fn, *args):
    return fn(*args)


FAKE = 0x10000  # an aligned non-null address; validation fails before any use


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, H=2, N=64, D=64, window=8,
         dilation=None, g=None, ng=0, scale=0.125, dtype=sa.SA_BF16):
    dil = None if dilation is None else np.asarray(dilation, dtype=np.int32)
    gg = None if g is None else np.asarray(g, dtype=np.int32)
    return lib.sa_forward(q, k, v, out, B, H, N, D, window,
                          None if dil is None else dil.ctypes.data_as(ctypes.c_void_p),
                          None if gg is None else gg.ctypes.data_as(ctypes.c_void_p),
                          ng, scale, dtype, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(q=None), sa.SA_ERR_INVALID_ARG),
    (dict(out=None), sa.SA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), sa.SA_ERR_INVALID_ARG),
    (dict(N=0), sa.SA_ERR_INVALID_ARG),
    (dict(N=-5), sa.SA_ERR_INVALID_ARG),
    (dict(B=0), sa.SA_ERR_INVALID_ARG),
    (dict(H=0), sa.SA_ERR_INVALID_ARG),
    (dict(window=-1), sa.SA_ERR_INVALID_ARG),
    (dict(dilation=[1, 0]), sa.SA_ERR_INVALID_ARG),
    (dict(g=[64], ng=1), sa.SA_ERR_INVALID_ARG),
    (dict(g=[-1], ng=1), sa.SA_ERR_INVALID_ARG),
    (dict(g=None, ng=3), sa.SA_ERR_INVALID_ARG),
    (dict(ng=-1), sa.SA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), sa.SA_ERR_INVALID_ARG),
    (dict(dtype=7), sa.SA_ERR_INVALID_ARG),
    (dict(D=96), sa.SA_ERR_UNSUPPORTED),
    (dict(D=32), sa.SA_ERR_UNSUPPORTED),
    (dict(N=1000, g=list(range(300)), ng=300), sa.SA_ERR_UNSUPPORTED),
])
def test_forward_rejects_bad_arguments(lib, kwargs, status):
    assert _fwd(lib, **kwargs) == status
    assert lib.sa_last_error().decode()


def _fwd_host(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, H=2, N=64, D=64, window=8,
              dilation=None, g=None, ng=0, scale=0.125, dtype=sa.SA_BF16, heads_per_group=0):
    dil = None if dilation is None else np.asarray(dilation, dtype=np.int32)
    gg = None if g is None else np.asarray(g, dtype=np.int32)
    return lib.sa_forward_host(q, k, v, out, None, B, H, N, D, window,
                               None if dil is None else dil.ctypes.data_as(ctypes.c_void_p),
                               None if gg is None else gg.ctypes.data_as(ctypes.c_void_p),
                               ng, scale, dtype, heads_per_group)


@pytest.mark.parametrize("kwargs,status", [
    (dict(q=None), sa.SA_ERR_INVALID_ARG),
    (dict(out=None), sa.SA_ERR_INVALID_ARG),
    (dict(N=0), sa.SA_ERR_INVALID_ARG),
    (dict(B=0), sa.SA_ERR_INVALID_ARG),
    (dict(H=0), sa.SA_ERR_INVALID_ARG),
    (dict(window=-1), sa.SA_ERR_INVALID_ARG),
    (dict(dilation=[1, 0]), sa.SA_ERR_INVALID_ARG),
    (dict(g=[64], ng=1), sa.SA_ERR_INVALID_ARG),
    (dict(g=None, ng=3), sa.SA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), sa.SA_ERR_INVALID_ARG),
    (dict(dtype=7), sa.SA_ERR_INVALID_ARG),
    (dict(heads_per_group=-1), sa.SA_ERR_INVALID_ARG),
    (dict(D=96), sa.SA_ERR_UNSUPPORTED),
    (dict(D=128, dtype=sa.SA_TF32), sa.SA_ERR_UNSUPPORTED),
    (dict(N=1000, g=list(range(300)), ng=300), sa.SA_ERR_UNSUPPORTED),
])
def test_host_entry_rejects_bad_arguments(lib, kwargs, status):
    """sa_forward_host checks every argument before touching the device (this
    runs without a GPU); host buffers need no alignment."""
    assert _fwd_host(lib, **kwargs) == status
    assert lib.sa_last_error().decode()


def test_count_pairs_rejects_bad_arguments(lib):
    assert lib.sa_count_pairs(0, 8, None, 1, None, 0, None, None) == sa.SA_ERR_INVALID_ARG
    g = np.array([5], dtype=np.int32)
    assert lib.sa_count_pairs(5, 8, None, 1, g.ctypes.data_as(ctypes.c_void_p), 1, None,
                              None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_count_pairs(5, 8, None, 1, None, 1, None, None) == sa.SA_ERR_INVALID_ARG
    with pytest.raises(sa.SaError) as e:
        sa.count_pairs(10, -2, None, 1)
    assert e.value.status == sa.SA_ERR_INVALID_ARG and "window" in str(e.value)


def test_last_error_is_thread_local(lib):
    import threading
    assert _fwd(lib, N=0) == sa.SA_ERR_INVALID_ARG
    msg_main = lib.sa_last_error().decode()
    seen = {}

    def worker():
        seen["before"] = lib.sa_last_error().decode()
        _fwd(lib, D=96)
        seen["after"] = lib.sa_last_error().decode()

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert seen["before"] == "" and "D = 96" in seen["after"]
    assert lib.sa_last_error().decode() == msg_main


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        sa.load(str(tmp_path / "nope.so"))


def test_split_p_choice(lib):
    """Automatic precision of the P V product: the five workloads keep single
    bf16 P; narrow windows and sharp scales split it; the setting overrides."""
    from sparse_long_context_banded_gb300 import inputs
    for number in (1, 2, 3, 4, 5):
        w = inputs.workload(number)
        assert not sa.uses_split_p(w.N, w.D, w.window, w.dilation, w.H, w.globals_,
                                   scale=w.scale), w.describe()
    assert sa.uses_split_p(4096, 64, 100, None, 1, [0])          # 51 keys at the edge
    assert not sa.uses_split_p(4096, 64, 254, None, 1, [0])      # 128 keys + 1 global
    assert sa.uses_split_p(640, 64, 128, None, 1, [5], scale=0.6)
    assert sa.uses_split_p(640, 64, 128, None, 1, [5], scale=-0.6)
    assert not sa.uses_split_p(640, 64, 512, None, 1, [5], scale=0.15)
    # dilation: a residue class shorter than the window limits the keys
    assert sa.uses_split_p(300, 64, 512, [8], 1, [])
    try:
        sa.set_pv_mode(sa.SA_PV_SINGLE)
        assert sa.get_pv_mode() == sa.SA_PV_SINGLE
        assert not sa.uses_split_p(640, 64, 128, None, 1, [5], scale=0.6)
        sa.set_pv_mode(sa.SA_PV_SPLIT)
        assert sa.uses_split_p(4096, 64, 1024, None, 1, [0])
    finally:
        sa.set_pv_mode(sa.SA_PV_AUTO)
    assert lib.sa_set_pv_mode(7) == sa.SA_ERR_INVALID_ARG
