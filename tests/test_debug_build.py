"""The SA_DEBUG build (include/sa_debug.h): device-side range checks of every
work description.

GPU (marked):
  - the check by itself (sa_debug_check_band_items) passes well-formed band
    items and counts each kind of out-of-range field; only the check kernel
    runs on those lists, never an attention kernel;
  - the debug library computes exactly what the release library computes
    (the checks change no arithmetic): bitwise-equal outputs and log-sum-exp
    on band + dilated + global problems, both tensor-core families (band
    tiles and global-row tiles in one launch), and the error word stays clear.
"""
import ctypes

import numpy as np
import pytest

from sparse_long_context_banded_gb300 import build, inputs, sa

pytestmark = pytest.mark.gpu


def _slots(N, dilations):
    """Residue classes as the scheduler lays them out: per dilation d, r = 0..d-1."""
    rows = []
    for d in dilations:
        for r in range(min(d, N)):
            rows.append([d, r, (N - r + d - 1) // d, 0])
    return np.array(rows, dtype=np.int32)


def _check(items, slots, slot_base=0, BH=2):
    lib = sa.load_debug()
    items = np.ascontiguousarray(items, dtype=np.int32)
    slots = np.ascontiguousarray(slots, dtype=np.int32)
    bad = ctypes.c_int(-1)
    st = lib.sa_debug_check_band_items(items.ctypes.data_as(ctypes.c_void_p), len(items),
                                       slots.ctypes.data_as(ctypes.c_void_p), len(slots),
                                       slot_base, BH, ctypes.byref(bad))
    assert st == sa.SA_OK, lib.sa_last_error().decode()
    return bad.value


def test_range_check_flags_each_bad_field():
    build.build(debug=True)
    N = 1000                                  # 8 query tiles of 128 rows (the last ragged)
    slots = _slots(N, [1, 2])                 # class 0: d=1 (len 1000); 1, 2: d=2 (len 500)
    good = [
        [0, 0, 0, 0, 0, 0, 4, 5],             # head 0, class 0, tiles 0-1, keys 0-4 / 0-5
        [1, 0, 6, 0, 2, 3, 7, 7],             # head 1, last query tiles, keys up to tile 7
        [1, 2, 2, 1, 0, 0, 3, -1],            # class 2 (len 500): second query tile empty
    ]
    assert _check(good, slots) == 0
    bad = [
        [2, 0, 0, 0, 0, 0, 4, 5],             # head == B*H
        [-1, 0, 0, 0, 0, 0, 4, 5],            # negative head
        [0, 3, 0, 0, 0, 0, 1, 1],             # class past the last one
        [0, 0, 8, 0, 0, 0, 4, 5],             # query tile past the class end (8*128 >= 1000)
        [0, 1, 0, 0, 0, 0, 4, 4],             # key tile 4 of a 500-long class (4*128 >= 500)
        [0, 0, 0, 0, -1, 0, 4, 5],            # negative first key tile
        [0, 0, 0, 0, 0, 0, 4, 8],             # second query tile's last key tile past the end
    ]
    assert _check(bad, slots) == len(bad)
    for row in bad:
        assert _check([row], slots) == 1, row
    assert _check(good + bad, slots) == len(bad)
    # the launch window: classes slot_base .. slot_base + 15 only
    many = _slots(20000, [17, 1])             # classes 0..16 (d=17), then 17 (d=1)
    item = [[0, 17, 0, 0, 0, 0, 1, 1]]
    assert _check(item, many, slot_base=0) == 1
    assert _check(item, many, slot_base=16) == 0


CASES = [
    # B, H, N, D, window, dilation, globals
    (1, 2, 3000, 64, 256, [1, 3], [0, 5, 2999]),
    (1, 2, 2304, 128, 1024, [1, 1], list(range(64))),
    (2, 1, 1500, 64, 200, [2], list(range(100))),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}D{}".format(*c[:4]))
def test_debug_build_matches_release_bitwise(case):
    import torch
    build.build()
    build.build(debug=True)
    B, H, N, D, window, dil, G = case
    w = inputs.custom(B, H, N, D, window, dilation=dil, globals_=G, dtype="bf16")
    q, k, v = inputs.draw_qkv(w, seed=99)
    dev = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda() for a in (q, k, v)]

    def run():
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        out = sa.forward(*dev, window, dil, G, lse=lse)
        sa.sync_status()
        return out.view(torch.int16).cpu().numpy(), lse.cpu().numpy()

    rel_out, rel_lse = run()
    saved = sa._lib
    sa._lib = sa.load_debug()
    try:
        dbg_out, dbg_lse = run()
    finally:
        sa._lib = saved
    assert np.array_equal(rel_out, dbg_out)
    assert np.array_equal(rel_lse.view(np.int32), dbg_lse.view(np.int32))
