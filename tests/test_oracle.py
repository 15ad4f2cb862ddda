"""The fp64 oracle against what the pages and mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle_pins
from oracle_pins import closed_form_counts
from sparse_long_context_banded_gb300 import inputs


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(oracle, pin):
    pin(oracle)


def test_global_set(oracle):
    assert oracle.global_set([5, 1, 5, 3, 1], 6).tolist() == [1, 3, 5]
    assert oracle.global_set([], 6).tolist() == []
    with pytest.raises(ValueError):
        oracle.global_set([6], 6)
    with pytest.raises(ValueError):
        oracle.global_set([-1], 6)


def test_duplicate_globals_are_a_set(oracle):
    q, k, v = (np.random.default_rng(s).standard_normal((1, 1, 40, 8)) for s in range(3))
    a, _ = oracle.forward_longformer(q, k, v, 6, [1], [3, 3, 17])
    b, _ = oracle.forward_longformer(q, k, v, 6, [1], [17, 3])
    assert np.array_equal(a, b)


def test_row_subset_matches_full(oracle):
    q, k, v = (np.random.default_rng(20 + s).standard_normal((2, 3, 50, 8)) for s in range(3))
    full, lse = oracle.forward_longformer(q, k, v, 8, [1, 2, 3], [4])
    rows = np.array([0, 49, 50 + 7, 2 * 3 * 50 - 1, 3 * 50 + 4])
    sub, sub_lse = oracle.forward_longformer(q, k, v, 8, [1, 2, 3], [4], rows=rows)
    assert np.array_equal(sub, full.reshape(-1, 8)[rows])
    assert np.array_equal(sub_lse, lse.reshape(-1)[rows])


def test_bf16_bits_read_exactly(oracle):
    x = [np.random.default_rng(30 + s).standard_normal((1, 2, 33, 16)).astype(np.float32)
         for s in range(3)]
    bits = [inputs.bf16_bits(a) for a in x]
    as_f32 = [inputs.bf16_bits_to_float32(b) for b in bits]
    a, _ = oracle.forward_longformer(*bits, 9, [1, 2], [0])
    b, _ = oracle.forward_longformer(*as_f32, 9, [1, 2], [0])
    assert np.array_equal(a, b)


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], dtype=np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 ties between 1+2^-7 and 1+2^-6: even (1+2^-6) wins.
    got = inputs.bf16_bits_to_float32(inputs.bf16_bits(vals))
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == np.float32(1.015625)
    assert got[3] == -2.5
    assert abs(got[4] - 3.0e-3) <= 3.0e-3 * 2 ** -8


@pytest.mark.parametrize("number", [1, 2, 3, 4])
def test_workload_pair_counts(oracle, number):
    """Materialised-mask counts equal the closed form at the workload shapes."""
    w = inputs.workload(number)
    per_head = oracle.count_pairs_longformer(w.N, w.window, w.dilation, w.globals_)
    for h, d in enumerate(w.dilation):
        assert per_head[h] == closed_form_counts(w.N, w.window, d, w.globals_)
    if number == 1:
        assert per_head.tolist() == [461054, 461054]


def test_long_context_count_closed_form():
    w = inputs.workload(5)
    assert closed_form_counts(w.N, w.window, 1, w.globals_) == 150793664


def test_gmat_workload_mask_rows(oracle):
    """Memory-prefix workload: GMAT rows equal Longformer-form rows (sampled)."""
    w = inputs.workload(3)
    q, k, v = (np.random.default_rng(60 + s).standard_normal((1, 1, w.N, 8)) for s in range(3))
    rows = np.array([0, 63, 64, 65, 200, 4000, w.N - 1])
    a, la = oracle.forward_gmat(q, k, v, w.memory, window=w.window, rows=rows)
    b, lb = oracle.forward_longformer(q, k, v, w.window, [1], w.globals_, rows=rows)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
