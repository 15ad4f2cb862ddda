"""Failure detection without a GPU fault.

Every wait in the kernels is bounded: when it runs out, the kernel sets the
device error word and returns, the context stays usable, and sa_sync_status
reports SA_ERR_TIMEOUT.  sa_check_stalled_wait runs one kernel whose wait is
never satisfied (a barrier nothing arrives on) with a short limit, which makes
the wait run out on purpose; nothing faults, traps or hangs.
"""
import numpy as np
import pytest

from sparse_long_context_banded_gb300 import build, sa


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sa.load()


@pytest.mark.parametrize("limit", [0, 2000001])
def test_rejects_limits_out_of_range(lib, limit):
    assert lib.sa_check_stalled_wait(limit, None) == sa.SA_ERR_INVALID_ARG
    assert b"limit_us" in lib.sa_last_error()


@pytest.mark.gpu
def test_stalled_wait_is_reported_and_context_survives(oracle):
    import torch

    from test_parity_gpu import assert_close, make, run_gpu

    sa.sync_status()  # nothing pending
    sa.check_stalled_wait(20000)
    with pytest.raises(sa.SaError) as e:
        sa.sync_status()
    assert e.value.status == sa.SA_ERR_TIMEOUT
    sa.sync_status()  # the word was cleared
    # the context is usable: a forward call still runs and is right
    q, k, v = make(1, 2, 500, 64, "bf16", seed=3)
    got, _ = run_gpu(q, k, v, 128, [1, 1], [0])
    ref, _ = oracle.forward_longformer(q, k, v, 128, [1, 1], [0])
    assert_close(got, ref, "after a stalled wait")
    torch.cuda.synchronize()
