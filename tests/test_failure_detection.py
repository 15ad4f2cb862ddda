"""Failure detection without a GPU fault.

Every wait in the kernels is bounded: when it runs out, the kernel sets the
device error word and returns, the context stays usable, and sa_sync_status
reports SA_ERR_TIMEOUT.  sa_check_stalled_wait runs one kernel whose wait is
never satisfied (a barrier nothing arrives on) with a short limit, which makes
the wait run out on purpose; nothing faults, traps or hangs.

An allocation failure is simulated by capping the library's device pool
(SA_POOL_MAX_BYTES) in a child process: a call whose scratch does not fit
returns SA_ERR_NO_MEMORY, and calls that fit still run and are right.
"""
import json
import os
import subprocess
import sys

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


_CHILD = r"""
import json, sys
import numpy as np, torch
from sparse_long_context_banded_gb300 import build, inputs, sa
build.build()
res = {}
def status_of(fn):
    try:
        fn()
        return sa.SA_OK
    except sa.SaError as e:
        return e.status
# scratch of 85 MB (split-K partials of 256 scattered global rows of 16 heads)
big = inputs.custom(1, 16, 65536, 128, 256, globals_=range(0, 65536, 256), dtype="bf16")
q, k, v = (torch.zeros(big.B, big.H, big.N, big.D, dtype=torch.bfloat16, device="cuda")
           for _ in range(3))
res["device"] = status_of(lambda: sa.forward(q, k, v, big.window, None, big.globals_))
hq = torch.zeros(1, 8, 65536, 128, dtype=torch.bfloat16)  # 4 x 134 MB device buffers
res["host"] = status_of(lambda: sa.forward_host(hq, hq, hq, 256, heads_per_group=8))
del q, k, v
# a call that fits, after the failures
small = inputs.custom(1, 2, 700, 64, 128, globals_=[0, 350], dtype="bf16")
a = inputs.draw_qkv(small, seed=8)
dev = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in a]
out = sa.forward(*dev, small.window, None, small.globals_)
sa.sync_status()
np.save(sys.argv[1], out.float().cpu().numpy())
res["small"] = sa.SA_OK
print(json.dumps(res))
"""


@pytest.mark.gpu
def test_pool_cap_gives_no_memory_and_context_survives(tmp_path, oracle):
    from sparse_long_context_banded_gb300 import inputs

    from test_parity_gpu import assert_close

    out_file = tmp_path / "small.npy"
    env = dict(os.environ, SA_POOL_MAX_BYTES=str(64 << 20))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CHILD, str(out_file)], env=env, cwd=root,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res == {"device": sa.SA_ERR_NO_MEMORY, "host": sa.SA_ERR_NO_MEMORY,
                   "small": sa.SA_OK}, res
    small = inputs.custom(1, 2, 700, 64, 128, globals_=[0, 350], dtype="bf16")
    q, k, v = inputs.draw_qkv(small, seed=8)
    ref, _ = oracle.forward_longformer(q, k, v, small.window, None, small.globals_)
    assert_close(np.load(out_file).astype(np.float64), ref, "after out-of-memory returns")
