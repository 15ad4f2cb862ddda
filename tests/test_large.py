"""A problem past 2^31 elements per tensor (GPU, marked).

B=1, H=136, N=131072, D=128 bf16: 2.28 G elements per tensor (4.6 GB; q, k, v
and the output hold 18.3 GB), so the rows of the last heads sit at element
offsets past 2^31 and every offset computed in 32 bits would wrap.  Window
1024, the 64-token global prefix, dilation 2 on every eighth head.  Inputs are
drawn on the device by torch's seeded generator (standard normal, bf16).  Rows
of the first head and of the last three heads (seams, the ragged tail, global
rows and random rows) are compared with the fp64 oracle, which gets that
head's q, k and v copied to the host, at the parity tolerance
(|gpu - oracle| <= 2e-3 + 1e-2 |oracle|; lse 1e-3 (1 + |oracle|)).
"""
import numpy as np
import pytest

from sparse_long_context_banded_gb300 import sa

from test_parity_gpu import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

B, H, N, D = 1, 136, 131072, 128
WINDOW = 1024
GLOBALS = list(range(64))
DIL = [2 if h % 8 == 7 else 1 for h in range(H)]


def _head_rows(rng):
    rows = {0, 1, 63, 64, 127, 128, 129, 1000, N // 2, N - 129, N - 128, N - 2, N - 1}
    rows |= set(int(x) for x in rng.integers(0, N, size=24))
    return np.array(sorted(rows), dtype=np.int64)


def test_past_two_to_the_31_elements(oracle):
    import torch

    assert B * H * N * D > 2 ** 31
    gen = torch.Generator(device="cuda").manual_seed(2031)
    q, k, v = (torch.randn(B, H, N, D, device="cuda", dtype=torch.bfloat16, generator=gen)
               for _ in range(3))
    lse = torch.empty(B, H, N, device="cuda")
    out = sa.forward(q, k, v, WINDOW, DIL, GLOBALS, lse=lse)
    sa.sync_status()
    rng = np.random.default_rng(31)
    for h in (0, H - 3, H - 2, H - 1):
        qh, kh, vh = (x[:, h:h + 1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
                      for x in (q, k, v))
        rows = _head_rows(rng)
        ref, ref_lse = oracle.forward_longformer(qh, kh, vh, WINDOW, [DIL[h]], GLOBALS,
                                                 scale=D ** -0.5, rows=rows)
        got = out[0, h].float().cpu().numpy().astype(np.float64)[rows]
        got_lse = lse[0, h].cpu().numpy().astype(np.float64)[rows]
        what = f"head {h} of {H} (first element {h * N * D:,})"
        assert_close(got, ref, what)
        assert_lse_close(got_lse, ref_lse, what)
    assert bool(torch.isfinite(out).all())
