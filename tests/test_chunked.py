"""GMAT chunked self-attention with a global memory ("GMAT: Global Memory
Augmentation for Transformers", subsection "Chunked self-attention").

CPU: the library's exact pair count against the oracle's materialised mask and
argument validation.  GPU (marked): the CUDA path through sa_forward_chunked
against the fp64 oracle's forward_gmat(chunk=C), every row, both the bf16
tensor-core path and the fp32 CUDA-core path; tolerance as in
test_parity_gpu (|gpu - oracle| <= 2e-3 + 1e-2 |oracle|).
"""
import numpy as np
import pytest

from sparse_long_context_banded_gb300 import inputs, sa

COUNT_CASES = [
    # N, memory, chunk
    (12, 0, 12), (48, 0, 12), (50, 0, 12), (53, 5, 12), (40, 40, 7), (40, 39, 7),
    (100, 3, 1), (257, 64, 128), (300, 0, 1000), (1000, 17, 100),
]


@pytest.mark.parametrize("case", COUNT_CASES, ids=lambda c: "N{}M{}C{}".format(*c))
def test_count_pairs_chunked_matches_oracle_mask(oracle, case):
    N, M, C = case
    sa.load()
    mask = oracle.mask_gmat(N, M, chunk=C)
    assert sa.count_pairs_chunked(N, M, C) == int(mask.sum())
    assert oracle.count_pairs_gmat(N, M, chunk=C) == int(mask.sum())


def test_count_pairs_chunked_closed_forms():
    sa.load()
    # no memory, chunks dividing N: k chunks of C^2 pairs
    assert sa.count_pairs_chunked(512 * 4, 0, 512) == 4 * 512 * 512
    # one chunk covering everything, or all memory: dense
    assert sa.count_pairs_chunked(300, 0, 300) == 300 * 300
    assert sa.count_pairs_chunked(300, 300, 5) == 300 * 300
    # (512 x 4, 64): memory rows dense, main rows their chunk plus the memory
    N = 64 + 4 * 512
    assert sa.count_pairs_chunked(N, 64, 512) == 64 * N + 4 * 512 * (64 + 512)


@pytest.mark.parametrize("args", [(100, -1, 10), (100, 101, 10), (100, 5, 0), (0, 0, 1)])
def test_count_pairs_chunked_rejects_bad_arguments(args):
    sa.load()
    with pytest.raises(sa.SaError) as e:
        sa.count_pairs_chunked(*args)
    assert e.value.status == sa.SA_ERR_INVALID_ARG


# (*) Rows with only a handful of keys: single bf16 weights in the P V product
# would not average out over so few terms (one-token chunks with 5 memory
# tokens give 6 keys per row), so the automatic choice splits P into two bf16
# parts there; the case runs in bf16 and in fp32.
GPU_CASES = [
    # B, H, N, D, memory, chunk, dtype
    (1, 2, 1000, 128, 16, 200, "bf16"),
    (1, 2, 777, 64, 0, 128, "bf16"),
    (1, 1, 1000, 64, 37, 100, "bf16"),      # memory and chunk not tile multiples
    (2, 1, 600, 128, 5, 1, "bf16"),         # one-token chunks: self plus memory (*)
    (2, 1, 600, 128, 5, 1, "fp32"),
    (2, 1, 600, 64, 5, 1, "bf16"),
    (2, 1, 600, 128, 5, 16, "bf16"),
    (1, 2, 300, 64, 0, 1000, "bf16"),       # one chunk: plain attention
    (1, 1, 200, 64, 200, 64, "bf16"),       # all memory: dense
    (1, 2, 64 + 4 * 512, 64, 64, 512, "bf16"),  # (512 x 4, 64)
    (1, 2, 1000, 64, 16, 200, "fp32"),
    (1, 1, 513, 128, 3, 77, "fp32"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", GPU_CASES, ids=lambda c: "B{}H{}N{}D{}M{}C{}{}".format(*c))
def test_chunked_matches_oracle(oracle, case):
    import torch

    from test_parity_gpu import assert_close, assert_lse_close, to_device

    B, H, N, D, M, C, dtype = case
    w = inputs.custom(B, H, N, D, 0, dtype=dtype, number=0)
    q, k, v = inputs.draw_qkv(w, seed=4242 + N + M + C)
    ref, ref_lse = oracle.forward_gmat(q, k, v, M, chunk=C)
    tq, tk, tv = (to_device(a, torch) for a in (q, k, v))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    out = sa.forward_chunked(tq, tk, tv, M, C, lse=lse)
    sa.sync_status()
    got = out.float().cpu().numpy().astype(np.float64)
    assert_close(got, ref, f"chunked {case}")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, f"chunked {case}")


def test_split_choice_for_short_chunks():
    """Chunks shorter than 128 keys (with the memory) split P automatically."""
    sa.load()
    assert sa.uses_split_p(600, 128, 0, None, 1, list(range(5)), chunk=1, n_memory=5)
    assert sa.uses_split_p(600, 128, 0, None, 1, list(range(5)), chunk=16, n_memory=5)
    # 984 main positions = 4 * 200 + 184: the shortest chunk row sees 184 + 16 keys
    assert not sa.uses_split_p(1000, 128, 0, None, 1, list(range(16)), chunk=200, n_memory=16)
    # 1001 main positions = 5 * 200 + 1: the last chunk row sees 1 + 16 keys
    assert sa.uses_split_p(1017, 64, 0, None, 1, list(range(16)), chunk=200, n_memory=16)
