"""Pins that tie the fp64 oracle to the pages and to mathematics.

Each ``pin_*`` takes an ``oracle.Oracle`` handle and raises AssertionError when
the oracle disagrees with something fixed outside it:

  * the printed worked example of the Longformer glossary page (mask counts),
  * an independent closed-form pair count (interval arithmetic, no mask),
  * a brute-force pure-Python evaluation on tiny inputs (its own predicate),
  * torch's scaled_dot_product_attention (fp64, CPU) where the pattern reduces
    to dense attention, or with a boolean mask built here,
  * invariants the method has: permuting GMAT memory tokens, softmax shift
    invariance (Unlimiformer, section 2.3, footnote on constants added to all
    softmax inputs), values shifted by a constant, the dilated band being an
    ordinary band on each residue class.

``tests/test_oracle.py`` runs them on the real oracle; ``tests/test_oracle_mutants.py``
runs them on deliberately broken copies and requires each copy to fail one.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# independent references

def closed_form_counts(N: int, window: int, dilation: int, globals_) -> int:
    """|mask| for one head by interval arithmetic (no mask is built).

    Row i outside the global set scores the band keys i + t*d with
    |t| <= window//2 clipped to [0, N) -- an interval of t -- plus every global
    key not already in that band.  A global row scores all N keys.
    """
    h, d = window // 2, dilation
    G = np.array(sorted(set(int(g) for g in globals_)), dtype=np.int64)
    i = np.arange(N, dtype=np.int64)
    t_lo = np.maximum(-h, -(i // d))
    t_hi = np.minimum(h, (N - 1 - i) // d)
    band = t_hi - t_lo + 1
    extra = np.zeros(N, dtype=np.int64)
    for g in G:
        diff = i - g
        inside = (np.abs(diff) <= h * d) & (diff % d == 0)
        extra += (~inside).astype(np.int64)
    per_row = band + extra
    if G.size:
        per_row[G] = N
    return int(per_row.sum())


def py_predicate(N, window, dilation, globals_, i, j) -> bool:
    """Membership of (i, j) in the Longformer mask, spelled out directly."""
    gs = set(globals_)
    if i in gs or j in gs:
        return True
    half = window // 2
    return abs(i - j) <= half * dilation and (i - j) % dilation == 0


def py_attention_row(q, k, v, allowed, scale):
    """One output row by plain Python loops (math.exp), fp64."""
    D = len(q)
    scores = {j: scale * sum(q[d] * k[j][d] for d in range(D)) for j in allowed}
    m = max(scores.values())
    w = {j: math.exp(s - m) for j, s in scores.items()}
    z = sum(w.values())
    return [sum(w[j] * v[j][d] for j in allowed) / z for d in range(D)]


def sdpa(q, k, v, mask=None, scale=None):
    """torch.nn.functional.scaled_dot_product_attention in fp64 on the CPU."""
    t = [torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (q, k, v)]
    m = None if mask is None else torch.from_numpy(np.asarray(mask, dtype=bool))
    return torch.nn.functional.scaled_dot_product_attention(
        *t, attn_mask=m, scale=scale).numpy()


def randn(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------
# pins

def pin_page_printed_counts(o):
    """Glossary worked example: window 512, global token 0 -> 0.5M/1.0M/2.0M
    scores against full attention's 1.0M/4.2M/16.8M at n = 1024/2048/4096."""
    rows = []
    with open(os.path.join(GOLDEN, "longformer_mask_counts.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                n, full, lf = line.split()
                rows.append((int(n), full, lf))
    assert len(rows) == 3
    for n, full, lf in rows:
        sparse = int(o.count_pairs_longformer(n, 512, [1], [0])[0])
        dense = int(o.count_pairs_longformer(n, 2 * n, [1], [0])[0])
        assert f"{sparse / 1e6:.1f}" == lf, (n, sparse, lf)
        assert f"{dense / 1e6:.1f}" == full, (n, dense, full)
        assert dense == n * n


def pin_closed_form_counts(o):
    cases = [
        (1024, 512, 1, [0]), (2048, 512, 1, [0]), (4096, 512, 1, [0]),
        (100, 0, 1, []), (100, 1, 1, [99]), (97, 10, 3, [5, 5, 40, 96]),
        (64, 7, 2, [0, 1, 63]), (130, 300, 1, [3]), (130, 300, 4, [3, 129]),
        (200, 16, 5, list(range(0, 200, 37))), (33, 4, 40, [16]),
    ]
    for N, w, d, G in cases:
        got = int(o.count_pairs_longformer(N, w, [d], G)[0])
        assert got == closed_form_counts(N, w, d, G), (N, w, d, G, got)


def pin_brute_force_masks(o):
    rng = np.random.default_rng(7)
    for trial in range(12):
        N = int(rng.integers(1, 65))
        w = int(rng.integers(0, 2 * N + 3))
        d = int(rng.integers(1, 5))
        G = sorted(set(int(x) for x in rng.integers(0, N, size=int(rng.integers(0, 4)))))
        m = o.mask_longformer(N, w, d, G)
        ref = np.array([[py_predicate(N, w, d, G, i, j) for j in range(N)] for i in range(N)])
        assert (m == ref).all(), (N, w, d, G)


def pin_brute_force_attention(o):
    rng = np.random.default_rng(11)
    for trial in range(4):
        N = int(rng.integers(8, 49))
        D = int(rng.choice([4, 8]))
        w = int(rng.integers(0, N))
        d = int(rng.integers(1, 4))
        G = sorted(set(int(x) for x in rng.integers(0, N, size=2)))
        q, k, v = (randn((1, 1, N, D), 100 + 3 * trial + s) for s in range(3))
        scale = 0.7
        out, lse = o.forward_longformer(q, k, v, w, [d], G, scale=scale)
        for i in range(N):
            allowed = [j for j in range(N) if py_predicate(N, w, d, G, i, j)]
            ref = py_attention_row(q[0, 0, i], k[0, 0], v[0, 0], allowed, scale)
            assert np.allclose(out[0, 0, i], ref, rtol=1e-12, atol=1e-12), (trial, i)
            s = [scale * float(np.dot(q[0, 0, i], k[0, 0, j])) for j in allowed]
            mx = max(s)
            ref_lse = mx + math.log(sum(math.exp(x - mx) for x in s))
            assert abs(lse[0, 0, i] - ref_lse) < 1e-12
        mask = np.array([[py_predicate(N, w, d, G, i, j) for j in range(N)] for i in range(N)])
        ref = sdpa(q, k, v, mask, scale)
        assert np.allclose(out, ref, rtol=1e-11, atol=1e-12)


def pin_dense_limit(o):
    """w >= 2N with d = 1 scores every pair; so does 'every position global'."""
    for N, D, G in ((37, 16, []), (128, 32, [0]), (200, 8, [5, 199])):
        q, k, v = (randn((2, 2, N, D), 500 + N + s) for s in range(3))
        ref = sdpa(q, k, v, None, 1 / math.sqrt(D))
        for w in (2 * N, 2 * N + 1, 10 * N):
            out, _ = o.forward_longformer(q, k, v, w, [1, 1], G)
            assert np.allclose(out, ref, rtol=1e-11, atol=1e-12), (N, w)
        out, _ = o.forward_longformer(q, k, v, 0, [3, 1], list(range(N)))
        assert np.allclose(out, ref, rtol=1e-11, atol=1e-12)


def pin_global_rows_dense(o):
    N, D = 90, 16
    G = [0, 7, 89]
    q, k, v = (randn((1, 2, N, D), 40 + s) for s in range(3))
    out, _ = o.forward_longformer(q, k, v, 6, [1, 2], G)
    ref = sdpa(q, k, v, None, 1 / math.sqrt(D))
    for g in G:
        assert np.allclose(out[:, :, g], ref[:, :, g], rtol=1e-11, atol=1e-12)
    # a non-global row sees only its band and the globals
    mask = np.zeros((N, N), dtype=bool)
    for h, d in enumerate([1, 2]):
        for i in range(N):
            mask[i] = [py_predicate(N, 6, d, G, i, j) for j in range(N)]
        ref_h = sdpa(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], mask, 1 / math.sqrt(D))
        assert np.allclose(out[:, h:h + 1], ref_h, rtol=1e-11, atol=1e-12)


def pin_global_projections(o):
    """Separate global projections (Longformer glossary, "How the Longformer
    attention works"): with qg, kg, vg = q, k, v the call is the plain pattern;
    the non-global rows never read the global projections; each global row is
    dense softmax attention of its qg row over kg, vg (a library routine)."""
    N, D = 70, 16
    G = [0, 33, 69]
    q, k, v, qg, kg, vg = (randn((1, 2, N, D), 60 + s) for s in range(6))
    plain, plain_lse = o.forward_longformer(q, k, v, 10, [1, 3], G)
    same, same_lse = o.forward_longformer(q, k, v, 10, [1, 3], G, global_proj=(q, k, v))
    assert np.array_equal(plain, same) and np.array_equal(plain_lse, same_lse)
    out, _ = o.forward_longformer(q, k, v, 10, [1, 3], G, global_proj=(qg, kg, vg))
    rest = [i for i in range(N) if i not in G]
    assert np.array_equal(out[:, :, rest], plain[:, :, rest])
    ref = sdpa(qg, kg, vg, None, 1 / math.sqrt(D))
    for g in G:
        assert np.allclose(out[:, :, g], ref[:, :, g], rtol=1e-11, atol=1e-12)
        # and not the plain projections' answer
        assert not np.allclose(out[:, :, g], plain[:, :, g], rtol=1e-3, atol=1e-3)


def pin_gmat_band_is_longformer_with_memory_globals(o):
    """GMAT (memory prefix dense both ways + band on main tokens) has the same
    mask as the Longformer form over all M+L positions with globals {0..M-1}."""
    for M, L, w in ((4, 40, 8), (8, 100, 16), (3, 7, 100), (64, 500, 256)):
        N = M + L
        a = o.mask_gmat(N, M, w)
        b = o.mask_longformer(N, w, 1, list(range(M)))
        assert (a == b).all(), (M, L, w)
        ref = np.zeros((N, N), dtype=bool)
        idx = np.arange(N)
        ref[:M, :] = True
        ref[:, :M] = True
        main = np.abs(idx[:, None] - idx[None, :]) <= w // 2
        ref[M:, M:] |= main[M:, M:]
        assert (a == ref).all()
    assert o.count_pairs_gmat(64 + 500, 64, 256) == closed_form_counts(564, 256, 1, range(64))


def pin_memory_permutation(o):
    """Permuting the memory tokens permutes their outputs and leaves the main
    sequence's outputs unchanged (memory attends and is attended densely)."""
    M, L, D = 6, 50, 8
    N = M + L
    q, k, v = (randn((1, 2, N, D), 70 + s) for s in range(3))
    perm = np.array([3, 0, 5, 1, 4, 2])
    full = np.concatenate([perm, np.arange(M, N)])
    for chunk in (None, 10):
        out, _ = o.forward_gmat(q, k, v, M, window=12, chunk=chunk)
        outp, _ = o.forward_gmat(q[:, :, full], k[:, :, full], v[:, :, full], M,
                                 window=12, chunk=chunk)
        assert np.allclose(outp[:, :, :M], out[:, :, perm], rtol=1e-12, atol=1e-12)
        assert np.allclose(outp[:, :, M:], out[:, :, M:], rtol=1e-12, atol=1e-12)


def pin_shift_invariance(o):
    N, D = 60, 8
    q, k, v = (randn((1, 1, N, D), 90 + s) for s in range(3))
    u = randn((D,), 95)
    G = [2, 30]
    out, _ = o.forward_longformer(q, k, v, 10, [2], G)
    out_k, _ = o.forward_longformer(q, k + u, v, 10, [2], G)
    assert np.allclose(out_k, out, rtol=1e-10, atol=1e-11)
    out_v, _ = o.forward_longformer(q, k, v + 0.375, 10, [2], G)
    assert np.allclose(out_v, out + 0.375, rtol=1e-12, atol=1e-12)


def pin_dilation_is_band_per_residue(o):
    """With no globals, dilation d is an ordinary (d = 1) band on each residue
    class r, r+d, r+2d, ... -- checked against SDPA with a band mask."""
    N, D, w = 61, 8, 10
    q, k, v = (randn((1, 1, N, D), 120 + s) for s in range(3))
    for d in (2, 3, 7):
        out, _ = o.forward_longformer(q, k, v, w, [d], [])
        for r in range(d):
            sub = np.arange(r, N, d)
            n = sub.size
            t = np.arange(n)
            band = np.abs(t[:, None] - t[None, :]) <= w // 2
            ref = sdpa(q[:, :, sub], k[:, :, sub], v[:, :, sub], band, 1 / math.sqrt(D))
            assert np.allclose(out[:, :, sub], ref, rtol=1e-11, atol=1e-12), (d, r)


def pin_chunked(o):
    """C x k chunks with no memory: block diagonal, each chunk is vanilla
    attention; k = 1 is vanilla attention over the whole sequence."""
    C, nchunks, D = 12, 4, 8
    N = C * nchunks
    q, k, v = (randn((1, 1, N, D), 140 + s) for s in range(3))
    out, _ = o.forward_gmat(q, k, v, 0, chunk=C)
    for c in range(nchunks):
        sl = slice(c * C, (c + 1) * C)
        ref = sdpa(q[:, :, sl], k[:, :, sl], v[:, :, sl], None, 1 / math.sqrt(D))
        assert np.allclose(out[:, :, sl], ref, rtol=1e-11, atol=1e-12)
    out1, _ = o.forward_gmat(q, k, v, 0, chunk=N)
    assert np.allclose(out1, sdpa(q, k, v, None, 1 / math.sqrt(D)), rtol=1e-11, atol=1e-12)
    # with memory: compare with SDPA under the mask written out here
    M = 5
    qm, km, vm = (randn((1, 1, M + N, D), 150 + s) for s in range(3))
    mask = np.zeros((M + N, M + N), dtype=bool)
    mask[:M, :] = True
    mask[:, :M] = True
    for c in range(nchunks):
        a, b = M + c * C, M + (c + 1) * C
        mask[a:b, a:b] = True
    outm, _ = o.forward_gmat(qm, km, vm, M, chunk=C)
    assert np.allclose(outm, sdpa(qm, km, vm, mask, 1 / math.sqrt(D)), rtol=1e-11, atol=1e-12)
    assert o.count_pairs_gmat(M + N, M, chunk=C) == int(mask.sum())


def pin_bf16_decode(o):
    """bf16 bit patterns decode to the values they encode: 0x3FC0 is 1.5, so
    attention over identical rows of 1.5 returns 1.5 exactly."""
    bits = np.full((1, 1, 2, 2), 0x3FC0, dtype=np.uint16)
    out, _ = o.forward_longformer(bits, bits, bits, 0, [1], [])
    assert np.array_equal(out, np.full((1, 1, 2, 2), 1.5))


def _lists_to_mask(idx, Nk):
    """Additive float mask from key lists: log(count) where listed, -inf elsewhere
    (entries outside [0, Nk) ignored)."""
    B, H, Nq, K = idx.shape
    cnt = np.zeros((B, H, Nq, Nk))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                for j in idx[b, h, i]:
                    if 0 <= j < Nk:
                        cnt[b, h, i, j] += 1
    with np.errstate(divide="ignore"):
        return np.log(cnt), cnt


def pin_gather_dense(o):
    """Per-query lists holding every key (each in its own shuffled order) give
    dense softmax attention of q over k, v (SDPA, fp64), and the log-sum-exp of
    the scaled score matrix (matmul + logsumexp)."""
    rng = np.random.default_rng(21)
    B, H, Nq, Nk, D = 1, 2, 9, 23, 16
    q, k, v = randn((B, H, Nq, D), 1), randn((B, H, Nk, D), 2), randn((B, H, Nk, D), 3)
    idx = np.stack([np.stack([np.stack([rng.permutation(Nk) for _ in range(Nq)])
                              for _ in range(H)]) for _ in range(B)]).astype(np.int32)
    out, lse = o.forward_gather(q, k, v, idx, scale=0.3)
    assert np.allclose(out, sdpa(q, k, v, None, 0.3), rtol=1e-11, atol=1e-12)
    sc = 0.3 * np.einsum("bhid,bhjd->bhij", q, k)
    ref_lse = sc.max(-1) + np.log(np.exp(sc - sc.max(-1, keepdims=True)).sum(-1))
    assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def pin_gather_lists_with_padding_and_repeats(o):
    """Ragged lists (padding -1 and indices >= Nk skipped) with repeated entries:
    the same as SDPA with an additive mask of log(times listed) -- a key listed
    twice weighs twice -- and rows with no valid entry give 0 and -inf."""
    rng = np.random.default_rng(22)
    B, H, Nq, Nk, D, K = 2, 2, 11, 30, 8, 12
    q, k, v = randn((B, H, Nq, D), 4), randn((B, H, Nk, D), 5), randn((B, H, Nk, D), 6)
    idx = rng.integers(0, Nk, size=(B, H, Nq, K)).astype(np.int32)
    idx[rng.random(idx.shape) < 0.2] = -1
    idx[rng.random(idx.shape) < 0.05] = Nk + 3
    idx[0, 1, 4] = -1                         # an empty row
    idx[1, 0, 2, :3] = [7, 7, 7]             # one key three times
    mask, cnt = _lists_to_mask(idx, Nk)
    assert cnt.max() >= 3
    out, lse = o.forward_gather(q, k, v, idx, scale=0.5)
    t = [torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(
        *t, attn_mask=torch.from_numpy(mask), scale=0.5).numpy()
    has = cnt.sum(-1) > 0
    assert np.allclose(out[has], ref[has], rtol=1e-11, atol=1e-12)
    assert (out[~has] == 0).all() and np.isneginf(lse[~has]).all() and (~has).sum() == 1
    sc = (0.5 * np.einsum("bhid,bhjd->bhij", q, k) + mask)[has]
    m = sc.max(-1)
    ref_lse = m + np.log(np.exp(sc - m[..., None]).sum(-1))
    assert np.allclose(lse[has], ref_lse, rtol=1e-12, atol=1e-12)


def pin_gather_band_is_longformer(o):
    """The Longformer pattern written as per-row key lists gives the mask-based
    Longformer forward (two code paths of the oracle that share no mask code),
    per head with different dilations."""
    N, D, w, dil, G = 57, 8, 12, [1, 3], [0, 20]
    q, k, v = (randn((1, 2, N, D), 70 + s) for s in range(3))
    masks = [o.mask_longformer(N, w, d, G) for d in dil]
    K = max(int(m.sum(1).max()) for m in masks)
    idx = np.full((1, 2, N, K), -1, dtype=np.int32)
    for h, m in enumerate(masks):
        for i in range(N):
            js = np.flatnonzero(m[i])[::-1]  # any order
            idx[0, h, i, :js.size] = js
    got, got_lse = o.forward_gather(q, k, v, idx, scale=0.25)
    ref, ref_lse = o.forward_longformer(q, k, v, w, dil, G, scale=0.25)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(got_lse, ref_lse, rtol=1e-12, atol=1e-13)


ALL_PINS = [
    pin_page_printed_counts, pin_closed_form_counts, pin_brute_force_masks,
    pin_brute_force_attention, pin_dense_limit, pin_global_rows_dense,
    pin_gmat_band_is_longformer_with_memory_globals, pin_memory_permutation,
    pin_shift_invariance, pin_dilation_is_band_per_residue, pin_chunked,
    pin_bf16_decode, pin_global_projections, pin_gather_dense,
    pin_gather_lists_with_padding_and_repeats, pin_gather_band_is_longformer,
]
