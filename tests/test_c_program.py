"""The library used from C: tests/c/host_call.c includes include/sa.h alone and
links libsa_gb300.so, with no Python or torch in the process.

CPU: the program compiles as C11 against the header and links against the
library (the header is plain C; every symbol it calls is exported).
GPU (marked): the program runs sa_forward_host on host buffers read from a file
of seeded inputs, and its output and log-sum-exp match the fp64 oracle at the
parity tolerance (|gpu - oracle| <= 2e-3 + 1e-2 |oracle|; lse 1e-3 (1 + |oracle|)).
"""
import os
import subprocess

import numpy as np
import pytest

from sparse_long_context_banded_gb300 import build, inputs, sa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "host_call.c")


def compile_program(tmp_path):
    build.build()
    exe = str(tmp_path / "host_call")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", build.INCLUDE, SRC, "-o", exe,
           "-L", build.BUILD, "-lsa_gb300", "-Wl,-rpath," + build.BUILD, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(compile_program(tmp_path))


@pytest.mark.gpu
@pytest.mark.parametrize("case", [
    # B, H, N, D, window, n_global, dtype, heads_per_group
    (1, 3, 2000, 128, 256, 64, "bf16", 1),
    (2, 2, 900, 64, 100, 3, "bf16", 0),
    (1, 2, 600, 64, 64, 1, "fp32", 2),
], ids=lambda c: "B{}H{}N{}D{}-{}".format(*c[:4], c[6]))
def test_c_program_host_call(tmp_path, case, oracle):
    from test_parity_gpu import assert_close, assert_lse_close

    B, H, N, D, window, ng, dtype, hpg = case
    exe = compile_program(tmp_path)
    w = inputs.custom(B, H, N, D, window, globals_=range(ng), dtype=dtype)
    q, k, v = inputs.draw_qkv(w, seed=77)
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(fin, "wb") as f:
        for a in (q, k, v):
            f.write(np.ascontiguousarray(a).tobytes())
    code = sa.SA_BF16 if dtype == "bf16" else sa.SA_FP32
    r = subprocess.run([exe, str(fin), str(fout), str(B), str(H), str(N), str(D), str(window),
                        str(ng), str(code), str(hpg)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    raw = np.fromfile(fout, dtype=np.uint8)
    n = B * H * N * D
    if dtype == "bf16":
        bits = raw[:2 * n].view(np.uint16).astype(np.uint32) << 16
        got = bits.view(np.float32).astype(np.float64)
        rest = raw[2 * n:]
    else:
        got = raw[:4 * n].view(np.float32).astype(np.float64)
        rest = raw[4 * n:]
    got = got.reshape(B, H, N, D)
    got_lse = rest.view(np.float32).astype(np.float64).reshape(B, H, N)
    ref, ref_lse = oracle.forward_longformer(q, k, v, window, None, list(range(ng)), scale=D ** -0.5)
    assert_close(got, ref, f"C program {case}")
    assert_lse_close(got_lse, ref_lse, f"C program {case}")
