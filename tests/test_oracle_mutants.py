"""Each plausible mistake planted in a copy of the oracle must fail a pin.

The mutants are textual edits of ``oracle/oracle.c`` compiled into a temporary
library; the committed oracle is never modified.
"""
import os

import pytest

import oracle as oracle_pkg
import oracle_pins

MUTANTS = {
    "band_strict": ("in_band = (dist <= half * (int64_t)dilation)",
                    "in_band = (dist < half * (int64_t)dilation)"),
    "band_full_width": ("int64_t half = window / 2; /* floor for w >= 0 */",
                        "int64_t half = window; /* floor for w >= 0 */"),
    "dilation_divisibility_dropped": ("&& (diff % dilation == 0)", "&& 1"),
    "dilation_span_not_scaled": ("dist <= half * (int64_t)dilation", "dist <= half"),
    "global_column_dropped": ("for (g = 0; g < n_globals; ++g) row[globals[g]] = 1;", ""),
    "global_row_not_dense": ("if (globals[g] == i) row_is_global = 1;", ""),
    "scale_dropped": ("s[j] = job->scale * acc;", "s[j] = acc;"),
    "key_index_transposed": (
        "acc += qi[d] * load_elem(ks, job->dtype, base + (int64_t)j * D + d);",
        "acc += qi[d] * load_elem(ks, job->dtype, base + (int64_t)i * D + d);"),
    "value_from_keys": (
        "o[d] += e * load_elem(vs, job->dtype, base + (int64_t)j * D + d);",
        "o[d] += e * load_elem(ks, job->dtype, base + (int64_t)j * D + d);"),
    "global_rows_plain_keys": ("      ks = job->kg;", "      ks = job->k;"),
    "no_normalise": ("for (d = 0; d < D; ++d) o[d] /= z;", ""),
    "lse_without_max": ("job->lse[r] = m + log(z);", "job->lse[r] = log(z);"),
    "gmat_memory_column_dropped": ("if (row_mem || col_mem)", "if (row_mem)"),
    "gmat_chunk_memory_column_dropped": ("if (i < M || j < M)", "if (i < M)"),
    "gmat_chunk_boundary_off": ("row[j] = (uint8_t)(((i - M) / C) == ((j - M) / C));",
                                "row[j] = (uint8_t)(((i - M + 1) / C) == ((j - M) / C));"),
    "bf16_decode_shift": ("uint32_t wide = ((uint32_t)bits) << 16;",
                          "uint32_t wide = ((uint32_t)bits) << 15;"),
    "gather_scale_dropped": ("s[t] = job->scale * dot;", "s[t] = dot;"),
    "gather_value_from_keys": (
        "o[d] += w * load_elem(job->v, job->dtype, kbase + (int64_t)list[t] * D + d);",
        "o[d] += w * load_elem(job->k, job->dtype, kbase + (int64_t)list[t] * D + d);"),
    "gather_first_query_of_head": ("int64_t qbase = flat * D;",
                                   "int64_t qbase = bh * (int64_t)job->Nq * D;"),
    "gather_head_offset_dropped": ("int64_t kbase = bh * (int64_t)job->Nk * D;",
                                   "int64_t kbase = 0;"),
    "gather_lse_without_max": ("job->lse[r] = top + log(total);",
                               "job->lse[r] = log(total);"),
    "gather_repeats_counted_once": (
        "      if (!gather_valid(list[t], job->Nk)) continue;\n      w = exp(s[t] - top);",
        "      if (!gather_valid(list[t], job->Nk)) continue;\n      if (t > 0 && list[t] == list[t - 1]) continue;\n      w = exp(s[t] - top);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle_pkg.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle_pkg.compile_library(str(path), str(tmp_path / "libmutant.so"))
    mutant = oracle_pkg.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, MemoryError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"

