"""The oracle's pins must catch plausible mistakes (runs without a GPU).

Each case plants one mistake in a temporary copy of the oracle's C source --
a dropped term, a wrong start value, a wrong rounding, a transposed index, a
reversed order -- builds it, and runs the pin suite (tests/test_oracle.py) in a
child process against that build.  The suite must fail for every mutant and pass
for the unmodified source built the same way.
"""
import os
import shutil
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "purlin_oracle.c")
HDR = os.path.join(ROOT, "oracle", "purlin_oracle.h")

MUTANTS = {
    "dropped_rank_term": ("for (int r = 1; r < R; ++r)\n        acc = acc +",
                          "for (int r = 2; r < R; ++r)\n        acc = acc +"),
    "fold_starts_from_plus_zero": ("float acc = load_elem(x[0], at, dtype);",
                                   "float acc = 0.0f + load_elem(x[0], at, dtype);"),
    "fold_in_reverse_rank_order": ("acc = acc + load_elem(x[r], at, dtype);",
                                   "acc = acc + load_elem(x[R - r], at, dtype);"),
    "bf16_ties_away_from_zero": ("dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))",
                                 "dropped >= 0x8000u"),
    "bf16_truncates": ("kept += 1u;", "kept += 0u;"),
    "f16_wrong_quantum": ("int q = E + top_bit(M) - 10;", "int q = E + top_bit(M) - 11;"),
    "f16_no_subnormals": ("if (q < -24) q = -24;", "if (q < -14) q = -14;"),
    "f16_widen_wrong_bias": ("mag = (float)(m + 1024) * pow2f(e - 25);",
                             "mag = (float)(m + 1024) * pow2f(e - 24);"),
    "allgather_reversed_ranks": ("uint64_t D = start_of(counts, out_displs, k);\n"
                                 "            memcpy((char*)out[j] + D * elem_bytes, in[k],",
                                 "uint64_t D = start_of(counts, out_displs, R - 1 - k);\n"
                                 "            memcpy((char*)out[j] + D * elem_bytes, in[R - 1 - k],"),
    "alltoall_transposed_counts": ("uint64_t c = send_counts[(size_t)s * R + j];",
                                   "uint64_t c = send_counts[(size_t)j * R + s];"),
    "alltoall_recv_displs_transposed": ("recv_displs[(size_t)j * R + s]",
                                        "recv_displs[(size_t)s * R + j]"),
    "reduce_scatter_ignores_displs": ("uint64_t d = start_of(recv_counts, in_displs, k);\n"
                                      "        for (uint64_t i = 0; i < recv_counts[k]; ++i)\n"
                                      "            store_elem(",
                                      "uint64_t d = start_of(recv_counts, 0, k);\n"
                                      "        for (uint64_t i = 0; i < recv_counts[k]; ++i)\n"
                                      "            store_elem("),
    "tree_drops_odd_carry": ("if (live & 1) v[next++] = v[live - 1];", ";"),
    "tree_is_a_left_fold": ("            int live = R;\n",
                            "            int live = R;\n"
                            "            for (int r = 1; r < R; ++r) v[0] = v[0] + v[r];\n"
                            "            live = 1;\n"),
    "bf16_nan_becomes_infinity": ("return (uint16_t)((u >> 16) | 0x0040u);",
                                  "return (uint16_t)((u >> 16) & 0xff80u);"),
    "f16_overflow_saturates": ("if (enc > 0x7c00u) enc = 0x7c00u;",
                               "if (enc > 0x7bffu) enc = 0x7bffu;"),
    "f16_nan_becomes_infinity": ("if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);",
                                 "if (a > 0x7f800000u) return (uint16_t)(sign | 0x7c00u);"),
    "allreduce_skips_last_output": ("        for (int j = 0; j < R; ++j)\n"
                                    "            store_elem(out[j], i, acc, dtype);",
                                    "        for (int j = 0; j + 1 < R; ++j)\n"
                                    "            store_elem(out[j], i, acc, dtype);"),
    "allgather_ignores_out_displs": ("uint64_t D = start_of(counts, out_displs, k);",
                                     "uint64_t D = start_of(counts, 0, k);"),
    "alltoall_ignores_send_displs": ("send_displs ? send_displs + (size_t)s * R : 0, j);",
                                     "0, j);"),
    "alltoall_ignores_recv_displs": ("uint64_t rd = recv_displs ? recv_displs[(size_t)j * R + s] : packed_recv;",
                                     "uint64_t rd = packed_recv;"),
    "packed_partitions_skip_one": ("for (int m = 0; m < k; ++m) s += counts[m];",
                                   "for (int m = 1; m < k; ++m) s += counts[m];"),
}


def _build(tmp_path, text):
    d = tmp_path / "src"
    d.mkdir()
    (d / "purlin_oracle.c").write_text(text)
    shutil.copy(HDR, d / "purlin_oracle.h")
    lib = d / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib), str(d / "purlin_oracle.c")],
                   check=True, capture_output=True)
    return str(lib)


def _run_pins(lib):
    env = dict(os.environ, PURLIN_ORACLE_LIB=lib)
    return subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle.py", "-x", "-q",
                           "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_unmodified_source_passes(tmp_path):
    r = _run_pins(_build(tmp_path, open(SRC).read()))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    r = _run_pins(_build(tmp_path, text.replace(old, new)))
    assert r.returncode != 0, f"pins did not catch {name}"
