"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Every mutant below is a plausible slip in the oracle's arithmetic (a dropped
term, a wrong sign, base or index, a transposed operand).  The copy is compiled
to a temporary library on the CPU and the pin suite is run against it through
MLA_ORACLE_LIB; the suite must fail for every mutant.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mla_oracle.c")

MUTANTS = {
    "drop_rope_term": ("double dot = 0.0;\n        for (int64_t c = 0; c < width; ++c) {",
                       "double dot = 0.0;\n        for (int64_t c = 0; c < d_v; ++c) {"),
    "softmax_sign": ("double w = exp(s[j] - m);", "double w = exp(m - s[j]);"),
    "no_logit_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "v_not_dequantized": ("o[c] += w * (g_e4m3[row[c]] * kv_scale);",
                          "o[c] += w * g_e4m3[row[c]];"),
    "v_wrong_columns": ("o[c] += w * (g_e4m3[row[c]] * kv_scale);",
                        "o[c] += w * (g_e4m3[row[c + d_rope]] * kv_scale);"),
    "lse_natural_log": ("*lse2 = (m + log(z)) / log(2.0);", "*lse2 = m + log(z);"),
    "window_exclusive": ("int64_t n = (int64_t)seq_lens[b] - q_len + t + 1;",
                         "int64_t n = (int64_t)seq_lens[b] - q_len + t;"),
    "e4m3_bias": ("v = ldexp(1.0 + (double)mant / 8.0, expo - 7);",
                  "v = ldexp(1.0 + (double)mant / 8.0, expo - 8);"),
    "e4m3_subnormal": ("v = ldexp((double)mant, -9);", "v = ldexp((double)mant, -10);"),
    "heads_transposed": ("local = attend_row(q_lat + (r * num_heads + h) * d_v,",
                         "local = attend_row(q_lat + (h * ((int64_t)batch * q_len) + r) * d_v,"),
    "merge_natural_base": ("double w = exp2(lse2_parts[s] - m);",
                           "double w = exp(lse2_parts[s] - m);"),
    "merge_lse_drop_sum": ("*lse2 = m + log2(wsum);", "*lse2 = m;"),
    "dcp_local_positions": ("while (n < seq_lens[b] && n * cp_world + cp_rank <= last)",
                            "while (n < seq_lens[b] && n <= last)"),
    "dcp_rank_offset_dropped": ("while (n < seq_lens[b] && n * cp_world + cp_rank <= last)",
                                "while (n < seq_lens[b] && n * cp_world <= last)"),
    "dcp_window_exclusive": ("int64_t last = (int64_t)glen[b] - q_len + t;",
                             "int64_t last = (int64_t)glen[b] - q_len + t - 1;"),
    "sparse_invalid_kept": ("if (slot < 0)\n            continue;\n        if ((int64_t)slot >= pool_rows)",
                            "if (slot < 0)\n            slot = 0;\n        if ((int64_t)slot >= pool_rows)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                    str(mutant_c), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, MLA_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
