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


# Planted mistakes in the Python side of the oracle (the DCP sharding and rank
# merge, and the second-cache join).  A mutated copy of oracle.py is loaded as
# its own module (over the same compiled C library) and put in place of the
# oracle the pins call; at least one pin must then fail.
PY_MUTANTS = {
    "dcp_shard_wrong_residue": ("if p % cp_world == cp_rank]",
                                "if p % cp_world == (cp_rank + 1) % cp_world]"),
    "dcp_merge_wrong_rank_lse": ("o[r], lse[r] = merge(op2[:, r, :], lp2[:, r])",
                                 "o[r], lse[r] = merge(op2[:, r, :], lp2[::-1, r])"),
    "extra_slot_shift_dropped": ("extra >= 0, extra + n_main, torch.full_like",
                                 "extra >= 0, extra, torch.full_like"),
    "extra_invalid_kept": ("torch.where(extra >= 0, extra + n_main, torch.full_like(extra, -1))",
                           "extra + n_main"),
}


def _python_pins(pins):
    """The pins of the DCP and second-cache oracle functions, with their cases."""
    yield lambda: pins.test_dcp_shares_merge_to_the_unsharded_decode(1, 2, [9, 1, 0, 6])
    yield lambda: pins.test_dcp_shares_merge_to_the_unsharded_decode(4, 3, [11, 2, 7, 3])
    yield lambda: pins.test_dcp_single_rank_is_the_plain_decode()
    yield lambda: pins.test_dcp_share_matches_brute_force(4, 3)
    yield lambda: pins.test_dcp_rank_without_visible_keys_gives_zero_and_minus_inf()
    yield lambda: pins.test_sparse_extra_matches_brute_force()
    yield lambda: pins.test_sparse_extra_with_no_valid_second_candidate_is_the_main_decode()
    yield lambda: pins.test_sparse_extra_equals_one_cache_holding_the_same_rows()


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_pins_catch_planted_python_mistake(name, tmp_path, monkeypatch):
    import importlib.util
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import test_oracle_pins as pins
    from oracle import oracle as real
    lib = real.build()
    old, new = PY_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "oracle.py")).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / "oracle_mutant.py"
    path.write_text(src.replace(old, new))
    monkeypatch.setenv("MLA_ORACLE_LIB", lib)
    spec = importlib.util.spec_from_file_location("oracle_mutant", path)
    mutant = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mutant)
    monkeypatch.setattr(pins, "oracle", mutant)
    failed = 0
    for pin in _python_pins(pins):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"python mutant {name} passed every pin"


def test_python_pins_pass_on_the_oracle_itself():
    # control for the harness above: the unmutated oracle passes every pin
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import test_oracle_pins as pins
    for pin in _python_pins(pins):
        pin()
