"""Planted mistakes in the oracle: each copy of oracle.c below carries one plausible
error (a wrong head mapping, a sign, an index, a dropped factor, a rounding rule, a
constant) and must make the pins that guard that part of the oracle fail.  The copies
are compiled in a scratch folder and the pins run in a child process against them
(PA_ORACLE_SRC); the real oracle is never touched."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text in oracle.c, replacement, occurrences to replace, pins expected to fail)
MUTANTS = [
    ("gqa_interleaved", "int32_t kvh = h / group;", "int32_t kvh = h % a->num_kv_heads;", 2,
     "dense_bruteforce"),
    ("gqa_interleaved_fp8", "            int32_t kvh = h / group;\n",
     "            int32_t kvh = h % num_kv_heads;\n", 1, "fp8_cache_decode"),
    ("lse_merge_sign", "exp(mp[p] - M)", "exp(M - mp[p])", 2, "v2_equals_v1"),
    ("row_off_by_one", "int32_t row = t % a->block_size;",
     "int32_t row = (t + 1) % a->block_size;", 1, "dense_bruteforce"),
    ("dropped_scale", "logit[t - t0] = a->scale * acc;", "logit[t - t0] = acc;", 1,
     "dense_bruteforce"),
    ("unnormalised_pv", "o[d] = acc / l;", "o[d] = acc;", 1, "dense_bruteforce"),
    ("causal_limit_off_by_one", "int32_t limit = L - q_len + j + 1;",
     "int32_t limit = L - q_len + j;", 1, "multi_query"),
    ("fp8_dropped_v_scale", "(or_e4m3_to_f64(v_cache[row + d]) * (double)v_scale)",
     "or_e4m3_to_f64(v_cache[row + d])", 1, "fp8_cache_decode"),
    ("fp8_table_row_bound", "    if (logical >= max_blocks_per_seq) { *bad = 1; return -1; }\n", "", 1,
     "fp8_decode_context_past"),
    ("ties_away_16bit", "double r = nearbyint(n);              /* default rounding mode: ties to even */",
     "double r = round(n);", 1, "rounding and not e4m3"),
    ("ties_away_e4m3", "    double r = nearbyint(n);\n    if (r >= 16.0)",
     "    double r = round(n);\n    if (r >= 16.0)", 1, "e4m3_rounding"),
    ("reshape_offset", "int64_t offset = slot % block_size;",
     "int64_t offset = (slot + 1) % block_size;", 1, "reshape_and_cache_matches"),
    ("splitmix64_constant", "*state += 0x9E3779B97F4A7C15ULL;", "*state += 0x9E3779B97F4A7C13ULL;",
     1, "splitmix64"),
]


@pytest.mark.parametrize("name,old,new,count,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_its_pins(tmp_path, name, old, new, count, pins):
    text = open(SRC).read()
    assert text.count(old) >= count, f"{name}: mutation site not found"
    mutant = tmp_path / "oracle.c"
    mutant.write_text(text.replace(old, new, count))
    env = dict(os.environ, PA_ORACLE_SRC=str(mutant))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-k", pins],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    # exit code 1: tests ran and some failed (2 would be a collection or build error)
    assert r.returncode == 1, f"{name}: pins '{pins}' did not fail\n{r.stdout[-2000:]}{r.stderr[-2000:]}"
    assert os.path.exists(tmp_path / "liboracle.so")


def test_unaltered_copy_passes_the_same_pins(tmp_path):
    """Control: the mechanism itself (a copy compiled elsewhere, loaded by the child
    process) leaves every pin above passing, so the failures are the mistakes'."""
    mutant = tmp_path / "oracle.c"
    mutant.write_text(open(SRC).read())
    env = dict(os.environ, PA_ORACLE_SRC=str(mutant))
    sel = " or ".join(sorted({m[4] for m in MUTANTS if " " not in m[4]} | {"rounding"}))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-k", sel],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "passed" in r.stdout and os.path.exists(tmp_path / "liboracle.so")
