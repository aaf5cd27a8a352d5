"""The oracle's pins are strong enough to catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/oracle.c`` (a dropped term,
a wrong sign, a swapped index, a wrong exponent bias, ties rounded away from
zero, a missing tile in the budget ...), builds the copy with gcc on the CPU,
and runs the oracle pin tests against it in a child process.  The pins must
fail for every mutant.  The real oracle is untouched.
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "sum_sign": ("acc += p;", "acc -= p;"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 0; k + 1 < K; ++k) {"),
    "swapped_operand_rows": ("dot(Ad + i * K, Bd + j * K, K, &r, &s);",
                             "dot(Ad + (j % M) * K, Bd + (i % N) * K, K, &r, &s);"),
    "scale_without_abs": ("mag += fabs(p);", "mag += p;"),
    "f16_exponent_bias": ("e - 25);", "e - 24);"),
    "f16_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "bf16_exponent_bias": ("e - 134);", "e - 133);"),
    "bf16_subnormal_scale": ("v = ldexp((double)m, -133);", "v = ldexp((double)m, -132);"),
    "ties_away_from_zero": ("double r = nearbyint(q);", "double r = round(q);"),
    "subnormal_ulp": ("eunit = emin - (p - 1);", "eunit = emin - p;"),
    "overflow_at_max_finite": ("if (fabs(v) > maxf)", "if (fabs(v) >= maxf)"),
    "budget_counts_a_twice": ("return num_stages * (a_tile + b_tile);",
                              "return num_stages * (a_tile + a_tile);"),
    "budget_one_stage_short": ("return num_stages * (a_tile + b_tile);",
                               "return (num_stages - 1) * (a_tile + b_tile) + a_tile;"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c = tmp_path / "oracle_mutant.c"
    so = tmp_path / "liboracle_mutant.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
                    str(c), "-o", str(so), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
