"""The oracle's pins are strong enough to catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/oracle.c`` (a dropped term,
a wrong sign, a swapped index, a wrong exponent bias, ties rounded away from
zero, a missing tile in the budget ...), builds the copy with gcc on the CPU,
and runs the oracle pin tests against it in a child process.  The same is
done for the acceptance helpers of ``oracle/__init__.py`` (the output spacing
``ulp`` of each format and the two legs of ``check``), whose mutated copy is
put first on the child's import path.  The pins must fail for every mutant.
The real oracle is untouched.
"""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PY = os.path.join(ROOT, "oracle", "__init__.py")

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


# Mistakes in the acceptance helpers every GPU parity test relies on.
PY_MUTANTS = {
    "bf16_precision_7": ('"bf16": (8, -126)', '"bf16": (7, -126)'),
    "f32_emin_off_by_one": ('"f32": (24, -126)', '"f32": (24, -125)'),
    "f16_emin_off_by_one": ('"f16": (11, -14)', '"f16": (11, -15)'),
    "ulp_exponent_off_by_one": ("np.maximum(e - 1, emin)", "np.maximum(e, emin)"),
    "ulp_zero_as_normal": ("np.where(a == 0, emin, np.maximum(e - 1, emin))", "np.maximum(e - 1, emin)"),
    "pages_leg_dropped": ("ratio = np.maximum(err / bound, err / pages)", "ratio = err / bound"),
    "pages_rtol_wrong": ("pages = 1e-2 + 1e-2 * np.abs(R)", "pages = 1e-2 + 1e-3 * np.abs(R)"),
    "pages_atol_wrong": ("pages = 1e-2 + 1e-2 * np.abs(R)", "pages = 2e-2 + 1e-2 * np.abs(R)"),
    "target_rel_wrong": ("bound = 1e-4 * S + 1e-5", "bound = 1e-3 * S + 1e-5"),
    "ulp_for_f32_output": ('if out_dtype != "f32":', "if True:"),
    "nan_accepted": ("np.where(np.isnan(ratio), np.inf, ratio)", "np.where(np.isnan(ratio), 0.0, ratio)"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_pins_catch_python_mutant(name, tmp_path):
    import oracle

    real_lib = oracle.build()
    old, new = PY_MUTANTS[name]
    src = open(PY).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    shutil.copy(SRC, pkg / "oracle.c")
    (pkg / "__init__.py").write_text(src.replace(old, new))
    env = dict(os.environ, ORACLE_PKG_ROOT=str(tmp_path), ORACLE_LIB=real_lib)
    probe = subprocess.run([sys.executable, "-c", "import sys; sys.path.insert(0, sys.argv[1]); import oracle; "
                            "print(oracle.__file__)", str(tmp_path)], capture_output=True, text=True, env=env)
    assert probe.stdout.strip() == str(pkg / "__init__.py")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"


def test_python_mutation_harness_runs_the_copy(tmp_path):
    # The child really imports the copy: an unmutated copy passes the pins,
    # and a copy whose ulp() raises fails them.
    import oracle

    real_lib = oracle.build()
    src = open(PY).read()
    for text, want_ok in ((src, True), (src.replace('p, emin = {', 'raise RuntimeError("planted"); p, emin = {'),
                                        False)):
        d = tmp_path / ("ok" if want_ok else "bad")
        (d / "oracle").mkdir(parents=True)
        shutil.copy(SRC, d / "oracle" / "oracle.c")
        (d / "oracle" / "__init__.py").write_text(text)
        env = dict(os.environ, ORACLE_PKG_ROOT=str(d), ORACLE_LIB=real_lib)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-k", "ulp",
                            os.path.join(ROOT, "tests", "test_oracle.py")],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
        assert (r.returncode == 0) == want_ok, r.stdout[-2000:]
