"""The pipeline timeline model against the numbers the pages print.

tests/golden/pipeline_model.txt holds the summary table of chapter 11
"Pipeline and autotuning", section 1.3 (8 iterations, issue 1, latency 30,
compute 20), the 16-iteration speedup of section 1.4 and the minimum depth.
"""

import math

import pytest

from software_pipelined_tiled_02_gb300 import pipeline_model as pm
from tests.conftest import golden_lines


def golden():
    g = {"rows": []}
    for t in golden_lines("pipeline_model.txt"):
        if t[0] == "params":
            g["params"] = tuple(int(x) for x in t[1:])
        elif t[0] == "row":
            g["rows"].append((int(t[1]), float(t[2]), float(t[3]), float(t[4]), float(t[5]), float(t[6])))
        else:
            g[t[0]] = float(t[1])
    return g


def test_summary_table_matches_pages():
    g = golden()
    it, issue, lat, comp = g["params"]
    rows = pm.table(it, issue, lat, comp, max_stages=4)
    for (s, mk, sp, ii, ci, u), (gs, gmk, gsp, gii, gci, gu) in zip(rows, g["rows"]):
        assert s == gs
        assert mk == gmk
        assert round(sp, 2) == gsp
        assert round(ii, 1) == gii
        assert round(ci, 1) == gci
        assert round(100 * u) == gu


def test_min_depth_and_long_loop_speedup():
    g = golden()
    assert pm.min_depth(30, 20) == g["min_depth"]
    s1 = pm.simulate(16, 1, 30, 20, 1).makespan
    s3 = pm.simulate(16, 1, 30, 20, 3).makespan
    assert round(s1 / s3, 2) == g["speedup16_stages3"]


def test_more_stages_never_slower_and_plateau():
    prev = math.inf
    for s in range(1, 9):
        mk = pm.simulate(32, 1, 30, 20, s).makespan
        assert mk <= prev
        prev = mk
    assert pm.simulate(32, 1, 30, 20, 3).makespan == pm.simulate(32, 1, 30, 20, 8).makespan


def test_steady_cost_formula_agrees_with_simulation():
    # The section 2.2 per-iteration cost is the slope of the simulated schedule.
    for lat, comp, s in ((30, 20, 1), (30, 20, 2), (30, 20, 3), (100, 20, 3), (5, 20, 2)):
        a = pm.simulate(200, 1, lat, comp, s).makespan
        b = pm.simulate(400, 1, lat, comp, s).makespan
        assert (b - a) / 200 == pytest.approx(pm.steady_cost(1, lat, comp, s), rel=0.02)


def test_fit_recovers_known_parameters():
    truth = {s: pm.steady_cost(0, 75.0, 25.0, s) for s in (1, 2, 3, 4, 6, 8)}
    f = pm.fit(truth)
    assert f["ratio"] == pytest.approx(3.0, abs=0.02)
    assert f["compute"] == pytest.approx(25.0, rel=0.01)
    assert f["min_depth"] == 4
