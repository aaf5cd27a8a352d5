"""Discrete-event model of a software-pipelined loop, and its fit to measurements.

The model of chapter 11 "Pipeline and autotuning", section 1.3 (and the
space-time diagram of section 2.2): each iteration copies a tile in and then
computes on it; a copy takes ``issue`` cycles of the copy port and its data
arrives ``latency`` cycles after it was issued; a compute takes ``compute``
cycles; there are ``stages`` buffers.  Greedy list schedule:

* copy i is issued as soon as the port is free and its buffer is free, i.e.
  when compute i - stages has finished (buffer reuse, section 5.2);
* compute i starts when its data has arrived and compute i - 1 has finished.

Reported per run: makespan, the mean gap between consecutive copy issues and
between consecutive compute starts, compute utilisation over the span from
the first compute start to the end, and the speedup over one stage.  The
section also gives the minimum sufficient depth 1 + ceil(latency / compute)
and the steady-state cost per iteration max(compute, issue,
(latency + compute) / depth) of section 2.2.

``fit`` inverts the model: given measured time per iteration against the
number of stages (the latency-vs-num_stages experiment of the
"01 · 改 num_stages" README), it finds the (latency, compute) pair whose
steady-state curve matches best, which gives an effective latency/compute
ratio for the real kernel and the depth the model says is enough.
"""

from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass
class Schedule:
    stages: int
    makespan: float
    issue_iv: float
    compute_iv: float
    compute_util: float
    copy_issue: list
    compute_start: list


def simulate(iterations: int, issue: float, latency: float, compute: float, stages: int) -> Schedule:
    """Greedy list schedule of `iterations` copy -> compute pairs over `stages` buffers."""
    if iterations < 1 or stages < 1:
        raise ValueError("iterations and stages must be >= 1")
    t_issue, c_start, c_end = [], [], []
    port_free = 0.0
    for i in range(iterations):
        buffer_free = c_end[i - stages] if i >= stages else 0.0
        t = max(port_free, buffer_free)
        t_issue.append(t)
        port_free = t + issue
        ready = t + latency
        s = max(ready, c_end[i - 1] if i else 0.0)
        c_start.append(s)
        c_end.append(s + compute)
    makespan = c_end[-1]
    gaps = lambda xs: (xs[-1] - xs[0]) / (len(xs) - 1) if len(xs) > 1 else 0.0  # noqa: E731
    util = iterations * compute / (makespan - c_start[0]) if makespan > c_start[0] else 1.0
    return Schedule(stages, makespan, gaps(t_issue), gaps(c_start), util, t_issue, c_start)


def min_depth(latency: float, compute: float) -> int:
    """Smallest depth that reaches the compute-bound steady state: 1 + ceil(latency / compute)."""
    return 1 + math.ceil(latency / compute)


def steady_cost(issue: float, latency: float, compute: float, depth: int) -> float:
    """Steady-state cycles per iteration: max(compute, issue, (latency + compute) / depth)."""
    return max(compute, issue, (latency + compute) / depth)


def table(iterations: int = 8, issue: float = 1, latency: float = 30, compute: float = 20, max_stages: int = 4):
    """Rows (stages, makespan, speedup, issue_iv, compute_iv, util) like the pages' summary."""
    base = simulate(iterations, issue, latency, compute, 1).makespan
    rows = []
    for s in range(1, max_stages + 1):
        r = simulate(iterations, issue, latency, compute, s)
        rows.append((s, r.makespan, base / r.makespan, r.issue_iv, r.compute_iv, r.compute_util))
    return rows


def fit(per_stage_time: dict, issue: float = 0.0):
    """Fit (latency, compute) of the steady-state model to measured time per
    iteration for each number of stages; times are in any consistent unit.

    Returns dict(latency, compute, ratio, min_depth, rms, predicted).  The fit
    is a grid search on latency/compute ratios with compute solved in closed
    form (least squares on a linear model for a fixed ratio)."""
    items = sorted((int(s), float(t)) for s, t in per_stage_time.items())
    if not items:
        raise ValueError("no measurements")
    best = None
    for k in range(0, 4001):
        ratio = k / 100.0  # latency = ratio * compute
        # time(S) = compute * max(1, (ratio + 1) / S)  (issue negligible)
        basis = [max(1.0, (ratio + 1.0) / s) for s, _ in items]
        num = sum(b * t for b, (_, t) in zip(basis, items))
        den = sum(b * b for b in basis)
        c = num / den
        pred = [max(c * b, issue) for b in basis]
        rms = math.sqrt(sum((p - t) ** 2 for p, (_, t) in zip(pred, items)) / len(items))
        if best is None or rms < best[0] - 1e-12:
            best = (rms, ratio, c, pred)
    rms, ratio, c, pred = best
    return {"latency": ratio * c, "compute": c, "ratio": ratio, "min_depth": min_depth(ratio * c, c),
            "rms": rms, "predicted": {s: p for (s, _), p in zip(items, pred)}}


if __name__ == "__main__":
    print("stages makespan speedup issue_iv compute_iv util")
    for s, mk, sp, ii, ci, u in table():
        print(f"{s:6d} {mk:8.0f} x{sp:5.2f} {ii:8.1f} {ci:10.1f} {100 * u:4.0f}%")
