"""Sweep of (block_M, block_N, block_K, num_stages) for one workload.

The autotuning procedure of the TileLang tutorial, chapter 11 "Pipeline and
autotuning", restated for this kernel:

* section 3.7: prune the space before building anything -- drop tiles that do
  not divide the problem (optional here, since the kernel handles ragged
  edges) and configs whose num_stages x (A tile + B tile) bound exceeds the
  per-block shared-memory budget (section 4.5), here the limit queried from
  the device, never a constant;
* section 3.5: run every surviving candidate on the same inputs, warm-up then
  timed repetitions, and check each against the reference program the
  pages use, torch.matmul on fp32 copies of the operands, at rtol = atol =
  1e-2 (the fp64 oracle is test infrastructure, kept out of this tool);
* section 3.8: read the config, not the latency: the winner (lowest mean
  time; ties within 1 % go to the smaller shared footprint, then to fewer
  stages) is written to a per-device cache directory as best_config.json,
  beside latency.json with every candidate's timing, footprint and check.
  A later search of the same workload on the same device reads the cached
  winner instead of timing anything; the switch
  TGEMM_AUTOTUNE_DISABLE_CACHE=1 (or --no-cache) forces a new search;
* the num_stages experiment of the "01-num-stages-ir-diff" README: latency
  and shared memory against num_stages for several tile shapes, where
  latency should plateau while shared memory keeps growing.

The prune is reported twice: with the pages' own budget, 228 KiB for
num_stages x (A tile + B tile) (section 4.5; 214 of 216 configs at 4096^3,
section 3.7), and with this device's queried limit and this kernel's rules
(its real footprint, the tile shapes it implements).

Usage (on a GB300):
    python -m software_pipelined_tiled_02_gb300.sweep --workload gemm_4096_f16_normal --space gb300
    python -m software_pipelined_tiled_02_gb300.sweep --workload gemm_4096_f16_normal --stage-curve
"""

from __future__ import annotations

import argparse
import itertools
import json
import os
import statistics
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import software_pipelined_tiled_02_gb300 as tg  # noqa: E402
from software_pipelined_tiled_02_gb300 import inputs  # noqa: E402

PAGES_SPACE = dict(block_M=(64, 128, 256), block_N=(64, 128, 256), block_K=(16, 32, 64), num_stages=(1, 2, 3, 4))
GB300_SPACE = dict(block_M=(128, 256), block_N=(64, 128, 192, 224, 256, 352, 384, 512), block_K=(32, 64, 128),
                   num_stages=(2, 3, 4, 5, 6, 8), cta_pair=(0, 1))


PAGES_BUDGET = 228 * 1024  # the pages' per-block shared-memory budget (H100)


def pages_prune_count(configs, M, N, K, dtype, budget=PAGES_BUDGET, divisible=True):
    """How many configs the pages' own rule keeps: the tile divides the
    problem and num_stages x (A tile + B tile) fits the budget."""
    kept = 0
    for c in configs:
        if divisible and (M % c["block_M"] or N % c["block_N"] or K % c["block_K"]):
            continue
        if tg.tgemm_smem_bound(dtype, c["block_M"], c["block_N"], c["block_K"], c["num_stages"]) <= budget:
            kept += 1
    return kept


def enumerate_space(space: dict):
    keys = ("block_M", "block_N", "block_K", "num_stages", "cta_pair", "split_k", "stream_operands", "multicast_b",
            "group_m")
    # group_m 0: the library's raster group (8)
    vals = [space.get(k, (1,) if k == "split_k" else (0,)) for k in keys]
    out = [dict(zip(keys, v)) for v in itertools.product(*vals)]
    # CTA pairs exist only for block_M = 256 tiles, and B is shared only between pairs.
    return [c for c in out if not (c["cta_pair"] and c["block_M"] != 256) and not (c["multicast_b"] and not c["cta_pair"])]


def prune(configs, M, N, K, dtype, out_dtype, smem_limit, divisible=True):
    """Split candidates into legal ones and rejects, before anything runs.

    Returns (legal, rejects) where rejects maps a reason to its configs."""
    legal, rejects = [], {"not_divisible": [], "smem_budget": [], "no_kernel": [], "other": []}
    for c in configs:
        if divisible and (M % c["block_M"] or N % c["block_N"] or K % c["block_K"]):
            rejects["not_divisible"].append(c)
            continue
        rc = tg.tgemm_validate_ex(M, N, K, dtype, out_dtype, c["block_M"], c["block_N"], c["block_K"],
                                  c["num_stages"], smem_limit, cta_pair=c.get("cta_pair", 0),
                                  split_k=c.get("split_k", 1), cluster_k=c.get("cluster_k", 0),
                                  stream_operands=c.get("stream_operands", 0), multicast_b=c.get("multicast_b", 0),
                                  group_m=c.get("group_m", 0))
        if rc == tg.OK:
            legal.append(c)
        elif rc == tg.ERR_SMEM_BUDGET:
            rejects["smem_budget"].append(c)
        elif rc == tg.ERR_NO_KERNEL:
            rejects["no_kernel"].append(c)
        else:
            rejects["other"].append(c)
    return legal, rejects


def _time(r):
    # CUDA event timestamps on GB300 advance in steps of about 2 us, so the
    # median of a short kernel's repetitions sits on one step; their mean
    # averages the steps out.  Rows written before the mean was recorded
    # rank by their median.
    return r["mean_ms"] if "mean_ms" in r else r["median_ms"]


def pick_best(rows):
    """Lowest mean time; within 1 % prefer the smaller shared footprint, then fewer stages."""
    ok = [r for r in rows if r.get("ok")]
    if not ok:
        return None
    fastest = min(_time(r) for r in ok)
    near = [r for r in ok if _time(r) <= fastest * 1.01]
    return min(near, key=lambda r: (r["smem_bytes"], r["num_stages"], _time(r)))


def cache_dir(device_name: str, workload: str) -> str:
    """Per-device, per-workload cache directory (TGEMM_CACHE_DIR, default ~/.cache/tgemm)."""
    base = os.environ.get("TGEMM_CACHE_DIR", os.path.join(os.path.expanduser("~"), ".cache", "tgemm"))
    safe = "".join(ch if ch.isalnum() else "_" for ch in device_name)
    return os.path.join(base, safe, workload)


def cache_path(device_name: str, workload: str, name: str = "best_config.json") -> str:
    return os.path.join(cache_dir(device_name, workload), name)


def cache_disabled() -> bool:
    return os.environ.get("TGEMM_AUTOTUNE_DISABLE_CACHE") == "1"


def load_cached(device_name: str, workload: str):
    if cache_disabled():
        return None
    try:
        with open(cache_path(device_name, workload)) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def write_cache(device_name: str, workload: str, best: dict, rows: list):
    """best_config.json (the winner) and latency.json (every candidate)."""
    os.makedirs(cache_dir(device_name, workload), exist_ok=True)
    keys = ("block_M", "block_N", "block_K", "num_stages", "cta_pair", "split_k", "cluster_k", "stream_operands",
            "grid_reduce", "multicast_b", "group_m", "prefetch", "mean_ms", "median_ms", "min_ms", "tflops",
            "smem_bytes", "smem_bound", "ok", "worst_error_ratio", "error")
    lat = [{k: r[k] for k in keys if k in r} for r in rows]
    for name, obj in (("best_config.json", best), ("latency.json", lat)):
        path = cache_path(device_name, workload, name)
        tmp = path + f".{os.getpid()}.tmp"
        with open(tmp, "w") as f:
            json.dump(obj, f, indent=1)
        os.replace(tmp, path)


class Runner:
    """Times candidates of one workload on the current GPU and checks them.

    The check is the autotuner's own: the pages compare every candidate with
    their reference program, ``torch.matmul`` on fp32 copies of the operands,
    at rtol = atol = 1e-2 (chapter 11, sections 3.5-3.6).  The fp64 oracle is
    test infrastructure and stays out of this tool.
    """

    def __init__(self, workload: str, reps: int = 20, warmup: int = 5):
        import torch

        self.torch = torch
        self.w = inputs.WORKLOADS[workload]
        self.name = workload
        w = self.w
        self.M, self.N, self.K = w["M"], w["N"], w["K"]
        self.A, self.B = inputs.workload_operands(workload)
        self.dA = inputs.bits_to_torch(self.A, w["dtype"]).cuda()
        self.dB = inputs.bits_to_torch(self.B, w["dtype"]).cuda()
        tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[w["out"]]
        self.C = torch.empty((self.M, self.N), dtype=tdt, device="cuda")
        self.flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")
        self.reps, self.warmup = reps, warmup
        with _no_tf32(torch):
            self.ref = self.dA.float() @ self.dB.float().t()

    def run(self, c: dict) -> dict:
        torch = self.torch
        w = self.w
        row = dict(c)
        try:
            plan = tg.Plan(self.M, self.N, self.K, w["dtype"], w["out"],
                           (c["block_M"], c["block_N"], c["block_K"]), c["num_stages"], pair=bool(c.get("cta_pair")),
                           prefetch=int(c.get("prefetch", 0)), split_k=int(c.get("split_k", 1) or 1),
                           cluster_k=int(c.get("cluster_k", 0)), stream_operands=bool(c.get("stream_operands")),
                           grid_reduce=bool(c.get("grid_reduce")), multicast_b=bool(c.get("multicast_b")),
                           group_m=int(c.get("group_m", 0)))
        except tg.TgemmError as e:
            row.update(ok=False, error=str(e))
            return row
        info = plan.info
        self.C.fill_(float("nan"))
        for _ in range(self.warmup):
            plan.run(self.dA, self.dB, self.C)
        torch.cuda.synchronize()
        times = []
        for _ in range(self.reps):
            self.flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            plan.run(self.dA, self.dB, self.C)
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        code, _ = plan.status()
        err = (self.C.float() - self.ref).abs()
        bound = 1e-2 + 1e-2 * self.ref.abs()
        worst = float((err / bound).max())  # NaN (an unwritten entry) fails the comparison below
        ok = worst <= 1.0
        med = statistics.median(times)
        mean = statistics.fmean(times)
        row.update(ok=bool(ok and code == tg.OK), worst_error_ratio=worst, mean_ms=mean, median_ms=med,
                   min_ms=min(times), tflops=2.0 * self.M * self.N * self.K / (mean * 1e-3) / 1e12,
                   smem_bytes=info["smem_bytes"],
                   smem_bound=info["smem_bound"], grid=info["grid"], tiles=info["num_tiles"])
        plan.close()
        return row


class _no_tf32:
    """Context manager: fp32 matmuls in full precision (no TF32) while it is open."""

    def __init__(self, torch):
        self.m = torch.backends.cuda.matmul

    def __enter__(self):
        self.saved = self.m.allow_tf32
        self.m.allow_tf32 = False

    def __exit__(self, *exc):
        self.m.allow_tf32 = self.saved


def main(argv=None):
    ap = argparse.ArgumentParser(description="tile / num_stages sweep")
    ap.add_argument("--workload", default="gemm_4096_f16_normal")
    ap.add_argument("--space", choices=("pages", "gb300"), default="gb300")
    ap.add_argument("--any-tile", action="store_true", help="keep tiles that do not divide the problem")
    ap.add_argument("--stage-curve", action="store_true", help="latency and smem vs num_stages for 3 tile shapes")
    ap.add_argument("--prefetch-curve", action="store_true",
                    help="latency vs the producer's prefetch distance at a fixed number of buffers")
    ap.add_argument("--tiles", default=None, help="only these tiles, e.g. 128x128x32,256x224x128")
    ap.add_argument("--stages", default=None, help="only these num_stages, e.g. 2,3,4")
    ap.add_argument("--split-k", default=None, help="K splits to try, e.g. 1,9,19 (default 1)")
    ap.add_argument("--stream", action="store_true", help="also try the L2 evict-first operand hint")
    ap.add_argument("--multicast", action="store_true", help="also try pair tiles with B shared by two pairs")
    ap.add_argument("--group-m", default=None, help="raster groups of M-blocks to try, e.g. 2,4,8 (default: the "
                                                    "library's 8)")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--out", default=None, help="write all rows as JSON here")
    ap.add_argument("--no-cache", action="store_true",
                    help="neither read nor write the per-device cache (same as TGEMM_AUTOTUNE_DISABLE_CACHE=1 "
                         "for reading)")
    args = ap.parse_args(argv)

    import torch

    tg.load()
    w = inputs.WORKLOADS[args.workload]
    M, N, K = w["M"], w["N"], w["K"]
    limit = tg.tgemm_smem_limit()
    dev = torch.cuda.get_device_name()
    report = {"workload": args.workload, "device": dev, "smem_limit": limit}
    if not (args.stage_curve or args.prefetch_curve or args.no_cache):
        cached = load_cached(dev, args.workload)
        if cached is not None:
            report.update(cache_hit=True, best=cached, cache=cache_dir(dev, args.workload))
            print("cache hit:", json.dumps(cached), flush=True)
            if args.out:
                with open(args.out, "w") as f:
                    json.dump(report, f, indent=1)
            return report
    report["cache_hit"] = False
    runner = Runner(args.workload, reps=args.reps)

    if args.prefetch_curve:
        curve = []
        for block, S in (((128, 128, 32), 6), ((128, 256, 64), 4)):
            for D in range(1, S + 1):
                c = dict(block_M=block[0], block_N=block[1], block_K=block[2], num_stages=S, prefetch=D)
                curve.append(runner.run(c))
        report["prefetch_curve"] = curve
        print("| tile | buffers (num_stages) | prefetch distance | median µs | TFLOP/s | parity |")
        print("|---|---|---|---|---|---|")
        for r in curve:
            print(f"| {r['block_M']}x{r['block_N']}x{r['block_K']} | {r['num_stages']} | {r['prefetch']} | "
                  f"{1e3 * r['median_ms']:.1f} | {r['tflops']:.0f} | {'ok' if r['ok'] else 'FAIL'} |")
    elif args.stage_curve:
        curve = []
        for block in ((128, 128, 32), (128, 256, 64), (256, 256, 64)):
            for S in (1, 2, 3, 4, 6, 8):
                c = dict(block_M=block[0], block_N=block[1], block_K=block[2], num_stages=S)
                rc = tg.tgemm_validate(M, N, K, w["dtype"], w["out"], *block, S, limit)
                if rc != tg.OK:
                    curve.append(dict(c, ok=False, rejected=tg.strerror(rc),
                                      smem_bound=tg.tgemm_smem_bound(w["dtype"], *block, S)))
                    continue
                curve.append(runner.run(c))
        report["stage_curve"] = curve
        print("| tile | num_stages | median µs | TFLOP/s | smem bound B | smem requested B | parity |")
        print("|---|---|---|---|---|---|---|")
        for r in curve:
            tile = f"{r['block_M']}x{r['block_N']}x{r['block_K']}"
            if "median_ms" in r:
                print(f"| {tile} | {r['num_stages']} | {1e3 * r['median_ms']:.1f} | {r['tflops']:.0f} | "
                      f"{r['smem_bound']} | {r['smem_bytes']} | {'ok' if r['ok'] else 'FAIL'} |")
            else:
                print(f"| {tile} | {r['num_stages']} | rejected before launch | - | {r['smem_bound']} | - | - |")
        # Fit the pipeline model of chapter 11 section 1.3 to each tile's curve.
        from software_pipelined_tiled_02_gb300 import pipeline_model

        fits = {}
        for block in sorted({(r["block_M"], r["block_N"], r["block_K"]) for r in curve}):
            pts = {r["num_stages"]: r["median_ms"] for r in curve
                   if (r["block_M"], r["block_N"], r["block_K"]) == block and "median_ms" in r}
            if len(pts) >= 2:
                f = pipeline_model.fit(pts)
                fits["x".join(map(str, block))] = {k: f[k] for k in ("ratio", "min_depth", "rms")}
                print(f"model fit {block}: latency/compute = {f['ratio']:.2f}, "
                      f"model's sufficient depth = {f['min_depth']}")
        report["model_fit"] = fits
    else:
        space = dict(PAGES_SPACE if args.space == "pages" else GB300_SPACE)
        if args.tiles:
            tiles = [tuple(int(v) for v in t.split("x")) for t in args.tiles.split(",")]
            space.update(block_M=sorted({t[0] for t in tiles}), block_N=sorted({t[1] for t in tiles}),
                         block_K=sorted({t[2] for t in tiles}))
        if args.stages:
            space["num_stages"] = tuple(int(v) for v in args.stages.split(","))
        if args.split_k:
            space["split_k"] = tuple(int(v) for v in args.split_k.split(","))
        if args.stream:
            space["stream_operands"] = (0, 1)
        if args.multicast:
            space["multicast_b"] = (0, 1)
        if args.group_m:
            space["group_m"] = tuple(int(v) for v in args.group_m.split(","))
        configs = enumerate_space(space)
        if args.tiles:
            configs = [c for c in configs if (c["block_M"], c["block_N"], c["block_K"]) in tiles]
        legal, rejects = prune(configs, M, N, K, w["dtype"], w["out"], limit, divisible=not args.any_tile)
        report["requested"] = len(configs)
        report["pages_prune"] = {"budget": PAGES_BUDGET, "kept": pages_prune_count(
            configs, M, N, K, w["dtype"], divisible=not args.any_tile)}
        report["legal"] = len(legal)
        report["rejected"] = {k: len(v) for k, v in rejects.items()}
        print(json.dumps({k: report[k] for k in ("workload", "device", "smem_limit", "requested", "pages_prune",
                                                 "legal", "rejected")}), flush=True)
        rows = [runner.run(c) for c in legal]
        report["rows"] = rows
        best = pick_best(rows)
        report["best"] = best
        for r in sorted(rows, key=lambda r: _time(r) if "median_ms" in r else 1e9)[:10]:
            print(json.dumps({k: r.get(k) for k in ("block_M", "block_N", "block_K", "num_stages", "cta_pair",
                                                    "stream_operands", "multicast_b", "group_m", "mean_ms",
                                                    "median_ms", "tflops", "smem_bytes", "ok")}), flush=True)
        if best and not args.no_cache:
            write_cache(dev, args.workload, best, rows)
            report["cache"] = cache_dir(dev, args.workload)
        print("best:", json.dumps(best), flush=True)
        bad = [r for r in rows if not r.get("ok")]
        if bad:
            print(f"{len(bad)} candidates failed parity or reported an error", flush=True)
    if args.out:
        with open(args.out, "w") as f:
            json.dump(report, f, indent=1)
    return report


if __name__ == "__main__":
    main()
