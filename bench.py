#!/usr/bin/env python
"""Throughput of the pipelined tiled GEMM on GB300, one JSON line.

A step is one C = A . B^T over the workload's seeded synthetic operands
(default: 4096^3 fp16 normal, fp16 output: the headline GEMM TFLOP/s
workload).  W untimed warm-up steps, then K timed steps; before every step
a 256 MiB buffer is written so that L2 (129 MB) holds no operand; each
step's kernel is bracketed by CUDA events on the launching stream and the
region by a barrier and a device synchronise on both sides.

Reported: value (TFLOP/s, 2*M*N*K per step / mean kernel time), an e2e
figure through tgemm_run_host (pinned host operands copied in and the result
copied out every step), the roofline of the kernel against the measured
dense tensor peak, SM clocks sampled during the timed region, and the CPU
oracle timed on a bounded sample of the same workload.

``--impl reference`` times the CPU oracle instead (the reference arm).
``--gpus N`` under torchrun runs N independent replicas (weak scaling).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/t) at fp16 4096³ and % of GB300 dense tensor peak"
FALLBACK_PEAK_TFLOPS = 1900.0
FALLBACK_PEAK_GBS = 6800.0
L2_FLUSH_BYTES = 256 * 1024 * 1024
CSRC = os.path.join(ROOT, "software_pipelined_tiled_02_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="gemm_4096_f16_normal")
    ap.add_argument("--block", default=None, help="bm,bn,bk (default: tuned table)")
    ap.add_argument("--stages", type=int, default=None)
    ap.add_argument("--pair", type=int, choices=(0, 1), default=None,
                    help="1: CTA pairs (clusters of 2) share each 256-row tile (default: tuned table)")
    ap.add_argument("--split-k", type=int, default=None, help="K splits per tile (default: tuned table)")
    ap.add_argument("--cluster-k", type=int, default=None,
                    help="K splits reduced inside the kernel by clusters of this many CTAs (default: tuned table)")
    ap.add_argument("--stream-operands", type=int, choices=(0, 1), default=None,
                    help="1: L2 evict-first hint on the operand loads (default: tuned table)")
    ap.add_argument("--grid-reduce", type=int, choices=(0, 1), default=None,
                    help="1: reduce K splits inside the GEMM kernel after a grid-wide barrier (default: tuned table)")
    ap.add_argument("--multicast-b", type=int, choices=(0, 1), default=None,
                    help="1: clusters of two CTA pairs share B through TMA multicast (default: tuned table)")
    ap.add_argument("--group-m", type=int, default=None,
                    help="M-blocks per raster group of the persistent schedule (default: tuned table; 0 = 8)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    ap.add_argument("--sustain-seconds", type=float, default=1.5,
                    help="length of the sustained leg reported beside the timed steps (0: skip)")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_max(values, dist, device):
    """Elementwise max over ranks of a list of floats."""
    if dist is None:
        return list(values)
    import torch

    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def aggregate(per_rank_flops, max_seconds, world):
    """Whole-job throughput (TFLOP/s): all ranks' work over the slowest rank's time."""
    if max_seconds <= 0:
        return 0.0
    return per_rank_flops * world / max_seconds / 1e12


def roofline_for(flops, algo_bytes, seconds, peaks):
    """The roofline object of one launch.  The bound is the one the launch's
    arithmetic intensity (FLOP per algorithmic byte) falls under: HBM below
    the ridge peak_flops / peak_bandwidth, the tensor pipe above it.  Both
    fractions are reported; `achieved`, `peak`, `unit` and `frac` follow the
    bound."""
    if peaks and peaks.get("bf16_tflops"):
        tflops, t_src = float(peaks["bf16_tflops"]), "measured"
    else:
        tflops, t_src = FALLBACK_PEAK_TFLOPS, "fallback"
    if peaks and peaks.get("hbm_gbs"):
        gbs, g_src = float(peaks["hbm_gbs"]), "measured"
    else:
        gbs, g_src = FALLBACK_PEAK_GBS, "fallback"
    achieved_tf = flops / seconds / 1e12
    achieved_gbs = algo_bytes / seconds / 1e9
    ridge = tflops * 1e12 / (gbs * 1e9)
    intensity = flops / algo_bytes
    common = {"tensor_frac": achieved_tf / tflops, "hbm_frac": achieved_gbs / gbs,
              "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge}
    if intensity < ridge:
        return {"bound": "hbm", "achieved": achieved_gbs, "peak": gbs, "unit": "GB/s", "frac": achieved_gbs / gbs,
                "peak_source": f"{g_src} HBM copy bandwidth", **common}
    return {"bound": "tensor", "achieved": achieved_tf, "peak": tflops, "unit": "TFLOP/s", "frac": achieved_tf / tflops,
            "peak_source": f"{t_src} dense bf16 burst (fp16 runs at the bf16 rate: nominal ratio 1)", **common}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def kernel_source_hash():
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def config_key(block, stages, pair, split_k, group_m=8, cluster_k=0, stream_operands=False, grid_reduce=False,
               multicast_b=False):
    """The launch configuration as the ncu summaries record it."""
    key = (f"{block[0]},{block[1]},{block[2]} S{stages} pair{int(bool(pair))} split{int(split_k)} "
           f"group{int(group_m) or 8}")
    key += f" cluster{int(cluster_k)}" if cluster_k and cluster_k > 1 else ""
    key += " stream" if stream_operands else ""
    key += " gridreduce" if grid_reduce else ""
    return key + (" mcast" if multicast_b else "")


def recorded_traffic(workload, config=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source and, when given, the same launch
    configuration (see config_key); else None."""
    path = os.path.join(PROFILES, f"tgemm_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None
    if config is not None and fields.get("config") != config:
        return None
    try:
        return int(float(fields["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summary()

    def summary(self, windows=None):
        windows = self.windows if windows is None else windows
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(t=t, sm=float(parts[2]), smax=float(parts[3]), power=float(parts[4]),
                                 active=parts[5], hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [r for r in rows if any(a - 0.05 <= r["t"] <= b + 0.05 for a, b in windows)]
        use = inside or rows
        reasons = set()
        for r in use:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in use), "sm_max_mhz": max(r["smax"] for r in use),
                "reasons": sorted(reasons), "samples": len(use), "in_timed_region": bool(inside),
                "power_w_max": max(r["power"] for r in use)}


# ------------------------------------------------------------------ arms

def cpu_baseline(A, B, w, seconds):
    """The oracle, as it stands, on whole rows of C until `seconds` elapse.

    The operands are decoded to binary64 once before timing (they are
    resident, as the GPU arm's operands are); the timed part is the oracle's
    in-order fp64 sums."""
    import oracle

    M, N, K = w["M"], w["N"], w["K"]
    oracle.build()
    cores = oracle.num_threads()
    Ad, Bd = oracle.decode(A, w["dtype"]), oracle.decode(B, w["dtype"])
    chunk = max(cores, 16)
    done, t0 = 0, time.perf_counter()
    while done < M and time.perf_counter() - t0 < seconds:
        n = min(chunk, M - done)
        oracle.gemm_decoded_rows(Ad, Bd, done, n)
        done += n
    dt = time.perf_counter() - t0
    flops = 2.0 * done * N * K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"rows 0..{done - 1} of C ({done}x{N}x{K} in-order fp64 multiply-adds, {dt:.1f} s, "
                      f"operands decoded once beforehand) of the same seeded {w['dtype']} workload"}


def run_reference(args, w, world, rank):
    """Reference arm: the CPU oracle timed on bounded samples of the workload."""
    if rank != 0:
        return None
    import oracle
    from software_pipelined_tiled_02_gb300 import inputs

    A, B = inputs.workload_operands(args.workload)
    oracle.build()
    cores = oracle.num_threads()
    M, N, K = w["M"], w["N"], w["K"]
    rows = min(M, max(16, cores))
    Ad, Bd = oracle.decode(A, w["dtype"]), oracle.decode(B, w["dtype"])
    for i in range(args.warmup):
        oracle.gemm_decoded_rows(Ad, Bd, (i * rows) % (M - rows + 1), rows)
    times = []
    for i in range(args.steps):
        r0 = (i * rows) % (M - rows + 1)
        t0 = time.perf_counter()
        oracle.gemm_decoded_rows(Ad, Bd, r0, rows)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    flops = 2.0 * rows * N * K
    value = flops * len(times) / total / 1e12
    sample = (f"{rows} rows of C per step ({rows}x{N}x{K} in-order fp64 multiply-adds, operands decoded once "
              f"beforehand) of the seeded {w['dtype']} workload")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(args, w, None, None),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def sustained_leg(plan, dA, dB, dC, flush, stream, dev, seconds, flops, sampler):
    """Flushed steps back to back for at least `seconds` of wall time; each
    step's kernel is bracketed by CUDA events on the launching stream."""
    import torch

    batch = 256
    t0 = time.time()
    times = []
    while True:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(batch)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            plan.run(dA, dB, dC, stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        times += [a.elapsed_time(b) for a, b in ev]
        if time.time() - t0 >= seconds:
            break
    t1 = time.time()
    if sampler:
        sampler.mark(t0, t1)
    mean = sum(times) / len(times)
    return {"value": flops / (mean / 1e3) / 1e12, "unit": "TFLOP/s", "steps": len(times),
            "seconds": t1 - t0, "ms_per_step": mean, "kernel_ms_median": statistics.median(times),
            "_window": (t0, t1)}


def config_block(args, w, block, stages):
    cfg = {"workload": args.workload, "M": w["M"], "N": w["N"], "K": w["K"], "operand_dtype": w["dtype"],
           "accumulate": "f32", "out_dtype": w["out"], "distribution": w["dist"], "seed": w["seed"],
           "l2": "256 MiB buffer written before every timed step (L2 is 129 MB)"}
    if block is not None:
        cfg.update({"block_M": block[0], "block_N": block[1], "block_K": block[2], "num_stages": stages})
    return cfg


def run_ours(args, w, world, rank, local):
    import torch

    import software_pipelined_tiled_02_gb300 as tg
    from software_pipelined_tiled_02_gb300 import inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    tg.load()
    M, N, K = w["M"], w["N"], w["K"]
    if args.block:
        block = tuple(int(x) for x in args.block.split(","))
        stages = args.stages or 4
        pair = bool(args.pair)
        split_k = args.split_k or 1
        group_m = args.group_m or 0
        cluster_k = args.cluster_k or 0
        stream_ops = bool(args.stream_operands)
        grid_red = bool(args.grid_reduce)
        mcast = bool(args.multicast_b)
    else:
        cfg = tg.default_config(M, N, K, w["dtype"], w["out"])
        block, stages, pair, split_k = cfg["block"], cfg["num_stages"], cfg["cta_pair"], cfg["split_k"]
        group_m = cfg["group_m"] if args.group_m is None else args.group_m
        if args.stages:
            stages = args.stages
        if args.pair is not None:
            pair = bool(args.pair)
        if args.split_k is not None:
            split_k = args.split_k
        cluster_k = cfg["cluster_k"] if args.cluster_k is None else args.cluster_k
        stream_ops = cfg["stream_operands"] if args.stream_operands is None else bool(args.stream_operands)
        grid_red = cfg["grid_reduce"] if args.grid_reduce is None else bool(args.grid_reduce)
        mcast = cfg["multicast_b"] if args.multicast_b is None else bool(args.multicast_b)
    A, B = inputs.workload_operands(args.workload)
    hA = inputs.bits_to_torch(A, w["dtype"])
    hB = inputs.bits_to_torch(B, w["dtype"])
    dA, dB = hA.to(dev), hB.to(dev)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[w["out"]]
    dC = torch.empty((M, N), dtype=tdt, device=dev)
    plan = tg.Plan(M, N, K, w["dtype"], w["out"], block, stages, pair=pair, split_k=split_k, group_m=group_m,
                   cluster_k=cluster_k, stream_operands=stream_ops, grid_reduce=grid_red, multicast_b=mcast)
    info = plan.info
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = 2.0 * M * N * K

    sampler = None if args.no_clocks else ClockSampler(local)
    if sampler:
        sampler.start()
        time.sleep(0.4)  # let the sampler start; the warm-up below then runs right before the timed region

    for _ in range(args.warmup):
        flush.zero_()
        plan.run(dA, dB, dC, stream)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        plan.run(dA, dB, dC, stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    t_wall1 = time.time()
    if sampler:
        sampler.mark(t_wall0, t_wall1)
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    code, detail = plan.status()
    if code != tg.OK:
        raise RuntimeError(f"kernel reported {tg.strerror(code)} {detail}")
    mean_ms = sum(kernel_ms) / len(kernel_ms)
    (max_mean_ms,) = reduce_max([mean_ms], dist, dev)
    value = aggregate(flops, max_mean_ms / 1e3, world)

    # Sustained leg, reported beside `value` (never replacing it): the same
    # flushed steps back to back for at least `--sustain-seconds`, long enough
    # for the clock sampler to see the GPU under this load.
    sustained = None
    if args.sustain_seconds > 0:
        sustained = sustained_leg(plan, dA, dB, dC, flush, stream, dev, args.sustain_seconds, flops, sampler)
        code, detail = plan.status()
        if code != tg.OK:
            raise RuntimeError(f"kernel reported {tg.strerror(code)} {detail} in the sustained leg")

    e2e = None
    if not args.no_e2e:
        # End to end through tgemm_run_host: every step copies its operands in
        # from pinned host memory, runs the kernel and copies C back out.
        # Consecutive steps alternate between two streams, each with its own
        # plan and device buffers, so step i+1's copies overlap step i's work,
        # as a caller streaming independent GEMMs would run them.
        pA, pB = hA.pin_memory(), hB.pin_memory()
        pCs = [torch.empty((M, N), dtype=tdt).pin_memory() for _ in range(2)]
        plans = [plan, tg.Plan(M, N, K, w["dtype"], w["out"], block, stages, pair=pair, split_k=split_k,
                               group_m=group_m, cluster_k=cluster_k, stream_operands=stream_ops,
                               grid_reduce=grid_red, multicast_b=mcast)]
        bufs = [(dA, dB, dC), (torch.empty_like(dA), torch.empty_like(dB), torch.empty_like(dC))]
        streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
        torch.cuda.synchronize(dev)
        for i in range(4):
            k = i & 1
            plans[k].run_host(pA, pB, pCs[k], *bufs[k], stream=streams[k])
        torch.cuda.synchronize(dev)
        e_steps = max(2, min(args.steps, 400))
        t_start, t_mid, t_end = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        tw0 = time.time()
        t_start.record(streams[0])
        streams[1].wait_event(t_start)
        for i in range(e_steps):
            k = i & 1
            plans[k].run_host(pA, pB, pCs[k], *bufs[k], stream=streams[k])
        t_mid.record(streams[1])
        streams[0].wait_event(t_mid)
        t_end.record(streams[0])
        torch.cuda.synchronize(dev)
        if sampler:
            sampler.mark(tw0, time.time())
        e_ms = t_start.elapsed_time(t_end) / e_steps
        (e_max,) = reduce_max([e_ms], dist, dev)
        e2e = {"value": aggregate(flops, e_max / 1e3, world), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(pA.numel() * pA.element_size() + pB.numel() * pB.element_size()),
               "d2h_bytes_per_step": int(pCs[0].numel() * pCs[0].element_size()), "steps": e_steps,
               "ms_per_step": e_max,
               "path": "tgemm_run_host (pinned host A,B -> device; kernel; C -> pinned host), consecutive steps "
                       "on two streams with two buffer sets"}
        for pl in plans:
            if pl.status()[0] != tg.OK:
                raise RuntimeError("kernel reported an error in the end-to-end leg")
        plans[1].close()

    clocks = sampler.stop() if sampler else None
    if clocks:
        clocks["windows"] = "timed steps, the sustained leg and the e2e leg (samples every 50 ms)"
    if sustained is not None and sampler is not None:
        sustained["clocks"] = sampler.summary(windows=[sustained.pop("_window")])
        mhz = sustained["clocks"].get("sm_mhz")
        if mhz:
            # time x clock: kernel cycles per step, comparable across clock levels
            sustained["mcycles_per_step"] = sustained["ms_per_step"] * mhz / 1e3
    elif sustained is not None:
        sustained.pop("_window", None)

    algo_bytes = (M * K + N * K) * 2 + M * N * (4 if w["out"] == "f32" else 2)
    two_kernels = info["split_k"] > 1 and info["cluster_k"] <= 1 and not info["grid_reduce"]
    roofline = roofline_for(flops, algo_bytes, mean_ms / 1e3, measured_peaks())
    roofline.update({"traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch, L2 clean "
                                     "at its start; output still in L2 when the launch ends is not counted",
                     "traffic": recorded_traffic(args.workload,
                                                 config_key(block, stages, pair, info["split_k"], group_m,
                                                            info["cluster_k"], info["stream_operands"],
                                                            info["grid_reduce"], info["multicast_b"])),
                     "kernel": ("tgemm_kernel + splitk_reduce_kernel, timed together per step"
                                if two_kernels else "tgemm_kernel"),
                     "flops_per_launch": flops, "algorithmic_bytes_per_launch": algo_bytes})

    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(A, B, w, args.cpu_seconds)
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": max_mean_ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
                "config": dict(config_block(args, w, block, stages), cta_pair=int(pair),
                               split_k=int(info["split_k"]), group_m=int(group_m) or 8,
                               cluster_k=int(info["cluster_k"]),
                               stream_operands=int(info["stream_operands"]),
                               grid_reduce=int(info["grid_reduce"]),
                               multicast_b=int(info["multicast_b"])), "roofline": roofline,
                "cpu_baseline": cpu,
                "e2e": e2e, "gpu_launches": args.steps * (2 if two_kernels else 1),
                "clocks": clocks,
                "sustained": sustained,
                "plan": {k: info[k] for k in ("grid", "num_tiles", "smem_bytes", "tmem_columns", "acc_stages")},
                "kernel_ms": {"min": min(kernel_ms), "median": statistics.median(kernel_ms), "max": max(kernel_ms)}}
    plan.close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return line


def main(argv=None):
    args = parse_args(argv)
    from software_pipelined_tiled_02_gb300 import inputs

    if args.workload not in inputs.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; one of {sorted(inputs.WORKLOADS)}")
    if args.warmup < 3 and args.impl == "ours":
        raise SystemExit("at least 3 warm-up steps are required")
    w = inputs.WORKLOADS[args.workload]
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, w, world, rank)
    else:
        line = run_ours(args, w, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
