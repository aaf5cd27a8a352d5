"""Host logic of bench.py on the CPU: aggregation over ranks (gloo,
world_size 2), the reference arm's rank rule, clock-sample parsing and the
profile-traffic lookup."""

import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, "gloo")
    # rank r measured (r + 1) ms per step: the job time is the slowest rank's
    (mx,) = bench.reduce_max([float(rank + 1)], dist, "cpu")
    value = bench.aggregate(1e12, mx / 1e3, world)
    with open(f"{out_path}.{rank}", "w") as f:
        json.dump({"max": mx, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_and_aggregate_gloo_two_ranks(tmp_path):
    port = _free_port()
    out = str(tmp_path / "r")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        d = json.load(open(f"{out}.{r}"))
        assert d["max"] == 2.0
        # 2 ranks x 1e12 FLOP over 2 ms = 1000 TFLOP/s
        assert d["value"] == pytest.approx(1000.0)


def test_aggregate_single_rank():
    assert bench.aggregate(2 * 4096 ** 3, 1e-4, 1) == pytest.approx(2 * 4096 ** 3 / 1e-4 / 1e12)
    assert bench.aggregate(1.0, 0.0, 1) == 0.0


def test_reference_arm_only_rank_zero_works():
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    w = {"M": 64, "N": 64, "K": 64, "dtype": "f16"}
    assert bench.run_reference(args, w, world=2, rank=1) is None


def test_reference_arm_line_shape():
    args = bench.parse_args(["--impl", "reference", "--steps", "2", "--warmup", "1", "--workload",
                             "gemm_128_f16_uniform"])
    from software_pipelined_tiled_02_gb300 import inputs

    line = bench.run_reference(args, inputs.WORKLOADS["gemm_128_f16_uniform"], world=1, rank=0)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["metric"] == bench.METRIC


def test_clock_summary_parsing():
    s = bench.ClockSampler(0)
    s.lines = [(10.0, "2026/12/02 10:00:00.000, 0, 1980, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active"),
               (10.1, "2026/12/02 10:00:00.100, 0, 1900, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active"),
               (20.0, "2026/12/02 10:00:10.000, 0, 600, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active")]
    s.mark(9.9, 10.2)
    d = s.summary()
    assert d["sm_mhz"] == pytest.approx(1940.0) and d["sm_max_mhz"] == 2070.0
    assert d["reasons"] == ["sw_power_cap"] and d["samples"] == 2 and d["in_timed_region"]


def test_recorded_traffic_requires_current_kernel(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    p = tmp_path / "tgemm_kernel_wl.md"
    p.write_text(f"- kernel_source_sha256: `{bench.kernel_source_hash()}`\n- dram_bytes_per_launch: 1234\n")
    assert bench.recorded_traffic("wl") == 1234
    p.write_text("- kernel_source_sha256: `deadbeef`\n- dram_bytes_per_launch: 1234\n")
    assert bench.recorded_traffic("wl") is None
    assert bench.recorded_traffic("absent") is None


def test_recorded_traffic_requires_same_launch_config(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    key = bench.config_key((256, 224, 64), 3, False, 1)
    assert key == "256,224,64 S3 pair0 split1 group8"
    assert bench.config_key((256, 224, 64), 3, False, 1, 4) == "256,224,64 S3 pair0 split1 group4"
    assert (bench.config_key((256, 352, 64), 5, True, 1, 8, 0, True, False, True) ==
            "256,352,64 S5 pair1 split1 group8 stream mcast")
    p = tmp_path / "tgemm_kernel_wl.md"
    p.write_text(f"- kernel_source_sha256: `{bench.kernel_source_hash()}`\n- config: `{key}`\n"
                 "- dram_bytes_per_launch: 99\n")
    assert bench.recorded_traffic("wl", key) == 99
    assert bench.recorded_traffic("wl", bench.config_key((256, 224, 128), 3, True, 1)) is None


def test_roofline_bound_follows_arithmetic_intensity():
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}  # ridge 250 FLOP/B
    # 4096^3 fp16 -> fp16: 1365 FLOP/B, tensor-bound
    f, b = 2 * 4096 ** 3, 3 * 4096 * 4096 * 2
    r = bench.roofline_for(f, b, 1e-4, peaks)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(f / 1e-4 / 1e12) and r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    # 512x512x32768 fp16 -> fp32: 252 FLOP/B ... just above this ridge; 200 FLOP/B is below it
    r = bench.roofline_for(200.0 * 1e9, 1e9, 1e-3, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(1e9 / 1e-3 / 1e9) and r["frac"] == pytest.approx(1000.0 / 8000.0)
    assert r["tensor_frac"] == pytest.approx(200.0 / 2000.0)
    # without measured peaks the recipe's fallbacks are used
    r = bench.roofline_for(f, b, 1e-4, None)
    assert r["peak"] == bench.FALLBACK_PEAK_TFLOPS and r["peak_source"].startswith("fallback")
