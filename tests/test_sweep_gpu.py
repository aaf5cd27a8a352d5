"""The sweep on the GPU: prune, time, check, cache, cache hit, forced re-search.

Chapter 11 "Pipeline and autotuning", sections 3.5-3.8: every candidate runs
and is compared with the pages' reference program (torch.matmul at rtol =
atol = 1e-2); the winner is written per device as best_config.json beside
latency.json; a later search reads the cached winner without timing; the
disable switch forces a new search.  The winner is then checked here against
the fp64 oracle.
"""

import json
import os

import pytest
import torch

import oracle
from software_pipelined_tiled_02_gb300 import inputs

pytestmark = pytest.mark.gpu

ARGS = ["--workload", "gemm_128_f16_uniform", "--tiles", "128x128x32,128x64x32", "--stages", "2,3",
        "--reps", "5"]


def test_sweep_times_checks_caches_and_reuses(cuda_lib, tmp_path, monkeypatch):
    from software_pipelined_tiled_02_gb300 import sweep

    monkeypatch.setenv("TGEMM_CACHE_DIR", str(tmp_path))
    monkeypatch.delenv("TGEMM_AUTOTUNE_DISABLE_CACHE", raising=False)
    rep = sweep.main(ARGS)
    assert rep["cache_hit"] is False
    assert rep["requested"] == 4 and rep["legal"] == 4 and rep["pages_prune"]["kept"] == 4
    assert all(r["ok"] for r in rep["rows"]), rep["rows"]
    dev = torch.cuda.get_device_name()
    best_path = sweep.cache_path(dev, "gemm_128_f16_uniform")
    lat_path = sweep.cache_path(dev, "gemm_128_f16_uniform", "latency.json")
    best = json.load(open(best_path))
    lat = json.load(open(lat_path))
    assert len(lat) == 4 and all(r["median_ms"] > 0 and r["smem_bytes"] > 0 and r["ok"] for r in lat)
    assert best == {k: v for k, v in sweep.pick_best(rep["rows"]).items()}

    # the winner, run again, meets the oracle's tolerance
    w = inputs.WORKLOADS["gemm_128_f16_uniform"]
    A, B = inputs.workload_operands("gemm_128_f16_uniform")
    plan = cuda_lib.Plan(128, 128, 128, "f16", "f32", (best["block_M"], best["block_N"], best["block_K"]),
                         best["num_stages"])
    C = plan.run(inputs.bits_to_torch(A, "f16").cuda(), inputs.bits_to_torch(B, "f16").cuda())
    torch.cuda.synchronize()
    assert plan.status()[0] == 0
    R, S = oracle.gemm(A, B, w["dtype"])
    ok, worst, _ = oracle.check(C.cpu().double().numpy(), R, S, "f32")
    assert ok, worst

    # a second search reads the cache and times nothing
    mtime = os.path.getmtime(lat_path)
    rep2 = sweep.main(ARGS)
    assert rep2["cache_hit"] is True and rep2["best"] == best and "rows" not in rep2
    assert os.path.getmtime(lat_path) == mtime

    # the switch forces a new search, which rewrites both files
    monkeypatch.setenv("TGEMM_AUTOTUNE_DISABLE_CACHE", "1")
    rep3 = sweep.main(ARGS)
    assert rep3["cache_hit"] is False and len(rep3["rows"]) == 4
    assert os.path.getmtime(lat_path) >= mtime and len(json.load(open(lat_path))) == 4
