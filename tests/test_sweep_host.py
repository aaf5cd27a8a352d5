"""Host logic of the sweep: pruning before launch, tie-break, cache switch."""

import oracle
import software_pipelined_tiled_02_gb300 as tg
from software_pipelined_tiled_02_gb300 import build as tbuild
from software_pipelined_tiled_02_gb300 import sweep

LIMIT = 227 * 1024


def setup_module(_):
    tbuild.build()
    tg.load()


def test_pages_space_prunes_over_budget_before_launch():
    cfgs = sweep.enumerate_space(sweep.PAGES_SPACE)
    assert len(cfgs) == 3 * 3 * 3 * 4  # the pages' grid without its `threads` axis
    assert all(c["cta_pair"] == 0 for c in cfgs)
    legal, rej = sweep.prune(cfgs, 4096, 4096, 4096, tg.F16, tg.F16, LIMIT)
    over = {(c["block_M"], c["block_N"], c["block_K"], c["num_stages"]) for c in rej["smem_budget"]}
    assert (256, 256, 64, 4) in over
    # every config the pages' bound puts over the limit is rejected, none is launched
    for c in cfgs:
        if oracle.smem_bound(c["block_M"], c["block_N"], c["block_K"], c["num_stages"], 2) > LIMIT:
            assert c not in legal
    # the kernel implements every tile shape of the pages' grid (block_M 64 included)
    assert not rej["no_kernel"]
    assert not rej["not_divisible"]
    assert len(legal) + sum(len(v) for v in rej.values()) == len(cfgs)


def test_divisibility_prune_is_optional():
    cfgs = [dict(block_M=128, block_N=192, block_K=64, num_stages=3)]
    legal, rej = sweep.prune(cfgs, 4096, 4096, 4096, tg.F16, tg.F16, LIMIT, divisible=True)
    assert not legal and rej["not_divisible"]
    legal, rej = sweep.prune(cfgs, 4096, 4096, 4096, tg.F16, tg.F16, LIMIT, divisible=False)
    assert legal == cfgs


def test_pick_best_tie_break():
    rows = [dict(ok=True, median_ms=1.000, smem_bytes=200000, num_stages=4),
            dict(ok=True, median_ms=1.005, smem_bytes=150000, num_stages=3),
            dict(ok=True, median_ms=1.005, smem_bytes=150000, num_stages=2),
            dict(ok=False, median_ms=0.5, smem_bytes=1, num_stages=1),
            dict(ok=True, median_ms=1.2, smem_bytes=1000, num_stages=1)]
    best = sweep.pick_best(rows)
    assert best["smem_bytes"] == 150000 and best["num_stages"] == 2
    assert sweep.pick_best([dict(ok=False)]) is None


def test_pick_best_ranks_by_mean():
    # CUDA event timestamps advance in steps of about 2 us: two candidates can share a
    # median while their means differ; the mean decides, and the footprint rule still
    # applies within 1 % of the fastest mean.
    rows = [dict(ok=True, mean_ms=0.0830, median_ms=0.0820, smem_bytes=200000, num_stages=6),
            dict(ok=True, mean_ms=0.0812, median_ms=0.0820, smem_bytes=210000, num_stages=6),
            dict(ok=True, mean_ms=0.0815, median_ms=0.0840, smem_bytes=150000, num_stages=3)]
    assert sweep.pick_best(rows)["smem_bytes"] == 150000   # within 1 % of 0.0812, smaller footprint
    rows[2]["mean_ms"] = 0.0830
    assert sweep.pick_best(rows)["smem_bytes"] == 210000   # the lowest mean alone


def test_raster_group_dimension():
    space = dict(block_M=(256,), block_N=(224,), block_K=(64,), num_stages=(6,), cta_pair=(1,), group_m=(2, 4, 8))
    cfgs = sweep.enumerate_space(space)
    assert sorted(c["group_m"] for c in cfgs) == [2, 4, 8]
    legal, rej = sweep.prune(cfgs, 4096, 4096, 4096, tg.F16, tg.F16, LIMIT, divisible=False)
    assert len(legal) == 3
    # without the key every config takes the library's group (0 = 8)
    assert all(c["group_m"] == 0 for c in sweep.enumerate_space(dict(space, group_m=(0,))))


def test_cache_switch(tmp_path, monkeypatch):
    monkeypatch.setenv("TGEMM_CACHE_DIR", str(tmp_path))
    p = sweep.cache_path("NVIDIA GB300", "wl")
    import json
    import os

    os.makedirs(os.path.dirname(p), exist_ok=True)
    json.dump({"block_M": 256}, open(p, "w"))
    assert sweep.load_cached("NVIDIA GB300", "wl") == {"block_M": 256}
    monkeypatch.setenv("TGEMM_AUTOTUNE_DISABLE_CACHE", "1")
    assert sweep.load_cached("NVIDIA GB300", "wl") is None


def test_gb300_space_has_pairs_only_for_256_rows():
    cfgs = sweep.enumerate_space(sweep.GB300_SPACE)
    pairs = [c for c in cfgs if c["cta_pair"]]
    assert pairs and all(c["block_M"] == 256 for c in pairs)
    legal, rej = sweep.prune(cfgs, 4096, 4096, 4096, tg.F16, tg.F16, LIMIT, divisible=False)
    # A pair CTA holds half of B: 256x256x64 fits 6 stages as a pair, 3 alone.
    key = lambda c: (c["block_M"], c["block_N"], c["block_K"], c["num_stages"], c["cta_pair"])  # noqa: E731
    ok = {key(c) for c in legal}
    assert (256, 256, 64, 6, 1) in ok and (256, 256, 64, 6, 0) not in ok and (256, 256, 64, 3, 0) in ok


def test_frozen_defaults_are_legal_and_chosen():
    from software_pipelined_tiled_02_gb300 import defaults

    for (M, N, K, dt, od), entry in defaults.FROZEN.items():
        cfg = defaults.choose(M, N, K, dt, od)
        assert all(cfg[k] == v for k, v in entry.items())
        assert set(cfg) == {"block", "num_stages"} | set(defaults.DEFAULT_OPTS)
        rc = tg.tgemm_validate_ex(M, N, K, dt, od, *cfg["block"], cfg["num_stages"], 232448,
                                  cta_pair=int(cfg["cta_pair"]), split_k=cfg["split_k"], group_m=cfg["group_m"],
                                  cluster_k=cfg["cluster_k"], stream_operands=int(cfg["stream_operands"]),
                                  grid_reduce=int(cfg["grid_reduce"]), stream_k=int(cfg["stream_k"]),
                                  multicast_b=int(cfg["multicast_b"]))
        assert rc == tg.OK, ((M, N, K), cfg, tg.strerror(rc))


def test_multicast_dimension_of_the_space():
    # B shared by two pairs exists only in pair mode and without a K split.
    space = dict(sweep.GB300_SPACE, multicast_b=(0, 1), split_k=(1, 2))
    cfgs = sweep.enumerate_space(space)
    assert all(c["cta_pair"] for c in cfgs if c["multicast_b"])
    assert any(c["multicast_b"] for c in cfgs)
    legal, rej = sweep.prune(cfgs, 4000, 3000, 5000, tg.F16, tg.F32, LIMIT, divisible=False)
    mc = [c for c in legal if c["multicast_b"]]
    assert mc and all(c["split_k"] == 1 for c in mc)
    key = lambda c: (c["block_M"], c["block_N"], c["block_K"], c["num_stages"], c["multicast_b"])  # noqa: E731
    assert (256, 352, 64, 5, 1) in {key(c) for c in legal}
    assert any(c["multicast_b"] and c["split_k"] == 2 for c in rej["other"])


def test_estimator_shares_b_only_where_rows_straddle_lines_and_rounds_hold():
    from software_pipelined_tiled_02_gb300 import defaults

    # the frozen ragged shape's reasoning, on its tile: misaligned pitch, 72 items = 2 rounds of 36
    assert defaults.multicast_pays(4000, 3000, 5000, (256, 352, 64))
    # the same shape with an aligned pitch (K = 5120): no
    assert not defaults.multicast_pays(4000, 3000, 5120, (256, 352, 64))
    # 4096 x 4096 with a misaligned K: 304 tiles are 4 rounds of 76 pairs, 152 items 5 rounds of 36
    assert not defaults.multicast_pays(4096, 4096, 4100, (256, 224, 128))
    # a shape outside the table gets it through choose(), and only on pair tiles
    cfg = defaults.choose(4000, 3000, 5008, tg.F16, tg.F32)
    assert cfg["block"] == (256, 352, 64)
    assert cfg["cta_pair"] and cfg["multicast_b"] and defaults.multicast_pays(4000, 3000, 5008, cfg["block"])
    # where the chosen pair tile's rounds would grow, no multicast: 2 x 37 tiles of 256x512 are one round of
    # 76 pairs but 37 items on 36 clusters; 16 x 14 tiles of 256x448 are 3 rounds, 112 items 4
    for M, N in ((512, 18944), (4096, 6144)):
        cfg = defaults.choose(M, N, 4104, tg.F16, tg.F16)
        assert cfg["cta_pair"] and not cfg["multicast_b"] and not defaults.multicast_pays(M, N, 4104, cfg["block"])
    # with an aligned pitch, never
    assert not defaults.choose(4096, 4096, 4096 + 64, tg.F16, tg.F16)["multicast_b"]


def test_wide_pair_tiles_only_in_pair_mode():
    cfgs = sweep.enumerate_space(sweep.GB300_SPACE)
    legal, rej = sweep.prune(cfgs, 8192, 8192, 8192, tg.BF16, tg.BF16, LIMIT, divisible=False)
    key = lambda c: (c["block_M"], c["block_N"], c["block_K"], c["num_stages"], c["cta_pair"])  # noqa: E731
    ok = {key(c) for c in legal}
    no_kernel = {key(c) for c in rej["no_kernel"]}
    assert (256, 512, 64, 4, 1) in ok and (256, 512, 64, 5, 1) not in ok   # 48 KB slots: four fit
    assert (256, 512, 64, 2, 0) in no_kernel and (128, 384, 64, 2, 0) in no_kernel


def test_pages_prune_count_matches_the_pages():
    # Chapter 11 section 3.7: 216 configs at 4096^3 (the grid below times the
    # two `threads` values), of which 214 are kept; the two rejects are
    # 256x256x64 at 4 stages (256 KiB > 228 KiB).
    cfgs = sweep.enumerate_space(sweep.PAGES_SPACE)
    kept = sweep.pages_prune_count(cfgs, 4096, 4096, 4096, tg.F16)
    assert 2 * len(cfgs) == 216 and 2 * kept == 214
    assert sweep.PAGES_BUDGET == 228 * 1024


def test_write_and_read_cache(tmp_path, monkeypatch):
    import json

    monkeypatch.setenv("TGEMM_CACHE_DIR", str(tmp_path))
    monkeypatch.delenv("TGEMM_AUTOTUNE_DISABLE_CACHE", raising=False)
    rows = [dict(block_M=128, block_N=128, block_K=32, num_stages=3, ok=True, median_ms=0.01, min_ms=0.009,
                 smem_bytes=1000, smem_bound=900, tflops=1.0, extra="dropped"),
            dict(block_M=128, block_N=64, block_K=32, num_stages=2, ok=False, error="x")]
    sweep.write_cache("NVIDIA GB300", "wl", rows[0], rows)
    assert sweep.load_cached("NVIDIA GB300", "wl") == rows[0]
    lat = json.load(open(sweep.cache_path("NVIDIA GB300", "wl", "latency.json")))
    assert len(lat) == 2 and "extra" not in lat[0] and lat[1]["ok"] is False
    monkeypatch.setenv("TGEMM_AUTOTUNE_DISABLE_CACHE", "1")
    assert sweep.load_cached("NVIDIA GB300", "wl") is None


def test_estimator_picks_the_measured_best_tiles():
    # Shapes outside the tuned table: the candidate the wave-count estimator
    # picks ran within 3 % of the fastest tile of a timed search on a GB300
    # with two producer warps (mean CUDA-event microseconds, fp16 in and out,
    # 256 MiB L2 flush before each launch; the block_K = 128 pair tiles were
    # timed as well but are no longer candidates).
    from software_pipelined_tiled_02_gb300 import defaults

    P, O = True, False
    measured = {
        (3072, 3072, 3072): {
            ((256, 256, 128), 3, P): 42.2, ((256, 512, 64), 4, P): 41.7, ((256, 448, 64), 4, P): 65.4,
            ((256, 384, 64), 4, P): 58.7, ((256, 352, 64), 5, P): 54.8, ((256, 224, 128), 3, P): 52.1,
            ((256, 256, 64), 6, P): 41.4, ((256, 224, 64), 6, P): 50.3, ((256, 192, 64), 6, P): 47.0,
            ((256, 128, 64), 8, P): 52.0, ((256, 256, 64), 3, O): 41.4, ((256, 224, 64), 3, O): 65.0,
            ((128, 256, 64), 4, O): 45.1, ((128, 128, 64), 4, O): 61.6},
        (6144, 6144, 6144): {
            ((256, 256, 128), 3, P): 273.8, ((256, 512, 64), 4, P): 281.4, ((256, 448, 64), 4, P): 306.6,
            ((256, 384, 64), 4, P): 315.1, ((256, 352, 64), 5, P): 291.4, ((256, 224, 128), 3, P): 271.5,
            ((256, 256, 64), 6, P): 267.5, ((256, 224, 64), 6, P): 266.4, ((256, 192, 64), 6, P): 285.2,
            ((256, 128, 64), 8, P): 362.5, ((256, 256, 64), 3, O): 280.6, ((256, 224, 64), 3, O): 312.5,
            ((128, 256, 64), 4, O): 317.1, ((128, 128, 64), 4, O): 485.9},
        (1024, 8192, 4096): {
            ((256, 256, 128), 3, P): 53.7, ((256, 512, 64), 4, P): 51.1, ((256, 448, 64), 4, P): 48.3,
            ((256, 384, 64), 4, P): 74.9, ((256, 352, 64), 5, P): 68.2, ((256, 224, 128), 3, P): 52.0,
            ((256, 256, 64), 6, P): 51.7, ((256, 224, 64), 6, P): 48.9, ((256, 192, 64), 6, P): 60.3,
            ((256, 128, 64), 8, P): 65.1, ((256, 256, 64), 3, O): 52.3, ((256, 224, 64), 3, O): 50.0,
            ((128, 256, 64), 4, O): 60.0, ((128, 128, 64), 4, O): 86.2},
        (8192, 1024, 4096): {
            ((256, 256, 128), 3, P): 54.1, ((256, 512, 64), 4, P): 50.2, ((256, 448, 64), 4, P): 80.4,
            ((256, 384, 64), 4, P): 73.1, ((256, 352, 64), 5, P): 67.3, ((256, 224, 128), 3, P): 67.6,
            ((256, 256, 64), 6, P): 51.9, ((256, 224, 64), 6, P): 63.8, ((256, 192, 64), 6, P): 60.2,
            ((256, 128, 64), 8, P): 66.3, ((256, 256, 64), 3, O): 52.8, ((256, 224, 64), 3, O): 84.4,
            ((128, 256, 64), 4, O): 58.5, ((128, 128, 64), 4, O): 76.6},
        (4096, 4096, 1024): {
            ((256, 256, 128), 3, P): 33.2, ((256, 512, 64), 4, P): 38.6, ((256, 448, 64), 4, P): 45.7,
            ((256, 384, 64), 4, P): 43.5, ((256, 352, 64), 5, P): 41.2, ((256, 224, 128), 3, P): 31.6,
            ((256, 256, 64), 6, P): 32.1, ((256, 224, 64), 6, P): 30.9, ((256, 192, 64), 6, P): 33.3,
            ((256, 128, 64), 8, P): 37.5, ((256, 256, 64), 3, O): 36.2, ((256, 224, 64), 3, O): 33.4,
            ((128, 256, 64), 4, O): 33.5, ((128, 128, 64), 4, O): 39.3},
        (2048, 2048, 2048): {
            ((256, 256, 128), 3, P): 22.1, ((256, 512, 64), 4, P): 31.1, ((256, 448, 64), 4, P): 29.0,
            ((256, 384, 64), 4, P): 26.8, ((256, 352, 64), 5, P): 25.0, ((256, 224, 128), 3, P): 28.7,
            ((256, 256, 64), 6, P): 21.3, ((256, 224, 64), 6, P): 27.1, ((256, 192, 64), 6, P): 26.9,
            ((256, 128, 64), 8, P): 24.9, ((256, 256, 64), 3, O): 29.6, ((256, 224, 64), 3, O): 28.9,
            ((128, 256, 64), 4, O): 21.5, ((128, 128, 64), 4, O): 26.9},
    }
    for (M, N, K), times in measured.items():
        cfg = defaults.choose(M, N, K, tg.F16, tg.F16)
        key = (cfg["block"], cfg["num_stages"], cfg["cta_pair"])
        assert key in times, ((M, N, K), key)
        assert times[key] <= 1.03 * min(times.values()), ((M, N, K), key, times[key], min(times.values()))
        assert tg.tgemm_validate_ex(M, N, K, tg.F16, tg.F16, *cfg["block"], cfg["num_stages"], 232448,
                                    cta_pair=int(cfg["cta_pair"])) == tg.OK


def test_accumulator_count_and_exposed_epilogues():
    from software_pipelined_tiled_02_gb300 import defaults

    # TMEM holds 512 columns; a tile keeps two accumulators when twice its columns fit
    assert defaults.accumulators((256, 256, 64), pair=True) == 2
    assert defaults.accumulators((256, 512, 64), pair=True) == 1      # two N-halves of 256
    assert defaults.accumulators((256, 256, 64), pair=False) == 1     # two M-halves of 256 columns
    assert defaults.accumulators((256, 128, 64), pair=False) == 2
    assert defaults.accumulators((128, 256, 64), pair=False) == 2
    # one accumulator exposes every tile's epilogue, two only the last one
    e = defaults.EPILOGUE_K
    one = defaults.estimate(4096, 4096, 1000, (256, 512, 64), 1.0, pair=True)      # 128 tiles: 2 waves
    two = defaults.estimate(4096, 4096, 1000, (256, 256, 64), 1.0, pair=True)      # 256 tiles: 4 waves
    assert one == 256 * 512 / 2 * (2 * 1000 + 2 * e)
    assert two == 256 * 256 / 2 * (4 * 1000 + 1 * e)

