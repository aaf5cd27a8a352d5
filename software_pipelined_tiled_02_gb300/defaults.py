"""Default tile and depth per problem, frozen from the sweep on GB300.

Chapter 11 "Pipeline and autotuning", section 3.8, recommends writing the
tuned config back as defaults per compute capability and keeping a switch to
turn tuning off.  ``FROZEN`` holds the sweep's winners (``sweep.py`` on a
GB300, compute capability 10.3, 152 SMs) for the measured workloads; other
shapes take the candidate tile with the smallest estimated makespan: whole
waves of persistent tiles (ceil(tiles / SMs)) times the tile's work over its
measured relative throughput.  The estimate only ranks candidates, as the
pages say of cost models; the sweep decides.
"""

from __future__ import annotations

# (M, N, K, operand dtype, out dtype) -> (block, num_stages[, cta_pair[, split_k[, group_m]]]);
# dtype codes 0 f16, 1 bf16, 2 f32; group_m is the persistent raster's group of
# M-blocks (0: the library's 8).  The figures are same-GPU, interleaved
# timings against the runner-up.
FROZEN = {
    (4096, 4096, 4096, 0, 0): ((256, 224, 128), 3, True, 1, 2),  # 1643 vs 1607 for one CTA 256x224x64, group 8
    (8192, 8192, 8192, 1, 1): ((256, 256, 128), 3, True),       # 1753 vs 1692 for one CTA 256x256x64
    (4000, 3000, 5000, 0, 2): ((256, 384, 64), 4, True),        # 94.0 vs 100.1 us for 256x224x64 S6 (96.9 vs 99.0 at S5)
    (512, 512, 32768, 0, 2): ((256, 256, 128), 3, True, 19),    # 514 vs 485 for 128x128x64 S6 split 9; 107 unsplit
    (128, 128, 128, 0, 2): ((128, 128, 32), 3),
}

# Candidate tiles: (block, depth, relative steady-state throughput per SM
# measured at full waves on GB300 with one CTA 256x256 = 1, CTA pair).  A
# pair computes one 256-row tile on two SMs.
CANDIDATES = (
    ((256, 256, 128), 3, 1.04, True),
    ((256, 384, 64), 4, 1.04, True),   # two N = 192 MMAs per k-step; measured on 4000x3000x5000
    ((256, 224, 64), 5, 1.00, True),
    ((256, 256, 64), 3, 1.00, False),
    ((256, 224, 64), 3, 0.98, False),
    ((256, 192, 64), 3, 0.90, False),
    ((128, 256, 64), 4, 0.90, False),
    ((128, 224, 64), 4, 0.86, False),
    ((256, 128, 64), 4, 0.80, False),
    ((128, 128, 64), 4, 0.60, False),
    ((128, 64, 64), 4, 0.35, False),
)

DEFAULT_SMS = 152


def estimate(M: int, N: int, K: int, block, rel: float, num_sms: int = DEFAULT_SMS, pair: bool = False) -> float:
    """Relative makespan of a persistent launch of this tile (arbitrary units).

    A pair works on one tile with two SMs: half as many tiles run at once,
    each in half the time."""
    bm, bn, _ = block
    tiles = -(-M // bm) * -(-N // bn)
    slots = num_sms // 2 if pair else num_sms
    waves = -(-tiles // slots)
    return waves * bm * bn * max(K, 1) / (2 if pair else 1) / rel


def choose(M: int, N: int, K: int, dtype: int, out_dtype: int, num_sms: int = DEFAULT_SMS) -> dict:
    """{block, num_stages, cta_pair, split_k, group_m} for a problem."""
    hit = FROZEN.get((M, N, K, dtype, out_dtype))
    if hit is not None:
        return {"block": hit[0], "num_stages": hit[1], "cta_pair": hit[2] if len(hit) > 2 else False,
                "split_k": hit[3] if len(hit) > 3 else 1, "group_m": hit[4] if len(hit) > 4 else 0}
    best = min(CANDIDATES, key=lambda c: (estimate(M, N, K, c[0], c[2], num_sms, c[3]), -c[2]))
    return {"block": best[0], "num_stages": best[1], "cta_pair": best[3], "split_k": 1, "group_m": 0}
