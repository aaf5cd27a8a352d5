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

# (M, N, K, operand dtype, out dtype) -> (block, num_stages[, cta_pair[, split_k]]);
# dtype codes 0 f16, 1 bf16, 2 f32.
FROZEN = {
    (4096, 4096, 4096, 0, 0): ((256, 224, 64), 3),      # 1584 TFLOP/s
    (8192, 8192, 8192, 1, 1): ((256, 256, 64), 3),      # 1849 TFLOP/s
    (4000, 3000, 5000, 0, 2): ((256, 192, 64), 3),      # 988 TFLOP/s
    (512, 512, 32768, 0, 2): ((128, 128, 64), 6, False, 9),  # 484 TFLOP/s; 107 unsplit (16 tiles for 152 SMs)
    (128, 128, 128, 0, 2): ((128, 128, 32), 3),
}

# Candidate tiles with their depth and relative steady-state throughput per
# SM (measured at full waves on GB300, 256x256 = 1).
CANDIDATES = (
    ((256, 256, 64), 3, 1.00),
    ((256, 224, 64), 3, 0.98),
    ((256, 192, 64), 3, 0.90),
    ((128, 256, 64), 4, 0.90),
    ((128, 224, 64), 4, 0.86),
    ((256, 128, 64), 4, 0.80),
    ((128, 128, 64), 4, 0.60),
    ((128, 64, 64), 4, 0.35),
)

DEFAULT_SMS = 152


def estimate(M: int, N: int, K: int, block, rel: float, num_sms: int = DEFAULT_SMS) -> float:
    """Relative makespan of a persistent launch of this tile (arbitrary units)."""
    bm, bn, _ = block
    tiles = -(-M // bm) * -(-N // bn)
    waves = -(-tiles // num_sms)
    return waves * bm * bn * max(K, 1) / rel


def choose(M: int, N: int, K: int, dtype: int, out_dtype: int, num_sms: int = DEFAULT_SMS) -> dict:
    """{block, num_stages, cta_pair, split_k} for a problem."""
    hit = FROZEN.get((M, N, K, dtype, out_dtype))
    if hit is not None:
        return {"block": hit[0], "num_stages": hit[1], "cta_pair": hit[2] if len(hit) > 2 else False,
                "split_k": hit[3] if len(hit) > 3 else 1}
    best = min(CANDIDATES, key=lambda c: (estimate(M, N, K, c[0], c[2], num_sms), -c[2]))
    return {"block": best[0], "num_stages": best[1], "cta_pair": False, "split_k": 1}
