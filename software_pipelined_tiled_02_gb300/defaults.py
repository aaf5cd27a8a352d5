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

# (M, N, K, operand dtype, out dtype) -> launch configuration; dtype codes 0
# f16, 1 bf16, 2 f32.  Keys left out take their defaults (DEFAULT_OPTS):
# cta_pair, split_k (K splits), group_m (the persistent raster's group of
# M-blocks; 0: the library's 8), cluster_k (> 1: K splits reduced inside the
# kernel by clusters of that many CTAs), stream_operands (L2 evict-first
# hint on the operand loads), grid_reduce (K splits reduced in the GEMM
# kernel after a grid-wide barrier) and multicast_b (clusters of two CTA
# pairs that share B through TMA multicast).  The comments give same-GPU, interleaved timings
# against the runner-up.
FROZEN = {
    # 1643 vs 1607 TFLOP/s for one CTA 256x224x64, group 8
    (4096, 4096, 4096, 0, 0): dict(block=(256, 224, 128), num_stages=3, cta_pair=True, group_m=2),
    # 1952-1976 vs 1897-1922 for pair 256x256x128 S3 and 1961-1968 for 256x448x64 (same GPU)
    (8192, 8192, 8192, 1, 1): dict(block=(256, 512, 64), num_stages=4, cta_pair=True),
    # 144 tiles of 256x352 fill two waves of 76 pairs, or with B shared by two pairs (multicast) 72
    # work items on 36 clusters of four: 84.0 us vs 88.9 for the pairs alone (same GPU), 89.1 for
    # 256x384x64 S4 with multicast; the 10,000-byte row pitch makes each B row two L2 requests
    (4000, 3000, 5000, 0, 2): dict(block=(256, 352, 64), num_stages=5, cta_pair=True, stream_operands=True,
                                   multicast_b=True),
    # 31.2 vs 33.3 us without the evict-first hint; 35.4 for 128x128x64 S6 split 9; 166 unsplit;
    # the in-kernel cluster reduction (128x256x64 S4, split 16, clusters of 4) 38.9;
    # the reduction in the GEMM kernel after a grid-wide barrier 33.3
    (512, 512, 32768, 0, 2): dict(block=(256, 256, 128), num_stages=3, cta_pair=True, split_k=19,
                                  stream_operands=True),
    (128, 128, 128, 0, 2): dict(block=(128, 128, 32), num_stages=3),
}

DEFAULT_OPTS = dict(cta_pair=False, split_k=1, group_m=0, cluster_k=0, stream_operands=False, grid_reduce=False,
                    stream_k=False, multicast_b=False)

# Candidate tiles: (block, depth, relative steady-state throughput per SM,
# CTA pair), measured on GB300 at whole waves.  A pair computes one 256-row
# tile on two SMs.  The throughputs follow the operand bytes each SM takes in
# per cycle at the full tensor rate (69 B for pair 256x224, 64 for 256x256, 48
# for 256x512): 4096^3 at 256x224 reaches 0.87 of peak, 8192^3 at 256x256
# 0.97-0.99, 6144^3 at 256x512 1727 against 1706 TFLOP/s for 256x256, and
# 1024x8192x4096 at 256x448 1397 against 1198 for 256x224x64.  Wide tiles keep
# one accumulator (no epilogue overlap), which their throughput includes.
CANDIDATES = (
    ((256, 256, 128), 3, 0.99, True),
    ((256, 512, 64), 4, 1.00, True),   # two N = 256 MMAs per k-step sharing A
    ((256, 448, 64), 4, 1.00, True),
    ((256, 384, 64), 4, 0.98, True),   # measured on 4000x3000x5000
    ((256, 352, 64), 5, 0.97, True),   # two N = 176 MMAs per k-step
    ((256, 224, 128), 3, 0.88, True),
    ((256, 256, 64), 3, 0.95, False),
    ((256, 224, 64), 3, 0.85, False),
    ((128, 256, 64), 4, 0.80, False),
    ((128, 128, 64), 4, 0.55, False),
    ((128, 64, 64), 4, 0.32, False),
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


# Clusters of four CTAs (two pairs) resident at once on a 152-SM GB300.
CLUSTERS_OF_FOUR = 36


def multicast_pays(M: int, N: int, K: int, block, num_sms: int = DEFAULT_SMS) -> bool:
    """B shared by two pairs (multicast_b) measured faster where a row of the
    16-bit operands is not a whole number of 128-byte L2 lines (each box row is
    then two L2 requests) and the work items, two M-adjacent tiles each, fill
    rounds of the resident clusters of four no worse than the tiles fill
    rounds of pairs: 4000x3000x5000, 83.9 against 88.3 us; 2000x3000x5000,
    46.1 against 47.2 us; 6000x3000x3000 (256x512 tiles), 75.8 either way.
    Where the rounds grow it was slower (4096^3: 104 against 84 us)."""
    if (K * 2) % 128 == 0:
        return False
    bm, bn, _ = block
    tiles_m, tiles_n = -(-M // bm), -(-N // bn)
    clusters = max(1, CLUSTERS_OF_FOUR * num_sms // DEFAULT_SMS)
    pair_rounds = -(-(tiles_m * tiles_n) // (num_sms // 2))
    mc_rounds = -(-(-(-tiles_m // 2) * tiles_n) // clusters)
    return mc_rounds <= pair_rounds


def choose(M: int, N: int, K: int, dtype: int, out_dtype: int, num_sms: int = DEFAULT_SMS) -> dict:
    """{block, num_stages, cta_pair, split_k, group_m, cluster_k, stream_operands, grid_reduce, stream_k,
    multicast_b} for a problem."""
    hit = FROZEN.get((M, N, K, dtype, out_dtype))
    if hit is not None:
        return dict(DEFAULT_OPTS, **hit)
    best = min(CANDIDATES, key=lambda c: (estimate(M, N, K, c[0], c[2], num_sms, c[3]), -c[2]))
    mc = best[3] and multicast_pays(M, N, K, best[0], num_sms)
    return dict(DEFAULT_OPTS, block=best[0], num_stages=best[1], cta_pair=best[3], multicast_b=mc)
