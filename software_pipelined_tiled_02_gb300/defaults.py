"""Default tile and depth per problem, frozen from the sweep on GB300.

Chapter 11 "Pipeline and autotuning", section 3.8, recommends writing the
tuned config back as defaults per compute capability and keeping a switch to
turn tuning off.  ``FROZEN`` holds the sweep's winners (``sweep.py`` on a
GB300, compute capability 10.3, 152 SMs) for the measured workloads; other
shapes take the candidate tile with the smallest estimated makespan: whole
waves of persistent tiles (ceil(tiles / SMs)) times the tile's work over its
measured relative throughput, plus the epilogues that no MMAs overlap.  The estimate only ranks candidates, as the
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
    # 82.1-82.3 us vs 83.7-84.0 for 256x224x128 S3 (same GPU, two GPUs); groups of 4 82.6-82.8
    (4096, 4096, 4096, 0, 0): dict(block=(256, 224, 64), num_stages=6, cta_pair=True, group_m=2),
    # 612-615 vs 631-633 us for 256x512x64 S4 and 638-641 for 256x448x64 (same GPU, two GPUs)
    (8192, 8192, 8192, 1, 1): dict(block=(256, 256, 64), num_stages=6, cta_pair=True),
    # 144 tiles of 256x352 fill two waves of 76 pairs, or with B shared by two pairs (multicast) 72
    # work items on 36 clusters of four: 82.4 us vs 88.6 for the pairs alone (same GPU), 89.4 for
    # 256x384x64 S4 with multicast, 97-98 for 256x224x64 S6; the 10,000-byte row pitch makes each
    # B row two L2 requests.  Raster groups of 4: 81.1-81.2 us vs 82.1 for 8, 82.2-82.3 for 2
    (4000, 3000, 5000, 0, 2): dict(block=(256, 352, 64), num_stages=5, cta_pair=True, stream_operands=True,
                                   multicast_b=True, group_m=4),
    # 8 tiles x 8 splits = 64 work units on 64 pairs: 29.1-29.3 us vs 29.5-29.6 for 9 splits (72 units),
    # 29.4-29.5 for 256x128x64 S8 split 9, 31.6-31.9 for 256x256x64 S6 split 16 and for one CTA
    # 128x256x64 split 19, 33.2 for 256x256x64 split 19; 9 splits with the reduction after a
    # grid-wide barrier 31.7-31.9; without the evict-first hint 34.6-34.9
    (512, 512, 32768, 0, 2): dict(block=(256, 128, 128), num_stages=4, cta_pair=True, split_k=8,
                                  stream_operands=True),
    (128, 128, 128, 0, 2): dict(block=(128, 128, 32), num_stages=3),
}

DEFAULT_OPTS = dict(cta_pair=False, split_k=1, group_m=0, cluster_k=0, stream_operands=False, grid_reduce=False,
                    stream_k=False, multicast_b=False)

# Candidate tiles: (block, depth, relative steady-state throughput per SM with
# a row pitch that is a multiple of 128 bytes, the same with one that is not,
# CTA pair).  Measured on GB300 at whole waves (76 pair tiles or 152 one-CTA
# tiles, fp16) at K = 16384 and K = 16392, less about 8 us of fixed launch
# cost; TFLOP/s aligned / misaligned: 256x512 pairs 1966 / 1881, 256x448 pairs
# 1952 / 1827, 256x256x64 pairs 1927 / 1612, 256x352 1926 / 1743, 256x384
# 1923 / 1757, one CTA 256x256x64 1953 / 1618, 256x224x64 pairs 1864 / 1520,
# one CTA 256x224x64 1886 / 1534, 128x256 1689 / 1181, 256x192x64 pairs
# 1656 / 1404, 128x128 1017 / 844, 128x64 536 / 484 (re-measured with two
# producer warps: each within 2 %, 256x192 pairs 3 % up).  A misaligned pitch makes
# each 128-byte box row two L2 requests, which narrow tiles (more operand
# rows per output) feel most.  A pair computes one 256-row tile on two SMs.
# The one-CTA 256x224 tile is entered at 0.94 aligned: at K = 1024 and 4096 it
# ran 6 % behind the 256x224x64 pair.  Wide tiles keep one accumulator (no
# epilogue overlap), which their throughput includes.  256x256x128 and
# 256x224x128 pairs (0.95 and 0.89 aligned) are left out: the same tiles at
# block_K = 64 and six stages are faster.
CANDIDATES = (
    ((256, 512, 64), 4, 1.00, 0.96, True),   # two N = 256 MMAs per k-step sharing A
    ((256, 448, 64), 4, 0.99, 0.93, True),
    ((256, 256, 64), 6, 0.98, 0.82, True),
    ((256, 384, 64), 4, 0.98, 0.89, True),
    ((256, 352, 64), 5, 0.98, 0.89, True),   # two N = 176 MMAs per k-step
    ((256, 256, 64), 3, 0.99, 0.82, False),
    ((256, 224, 64), 6, 0.95, 0.77, True),
    ((256, 224, 64), 3, 0.94, 0.78, False),
    ((128, 256, 64), 4, 0.86, 0.60, False),
    ((256, 192, 64), 6, 0.84, 0.71, True),
    ((128, 128, 64), 4, 0.52, 0.43, False),
    ((128, 64, 64), 4, 0.27, 0.25, False),
)

DEFAULT_SMS = 152


# An epilogue that no MMAs overlap costs about as much as this many K-steps of the
# tile's own MMAs (its output and its MMA rate both scale with block_N).  Fitted to
# the timed searches below the tuned table: 6144^3 needs more than 143 to prefer
# 256x256 pairs (2 accumulators) to 256x512 (1), 8192x1024x4096 less than 168 to
# keep 256x512.
EPILOGUE_K = 155


def accumulators(block, pair: bool = False) -> int:
    """Accumulators a tile keeps in TMEM (512 columns): two when twice its
    columns fit, so that a tile's epilogue overlaps the next tile's MMAs."""
    bm, bn, _ = block
    cols = (1 if pair or bm < 256 else 2) * bn
    return 2 if 2 * cols <= 512 else 1


def estimate(M: int, N: int, K: int, block, rel: float, num_sms: int = DEFAULT_SMS, pair: bool = False) -> float:
    """Relative makespan of a persistent launch of this tile (arbitrary units).

    A pair works on one tile with two SMs: half as many tiles run at once,
    each in half the time.  Every tile's epilogue is exposed with one
    accumulator, only the last with two."""
    bm, bn, _ = block
    tiles = -(-M // bm) * -(-N // bn)
    slots = num_sms // 2 if pair else num_sms
    waves = -(-tiles // slots)
    exposed = waves if accumulators(block, pair) == 1 else 1
    return bm * bn / (2 if pair else 1) * (waves * max(K, 1) / rel + EPILOGUE_K * exposed)


# Clusters of four CTAs (two pairs) resident at once on a 152-SM GB300.
CLUSTERS_OF_FOUR = 36


def multicast_pays(M: int, N: int, K: int, block, num_sms: int = DEFAULT_SMS) -> bool:
    """B shared by two pairs (multicast_b) measured faster where a row of the
    16-bit operands is not a whole number of 128-byte L2 lines (each box row is
    then two L2 requests) and the work items, two M-adjacent tiles each, fill
    rounds of the resident clusters of four no worse than the tiles fill
    rounds of pairs: 4000x3000x5000, 82.4 against 88.6 us; 2000x3000x5000,
    46.1 against 47.2 us; 6000x3000x3000 (256x512 tiles), 75.8 either way.
    Where the rounds grow it was slower (4096^3, 256x224x128 tiles: 101.4
    against 83.5 us)."""
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
    col = 2 if (K * 2) % 128 == 0 else 3  # 16-bit operands: a row pitch of 2K bytes
    best = min(CANDIDATES, key=lambda c: (estimate(M, N, K, c[0], c[col], num_sms, c[4]), -c[col]))
    mc = best[4] and multicast_pays(M, N, K, best[0], num_sms)
    return dict(DEFAULT_OPTS, block=best[0], num_stages=best[1], cta_pair=best[4], multicast_b=mc)
