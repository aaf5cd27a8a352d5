"""A seeded random sweep of shapes and launch configurations against the oracle.

Each case draws operand and output dtypes, a ragged shape (the only
constraint is the 16-byte row-pitch rule), a tile, a depth the shared memory
admits, CTA pairs, a K split, a producer lead and a raster group.  It then compares the
kernel's C with the fp64 oracle element by element, to the tolerance of
oracle.check.  The draws come from one fixed seed, so a failure names a
reproducible case.
"""

import os

import numpy as np
import pytest
import torch

import oracle
from software_pipelined_tiled_02_gb300 import inputs

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
SINGLE_TILES = [(128, 128, 32), (128, 256, 64), (256, 128, 64), (128, 64, 16), (256, 224, 64), (128, 128, 128),
                (256, 96, 128), (128, 32, 64), (256, 256, 64), (128, 192, 64), (64, 128, 32), (64, 256, 64),
                (64, 64, 128)]
PAIR_TILES = [(256, 256, 128), (256, 224, 128), (256, 256, 64), (256, 128, 32), (256, 64, 16), (256, 32, 64),
              (256, 192, 128), (256, 160, 64), (256, 512, 64), (256, 448, 128), (256, 384, 64), (256, 320, 32),
              (256, 352, 64), (256, 416, 128), (256, 480, 32)]
N_CASES = int(os.environ.get("TGEMM_SWEEP_CASES", "400"))  # more for a longer soak
SEED = int(os.environ.get("TGEMM_SWEEP_SEED", "20261202"))   # another seed draws other cases


def draw_cases(tg, n=N_CASES, seed=SEED):
    rng = np.random.default_rng(seed)
    limit = tg.tgemm_smem_limit()
    cases = []
    while len(cases) < n:
        dtype = str(rng.choice(["f16", "bf16"]))
        out = str(rng.choice(["f32", dtype]))
        pair = bool(rng.random() < 0.35)
        block = PAIR_TILES[rng.integers(len(PAIR_TILES))] if pair else SINGLE_TILES[rng.integers(len(SINGLE_TILES))]
        M = int(rng.integers(1, 521))
        n_align = 4 if out == "f32" else 8
        N = int(rng.integers(1, 521 // n_align + 1)) * n_align
        K = int(rng.integers(1, 1041 // 8 + 1)) * 8
        split = int(rng.choice([1, 1, 1, 2, 3, 4, 5, 8]))
        stages = int(rng.integers(1, 9))
        cluster = int(rng.choice([0, 0, 0, 2, 4]))  # K splits reduced inside the kernel
        stream = int(rng.random() < 0.3)            # L2 evict-first operand loads
        mcast = int(pair and rng.random() < 0.3)    # two pairs sharing B through multicast
        if mcast:
            split, cluster = 1, 0                   # it takes neither a K split nor the cluster reduction
        if tg.tgemm_validate_ex(M, N, K, dtype, out, *block, stages, limit, cta_pair=int(pair),
                                split_k=split, cluster_k=cluster, stream_operands=stream, multicast_b=mcast) != tg.OK:
            continue
        prefetch = int(rng.integers(1, stages + 1)) if rng.random() < 0.25 else 0
        group = int(rng.choice([0, 0, 1, 2, 3, 16]))
        cases.append((M, N, K, dtype, out, block, stages, pair, split, prefetch, group, cluster, stream, mcast,
                      int(rng.integers(1 << 30))))
    return cases


def test_random_sweep_matches_oracle(cuda_lib):
    tg = cuda_lib
    failures = []
    for i, case in enumerate(draw_cases(tg)):
        M, N, K, dtype, out, block, stages, pair, split, prefetch, group, cluster, stream, mcast, seed = case
        A, B = inputs.operands(seed, M, N, K, dtype, "normal")
        plan = tg.Plan(M, N, K, dtype, out, block, stages, pair=pair, split_k=split, prefetch=prefetch,
                       group_m=group, cluster_k=cluster, stream_operands=stream, multicast_b=mcast)
        C = torch.full((M, N), float("nan"), dtype=TORCH[out], device="cuda")
        plan.run(inputs.bits_to_torch(A, dtype).cuda(), inputs.bits_to_torch(B, dtype).cuda(), C)
        torch.cuda.synchronize()
        code = plan.status()[0]
        plan.close()
        R, S = oracle.gemm(A, B, dtype)
        ok, worst, idx = oracle.check(C.float().cpu().double().numpy(), R, S, out)
        if code != 0 or not ok:
            failures.append((i, case, code, worst))
    assert not failures, failures
