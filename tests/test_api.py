"""Host-side tests of the C ABI: loading, exports, validation, budget.

No kernel is launched and no GPU is needed: these call only the functions
that are pure host logic, plus tgemm_plan on a machine without a device
(which must fail with a status, not crash).
"""

import itertools
import os
import re

import pytest
import torch

import oracle
import software_pipelined_tiled_02_gb300 as tg
from software_pipelined_tiled_02_gb300 import build as tbuild
from tests.conftest import ROOT, golden_lines

LIMIT_227K = 227 * 1024  # cudaDevAttrMaxSharedMemoryPerBlockOptin on sm_100/sm_103
PAGES_BUDGET = 228 * 1024


@pytest.fixture(scope="module")
def lib():
    tbuild.build()
    return tg.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "tgemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tgemm_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function(lib):
    declared = header_functions()
    assert len(declared) >= 13
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/tgemm.h but not exported"
    assert sorted(tg.SYMBOLS) == declared


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "tgemm.h"

int main(void)
{
    /* pair, group, split, prefetch, cluster, stream, grid, stream-K, multicast B */
    tgemm_plan_opts opts = {1, 2, 1, 0, 0, 0, 0, 0, 0};
    int64_t bound = tgemm_smem_bound(TGEMM_F16, 128, 128, 32, 3);
    int one = tgemm_validate(4096, 4096, 4096, TGEMM_F16, TGEMM_F16, 256, 224, 64, 3, 232448);
    int pair = tgemm_validate_ex(4096, 4096, 4096, TGEMM_F16, TGEMM_F16, 256, 224, 128, 3, 232448, &opts);
    int over = tgemm_validate(4000, 3000, 5000, TGEMM_F16, TGEMM_F32, 256, 256, 64, 4, 232448);
    const char *msg = tgemm_strerror(TGEMM_ERR_SMEM_BUDGET);
    printf("%lld %d %d %d %s\n", (long long)bound, one, pair, over, msg);
    return bound == 3 * (128 * 32 + 32 * 128) * 2 && one == TGEMM_OK && pair == TGEMM_OK &&
                   over == TGEMM_ERR_SMEM_BUDGET && strlen(msg) > 0
               ? 0
               : 1;
}
"""


def test_header_is_c_and_links(lib, tmp_path):
    """The public header compiles as strict C99 and a C program links and calls the library."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(tg.LIB_PATH)
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-L", libdir, "-ltgemm", "-Wl,-rpath," + libdir, "-o", str(exe)]
    out = subprocess.run(cmd, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr


def test_strerror_covers_every_code(lib):
    texts = {tg.strerror(c) for c in range(9)}
    assert len(texts) == 9
    assert tg.strerror(99) == "unknown status code"
    assert tg.strerror(-tg.ERR_CUDA) == tg.strerror(tg.ERR_CUDA)


def test_smem_bound_matches_oracle_and_pages(lib):
    # The library's bound and the oracle's are separate code; the pages'
    # printed values pin both.
    for t in golden_lines("smem_budget.txt"):
        if t[0] == "tile":
            bm, bn, bk, eb, per, _ = map(int, t[1:])
            assert tg.tgemm_smem_bound(tg.F16, bm, bn, bk, 1) == per
    for bm, bn, bk, s in itertools.product((64, 128, 256), (32, 64, 128, 256), (16, 32, 64), (1, 2, 3, 4, 6, 8)):
        for dt in (tg.F16, tg.BF16):
            assert tg.tgemm_smem_bound(dt, bm, bn, bk, s) == oracle.smem_bound(bm, bn, bk, s, 2)


def test_smem_bytes_cover_the_bound(lib):
    for bm, bn, bk, s in itertools.product((128, 256), (32, 64, 96, 128, 256), (16, 32, 64), (1, 2, 3, 4, 6)):
        for out in (tg.F16, tg.F32):
            b = tg.tgemm_smem_bytes(tg.F16, out, bm, bn, bk, s)
            assert b >= tg.tgemm_smem_bound(tg.F16, bm, bn, bk, s)
            assert b % 16 == 0 or b > 0


def test_over_budget_config_rejected(lib):
    # 256x256x64 at num_stages = 4 needs 256 KiB (chapter 11 section 4.5): it
    # must be rejected before anything is launched, at the GB300 limit and at
    # the pages' 228 KiB figure; 3 stages fit the bound.
    for limit in (LIMIT_227K, PAGES_BUDGET):
        assert tg.tgemm_validate(4000, 3000, 5000, tg.F16, tg.F32, 256, 256, 64, 4, limit) == tg.ERR_SMEM_BUDGET
    assert tg.tgemm_smem_bound(tg.F16, 256, 256, 64, 3) <= LIMIT_227K


def test_validate_rules(lib):
    V = tg.tgemm_validate
    L = LIMIT_227K
    assert V(128, 128, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.OK
    assert V(4096, 4096, 4096, tg.F16, tg.F16, 128, 256, 64, 4, L) == tg.OK
    assert V(8192, 8192, 8192, tg.BF16, tg.BF16, 128, 256, 64, 4, L) == tg.OK
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 128, 64, 6, L) == tg.OK
    # dtypes
    assert V(128, 128, 128, tg.F32, tg.F32, 128, 128, 32, 3, L) == tg.ERR_UNSUPPORTED_DTYPE
    assert V(128, 128, 128, tg.F16, tg.BF16, 128, 128, 32, 3, L) == tg.ERR_UNSUPPORTED_DTYPE
    assert V(128, 128, 128, 7, tg.F32, 128, 128, 32, 3, L) == tg.ERR_UNSUPPORTED_DTYPE
    # sizes and depth
    assert V(-1, 128, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.ERR_INVALID_ARG
    assert V(128, 128, -8, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.ERR_INVALID_ARG
    assert V(2 ** 31, 128, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.ERR_INVALID_ARG
    # tile-rounded coordinates must stay 32-bit: 2^31 - 257 is the largest M, N or K
    big = 2 ** 31 - 257
    assert V(big - 7, 128, 128, tg.F16, tg.F32, 256, 128, 32, 3, L) == tg.OK
    assert V(big + 7, 128, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.ERR_INVALID_ARG
    assert V(128, big - 3, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.OK
    assert V(128, big + 5, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.ERR_INVALID_ARG
    assert V(128, 128, big - 7, tg.F16, tg.F32, 128, 128, 128, 3, L) == tg.OK
    assert V(128, 128, big + 9, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.ERR_INVALID_ARG
    # at most 2^30 output tiles: a 2^22 x 2^23 C in 128 x 32 tiles is 2^15 x 2^18 = 2^33 tiles
    assert V(2 ** 22, 2 ** 23, 64, tg.F16, tg.F32, 128, 32, 32, 3, L) == tg.ERR_INVALID_ARG
    assert V(2 ** 22, 2 ** 20, 64, tg.F16, tg.F32, 128, 32, 32, 3, L) == tg.OK  # 2^15 x 2^15 tiles
    assert V(128, 128, 128, tg.F16, tg.F32, 128, 128, 32, 0, L) == tg.ERR_INVALID_ARG
    # empty products and the empty reduction are valid
    assert V(0, 128, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.OK
    assert V(128, 0, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.OK
    assert V(128, 128, 0, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.OK
    # row pitch must be 16-byte aligned for the TMA engine
    assert V(128, 128, 12, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.ERR_ALIGNMENT
    assert V(128, 130, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.ERR_ALIGNMENT
    assert V(128, 132, 128, tg.F16, tg.F32, 128, 128, 32, 3, L) == tg.OK      # 528-byte fp32 rows
    assert V(128, 132, 128, tg.F16, tg.F16, 128, 128, 32, 3, L) == tg.ERR_ALIGNMENT  # 264-byte fp16 rows
    # tile shapes the kernel implements
    assert V(128, 128, 128, tg.F16, tg.F32, 64, 128, 32, 3, L) == tg.OK  # M = 64 instructions
    assert V(128, 128, 128, tg.F16, tg.F32, 96, 128, 32, 3, L) == tg.ERR_NO_KERNEL
    assert V(128, 128, 128, tg.F16, tg.F32, 32, 128, 32, 3, L) == tg.ERR_NO_KERNEL
    assert V(128, 128, 128, tg.F16, tg.F32, 128, 48, 32, 3, L) == tg.ERR_NO_KERNEL
    assert V(128, 128, 128, tg.F16, tg.F32, 128, 512, 32, 3, L) == tg.ERR_NO_KERNEL
    assert V(128, 128, 128, tg.F16, tg.F32, 128, 128, 128, 1, L) == tg.OK  # two 64-wide K-panels per slot
    assert V(128, 128, 256, tg.F16, tg.F32, 128, 128, 256, 1, L) == tg.ERR_NO_KERNEL
    assert V(128, 128, 128, tg.F16, tg.F32, 128, 128, 8, 3, L) == tg.ERR_NO_KERNEL
    # depth is bounded only by the budget
    assert V(128, 128, 128, tg.F16, tg.F32, 128, 128, 32, 12, L) == tg.OK
    assert V(128, 128, 128, tg.F16, tg.F32, 128, 128, 32, 14, L) == tg.ERR_SMEM_BUDGET
    assert V(128, 128, 128, tg.F16, tg.F32, 128, 128, 32, 10 ** 6, L) == tg.ERR_SMEM_BUDGET


def test_validate_ex_options(lib):
    V = tg.tgemm_validate_ex
    L = LIMIT_227K
    # CTA pairs need 256-row tiles; each CTA of the pair is a block for the budget
    assert V(4096, 4096, 4096, tg.F16, tg.F16, 256, 224, 128, 3, L, cta_pair=1) == tg.OK
    assert V(4096, 4096, 4096, tg.F16, tg.F16, 128, 224, 64, 3, L, cta_pair=1) == tg.ERR_NO_KERNEL
    # split-K: at most 64 splits, and fp32 partial staging counts against the budget
    assert V(512, 512, 32768, tg.F16, tg.F32, 256, 256, 128, 3, L, cta_pair=1, split_k=19) == tg.OK
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 128, 64, 4, L, split_k=65) == tg.ERR_INVALID_ARG
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 128, 64, 4, L, split_k=-1) == tg.ERR_INVALID_ARG
    # the workspace row of split s (s * ceil(M / bm) * bm + r) must stay a 32-bit coordinate
    M = 2 ** 26
    assert V(M, 4, 64 * 32, tg.F16, tg.F32, 128, 32, 32, 4, L, split_k=31) == tg.OK      # 31 * 2^26 < 2^31
    assert V(M, 4, 64 * 32, tg.F16, tg.F32, 128, 32, 32, 4, L, split_k=32) == tg.ERR_INVALID_ARG
    # option ranges, as tgemm_plan_ex checks them
    assert V(512, 512, 512, tg.F16, tg.F32, 128, 128, 64, 4, L, cta_pair=2) == tg.ERR_INVALID_ARG
    assert V(512, 512, 512, tg.F16, tg.F32, 128, 128, 64, 4, L, group_m=-1) == tg.ERR_INVALID_ARG
    assert V(512, 512, 512, tg.F16, tg.F32, 128, 128, 64, 4, L, group_m=4097) == tg.ERR_INVALID_ARG
    assert V(512, 512, 512, tg.F16, tg.F32, 128, 128, 64, 4, L, prefetch=5) == tg.ERR_INVALID_ARG
    assert V(512, 512, 512, tg.F16, tg.F32, 128, 128, 64, 4, L, prefetch=4) == tg.OK
    # a split count above the number of k-blocks is cut down first, so it is not an error
    assert V(M, 4, 2 * 32, tg.F16, tg.F32, 128, 32, 32, 4, L, split_k=64) == tg.OK


def test_validate_ex_stream_operands_and_grid_reduce(lib):
    V = tg.tgemm_validate_ex
    for v, want in ((0, tg.OK), (1, tg.OK), (2, tg.ERR_INVALID_ARG), (-1, tg.ERR_INVALID_ARG)):
        assert V(512, 512, 512, tg.F16, tg.F32, 128, 128, 64, 4, LIMIT_227K, stream_operands=v) == want
        assert V(512, 512, 512, tg.F16, tg.F32, 128, 128, 64, 4, LIMIT_227K, split_k=4, grid_reduce=v) == want


def test_validate_ex_stream_k_rules(lib):
    V = tg.tgemm_validate_ex
    L = LIMIT_227K
    assert V(4000, 3000, 5000, tg.F16, tg.F32, 256, 352, 64, 5, L, cta_pair=1, stream_k=1) == tg.OK
    assert V(4000, 3000, 5000, tg.F16, tg.F32, 256, 352, 64, 5, L, cta_pair=1, stream_k=2) == tg.ERR_INVALID_ARG
    # the tail is shared by k-blocks: not combined with a K split or the cluster reduction
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 256, 64, 4, L, split_k=2, stream_k=1) == tg.ERR_INVALID_ARG
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 256, 64, 4, L, split_k=8, cluster_k=4,
             stream_k=1) == tg.ERR_INVALID_ARG


def test_validate_ex_multicast_rules(lib):
    V = tg.tgemm_validate_ex
    L = LIMIT_227K
    assert V(4000, 3000, 5000, tg.F16, tg.F32, 256, 352, 64, 5, L, cta_pair=1, multicast_b=1) == tg.OK
    assert V(4000, 3000, 5000, tg.F16, tg.F32, 256, 352, 64, 5, L, cta_pair=1, multicast_b=2) == tg.ERR_INVALID_ARG
    # two CTA pairs per cluster: pairs only, one K split, no stream-K tail or in-kernel reduction
    assert V(4000, 3000, 5000, tg.F16, tg.F32, 256, 352, 64, 5, L, multicast_b=1) == tg.ERR_INVALID_ARG
    assert V(512, 512, 32768, tg.F16, tg.F32, 256, 256, 128, 3, L, cta_pair=1, split_k=19,
             multicast_b=1) == tg.ERR_INVALID_ARG
    assert V(512, 512, 32768, tg.F16, tg.F32, 256, 256, 128, 3, L, cta_pair=1, split_k=1, multicast_b=1) == tg.OK
    assert V(4000, 3000, 5000, tg.F16, tg.F32, 256, 352, 64, 5, L, cta_pair=1, stream_k=1,
             multicast_b=1) == tg.ERR_INVALID_ARG
    assert V(512, 512, 4096, tg.F16, tg.F32, 256, 256, 64, 4, L, cta_pair=1, split_k=2, grid_reduce=1,
             multicast_b=1) == tg.ERR_INVALID_ARG
    # the smallest pair tile: a 16-row B box in two 8-row parts
    assert V(512, 64, 512, tg.F16, tg.F16, 256, 32, 64, 4, L, cta_pair=1, multicast_b=1) == tg.OK
    # the second tile of the last cluster may lie one 256-row block past M: M stays 512 below the limit
    big = (1 << 31) - 1 - 256
    assert V(big - 512, 64, 64, tg.F16, tg.F16, 256, 32, 64, 4, L, cta_pair=1, multicast_b=1) == tg.OK
    assert V(big - 511, 64, 64, tg.F16, tg.F16, 256, 32, 64, 4, L, cta_pair=1, multicast_b=1) == tg.ERR_INVALID_ARG
    assert V(big - 511, 64, 64, tg.F16, tg.F16, 256, 32, 64, 4, L, cta_pair=1) == tg.OK


def stream_k_tail(T, G, KB):
    """The stream-K tail as the header states it: tiles past the last whole
    wave of G workers, if each worker gets at least two of their k-blocks;
    worker w takes iterations [I*w/G, I*(w+1)/G) of the I = R*KB total."""
    R = T % G
    if R == 0 or R * KB < 2 * G:
        return None
    I = R * KB
    return [(I * w // G, I * (w + 1) // G) for w in range(G)]


def test_stream_k_tail_partition_by_brute_force():
    # Every tail tile is covered exactly once, in k order, by consecutive
    # workers; no worker touches more than two tail tiles; the kernel's closed
    # forms for a tile's first and last worker (ceil(G*(t*KB+1)/I) - 1 and
    # ceil(G*(t+1)*KB/I) - 1) agree with a search.
    for G in (1, 3, 76, 152):
        for T in range(1, 330, 7):
            for KB in (1, 2, 5, 33, 79, 128):
                ranges = stream_k_tail(T, G, KB)
                if ranges is None:
                    continue
                R, I = T % G, (T % G) * KB
                owners = {}
                for w, (s0, s1) in enumerate(ranges):
                    if s0 < s1:
                        assert (s1 - 1) // KB - s0 // KB <= 1
                    for k in range(s0, s1):
                        owners.setdefault(k // KB, []).append((w, k % KB))
                for t in range(R):
                    ks = [k for _, k in owners[t]]
                    assert ks == list(range(KB))
                    ws = [w for w, _ in owners[t]]
                    assert ws == sorted(ws)
                    assert -(-(G * (t * KB + 1)) // I) - 1 == ws[0]
                    assert -(-(G * (t + 1) * KB) // I) - 1 == ws[-1]


def test_validate_ex_cluster_k_rules(lib):
    # Splits reduced inside the kernel by clusters of cluster_k CTAs.
    V = tg.tgemm_validate_ex
    L = LIMIT_227K
    ok = dict(split_k=16, cluster_k=4)
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 256, 64, 4, L, **ok) == tg.OK
    assert V(512, 512, 32768, tg.F16, tg.F16, 128, 256, 64, 4, L, **ok) == tg.OK
    for c in (0, 1, 2, 4, 8):
        assert V(512, 512, 32768, tg.F16, tg.F32, 128, 256, 64, 4, L, split_k=16, cluster_k=c) == tg.OK
    for c in (3, 5, 16, -1):  # only 2, 4 and 8 (portable cluster sizes) or off
        assert V(512, 512, 32768, tg.F16, tg.F32, 128, 256, 64, 4, L, split_k=16, cluster_k=c) == tg.ERR_INVALID_ARG
    # one CTA per 128-row tile only
    assert V(512, 512, 32768, tg.F16, tg.F32, 256, 256, 128, 3, L, cta_pair=1, **ok) == tg.ERR_INVALID_ARG
    assert V(512, 512, 32768, tg.F16, tg.F32, 256, 128, 64, 3, L, **ok) == tg.ERR_INVALID_ARG
    # a whole number of clusters per tile, after the split count is cut to the k-blocks
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 256, 64, 4, L, split_k=18, cluster_k=4) == tg.ERR_INVALID_ARG
    assert V(512, 512, 64 * 6, tg.F16, tg.F32, 128, 256, 64, 4, L, split_k=8, cluster_k=4) == tg.ERR_INVALID_ARG
    assert V(512, 512, 64 * 8, tg.F16, tg.F32, 128, 256, 64, 4, L, split_k=8, cluster_k=4) == tg.OK
    # slices of block_N / cluster_k columns must be whole 32-column chunks
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 128, 64, 4, L, split_k=16, cluster_k=8) == tg.ERR_INVALID_ARG
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 96, 64, 4, L, split_k=16, cluster_k=2) == tg.ERR_INVALID_ARG
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 224, 64, 4, L, split_k=16, cluster_k=2) == tg.ERR_INVALID_ARG
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 192, 64, 4, L, split_k=16, cluster_k=2) == tg.OK  # 96
    # the exchanged partials (128 x block_N x 4 bytes) must fit the operand ring
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 256, 64, 2, L, **ok) == tg.ERR_SMEM_BUDGET  # 96 KB < 128 KB
    assert V(512, 512, 32768, tg.F16, tg.F32, 128, 256, 64, 3, L, **ok) == tg.OK              # 144 KB


def test_budget_rule_agrees_with_oracle_over_the_grid(lib):
    # Whatever the real footprint adds, a config whose pages' bound exceeds
    # the limit is always rejected, and the rejection is monotone in depth.
    for bm, bn, bk in itertools.product((128, 256), (64, 128, 256), (16, 32, 64)):
        prev_ok = True
        for s in range(1, 16):
            rc = tg.tgemm_validate(4096, 4096, 4096, tg.F16, tg.F16, bm, bn, bk, s, LIMIT_227K)
            if oracle.smem_bound(bm, bn, bk, s, 2) > LIMIT_227K:
                assert rc == tg.ERR_SMEM_BUDGET
            assert rc in (tg.OK, tg.ERR_SMEM_BUDGET)
            if not prev_ok:
                assert rc == tg.ERR_SMEM_BUDGET
            prev_ok = rc == tg.OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_plan_without_device_fails_cleanly(lib):
    rc, h = tg.tgemm_plan(128, 128, 128, tg.F16, tg.F32, 128, 128, 32, 3)
    assert rc == tg.ERR_CUDA and h is None
    # argument errors are reported before any device query
    rc, h = tg.tgemm_plan(128, 128, 128, tg.F16, tg.F32, 128, 128, 32, 0)
    assert rc == tg.ERR_INVALID_ARG and h is None
    rc, h = tg.tgemm_plan(128, 128, 128, tg.F16, tg.F32, 96, 128, 32, 2)
    assert rc == tg.ERR_NO_KERNEL and h is None
    assert tg.tgemm_smem_limit() < 0
    assert tg.tgemm_destroy(None) == tg.OK


def test_null_plan_arguments(lib):
    assert lib.tgemm_run(None, None, None, None, None) == tg.ERR_INVALID_ARG
    assert lib.tgemm_status(None, None) == tg.ERR_INVALID_ARG
    assert lib.tgemm_get_plan_info(None, None) == tg.ERR_INVALID_ARG
    assert lib.tgemm_plan(None, 1, 1, 8, 0, 2, 128, 128, 32, 1) == tg.ERR_INVALID_ARG


def test_missing_library_raises(tmp_path):
    with pytest.raises(RuntimeError):
        tg._lib_saved = tg._lib
        tg._lib = None
        try:
            tg.load(str(tmp_path / "nope.so"))
        finally:
            tg._lib = tg._lib_saved
