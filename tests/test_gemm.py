"""GPU parity: the sm_103a kernel against the CPU oracle, element by element.

Acceptance (oracle.check): |C - R| <= 1e-4 * S + 1e-5 (+ one output ulp for
16-bit output) and the pages' rtol = atol = 1e-2; integer-valued inputs must
match exactly.  Small problems are compared in full; the full-size workloads
are compared on sampled entries (whole first/last rows and columns plus
random entries) that the oracle computes one by one; the pages' workloads
are compared in full, in the launch configuration the benchmark times.
"""

import numpy as np
import pytest
import torch

import oracle
from software_pipelined_tiled_02_gb300 import inputs

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def to_dev(bits, dtype):
    return inputs.bits_to_torch(bits, dtype).cuda()


def run(tg, A, B, dtype, out, block, stages, pair=False, split_k=1, group_m=0, cluster_k=0, stream_operands=False,
        multicast_b=False):
    M, K = A.shape
    N = B.shape[0]
    plan = tg.Plan(M, N, K, dtype, out, block, stages, pair=pair, split_k=split_k, group_m=group_m,
                   cluster_k=cluster_k, stream_operands=stream_operands, multicast_b=multicast_b)
    dA, dB = to_dev(A, dtype), to_dev(B, dtype)
    C = torch.full((M, N), float("nan"), dtype=TORCH[out], device="cuda")
    plan.run(dA, dB, C)
    torch.cuda.synchronize()
    rc, detail = plan.status()
    assert rc == 0, f"kernel status {rc} {detail}"
    plan.close()
    return C


def as_f64(C):
    return C.float().cpu().double().numpy()


def assert_close(C, R, S, out):
    ok, worst, idx = oracle.check(C, R, S, out)
    assert ok, f"worst error/bound {worst:.3g} at flat index {idx}: got {np.ravel(C)[idx]!r} want {np.ravel(R)[idx]!r}"


# ------------------------------------------------------------ small, full compare

def test_gemm_128_f16_uniform_tile_128x128x32_s3(cuda_lib):
    w = inputs.WORKLOADS["gemm_128_f16_uniform"]
    A, B = inputs.workload_operands("gemm_128_f16_uniform")
    C = as_f64(run(cuda_lib, A, B, "f16", "f32", w["tile"], w["stages"]))
    R, S = oracle.gemm(A, B, "f16")
    assert_close(C, R, S, "f32")


CONFIGS = [
    ((64, 128, 32), 3),     # M = 64 instructions: 16 accumulator rows per TMEM lane quarter
    ((64, 256, 64), 4),
    ((64, 64, 16), 2),
    ((64, 96, 128), 3),
    ((128, 128, 32), 3),
    ((128, 256, 64), 4),
    ((256, 128, 64), 3),
    ((128, 64, 16), 2),
    ((128, 96, 32), 1),
    ((256, 256, 64), 3),
    ((128, 32, 64), 5),
    ((128, 128, 128), 3),
    ((256, 96, 128), 2),
]
SHAPES = [(300, 200, 136), (257, 96, 72), (129, 264, 1032), (1, 32, 8), (64, 512, 16)]


@pytest.mark.parametrize("block,stages", CONFIGS, ids=lambda v: str(v))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype,out", [("f16", "f32"), ("bf16", "bf16"), ("f16", "f16"), ("bf16", "f32")])
def test_small_shapes_all_tiles(cuda_lib, block, stages, shape, dtype, out):
    M, N, K = shape
    A, B = inputs.operands(100 + M + N + K, M, N, K, dtype, "uniform")
    C = as_f64(run(cuda_lib, A, B, dtype, out, block, stages))
    R, S = oracle.gemm(A, B, dtype)
    assert_close(C, R, S, out)


@pytest.mark.parametrize("block,stages", CONFIGS, ids=lambda v: str(v))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_integer_inputs_bit_exact(cuda_lib, block, stages, dtype):
    M, N, K = 300, 520, 2056
    A, B = inputs.operands(40, M, N, K, dtype, "int", lo=-4, hi=4)
    C = as_f64(run(cuda_lib, A, B, dtype, "f32", block, stages))
    R, _ = oracle.gemm(A, B, dtype)
    assert np.array_equal(C, R)


# ------------------------------------------------------------ CTA-pair mode

PAIR_CONFIGS = [
    ((256, 512, 64), 4),     # two N = 256 MMAs per k-step sharing A
    ((256, 384, 128), 2),    # two N = 192 MMAs, two K-panels per slot
    ((256, 352, 64), 4),     # two N = 176 MMAs: 88 B rows per CTA and N-half
    ((256, 288, 32), 5),     # two N = 144 MMAs
    ((256, 256, 128), 3),
    ((256, 224, 128), 3),
    ((256, 256, 64), 4),
    ((256, 224, 64), 6),
    ((256, 128, 32), 3),
    ((256, 64, 16), 2),
    ((256, 32, 64), 1),
]


@pytest.mark.parametrize("block,stages", PAIR_CONFIGS, ids=lambda v: str(v))
@pytest.mark.parametrize("shape", SHAPES + [(520, 704, 264)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype,out", [("f16", "f32"), ("bf16", "bf16"), ("f16", "f16")])
def test_pair_small_shapes(cuda_lib, block, stages, shape, dtype, out):
    M, N, K = shape
    A, B = inputs.operands(200 + M + N + K, M, N, K, dtype, "uniform")
    C = as_f64(run(cuda_lib, A, B, dtype, out, block, stages, pair=True))
    R, S = oracle.gemm(A, B, dtype)
    assert_close(C, R, S, out)


@pytest.mark.parametrize("block,stages", PAIR_CONFIGS, ids=lambda v: str(v))
def test_pair_integer_inputs_bit_exact(cuda_lib, block, stages):
    M, N, K = 600, 520, 2056
    A, B = inputs.operands(41, M, N, K, "bf16", "int", lo=-4, hi=4)
    C = as_f64(run(cuda_lib, A, B, "bf16", "f32", block, stages, pair=True))
    R, _ = oracle.gemm(A, B, "bf16")
    assert np.array_equal(C, R)


def test_pair_matches_single_cta_bitwise(cuda_lib):
    # The pair issues the same K-ordered MMAs over the same tile as one CTA
    # with two M-halves; the fp32 accumulation must come out bit for bit.
    M, N, K = 1024, 1024, 1024
    A, B = inputs.operands(42, M, N, K, "f16", "normal")
    one = run(cuda_lib, A, B, "f16", "f32", (256, 128, 64), 3, pair=False)
    two = run(cuda_lib, A, B, "f16", "f32", (256, 128, 64), 3, pair=True)
    assert torch.equal(one.view(torch.int32), two.view(torch.int32))


def test_pair_rejects_other_block_m(cuda_lib):
    rc, h = cuda_lib.tgemm_plan_ex(512, 512, 512, "f16", "f32", 128, 128, 64, 3, cta_pair=1)
    assert rc == cuda_lib.ERR_NO_KERNEL and h is None
    rc, h = cuda_lib.tgemm_plan_ex(512, 512, 512, "f16", "f32", 256, 128, 64, 3, cta_pair=2)
    assert rc == cuda_lib.ERR_INVALID_ARG and h is None


@pytest.mark.parametrize("name,block,stages", [("gemm_4096_f16_normal", (256, 256, 64), 6),
                                               ("gemm_8192_bf16_normal", (256, 224, 64), 6)])
def test_pair_full_size_sampled(cuda_lib, name, block, stages):
    w, A, B, C = full_size(cuda_lib, name, block, stages, pair=True)
    rows, cols = sample_entries(w["M"], w["N"], 4096, 6)
    R, S = oracle.gemm_entries(A, B, w["dtype"], rows, cols)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    assert_close(as_f64(got), R, S, w["out"])


# ------------------------------------------------------------ two pairs sharing B (multicast)

MCAST_CONFIGS = [
    ((256, 352, 64), 5),     # a CTA's 88 B rows per N-half in multicast parts of 48 and 40
    ((256, 512, 64), 4),
    ((256, 384, 128), 2),    # two K-panels per slot
    ((256, 256, 64), 4),
    ((256, 224, 128), 3),    # parts of 56 and 56
    ((256, 64, 16), 2),      # a 32-row box: parts of 16 and 16
    ((256, 32, 64), 1),      # the smallest box (16 rows), a one-slot ring
]
# tiles_m odd (the cluster's second tile lies past M), one M-block, ragged edges
MCAST_SHAPES = [(520, 704, 264), (257, 96, 72), (300, 200, 136), (1, 32, 8), (1300, 704, 512)]


@pytest.mark.parametrize("block,stages", MCAST_CONFIGS, ids=lambda v: str(v))
@pytest.mark.parametrize("shape", MCAST_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype,out", [("f16", "f32"), ("bf16", "bf16"), ("f16", "f16")])
def test_multicast_small_shapes(cuda_lib, block, stages, shape, dtype, out):
    M, N, K = shape
    A, B = inputs.operands(300 + M + N + K, M, N, K, dtype, "uniform")
    C = as_f64(run(cuda_lib, A, B, dtype, out, block, stages, pair=True, multicast_b=True))
    R, S = oracle.gemm(A, B, dtype)
    assert_close(C, R, S, out)


@pytest.mark.parametrize("block,stages", MCAST_CONFIGS, ids=lambda v: str(v))
def test_multicast_integer_exact_and_equal_to_pairs(cuda_lib, block, stages):
    # Same MMAs in the same order as plain CTA pairs: the fp32 results agree
    # bit for bit, and integer inputs are exact.
    M, N, K = 1800, 1000, 1032
    A, B = inputs.operands(43, M, N, K, "bf16", "int", lo=-4, hi=4)
    two = run(cuda_lib, A, B, "bf16", "f32", block, stages, pair=True)
    four = run(cuda_lib, A, B, "bf16", "f32", block, stages, pair=True, multicast_b=True)
    R, _ = oracle.gemm(A, B, "bf16")
    assert np.array_equal(as_f64(four), R)
    A, B = inputs.operands(44, M, N, K, "f16", "normal")
    two = run(cuda_lib, A, B, "f16", "f32", block, stages, pair=True)
    four = run(cuda_lib, A, B, "f16", "f32", block, stages, pair=True, multicast_b=True)
    assert torch.equal(two.view(torch.int32), four.view(torch.int32))


def test_multicast_plan_geometry(cuda_lib):
    # Clusters of four CTAs; a work item is two M-adjacent tiles of one N-block.
    plan = cuda_lib.Plan(4000, 3000, 5000, "f16", "f32", (256, 352, 64), 5, pair=True, multicast_b=True)
    info = plan.info
    assert info["multicast_b"] == 1 and info["cta_pair"] == 1
    assert info["grid"] % 4 == 0 and info["num_units"] == 8 * 9
    plan.close()
    rc, h = cuda_lib.tgemm_plan_ex(512, 512, 512, "f16", "f32", 256, 256, 64, 3, cta_pair=0, multicast_b=1)
    assert rc == cuda_lib.ERR_INVALID_ARG and h is None
    rc, h = cuda_lib.tgemm_plan_ex(512, 512, 4096, "f16", "f32", 256, 256, 64, 3, cta_pair=1, split_k=4,
                                   multicast_b=1)
    assert rc == cuda_lib.ERR_INVALID_ARG and h is None


# ------------------------------------------------------------ split-K

SPLIT_CONFIGS = [((128, 128, 64), 4, 4, False), ((128, 64, 32), 3, 7, False), ((256, 128, 64), 3, 3, False),
                 ((256, 256, 64), 4, 2, True), ((128, 32, 16), 2, 64, False), ((128, 128, 128), 3, 3, False),
                 ((256, 224, 128), 2, 2, True)]


@pytest.mark.parametrize("block,stages,splits,pair", SPLIT_CONFIGS, ids=lambda v: str(v))
@pytest.mark.parametrize("shape", [(300, 200, 1032), (520, 264, 4096), (64, 32, 8), (257, 96, 200)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype,out", [("f16", "f32"), ("bf16", "bf16"), ("f16", "f16")])
def test_split_k_parity(cuda_lib, block, stages, splits, pair, shape, dtype, out):
    M, N, K = shape
    A, B = inputs.operands(300 + M + K, M, N, K, dtype, "uniform")
    C = as_f64(run(cuda_lib, A, B, dtype, out, block, stages, pair, splits))
    R, S = oracle.gemm(A, B, dtype)
    assert_close(C, R, S, out)


def test_split_k_integer_exact_and_stage_invariant(cuda_lib):
    M, N, K = 512, 512, 8192
    A, B = inputs.operands(43, M, N, K, "f16", "int", lo=-4, hi=4)
    R, _ = oracle.gemm(A, B, "f16")
    outs = [run(cuda_lib, A, B, "f16", "f32", (128, 128, 64), s, split_k=8) for s in (1, 2, 4, 6)]
    assert np.array_equal(as_f64(outs[0]), R)
    for C in outs[1:]:
        assert torch.equal(C.view(torch.int32), outs[0].view(torch.int32))


def test_split_k_plan_reports_effective_splits(cuda_lib):
    # 3 k-blocks cannot be cut 8 ways: one k-block per split at most.
    plan = cuda_lib.Plan(256, 256, 192, "f16", "f32", (128, 128, 64), 2, split_k=8)
    assert plan.info["split_k"] == 3 and plan.info["num_units"] == 4 * 3
    plan.close()
    plan = cuda_lib.Plan(256, 256, 64, "f16", "f32", (128, 128, 64), 2, split_k=8)
    assert plan.info["split_k"] == 1
    plan.close()
    rc, h = cuda_lib.tgemm_plan_ex(256, 256, 256, "f16", "f32", 128, 128, 64, 2, split_k=65)
    assert rc == cuda_lib.ERR_INVALID_ARG and h is None


# ------------------------------------------------------------ degenerate cases

def test_empty_product_is_a_noop(cuda_lib):
    for M, N in ((0, 64), (64, 0)):
        plan = cuda_lib.Plan(M, N, 64, "f16", "f32", (128, 128, 32), 3)
        A = torch.zeros((M, 64), dtype=torch.float16, device="cuda")
        B = torch.zeros((N, 64), dtype=torch.float16, device="cuda")
        C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        plan.run(A, B, C)
        torch.cuda.synchronize()
        assert plan.status()[0] == 0


@pytest.mark.parametrize("out", ["f32", "f16"])
def test_empty_reduction_gives_zeros(cuda_lib, out):
    M, N = 200, 136
    plan = cuda_lib.Plan(M, N, 0, "f16", out, (128, 128, 32), 3)
    A = torch.empty((M, 0), dtype=torch.float16, device="cuda")
    B = torch.empty((N, 0), dtype=torch.float16, device="cuda")
    C = torch.full((M, N), 7.0, dtype=TORCH[out], device="cuda")
    plan.run(A, B, C)
    torch.cuda.synchronize()
    assert plan.status()[0] == 0
    assert not C.any()


def test_k_smaller_than_block_k(cuda_lib):
    M, N, K = 130, 70 * 4, 8
    A, B = inputs.operands(9, M, N, K, "f16", "uniform")
    C = as_f64(run(cuda_lib, A, B, "f16", "f32", (128, 256, 64), 4))
    R, S = oracle.gemm(A, B, "f16")
    assert_close(C, R, S, "f32")


def test_output_not_written_outside_c(cuda_lib):
    # C is a view into a larger buffer: the guard bands around it must survive.
    M, N, K = 200, 136, 64
    A, B = inputs.operands(12, M, N, K, "f16", "uniform")
    plan = cuda_lib.Plan(M, N, K, "f16", "f32", (128, 128, 32), 3)
    big = torch.full((M + 64, N), -5.0, dtype=torch.float32, device="cuda")
    C = big[32:32 + M]
    plan.run(to_dev(A, "f16"), to_dev(B, "f16"), C)
    torch.cuda.synchronize()
    assert torch.all(big[:32] == -5.0) and torch.all(big[32 + M:] == -5.0)
    R, S = oracle.gemm(A, B, "f16")
    assert_close(as_f64(C), R, S, "f32")


def test_plans_of_different_footprints_coexist(cuda_lib):
    # A plan created after a larger one must not shrink what the larger one may launch with.
    M, N, K = 256, 256, 256
    A, B = inputs.operands(8, M, N, K, "f16", "uniform")
    dA, dB = to_dev(A, "f16"), to_dev(B, "f16")
    big = cuda_lib.Plan(M, N, K, "f16", "f32", (256, 256, 64), 3)
    small = cuda_lib.Plan(M, N, K, "f16", "f32", (128, 64, 16), 1)
    assert big.info["smem_bytes"] > small.info["smem_bytes"]
    R, S = oracle.gemm(A, B, "f16")
    for plan in (big, small, big):
        C = plan.run(dA, dB)
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        assert_close(as_f64(C), R, S, "f32")


def test_plan_rejects_over_budget_on_device(cuda_lib):
    rc, h = cuda_lib.tgemm_plan(4000, 3000, 5000, "f16", "f32", 256, 256, 64, 4)
    assert rc == cuda_lib.ERR_SMEM_BUDGET and h is None
    assert cuda_lib.tgemm_smem_limit() >= 200 * 1024


def test_misaligned_pointer_rejected_before_launch(cuda_lib):
    plan = cuda_lib.Plan(128, 128, 64, "f16", "f32", (128, 128, 32), 3)
    A = torch.zeros(128 * 64 + 8, dtype=torch.float16, device="cuda")
    B = torch.zeros((128, 64), dtype=torch.float16, device="cuda")
    C = torch.zeros((128, 128), dtype=torch.float32, device="cuda")
    rc = cuda_lib.tgemm_run(plan.handle, A.data_ptr() + 2, B.data_ptr(), C.data_ptr(), 0)
    assert rc == cuda_lib.ERR_ALIGNMENT


def test_run_host_end_to_end(cuda_lib):
    M, N, K = 384, 256, 320
    A, B = inputs.operands(21, M, N, K, "bf16", "normal")
    plan = cuda_lib.Plan(M, N, K, "bf16", "bf16", (128, 128, 64), 4)
    hA = inputs.bits_to_torch(A, "bf16").pin_memory()
    hB = inputs.bits_to_torch(B, "bf16").pin_memory()
    hC = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    dA = torch.empty_like(hA, device="cuda")
    dB = torch.empty_like(hB, device="cuda")
    dC = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    plan.run_host(hA, hB, hC, dA, dB, dC)
    torch.cuda.synchronize()
    assert plan.status()[0] == 0
    R, S = oracle.gemm(A, B, "bf16")
    assert_close(hC.float().double().numpy(), R, S, "bf16")


# ------------------------------------------------------------ full-size workloads

def sample_entries(M, N, n_random, seed):
    rng = np.random.default_rng(seed)
    rows = [np.zeros(N, np.int64), np.full(N, M - 1), np.arange(M), np.arange(M), rng.integers(0, M, n_random)]
    cols = [np.arange(N), np.arange(N), np.zeros(M, np.int64), np.full(M, N - 1), rng.integers(0, N, n_random)]
    return np.concatenate(rows), np.concatenate(cols)


def full_size(cuda_lib, name, block=None, stages=None, pair=False, split_k=1):
    """The workload in the launch configuration the benchmark times (the tuned default)."""
    w = inputs.WORKLOADS[name]
    A, B = inputs.workload_operands(name)
    group_m = cluster_k = 0
    stream_operands = multicast_b = False
    if block is None:
        cfg = cuda_lib.default_config(w["M"], w["N"], w["K"], w["dtype"], w["out"])
        block, stages, pair, split_k = cfg["block"], cfg["num_stages"], cfg["cta_pair"], cfg["split_k"]
        group_m, cluster_k = cfg["group_m"], cfg["cluster_k"]
        stream_operands, multicast_b = cfg["stream_operands"], cfg["multicast_b"]
    C = run(cuda_lib, A, B, w["dtype"], w["out"], block, stages, pair, split_k, group_m, cluster_k, stream_operands,
            multicast_b)
    return w, A, B, C


@pytest.mark.parametrize("name", ["gemm_4096_f16_normal", "gemm_8192_bf16_normal",
                                  "gemm_512x512x32768_f16_uniform", "gemm_4000x3000x5000_f16_uniform"])
def test_full_size_complete(cuda_lib, name):
    # Every element of the workload in the benchmark's launch configuration
    # against the oracle (8192^3: about half a minute of fp64 on 16 cores).
    w, A, B, C = full_size(cuda_lib, name)
    R, S = oracle.gemm(A, B, w["dtype"])
    assert_close(as_f64(C), R, S, w["out"])


def test_long_k_integer_exact(cuda_lib):
    w, A, B, C = full_size(cuda_lib, "gemm_512x512x32768_f16_int")
    R, _ = oracle.gemm(A, B, w["dtype"])
    assert np.array_equal(as_f64(C), R)


# ------------------------------------------------------------ large coordinates

@pytest.mark.parametrize("M,N,K,block,stages,split,nrand", [
    (1 << 20, 64, 64, (128, 64, 64), 4, 1, 4096),      # a million rows: tile row coordinates up to 2^20
    (128, 96, 1 << 19, (128, 96, 64), 6, 16, 128),     # a half-million-deep reduction, split 16 ways
    (96, 1 << 18, 128, (128, 256, 64), 4, 1, 4096),    # a quarter-million columns
])
def test_large_coordinates_sampled(cuda_lib, M, N, K, block, stages, split, nrand):
    A, B = inputs.operands(51, M, N, K, "bf16", "uniform")
    C = run(cuda_lib, A, B, "bf16", "f32", block, stages, split_k=split)
    rows, cols = sample_entries(M, N, nrand, 9)
    if M * N > 1 << 20:  # whole first/last rows and columns of a huge C: keep a strided subset
        keep = np.arange(rows.size) % 8 == 0
        rows, cols = rows[keep], cols[keep]
    R, S = oracle.gemm_entries(A, B, "bf16", rows, cols)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    assert_close(as_f64(got), R, S, "f32")


@pytest.mark.parametrize("M,N,K,block,stages,nrand", [
    ((1 << 20) + 100, 64, 64, (256, 64, 64), 4, 4096),  # odd M-block count: the last second tile past row 2^20
    (300, 1 << 18, 128, (256, 512, 64), 4, 4096),       # a quarter-million columns, 512-wide pair tiles
])
def test_multicast_large_coordinates_sampled(cuda_lib, M, N, K, block, stages, nrand):
    A, B = inputs.operands(52, M, N, K, "bf16", "uniform")
    C = run(cuda_lib, A, B, "bf16", "f32", block, stages, pair=True, multicast_b=True)
    rows, cols = sample_entries(M, N, nrand, 10)
    keep = np.arange(rows.size) % 8 == 0  # whole first/last rows and columns of a huge C: a strided subset
    rows, cols = rows[keep], cols[keep]
    R, S = oracle.gemm_entries(A, B, "bf16", rows, cols)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    assert_close(as_f64(got), R, S, "f32")


def test_gemm_convenience_api_uses_tuned_defaults(cuda_lib):
    M, N, K = 512, 512, 32768
    A, B = inputs.operands(52, M, N, K, "f16", "uniform")
    dA, dB = to_dev(A, "f16"), to_dev(B, "f16")
    C = cuda_lib.gemm(dA, dB, out_dtype=torch.float32)  # frozen default: split-K
    C2 = cuda_lib.gemm(dA, dB, out_dtype=torch.float32)  # cached plan
    torch.cuda.synchronize()
    R, S = oracle.gemm(A, B, "f16")
    assert_close(as_f64(C), R, S, "f32")
    assert torch.equal(C, C2)
    with pytest.raises(cuda_lib.TgemmError):
        cuda_lib.gemm(dA.float(), dB.float())
    with pytest.raises(ValueError):
        cuda_lib.gemm(dA, dB[:, :-8])


def test_run_host_argument_errors(cuda_lib):
    plan = cuda_lib.Plan(128, 128, 64, "f16", "f32", (128, 128, 32), 3)
    x = torch.zeros(128 * 128, dtype=torch.float32, device="cuda").data_ptr()
    assert cuda_lib.tgemm_run_host(plan.handle, 0, 0, 0, x, x, x) == cuda_lib.ERR_INVALID_ARG
    assert cuda_lib.tgemm_run_host(None, 0, 0, 0, 0, 0, 0) == cuda_lib.ERR_INVALID_ARG
    # the binding checks every buffer against the plan before the library copies anything
    dA = torch.zeros(128, 64, dtype=torch.float16, device="cuda")
    dB = torch.zeros(128, 64, dtype=torch.float16, device="cuda")
    dC = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    hA, hB, hC = dA.cpu(), dB.cpu(), dC.cpu()
    with pytest.raises(ValueError):
        plan.run_host(hA[:64], hB, hC, dA, dB, dC)           # host A too small
    with pytest.raises(ValueError):
        plan.run_host(hA, hB, hC.half(), dA, dB, dC)          # host C of the wrong dtype
    with pytest.raises(ValueError):
        plan.run_host(dA, hB, hC, dA, dB, dC)                 # a device tensor where host A belongs
    with pytest.raises(ValueError):
        plan.run_host(hA, hB, hC, dA, dB, dC[:64])            # device C too small
    plan.run_host(hA, hB, hC, dA, dB, dC)
    torch.cuda.synchronize()
    assert plan.status()[0] == 0 and not hC.any()
    plan.close()


# ------------------------------------------------------------ split K reduced inside the kernel

# (block, num_stages, split_k, cluster_k): clusters of 2, 4 and 8 CTAs, one to
# three clusters per tile (outer = split_k / cluster_k), slices of 128, 64 and
# 32 columns.
CSPLIT_CONFIGS = [
    ((128, 256, 64), 4, 16, 4),
    ((128, 256, 64), 3, 8, 8),
    ((128, 256, 128), 2, 4, 4),
    ((128, 256, 64), 4, 6, 2),
    ((128, 128, 64), 4, 8, 4),
    ((128, 64, 32), 5, 2, 2),
    ((128, 256, 32), 6, 24, 8),
    ((128, 192, 64), 4, 4, 2),     # 96-column slices
    ((128, 192, 32), 6, 6, 2),
]


def csplit_k(block, split_k, per_split):
    # per_split k-blocks per split, the last k-block ragged (8 columns short,
    # zero-filled by the loads), so that the split count stays split_k
    return per_split * split_k * block[2] - 8


@pytest.mark.parametrize("block,stages,split_k,cluster_k", CSPLIT_CONFIGS, ids=lambda v: str(v))
@pytest.mark.parametrize("shape", [(300, 520, 2), (129, 264, 3), (512, 512, 4), (1, 64, 1)],
                         ids=lambda s: "%dx%dxk%d" % s)
@pytest.mark.parametrize("dtype,out", [("f16", "f32"), ("bf16", "bf16"), ("f16", "f16")])
def test_cluster_split_parity(cuda_lib, block, stages, split_k, cluster_k, shape, dtype, out):
    M, N, per = shape
    K = csplit_k(block, split_k, per)
    assert cuda_lib.tgemm_validate_ex(M, N, K, dtype, out, *block, stages, 232448, split_k=split_k,
                                      cluster_k=cluster_k) == cuda_lib.OK
    A, B = inputs.operands(300 + M + N + K, M, N, K, dtype, "uniform")
    C = as_f64(run(cuda_lib, A, B, dtype, out, block, stages, split_k=split_k, cluster_k=cluster_k))
    R, S = oracle.gemm(A, B, dtype)
    assert_close(C, R, S, out)


@pytest.mark.parametrize("block,stages,split_k,cluster_k", CSPLIT_CONFIGS, ids=lambda v: str(v))
def test_cluster_split_integer_exact_repeatable_and_stage_invariant(cuda_lib, block, stages, split_k, cluster_k):
    # Integer inputs: every order of summation gives the exact result.  The
    # same plan launched again (its counters reset by the last cluster of each
    # tile) and plans of other depths give the same bits.
    M, N, K = 300, 520, csplit_k(block, split_k, 3)
    A, B = inputs.operands(41, M, N, K, "f16", "int", lo=-4, hi=4)
    dA, dB = to_dev(A, "f16"), to_dev(B, "f16")
    R, _ = oracle.gemm(A, B, "f16")
    outs = []
    for s in sorted({1, 2, stages}):
        try:
            plan = cuda_lib.Plan(M, N, K, "f16", "f32", block, s, split_k=split_k, cluster_k=cluster_k)
        except cuda_lib.TgemmError as e:  # a ring too small for the exchange at this depth
            assert e.code == cuda_lib.ERR_SMEM_BUDGET and s < stages
            continue
        assert plan.info["cluster_k"] == cluster_k
        for _ in range(2):
            outs.append(plan.run(dA, dB))
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        plan.close()
    assert outs
    assert np.array_equal(as_f64(outs[0]), R)
    for C in outs[1:]:
        assert torch.equal(C, outs[0])
    # random values: bit-identical across depths and launches as well
    A, B = inputs.operands(42, M, N, K, "bf16", "normal")
    dA, dB = to_dev(A, "bf16"), to_dev(B, "bf16")
    outs = []
    for s in sorted({1, 2, stages}):
        if cuda_lib.tgemm_validate_ex(M, N, K, "bf16", "bf16", *block, s, 232448, split_k=split_k,
                                      cluster_k=cluster_k) != cuda_lib.OK:
            continue
        plan = cuda_lib.Plan(M, N, K, "bf16", "bf16", block, s, split_k=split_k, cluster_k=cluster_k)
        outs += [plan.run(dA, dB), plan.run(dA, dB)]
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        plan.close()
    for C in outs[1:]:
        assert torch.equal(C.view(torch.int16), outs[0].view(torch.int16))


def test_cluster_split_long_k_full_and_integer(cuda_lib):
    # The long-reduction workload in cluster mode, whatever the tuned default is.
    for name in ("gemm_512x512x32768_f16_uniform", "gemm_512x512x32768_f16_int"):
        w = inputs.WORKLOADS[name]
        A, B = inputs.workload_operands(name)
        C = as_f64(run(cuda_lib, A, B, w["dtype"], w["out"], (128, 256, 64), 4, split_k=16, cluster_k=4))
        R, S = oracle.gemm(A, B, w["dtype"])
        if w["dist"] == "int":
            assert np.array_equal(C, R)
        else:
            assert_close(C, R, S, w["out"])


@pytest.mark.parametrize("block,stages,pair,split_k,shape", [
    ((256, 256, 128), 3, True, 19, (512, 512, 32768)),   # the long-K default
    ((128, 128, 64), 4, False, 5, (300, 520, 2056)),     # one CTA, ragged M, persistent with several units per CTA
    ((256, 224, 64), 3, True, 3, (1000, 1040, 4104)),    # more units than pairs
    ((64, 256, 32), 2, False, 64, (129, 264, 8192)),     # the most splits, M = 64 tiles
])
@pytest.mark.parametrize("out", ["f32", "f16"])
def test_in_kernel_split_reduction_equals_second_kernel(cuda_lib, block, stages, pair, split_k, shape, out):
    # The grid-wide reduction inside the GEMM kernel adds the partials in the
    # same order as the separate reduction kernel: the same bits, launch after
    # launch (its barrier resets itself), and within the oracle's tolerance.
    M, N, K = shape
    A, B = inputs.operands(91 + split_k, M, N, K, "f16", "uniform")
    dA, dB = to_dev(A, "f16"), to_dev(B, "f16")
    res = []
    for gr in (True, False):
        plan = cuda_lib.Plan(M, N, K, "f16", out, block, stages, pair=pair, split_k=split_k, grid_reduce=gr)
        assert plan.info["grid_reduce"] == int(gr) and plan.info["split_k"] > 1
        for _ in range(3 if gr else 1):
            res.append(plan.run(dA, dB))
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        plan.close()
    for C in res[1:]:
        assert torch.equal(C.view(torch.int32 if out == "f32" else torch.int16),
                           res[0].view(torch.int32 if out == "f32" else torch.int16))
    R, S = oracle.gemm(A, B, "f16")
    assert_close(as_f64(res[0]), R, S, out)


def test_gemm_from_several_host_threads(cuda_lib):
    # gemm() holds its plan cache's lock for the lookup only and each plan's own
    # lock for the enqueue: threads on different plans run side by side, and
    # threads sharing a plan take turns.  Every result must still be right.
    import threading

    shapes = [(256, 512, 1024), (384, 256, 512), (256, 512, 1024), (512, 768, 256)]
    work = []
    for i, (M, N, K) in enumerate(shapes):
        A, B = inputs.operands(700 + i, M, N, K, "f16", "uniform")
        work.append((A, B, to_dev(A, "f16"), to_dev(B, "f16")))
    results, errors = [None] * len(work), []

    def worker(i):
        try:
            _, _, dA, dB = work[i]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                outs = [cuda_lib.gemm(dA, dB, out_dtype=torch.float32, stream=stream) for _ in range(20)]
            stream.synchronize()
            results[i] = outs
        except Exception as e:  # reported below, in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(work))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (A, B, _, _), outs in zip(work, results):
        R, S = oracle.gemm(A, B, "f16")
        for C in outs:
            assert torch.equal(C, outs[0])
        assert_close(as_f64(outs[0]), R, S, "f32")


# ------------------------------------------------------------ stream-K tail of the persistent schedule

SK_CASES = [
    # (shape, block, stages, pair): tiles past the last whole wave of workers are
    # shared out by k-blocks (the persistent grid has one worker per SM or pair)
    ((4000, 3000, 5000), (256, 352, 64), 5, True),    # the ragged default: 144 tiles on 76 pairs
    ((3000, 2080, 1032), (256, 256, 128), 3, True),   # 108 tiles: 32 past one wave of pairs
    ((2304, 2304, 4096), (256, 256, 64), 3, True),    # 81 tiles: 5 past the wave, each in ~15 pieces
    ((2000, 2080, 1032), (128, 128, 64), 4, False),   # 272 tiles on 152 CTAs
    ((3000, 2080, 1032), (256, 128, 64), 3, False),   # one CTA, two M-halves per tile
    ((2000, 1304, 2048), (64, 256, 64), 4, False),    # 64-row tiles
]


@pytest.mark.parametrize("shape,block,stages,pair", SK_CASES, ids=lambda v: str(v))
@pytest.mark.parametrize("dtype,out", [("f16", "f32"), ("bf16", "bf16")])
def test_stream_k_parity(cuda_lib, shape, block, stages, pair, dtype, out):
    M, N, K = shape
    A, B = inputs.operands(800 + M % 97, M, N, K, dtype, "uniform")
    plan = cuda_lib.Plan(M, N, K, dtype, out, block, stages, pair=pair, stream_k=True)
    assert plan.info["stream_k_tiles"] > 0
    plan.close()
    C = as_f64(run_sk(cuda_lib, A, B, dtype, out, block, stages, pair))
    R, S = oracle.gemm(A, B, dtype)
    assert_close(C, R, S, out)


def run_sk(tg, A, B, dtype, out, block, stages, pair):
    M, K = A.shape
    N = B.shape[0]
    plan = tg.Plan(M, N, K, dtype, out, block, stages, pair=pair, stream_k=True)
    C = torch.full((M, N), float("nan"), dtype=TORCH[out], device="cuda")
    plan.run(to_dev(A, dtype), to_dev(B, dtype), C)
    torch.cuda.synchronize()
    rc, detail = plan.status()
    assert rc == 0, f"kernel status {rc} {detail}"
    plan.close()
    return C


@pytest.mark.parametrize("shape,block,stages,pair", SK_CASES, ids=lambda v: str(v))
def test_stream_k_integer_exact_repeatable_and_stage_invariant(cuda_lib, shape, block, stages, pair):
    M, N, K = shape
    A, B = inputs.operands(43, M, N, K, "f16", "int", lo=-4, hi=4)
    dA, dB = to_dev(A, "f16"), to_dev(B, "f16")
    outs = []
    for s in sorted({1, 2, stages}):
        plan = cuda_lib.Plan(M, N, K, "f16", "f32", block, s, pair=pair, stream_k=True)
        for _ in range(2):  # the tail's counters reset themselves between launches
            outs.append(plan.run(dA, dB))
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        plan.close()
    R, _ = oracle.gemm(A, B, "f16")
    assert np.array_equal(as_f64(outs[0]), R)
    for C in outs[1:]:
        assert torch.equal(C, outs[0])
    # random values: the pieces are added in a fixed order, so the bits repeat too
    A, B = inputs.operands(44, M, N, K, "bf16", "normal")
    dA, dB = to_dev(A, "bf16"), to_dev(B, "bf16")
    outs = []
    for s in sorted({2, stages}):
        plan = cuda_lib.Plan(M, N, K, "bf16", "f32", block, s, pair=pair, stream_k=True)
        outs += [plan.run(dA, dB), plan.run(dA, dB)]
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        plan.close()
    for C in outs[1:]:
        assert torch.equal(C.view(torch.int32), outs[0].view(torch.int32))
