"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against something fixed outside it:
hand-worked products, exact integer arithmetic, identity and zero matrices,
numpy's and torch's own conversions, numpy's float64 matmul, and the numbers
the tutorial pages print for the shared-memory budget and the config space.
"""

import fractions
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from software_pipelined_tiled_02_gb300 import inputs
from tests.conftest import golden_lines, hand_cases


def f16bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


# ---------------------------------------------------------------- GEMM pins

@pytest.mark.parametrize("case", hand_cases(), ids=lambda c: c["name"])
def test_hand_cases(case):
    A = f16bits(case["A"])
    B = f16bits(case["B"])
    R, S = oracle.gemm(A, B, "f16")
    assert R.shape == (case["M"], case["N"])
    assert np.array_equal(R, np.array(case["C"]))
    if case["S"]:
        assert np.array_equal(S, np.array(case["S"]))


def test_transpose_distinguishes():
    # A . B^T and A . B differ on the 2x2 hand case; the oracle is the former.
    A = f16bits([[1, 2], [3, 4]])
    B = f16bits([[5, 6], [7, 8]])
    R, _ = oracle.gemm(A, B, "f16")
    assert not np.array_equal(R, np.array([[19, 22], [43, 50]]))


def test_brute_force_tiny_exact_rationals():
    # Brute force with exact rational arithmetic on a 4x5x3 case of fp16
    # values with fractional parts: every product and partial sum is exact in
    # float64, so the oracle must agree exactly.
    rng = np.random.default_rng(7)
    vals = rng.integers(-64, 64, size=(4 + 5, 3)) / 16.0
    A = f16bits(vals[:4])
    B = f16bits(vals[4:])
    Av = A.view(np.float16).astype(object)
    Bv = B.view(np.float16).astype(object)
    R, S = oracle.gemm(A, B, "f16")
    for i in range(4):
        for j in range(5):
            exact = sum(fractions.Fraction(float(Av[i, k])) * fractions.Fraction(float(Bv[j, k]))
                        for k in range(3))
            mag = sum(abs(fractions.Fraction(float(Av[i, k])) * fractions.Fraction(float(Bv[j, k])))
                      for k in range(3))
            assert fractions.Fraction(R[i, j]) == exact
            assert fractions.Fraction(S[i, j]) == mag


def test_identity_and_zero():
    A = inputs.matrix_bits(11, 0, 6, 9, "f16", "uniform")
    eye = f16bits(np.eye(9))
    R, _ = oracle.gemm(A, eye, "f16")
    assert np.array_equal(R, A.view(np.float16).astype(np.float64))
    Z = f16bits(np.zeros((7, 9)))
    R0, S0 = oracle.gemm(A, Z, "f16")
    assert not R0.any() and not S0.any()
    R1, _ = oracle.gemm(Z[:3], A, "f16")
    assert not R1.any()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_integer_inputs_are_exact(dtype):
    # Small-integer operands in [-4, 4]: |sum| <= 16*K, exact in float64 and
    # in int64; numpy's integer matmul is exact.
    M, N, K = 33, 17, 1000
    A, B = inputs.operands(40, M, N, K, dtype, "int", lo=-4, hi=4)
    Ai = oracle.decode(A, dtype).astype(np.int64)
    Bi = oracle.decode(B, dtype).astype(np.int64)
    R, S = oracle.gemm(A, B, dtype)
    assert np.array_equal(R, (Ai @ Bi.T).astype(np.float64))
    assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi).T).astype(np.float64))


@pytest.mark.parametrize("shape", [(5, 7, 3), (1, 13, 40), (19, 1, 8), (64, 48, 200)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_matches_numpy_float64(shape, dtype):
    # Non-square shapes catch swapped indices; numpy's float64 matmul is an
    # independent library routine (its summation order differs, so the two
    # agree to float64 rounding, far below the kernel tolerance).
    M, N, K = shape
    A, B = inputs.operands(3, M, N, K, dtype, "normal")
    Ad = torch.from_numpy(A.view(np.int16)).view(
        torch.float16 if dtype == "f16" else torch.bfloat16).double().numpy()
    Bd = torch.from_numpy(B.view(np.int16)).view(
        torch.float16 if dtype == "f16" else torch.bfloat16).double().numpy()
    R, S = oracle.gemm(A, B, dtype)
    ref = Ad @ Bd.T
    assert np.all(np.abs(R - ref) <= 1e-12 * (np.abs(Ad) @ np.abs(Bd).T) + 1e-300)
    assert np.allclose(S, np.abs(Ad) @ np.abs(Bd).T, rtol=1e-12, atol=0)


def test_entries_and_rows_agree_with_full():
    M, N, K = 37, 29, 70
    A, B = inputs.operands(5, M, N, K, "f16", "uniform")
    R, S = oracle.gemm(A, B, "f16")
    rows = np.array([0, 36, 5, 17, 36])
    cols = np.array([0, 28, 11, 3, 0])
    r, s = oracle.gemm_entries(A, B, "f16", rows, cols)
    assert np.array_equal(r, R[rows, cols]) and np.array_equal(s, S[rows, cols])
    assert np.array_equal(oracle.gemm_rows(A, B, "f16", 10, 5), R[10:15])
    Ad, Bd = oracle.decode(A, "f16"), oracle.decode(B, "f16")
    assert np.array_equal(oracle.gemm_decoded_rows(Ad, Bd, 3, 30), R[3:33])


def test_degenerate_shapes():
    A = f16bits(np.ones((0, 4)))
    B = f16bits(np.ones((3, 4)))
    R, _ = oracle.gemm(A, B, "f16")
    assert R.shape == (0, 3)
    # K = 0: the empty sum is zero.
    R, S = oracle.gemm(f16bits(np.ones((2, 0))), f16bits(np.ones((3, 0))), "f16")
    assert R.shape == (2, 3) and not R.any() and not S.any()


def test_flop_count():
    # TFLOPS = 2*M*N*K / t ("Stage 04 - GEMM main line", exercise 3).
    assert oracle.flops(4096, 4096, 4096) == 137438953472.0
    assert oracle.flops(512, 512, 32768) == 2 * 512 * 512 * 32768
    assert oracle.flops(4000, 3000, 5000) == 1.2e11


# ------------------------------------------------------- conversion pins

def test_f16_decode_all_patterns():
    x = np.arange(65536, dtype=np.uint16)
    d = oracle.decode(x, "f16")
    ref = x.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(d), nan)
    assert np.array_equal(d[~nan], ref[~nan])
    assert np.array_equal(np.signbit(d[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_all_patterns():
    x = np.arange(65536, dtype=np.uint16)
    d = oracle.decode(x, "bf16")
    ref = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(d), nan)
    assert np.array_equal(d[~nan], ref[~nan])
    assert np.array_equal(np.signbit(d[~nan]), np.signbit(ref[~nan]))


def _neighbourhood(values):
    """Values, midpoints between consecutive values, and points just off the midpoints."""
    v = np.unique(values[np.isfinite(values)])
    mid = (v[:-1] + v[1:]) / 2
    up = np.nextafter(mid, np.inf)
    dn = np.nextafter(mid, -np.inf)
    return np.concatenate([v, mid, up, dn])


def test_round_f16_matches_numpy():
    allv = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    pts = _neighbourhood(allv)
    rng = np.random.default_rng(1)
    rnd = rng.standard_normal(200000) * np.exp2(rng.integers(-30, 17, size=200000))
    pts = np.concatenate([pts, rnd, [65504.0, 65519.99, 65520.0, 65536.0, 1e9, -1e9,
                                     2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26, 0.0, -0.0]])
    mine = oracle.round_to(pts, "f16")
    with np.errstate(over="ignore"):
        ref = pts.astype(np.float16).view(np.uint16)
    assert np.array_equal(mine, ref)


def test_round_bf16_matches_torch_on_f32_values():
    # torch rounds float32 -> bfloat16 to nearest even; for float64 inputs that
    # are float32 numbers that is a single rounding, comparable bit for bit.
    allv = torch.from_numpy(np.arange(65536, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).double().numpy()
    pts = _neighbourhood(allv)
    pts = pts[np.abs(pts) < 3.4e38]
    pts32 = pts.astype(np.float32)
    pts = pts32.astype(np.float64)  # keep only float32-representable points
    rng = np.random.default_rng(2)
    extra = (rng.standard_normal(200000) * np.exp2(rng.integers(-140, 120, size=200000))).astype(np.float32)
    pts = np.concatenate([pts, extra.astype(np.float64)])
    mine = oracle.round_to(pts, "bf16")
    ref = torch.from_numpy(pts.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_round_ties_to_even_by_hand():
    # 1 + 2^-11 lies halfway between 1 and 1 + 2^-10 in fp16: ties go to the
    # even significand (1.0); 1 + 3*2^-11 goes up to 1 + 2^-9.
    assert oracle.round_to([1 + 2.0 ** -11], "f16")[0] == 0x3C00
    assert oracle.round_to([1 + 3 * 2.0 ** -11], "f16")[0] == 0x3C02
    # bf16 keeps 8 significant bits: 1 + 2^-8 ties to 1.0, 1 + 3*2^-8 to 1 + 2^-6.
    assert oracle.round_to([1 + 2.0 ** -8], "bf16")[0] == 0x3F80
    assert oracle.round_to([1 + 3 * 2.0 ** -8], "bf16")[0] == 0x3F82
    # Overflow: the halfway point past the largest finite value becomes inf.
    assert oracle.round_to([65520.0], "f16")[0] == 0x7C00
    assert oracle.round_to([-65520.0], "f16")[0] == 0xFC00


# ------------------------------------------------- budget and config pins

def test_smem_budget_numbers_from_pages():
    for t in golden_lines("smem_budget.txt"):
        if t[0] == "tile":
            bm, bn, bk, eb, per, smax = map(int, t[1:])
            assert oracle.smem_bound(bm, bn, bk, 1, eb) == per
            assert oracle.max_stages(bm, bn, bk, 228 * 1024, eb) == smax
        elif t[0] == "stages":
            bm, bn, bk, s, foot, pct = map(int, t[1:7])
            fits = t[7] == "yes"
            got = oracle.smem_bound(bm, bn, bk, s, 2)
            assert got == foot
            assert round(100 * got / (228 * 1024)) == pct
            assert (got <= 228 * 1024) == fits


def test_config_space_count_from_pages():
    spec = {t[0]: t[1:] for t in golden_lines("config_space.txt") if t[0] != "reject"}
    rejects = {tuple(map(int, t[1:])) for t in golden_lines("config_space.txt") if t[0] == "reject"}
    M, N, K = map(int, spec["problem"])
    budget = int(spec["budget"][0])
    grid = list(itertools.product((64, 128, 256), (64, 128, 256), (16, 32, 64), (1, 2, 3, 4), (128, 256)))
    assert len(grid) == int(spec["requested"][0])
    legal, rejected = [], set()
    for bm, bn, bk, s, th in grid:
        if M % bm or N % bn or K % bk:
            rejected.add((bm, bn, bk, s, th))
        elif oracle.smem_bound(bm, bn, bk, s, 2) > budget:
            rejected.add((bm, bn, bk, s, th))
        else:
            legal.append((bm, bn, bk, s, th))
    assert len(legal) == int(spec["legal"][0])
    assert rejected == rejects


# ------------------------------------------------------- acceptance helper

def test_check_accepts_within_and_rejects_outside():
    R = np.array([1.0, -2.0, 100.0])
    S = np.array([10.0, 10.0, 1000.0])
    ok, worst, _ = oracle.check(R + 0.5 * (1e-4 * S + 1e-5), R, S, "f32")
    assert ok and worst <= 0.5 + 1e-9
    ok, _, idx = oracle.check(R + np.array([0, 0, 0.2]), R, S, "f32")
    assert not ok and idx == 2
    # 16-bit output: one output ulp is allowed on top.
    ok, _, _ = oracle.check(np.array([1.0 + 2.0 ** -10]), np.array([1.0]), np.array([0.0]), "f16")
    assert ok
    ok, _, _ = oracle.check(np.array([1.0 + 2.0 ** -8]), np.array([1.0]), np.array([0.0]), "f16")
    assert not ok
    ok, _, _ = oracle.check(np.array([np.nan]), np.array([1.0]), np.array([1.0]), "f32")
    assert not ok


def test_check_pages_leg_alone_rejects():
    # A huge error scale S makes the target's bound 1e-4*S + 1e-5 loose; the
    # pages' own check (rtol = atol = 1e-2 against torch.matmul) must still
    # reject an output that is 0.5 away from a zero reference.
    R, S = np.array([0.0]), np.array([1e4])
    ok, worst, _ = oracle.check(np.array([0.5]), R, S, "f32")
    assert not ok and worst == pytest.approx(0.5 / 1e-2)
    # Its absolute part is 1e-2: 0.009 passes, 0.011 fails.
    assert oracle.check(np.array([0.009]), R, S, "f32")[0]
    assert not oracle.check(np.array([0.011]), R, S, "f32")[0]
    # Its relative part is 1e-2 * |R|: at R = 100 an error of 1.0 passes
    # (bound 1.01) and 1.02 fails.
    R, S = np.array([100.0]), np.array([1e8])
    assert oracle.check(R + 1.0, R, S, "f32")[0]
    assert not oracle.check(R + 1.02, R, S, "f32")[0]
    assert not oracle.check(-R, R, S, "bf16")[0]


def test_check_bf16_output_allows_one_bf16_ulp():
    # bfloat16 keeps 8 significand bits: its spacing at 1.0 is 2^-7.
    R, S = np.array([1.0]), np.array([0.0])
    assert oracle.check(np.array([1.0 + 2.0 ** -7]), R, S, "bf16")[0]
    assert not oracle.check(np.array([1.0 + 2.0 ** -6]), R, S, "bf16")[0]
    assert oracle.check(np.array([3.0 + 2.0 ** -6]), np.array([3.0]), S, "bf16")[0]
    assert not oracle.check(np.array([3.0 + 2.0 ** -5]), np.array([3.0]), S, "bf16")[0]


def test_check_f32_output_gets_no_ulp():
    # The raw fp32 accumulator is compared with 1e-4*S + 1e-5 alone: at
    # R = 2^20 (binary32 spacing 2^-3) an error of one fp32 ulp is rejected
    # when S = 0, although the pages' relative bound (about 1e4) is far away.
    R, S = np.array([2.0 ** 20]), np.array([0.0])
    assert not oracle.check(R + 2.0 ** -3, R, S, "f32")[0]


def test_check_rejects_infinities_against_finite():
    R, S = np.array([1.0, 1.0]), np.array([1.0, 1.0])
    assert not oracle.check(np.array([np.inf, 1.0]), R, S, "f32")[0]
    assert not oracle.check(np.array([1.0, -np.inf]), R, S, "f16")[0]


# -------------------------------------------------- output spacing (ulp)

# IEEE 754 fixes each format's spacing.  binary16: p = 11 significand bits,
# emin = -14.  bfloat16: p = 8, with binary32's exponent range (emin = -126).
# binary32: p = 24, emin = -126.  For |x| in [2^e, 2^(e+1)) with e >= emin the
# spacing is 2^(e - p + 1); below 2^emin (subnormals and zero) it is the
# subnormal step 2^(emin - p + 1).
ULP_FIXED = [
    ("f16", 1.0, 2.0 ** -10), ("f16", 1.5, 2.0 ** -10), ("f16", -3.0, 2.0 ** -9), ("f16", 65504.0, 32.0),
    ("f16", 2.0 ** -14, 2.0 ** -24), ("f16", 2.0 ** -20, 2.0 ** -24), ("f16", 0.0, 2.0 ** -24),
    ("bf16", 1.0, 2.0 ** -7), ("bf16", 3.0, 2.0 ** -6), ("bf16", -0.75, 2.0 ** -8),
    ("bf16", 2.0 ** -126, 2.0 ** -133), ("bf16", 2.0 ** -130, 2.0 ** -133), ("bf16", 0.0, 2.0 ** -133),
    ("bf16", 2.0 ** 127, 2.0 ** 120),
    ("f32", 1.0, 2.0 ** -23), ("f32", 3.0, 2.0 ** -22), ("f32", 2.0 ** -126, 2.0 ** -149),
    ("f32", 1e-40, 2.0 ** -149), ("f32", 0.0, 2.0 ** -149), ("f32", 2.0 ** 127, 2.0 ** 104),
]


@pytest.mark.parametrize("fmt,x,want", ULP_FIXED, ids=lambda v: str(v))
def test_ulp_fixed_values(fmt, x, want):
    assert oracle.ulp(np.array([x]), fmt)[0] == want


def test_ulp_matches_numpy_spacing_f16_f32():
    # numpy's nextafter-based spacing of float16 / float32 numbers, across
    # normal and subnormal magnitudes of both signs.
    rng = np.random.default_rng(11)
    for fmt, npt, lo, hi in (("f16", np.float16, -30, 15), ("f32", np.float32, -160, 127)):
        mags = np.ldexp(rng.uniform(1.0, 2.0, 4000), rng.integers(lo, hi, 4000))
        x = (mags * rng.choice([-1.0, 1.0], 4000)).astype(npt)
        x = x[np.isfinite(x) & (x != 0)]
        with np.errstate(over="ignore"):
            want = np.spacing(np.abs(x)).astype(np.float64)  # gap above |x|
        x, want = x[np.isfinite(want)], want[np.isfinite(want)]  # the largest finite value has no upper neighbour
        assert np.array_equal(oracle.ulp(x.astype(np.float64), fmt), want)


def test_ulp_matches_bf16_neighbours_from_bits():
    # bfloat16 is the upper half of binary32: the value of pattern b is the
    # float32 with bits b << 16, and its spacing is value(b + 1) - value(b).
    rng = np.random.default_rng(12)
    b = rng.integers(0x0001, 0x7F7F, 20000).astype(np.uint32)  # positive finite, below the largest
    b = np.concatenate([b, np.array([0x0001, 0x007F, 0x0080, 0x3F80, 0x7F7E], np.uint32)])
    val = (b << 16).view(np.float32).astype(np.float64)
    nxt = ((b + 1) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(oracle.ulp(val, "bf16"), nxt - val)
    assert np.array_equal(oracle.ulp(-val, "bf16"), nxt - val)
