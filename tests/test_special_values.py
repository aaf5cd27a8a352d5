"""Non-finite values through the GPU path.

The pages say nothing about NaN or infinity.  The reading taken is IEEE-754
arithmetic throughout: a NaN operand makes its whole row (or column) of C NaN,
an infinite operand gives a signed infinity, infinity times zero and
+inf + -inf give NaN, and rounding to fp16 overflows to infinity.

The expected values are the definition written out in fp64 on the CPU, every
product A[i,k]*B[j,k] formed and summed with numpy's elementwise operations
(no BLAS, which may take shortcuts with zeros).  The finite operands are small
integers, so every finite sum is exact in fp32 and in any order; the
non-finite results do not depend on the order either.
"""

import numpy as np
import pytest
import torch

from software_pipelined_tiled_02_gb300 import inputs

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}

# (block, num_stages, cta_pair, split_k, options): one CTA (64- and 128-row
# tiles), pairs with one and two K-panels per slot and a wide tile (also with
# two pairs sharing B through multicast), and the
# split-K paths whose partials meet in the second kernel, in the GEMM kernel
# after a grid-wide barrier, or in a cluster through distributed shared memory
CONFIGS = [
    ((128, 128, 32), 3, False, 1, {}),
    ((64, 128, 64), 4, False, 1, {}),
    ((256, 224, 64), 6, True, 1, {}),
    ((256, 224, 128), 3, True, 1, {"stream_operands": True}),
    ((256, 352, 64), 4, True, 1, {}),
    ((256, 352, 64), 4, True, 1, {"multicast_b": True}),
    ((256, 256, 128), 3, True, 3, {}),
    ((128, 128, 64), 4, False, 2, {}),
    ((256, 256, 64), 3, True, 3, {"grid_reduce": True}),
    ((128, 256, 64), 3, False, 6, {"cluster_k": 2}),
]


def operands_with_specials(dtype, M, N, K):
    A, B = inputs.operands(41, M, N, K, dtype, "int", lo=-4, hi=4)
    At = inputs.bits_to_torch(A, dtype).clone()
    Bt = inputs.bits_to_torch(B, dtype).clone()
    At[3, 5] = float("nan")            # row 3 of C: NaN
    Bt[7, 200] = float("nan")          # column 7: NaN
    Bt[9, 9] = float("inf")            # column 9: +-inf by the sign of A[i, 9], NaN where it is 0
    At[11, 9] = 0.0
    Bt[20, 30] = float("-inf")         # column 20: -inf*A[i,30] + inf*A[i,31]
    Bt[20, 31] = float("inf")
    At[40, :] = 64.0                   # row 40 and column 50: sums beyond the fp16 range
    Bt[50, :] = 64.0
    return At, Bt


def reference(At, Bt, out):
    A64 = At.double().numpy()
    B64 = Bt.double().numpy()
    M, N = A64.shape[0], B64.shape[0]
    R = np.empty((M, N))
    with np.errstate(invalid="ignore", over="ignore"):
        for i in range(0, M, 32):
            R[i:i + 32] = (A64[i:i + 32, None, :] * B64[None, :, :]).sum(axis=-1)
    return torch.from_numpy(R).to(TORCH[out])


@pytest.mark.parametrize("block,stages,pair,split,opts", CONFIGS, ids=lambda v: str(v))
@pytest.mark.parametrize("dtype,out", [("f16", "f32"), ("f16", "f16"), ("bf16", "bf16")])
def test_nan_and_inf_follow_ieee(cuda_lib, block, stages, pair, split, opts, dtype, out):
    M, N, K = 300, 264, 384  # 16-bit C rows must be whole 16-byte units
    At, Bt = operands_with_specials(dtype, M, N, K)
    plan = cuda_lib.Plan(M, N, K, dtype, out, block, stages, pair=pair, split_k=split, **opts)
    C = torch.full((M, N), 5.0, dtype=TORCH[out], device="cuda")
    plan.run(At.cuda(), Bt.cuda(), C)
    torch.cuda.synchronize()
    assert plan.status()[0] == 0
    plan.close()
    C = C.cpu()
    E = reference(At, Bt, out)
    # the pattern is what the test is about: make sure it is there
    assert torch.isnan(E[3]).all() and torch.isnan(E[:, 7]).all()
    assert torch.isinf(E[:, 9]).any() and torch.isnan(E[11, 9])
    if out == "f16":
        assert torch.isinf(E[40, 50])
    nan_c, nan_e = torch.isnan(C), torch.isnan(E)
    assert torch.equal(nan_c, nan_e), f"NaN at {int((nan_c != nan_e).sum())} differing positions"
    keep = ~nan_e
    bad = (C[keep] != E[keep]).nonzero()
    assert bad.numel() == 0, f"{bad.numel()} non-NaN entries differ, e.g. got {C[keep][bad[0]]} want {E[keep][bad[0]]}"
