"""The allocation-free entry point, tgemm_run_noalloc.

It is for callers that cannot allocate device memory (code where cudaMalloc
is unavailable or forbidden, such as an allocator's own hooks or a service
with a fixed device footprint): the kernel's status record lives in a
fixed array inside the library instead of a buffer that tgemm_plan would
cudaMalloc.  These tests call it through the C ABI and compare its output
with the plan-based entry point's on the same inputs, twice in a row (the
second call finds the previous call's record in the shared array and must
clear it).  This file is collected last on purpose, and it must also pass
when run alone in a fresh process.
"""

import numpy as np
import pytest
import torch

import oracle
from software_pipelined_tiled_02_gb300 import inputs

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.mark.parametrize("shape,dtype,out,block,stages", [
    ((300, 200, 136), "f16", "f32", (128, 128, 32), 3),
    ((1000, 1040, 2056), "bf16", "bf16", (256, 224, 64), 3),
    ((4096, 4096, 4096), "f16", "f16", (256, 224, 64), 3),
    ((520, 704, 5000), "f16", "f32", (128, 128, 128), 3),
])
def test_noalloc_matches_plan_entry_point_twice(cuda_lib, shape, dtype, out, block, stages):
    tg = cuda_lib
    M, N, K = shape
    A, B = inputs.operands(61, M, N, K, dtype, "normal")
    dA = inputs.bits_to_torch(A, dtype).cuda()
    dB = inputs.bits_to_torch(B, dtype).cuda()
    plan = tg.Plan(M, N, K, dtype, out, block, stages)
    ref = plan.run(dA, dB)
    torch.cuda.synchronize()
    assert plan.status()[0] == tg.OK
    rows = np.random.default_rng(3).integers(0, M, 512)
    cols = np.random.default_rng(4).integers(0, N, 512)
    R, S = oracle.gemm_entries(A, B, dtype, rows, cols)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=TORCH[out], device="cuda")
        rc, status = tg.tgemm_run_noalloc(M, N, K, dtype, out, *block, stages, dA.data_ptr(), dB.data_ptr(),
                                          C.data_ptr(), stream)
        assert rc == tg.OK, tg.strerror(rc)
        assert status == tg.OK, f"call {call}: kernel status {status}"
        # Same kernel, same inputs: the outputs agree with the plan path's,
        # and both meet the oracle tolerance of the other GPU tests.
        assert torch.equal(C, ref), f"call {call} differs from the plan-based entry point"
        got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].float().cpu().double().numpy()
        ok, worst, _ = oracle.check(got, R, S, out)
        assert ok, worst
    plan.close()


def test_noalloc_without_status_is_asynchronous_and_correct(cuda_lib):
    tg = cuda_lib
    M, N, K = 257, 96, 72
    A, B = inputs.operands(62, M, N, K, "f16", "uniform")
    dA = inputs.bits_to_torch(A, "f16").cuda()
    dB = inputs.bits_to_torch(B, "f16").cuda()
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    rc, status = tg.tgemm_run_noalloc(M, N, K, "f16", "f32", 128, 64, 16, 2, dA.data_ptr(), dB.data_ptr(),
                                      C.data_ptr(), torch.cuda.current_stream().cuda_stream, want_status=False)
    assert rc == tg.OK and status is None
    torch.cuda.synchronize()
    R, S = oracle.gemm(A, B, "f16")
    ok, worst, _ = oracle.check(C.cpu().double().numpy(), R, S, "f32")
    assert ok, worst


def test_noalloc_rejects_what_the_plan_rejects(cuda_lib):
    tg = cuda_lib
    x = torch.zeros(1024 * 1024, dtype=torch.float16, device="cuda")
    p = x.data_ptr()
    assert tg.tgemm_run_noalloc(4000, 3000, 5000, "f16", "f32", 256, 256, 64, 4, p, p, p)[0] == tg.ERR_SMEM_BUDGET
    assert tg.tgemm_run_noalloc(128, 128, 12, "f16", "f32", 128, 128, 32, 3, p, p, p)[0] == tg.ERR_ALIGNMENT
    assert tg.tgemm_run_noalloc(128, 128, 64, "f16", "f32", 96, 128, 32, 3, p, p, p)[0] == tg.ERR_NO_KERNEL
    assert tg.tgemm_run_noalloc(128, 128, 64, "f16", "f32", 128, 128, 32, 3, p + 2, p, p)[0] == tg.ERR_ALIGNMENT
    assert tg.tgemm_run_noalloc(0, 128, 64, "f16", "f32", 128, 128, 32, 3, 0, 0, 0) == (tg.OK, tg.OK)


def test_noalloc_status_rejected_on_a_capturing_stream(cuda_lib):
    # Reading the status back waits for the stream, which a capturing stream
    # forbids: the call refuses before enqueueing anything.
    tg = cuda_lib
    x = torch.zeros(128 * 128, dtype=torch.float32, device="cuda")
    p = x.data_ptr()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        rc, _ = tg.tgemm_run_noalloc(128, 128, 64, "f16", "f32", 128, 128, 32, 3, p, p, p, side.cuda_stream,
                                     want_status=True)
    assert rc == tg.ERR_INVALID_ARG
