"""The kernel's bounded waits: a stalled pipeline reports, it does not hang.

The test hook makes every CTA's MMA warp wait on a barrier that nothing
arrives on; with a 50 ms watchdog the kernel must return, report
TGEMM_ERR_TIMEOUT through the plan's status word, and leave the context
usable (the next run on the same plan is correct).  No fault or trap is
involved.
"""

import pytest
import torch

import oracle
from software_pipelined_tiled_02_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("block,stages,pair,split_k,cluster_k", [
    ((128, 128, 32), 3, False, 1, 0), ((128, 256, 64), 1, False, 1, 0), ((256, 256, 64), 4, True, 1, 0),
    ((128, 256, 64), 4, False, 8, 4),  # K splits reduced in the kernel by clusters of 4: both cluster levels
    ((256, 256, 64), 3, True, 4, -1),  # K splits reduced in the kernel after a grid-wide barrier
    ((64, 64, 32), 4, False, 1, -2),   # a stream-K tail (1024 x 1024: 256 tiles on 152 CTAs)
    ((256, 352, 64), 4, True, 1, -3),  # clusters of two pairs sharing B through multicast
])
def test_stall_reports_timeout_and_context_survives(cuda_lib, block, stages, pair, split_k, cluster_k):
    grid_reduce, stream_k, multicast_b = cluster_k == -1, cluster_k == -2, cluster_k == -3
    cluster_k = max(cluster_k, 0)
    M, N, K = (1024, 1024, 512) if stream_k else (512, 512, 512)
    A, B = inputs.operands(31, M, N, K, "f16", "uniform")
    dA = inputs.bits_to_torch(A, "f16").cuda()
    dB = inputs.bits_to_torch(B, "f16").cuda()
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    plan = cuda_lib.Plan(M, N, K, "f16", "f32", block, stages, pair=pair, split_k=split_k, cluster_k=cluster_k,
                         grid_reduce=grid_reduce, stream_k=stream_k, multicast_b=multicast_b)
    if stream_k:
        assert plan.info["stream_k_tiles"] > 0
    plan.set_watchdog_ns(50_000_000)
    plan.debug_stall(True)
    plan.run(dA, dB, C)
    torch.cuda.synchronize()
    code, detail = plan.status()
    assert code == cuda_lib.ERR_TIMEOUT
    assert detail[1] in (0, 1, 2)  # the role that gave up first
    # status is cleared by reading it
    assert plan.status()[0] == 0
    # the context is still good: a normal run on the same plan is correct
    plan.debug_stall(False)
    plan.set_watchdog_ns(0)
    plan.run(dA, dB, C)
    torch.cuda.synchronize()
    assert plan.status()[0] == 0
    R, S = oracle.gemm(A, B, "f16")
    ok, worst, _ = oracle.check(C.cpu().double().numpy(), R, S, "f32")
    assert ok, worst
