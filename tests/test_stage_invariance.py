"""Bit-identity across num_stages at a fixed tile.

Pipelining changes when data arrives, never what is summed or in which order
(chapter 11 "Pipeline and autotuning", section 2.4: throughput, not the
result).  The kernel's summation order depends only on the tile shape, so
every depth must give the same bits, including the unpipelined num_stages=1.
"""

import pytest
import torch

from software_pipelined_tiled_02_gb300 import inputs

pytestmark = pytest.mark.gpu


def bits(C):
    return C.view(torch.int32 if C.element_size() == 4 else torch.int16)


def outputs_over_stages(tg, M, N, K, dtype, out, block, stage_list, seed, pair=False, group_m=0, split_k=1,
                        dist="normal", kw=None, cluster_k=0, multicast_b=False, stream_operands=False):
    A, B = inputs.operands(seed, M, N, K, dtype, dist, **(kw or {}))
    dA = inputs.bits_to_torch(A, dtype).cuda()
    dB = inputs.bits_to_torch(B, dtype).cuda()
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[out]
    res = []
    for s in stage_list:
        plan = tg.Plan(M, N, K, dtype, out, block, s, pair=pair, group_m=group_m, split_k=split_k,
                       cluster_k=cluster_k, multicast_b=multicast_b, stream_operands=stream_operands)
        C = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        plan.run(dA, dB, C)
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        res.append(C)
        plan.close()
    return res


@pytest.mark.parametrize("block,stage_list", [
    ((128, 128, 32), (1, 2, 3, 4, 6)),
    ((128, 256, 64), (1, 2, 3, 4)),
    ((256, 128, 64), (1, 2, 3)),
    ((128, 64, 16), (1, 2, 4, 8)),
    ((128, 128, 128), (1, 2, 3)),
    ((64, 128, 64), (1, 2, 4, 6)),
])
@pytest.mark.parametrize("dtype,out", [("f16", "f32"), ("bf16", "bf16")])
def test_bit_identical_across_stages(cuda_lib, block, stage_list, dtype, out):
    res = outputs_over_stages(cuda_lib, 1000, 1040, 2056, dtype, out, block, stage_list, seed=77)
    for s, C in zip(stage_list[1:], res[1:]):
        assert torch.equal(bits(C), bits(res[0])), f"num_stages={s} differs"


@pytest.mark.parametrize("name", ["gemm_4096_f16_normal", "gemm_8192_bf16_normal",
                                  "gemm_4000x3000x5000_f16_uniform", "gemm_512x512x32768_f16_uniform"])
def test_bit_identical_across_stages_benchmark_config(cuda_lib, name):
    # The launch configuration the benchmark times (tile, CTA pair, raster
    # group, K splits, multicast, load hint), at every depth that fits its tile.
    w = inputs.WORKLOADS[name]
    cfg = cuda_lib.default_config(w["M"], w["N"], w["K"], w["dtype"], w["out"])
    stage_list = [s for s in (1, 2, 3, 4, 5, 6) if s <= cfg["num_stages"] and
                  cuda_lib.tgemm_validate_ex(w["M"], w["N"], w["K"], w["dtype"], w["out"], *cfg["block"], s, 232448,
                                             cta_pair=int(cfg["cta_pair"]), split_k=cfg["split_k"],
                                             cluster_k=cfg["cluster_k"], multicast_b=int(cfg["multicast_b"]),
                                             stream_operands=int(cfg["stream_operands"])) == cuda_lib.OK]
    assert len(stage_list) >= 2 and stage_list[-1] == cfg["num_stages"]
    res = outputs_over_stages(cuda_lib, w["M"], w["N"], w["K"], w["dtype"], w["out"], cfg["block"], stage_list,
                              w["seed"], pair=cfg["cta_pair"], group_m=cfg["group_m"], split_k=cfg["split_k"],
                              dist=w["dist"], kw=w.get("kw"), cluster_k=cfg["cluster_k"],
                              multicast_b=cfg["multicast_b"], stream_operands=cfg["stream_operands"])
    for s, C in zip(stage_list[1:], res[1:]):
        assert torch.equal(bits(C), bits(res[0])), f"num_stages={s} differs"


def test_bit_identical_across_stages_4096(cuda_lib):
    res = outputs_over_stages(cuda_lib, 4096, 4096, 4096, "f16", "f16", (128, 128, 32), (1, 2, 3, 4, 6), seed=2)
    for C in res[1:]:
        assert torch.equal(bits(C), bits(res[0]))


@pytest.mark.parametrize("block,stage_list", [((256, 256, 64), (1, 2, 4, 6)), ((256, 128, 32), (1, 3, 8)),
                                              ((256, 224, 128), (1, 2, 3)), ((256, 512, 64), (1, 2, 4)),
                                              ((256, 224, 64), (1, 3, 6)), ((256, 128, 128), (1, 2, 4)),
                                              ((256, 352, 64), (1, 2, 4)),
                                              ((256, 448, 128), (1, 2))])
def test_bit_identical_across_stages_pair(cuda_lib, block, stage_list):
    res = outputs_over_stages(cuda_lib, 1000, 1040, 2056, "bf16", "f32", block, stage_list, seed=78, pair=True)
    for s, C in zip(stage_list[1:], res[1:]):
        assert torch.equal(bits(C), bits(res[0])), f"num_stages={s} differs"


@pytest.mark.parametrize("block,stage_list", [((256, 352, 64), (1, 2, 5)), ((256, 224, 128), (1, 3))])
def test_bit_identical_across_stages_multicast(cuda_lib, block, stage_list):
    # Two pairs sharing B through multicast: every depth gives the bits of
    # plain CTA pairs (odd tiles_m: the cluster's last second tile lies past M).
    res = outputs_over_stages(cuda_lib, 1300, 1040, 2056, "bf16", "f32", block, stage_list, seed=79, pair=True,
                              multicast_b=True)
    ref = outputs_over_stages(cuda_lib, 1300, 1040, 2056, "bf16", "f32", block, stage_list[:1], seed=79, pair=True)
    for s, C in zip(stage_list, res):
        assert torch.equal(bits(C), bits(ref[0])), f"num_stages={s} differs"


def test_bit_identical_across_prefetch_distances(cuda_lib):
    # The producer's lead D (1 = serial copy/compute, 2 = the two-stage manual
    # schedule, ... S = the full ring) changes timing only.
    M, N, K = 1000, 1040, 2056
    A, B = inputs.operands(79, M, N, K, "f16", "normal")
    dA = inputs.bits_to_torch(A, "f16").cuda()
    dB = inputs.bits_to_torch(B, "f16").cuda()
    res = []
    for D in (1, 2, 3, 5, 6):
        plan = cuda_lib.Plan(M, N, K, "f16", "f32", (128, 128, 32), 6, prefetch=D)
        assert plan.info["prefetch"] == D
        C = plan.run(dA, dB)
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        res.append(C)
        plan.close()
    for C in res[1:]:
        assert torch.equal(bits(C), bits(res[0]))
    rc, h = cuda_lib.tgemm_plan_ex(M, N, K, "f16", "f32", 128, 128, 32, 4, prefetch=5)
    assert rc == cuda_lib.ERR_INVALID_ARG and h is None


def test_bit_identical_across_prefetch_distances_two_panel_pair(cuda_lib):
    # The same with 128-column k-blocks (two K-panels per slot) in CTA pairs.
    M, N, K = 1000, 1040, 2056
    A, B = inputs.operands(80, M, N, K, "bf16", "normal")
    dA = inputs.bits_to_torch(A, "bf16").cuda()
    dB = inputs.bits_to_torch(B, "bf16").cuda()
    res = []
    for D in (1, 2, 3):
        plan = cuda_lib.Plan(M, N, K, "bf16", "bf16", (256, 224, 128), 3, pair=True, prefetch=D)
        C = plan.run(dA, dB)
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        res.append(C)
        plan.close()
    for C in res[1:]:
        assert torch.equal(bits(C), bits(res[0]))


def test_bit_identical_across_raster_groups(cuda_lib):
    # group_m only changes which CTA computes which tile, never a sum.
    M, N, K = 2000, 2080, 1032
    A, B = inputs.operands(81, M, N, K, "f16", "normal")
    dA = inputs.bits_to_torch(A, "f16").cuda()
    dB = inputs.bits_to_torch(B, "f16").cuda()
    for pair, block in ((False, (256, 224, 64)), (True, (256, 224, 128))):
        res = []
        for gm in (1, 2, 8, 16):
            plan = cuda_lib.Plan(M, N, K, "f16", "f16", block, 3, pair=pair, group_m=gm)
            C = plan.run(dA, dB)
            torch.cuda.synchronize()
            assert plan.status()[0] == 0
            res.append(C)
            plan.close()
        for C in res[1:]:
            assert torch.equal(bits(C), bits(res[0]))


@pytest.mark.parametrize("block,stages,pair,split_k", [((128, 256, 64), 4, False, 1), ((256, 224, 128), 3, True, 1),
                                                       ((256, 384, 64), 4, True, 1), ((256, 256, 128), 3, True, 5)])
def test_stream_operands_changes_nothing_but_the_cache_policy(cuda_lib, block, stages, pair, split_k):
    # The evict-first hint on the operand loads only steers L2 replacement.
    M, N, K = 1000, 1040, 2056
    A, B = inputs.operands(83, M, N, K, "f16", "normal")
    dA = inputs.bits_to_torch(A, "f16").cuda()
    dB = inputs.bits_to_torch(B, "f16").cuda()
    res = []
    for stream in (False, True):
        plan = cuda_lib.Plan(M, N, K, "f16", "f32", block, stages, pair=pair, split_k=split_k, stream_operands=stream)
        assert plan.info["stream_operands"] == int(stream)
        res.append(plan.run(dA, dB))
        torch.cuda.synchronize()
        assert plan.status()[0] == 0
        plan.close()
    assert torch.equal(bits(res[0]), bits(res[1]))
