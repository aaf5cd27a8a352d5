"""Back-to-back launches in one stream.

Every GEMM launch, and the split-K reduction after it, is a programmatic
dependent of the kernel before it in the stream: it may start while that kernel
finishes, and it waits in griddepcontrol.wait for that kernel's writes before
it reads A and B or writes C.  A chain launched without synchronisation must
therefore give the bits of the same chain with a synchronisation after every
launch, whatever reads or writes the buffers of the launch before it (read
after write, write after read, write after write).  Buffers start as NaN, so
a launch that ran ahead of its producer would leave NaN or stale values.
"""

import pytest
import torch

pytestmark = pytest.mark.gpu


def bits(C):
    return C.view(torch.int32 if C.element_size() == 4 else torch.int16)


def weights(rows, cols, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    # entries of size about 1/sqrt(cols) keep a chain of products near unit scale in fp16
    return (torch.randn(rows, cols, device="cuda", generator=g) / cols ** 0.5).to(torch.float16)


def nan_like(rows, cols, dtype=torch.float16):
    return torch.full((rows, cols), float("nan"), dtype=dtype, device="cuda")


def chain(tg, sync):
    """Five dependent products, each reading the previous output as A: pair and
    one-CTA tiles, a split-K plan (GEMM + reduction) and its consumer."""
    X0 = weights(2048, 1024, 1) * 1024 ** 0.5
    Ws = [weights(1536, 1024, 2), weights(1024, 1536, 3), weights(2048, 1024, 4), weights(512, 2048, 5),
          weights(256, 512, 6)]
    plans = [
        tg.Plan(2048, 1536, 1024, "f16", "f16", (256, 224, 64), 6, pair=True, group_m=2),
        tg.Plan(2048, 1024, 1536, "f16", "f16", (256, 256, 64), 3),
        tg.Plan(2048, 2048, 1024, "f16", "f16", (256, 256, 64), 6, pair=True),
        tg.Plan(2048, 512, 2048, "f16", "f16", (256, 128, 128), 4, pair=True, split_k=4),
        tg.Plan(2048, 256, 512, "f16", "f16", (128, 128, 32), 3),
    ]
    outs = [nan_like(2048, W.shape[0]) for W in Ws]
    torch.cuda.synchronize()
    X = X0
    for plan, W, Y in zip(plans, Ws, outs):
        plan.run(X, W, Y)
        if sync:
            torch.cuda.synchronize()
        X = Y
    torch.cuda.synchronize()
    for plan in plans:
        assert plan.status()[0] == 0
        plan.close()
    return outs


def test_dependent_chain_matches_synchronised_chain(cuda_lib):
    ref = chain(cuda_lib, sync=True)
    for _ in range(3):
        got = chain(cuda_lib, sync=False)
        for i, (a, b) in enumerate(zip(got, ref)):
            assert not torch.isnan(a.float()).any(), f"product {i} left NaN"
            assert torch.equal(bits(a), bits(b)), f"product {i} differs"


def test_operand_written_by_torch_just_before(cuda_lib):
    # A PyTorch kernel (no trigger of its own) writes A right before the GEMM reads it.
    tg = cuda_lib
    src = weights(1024, 2048, 7)
    B = weights(1536, 2048, 8)
    plan = tg.Plan(1024, 1536, 2048, "f16", "f16", (256, 224, 64), 6, pair=True)
    ref = nan_like(1024, 1536)
    plan.run(src, B, ref)
    torch.cuda.synchronize()
    for _ in range(3):
        A = nan_like(1024, 2048)
        C = nan_like(1024, 1536)
        torch.cuda.synchronize()
        A.copy_(src)
        plan.run(A, B, C)
        torch.cuda.synchronize()
        assert torch.equal(bits(C), bits(ref))
    plan.close()


def test_write_after_read_and_write_after_write(cuda_lib):
    # GEMM 1 reads A; GEMM 2 then writes its output into A's buffer (write after read).
    # GEMMs 3 and 4 write the same C from different inputs (write after write): C must
    # end as GEMM 4's product.
    tg = cuda_lib
    A = weights(2048, 1024, 9) * 1024 ** 0.5
    A_keep = A.clone()
    B1, W2 = weights(2048, 1024, 10), weights(1024, 1024, 11)
    X = weights(2048, 1024, 12) * 1024 ** 0.5
    p1 = tg.Plan(2048, 2048, 1024, "f16", "f16", (256, 256, 64), 6, pair=True)
    p2 = tg.Plan(2048, 1024, 1024, "f16", "f16", (256, 256, 64), 3)
    C1_ref, A2_ref, C_ref = nan_like(2048, 2048), nan_like(2048, 1024), nan_like(2048, 2048)
    p1.run(A_keep, B1, C1_ref)
    p2.run(X, W2, A2_ref)
    p1.run(X, B1, C_ref)
    torch.cuda.synchronize()
    for _ in range(3):
        Abuf = A_keep.clone()
        C1, C = nan_like(2048, 2048), nan_like(2048, 2048)
        torch.cuda.synchronize()
        p1.run(Abuf, B1, C1)   # reads Abuf
        p2.run(X, W2, Abuf)    # overwrites Abuf
        p1.run(Abuf, B1, C)    # C from the new Abuf ...
        p1.run(X, B1, C)       # ... then overwritten from X
        torch.cuda.synchronize()
        assert torch.equal(bits(C1), bits(C1_ref))
        assert torch.equal(bits(Abuf), bits(A2_ref))
        assert torch.equal(bits(C), bits(C_ref))
    for p in (p1, p2):
        assert p.status()[0] == 0
        p.close()
