"""GPU building blocks against plain references: the tcgen05 GEMM of the parent
projection (D = A . B^T, bf16 in, fp32 accumulate) against a float64 matmul of the
same bf16 values; the bounded device-side waits against a wait that never ends."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from diffusion_drafter_draft_gb300 import _build
    _build.build()
    import diffusion_drafter_draft_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (1, 128, 64), (200, 256, 200), (64, 4096, 4096),
                                   (768, 512, 4096), (300, 384, 2560),
                                   # 128 x 160 tiles with a 6-stage ring (one wave of 128 CTAs)
                                   (1024, 2560, 512), (1001, 2560, 136)])
def test_tcgen05_gemm_matches_float64(dd, M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D = dd.gemm_bf16(A.cuda(), B.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = A.double() @ B.double().T
    err = (D.cpu().double() - ref).abs().max().item()
    assert err <= 1e-4 * max(1.0, ref.abs().max().item()), err


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_waits_time_out_and_leave_the_context_usable(dd, which):
    """The library's wait helpers wait for something nothing signals (0: an
    mbarrier phase, 1: a grid-barrier target one CTA above the grid); each gives up
    after 20 ms with DARTREE_ETIMEOUT in the status word, and later work runs."""
    import time
    ws = dd.new_workspace(4096, torch.device("cuda"))
    dd.clear_status(ws)
    t0 = time.time()
    dd.selftest_wait(ws, which, 20000)
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    assert dd.read_status(ws) == dd.ETIMEOUT
    dd.clear_status(ws)
    x = torch.randn(4, 1000, device="cuda")
    tok, val = dd.topk(x, 8, ws=ws)
    torch.cuda.synchronize()
    ref = torch.topk(x, 8, dim=1)
    assert torch.equal(val, ref.values)
    assert dd.read_status(ws) == 0
