"""GPU building blocks against plain references: the tcgen05 GEMM of the parent
projection (D = A . B^T, bf16 in, fp32 accumulate) against a float64 matmul of the
same bf16 values."""
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
