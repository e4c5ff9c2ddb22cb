"""The tcgen05 GEMM engine in isolation, against a float64 matmul of the same bf16 inputs."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _ref(A, B, mn):
    Bk = B.double() if mn in (0, 3, 5, 6, 7, 8) else B.double().T
    return A.double() @ Bk.T


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (128, 256, 64), (200, 136, 200), (16, 64, 64),
                                   (300, 1000, 2816)])
@pytest.mark.parametrize("mn", [0, 1, 3])
def test_gemm_matches_matmul(M, N, K, mn):
    from block_diffusion_text_gb300 import dg
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn((N, K) if mn in (0, 3) else (K, N), device="cuda", generator=g).to(torch.bfloat16)
    D = dg.debug_gemm(A, B, mn)
    torch.cuda.synchronize()
    ref = _ref(A, B, mn)
    err = (D.double() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (16, 64, 64), (300, 2816, 256), (512, 200, 640)])
def test_pair_gemm_mn_major_b(M, N, K):
    """The CTA-pair engine with B [K][N] (each CTA holds 128 of the 256 columns of a tile)."""
    from block_diffusion_text_gb300 import dg
    g = torch.Generator(device="cuda").manual_seed(M + 3 * N)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, device="cuda", generator=g).to(torch.bfloat16)
    D = dg.debug_gemm(A, B, 4)
    torch.cuda.synchronize()
    ref = _ref(A, B, 4)
    err = (D.double() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err


@pytest.mark.parametrize("M,N,K", [(256, 4096, 2816), (256, 1024, 1024), (200, 136, 512), (16, 64, 256),
                                   (300, 200, 1000)])
@pytest.mark.parametrize("mode", [5, 6, 7, 8])
def test_cluster_splitk_gemm(M, N, K, mode):
    """The cluster split-K engine of the small projections: 2 or 4 CTAs of a cluster compute the K
    slices of one tile and sum them in the owners' shared memory (ragged M, N and K included)."""
    from block_diffusion_text_gb300 import dg
    g = torch.Generator(device="cuda").manual_seed(M * 5 + N + mode)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    D = dg.debug_gemm(A, B, mode)
    torch.cuda.synchronize()
    ref = _ref(A, B, mode)
    err = (D.double() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err
