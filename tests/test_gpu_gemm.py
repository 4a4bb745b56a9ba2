"""The layer's tensor-core GEMM (dualkv_gemm, csrc/gemm.cu) against fp64
products of the same bf16 inputs (torch on the CPU), for its three operand
layouts, with ragged tiles in every dimension, the residual add, K = 0, and
two calls in a row on a persistent grid of more tiles than SMs.  Outputs of
more than two 256 x 256 tiles per SM take the 256-row tile kernel, smaller
ones the 128-row kernel; both are covered.

Bounds: bf16 results are one rounding of an fp32 sum, so rel-L2 <= 4e-3
(the RMS relative error of bf16 rounding is about 1.1e-3); fp32 results
(kind 2) rel-L2 <= 1e-5."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _bf16(shape, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def _rel(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("M,N,K", [(300, 264, 200), (1024, 768, 512), (128, 256, 64), (17, 8, 8), (4096, 512, 72)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_kind0_x_wT(M, N, K, accumulate):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    A, B, Y0 = _bf16((M, K), 1), _bf16((N, K), 2), _bf16((M, N), 3)
    Y = Y0.cuda() if accumulate else torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    D.dualkv_gemm(0, A.cuda(), B.cuda(), Y, accumulate=accumulate)
    ref = A.double() @ B.double().T + (Y0.double() if accumulate else 0.0)
    assert D.dualkv_last_device_error()[0] == 0
    assert torch.isfinite(Y.float()).all()
    assert _rel(Y, ref) <= 4e-3


@pytest.mark.parametrize("M,N,K", [(300, 264, 200), (1000, 512, 384), (17, 8, 8)])
def test_kind1_dy_w(M, N, K):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    A, B = _bf16((M, K), 4), _bf16((K, N), 5)
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    D.dualkv_gemm(1, A.cuda(), B.cuda(), Y)
    assert D.dualkv_last_device_error()[0] == 0
    assert _rel(Y, A.double() @ B.double()) <= 4e-3


@pytest.mark.parametrize("M,N,K", [(264, 136, 300), (512, 768, 1000), (8, 8, 17), (256, 256, 0)])
def test_kind2_dyT_x(M, N, K):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    A, B = _bf16((K, M), 6), _bf16((K, N), 7)
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    D.dualkv_gemm(2, A.cuda(), B.cuda(), Y)
    assert D.dualkv_last_device_error()[0] == 0
    ref = A.double().T @ B.double()
    if K == 0:
        assert torch.equal(Y.cpu(), torch.zeros(M, N))
    else:
        assert _rel(Y, ref) <= 1e-5


def test_many_tiles_twice_in_a_row():
    """More tiles than SMs (each CTA walks several tiles through both TMEM
    accumulators); a second call on the same buffers gives the same bits."""
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    M, N, K = 8192, 2048, 256
    A, B = _bf16((M, K), 8).cuda(), _bf16((N, K), 9).cuda()
    Y1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Y2 = torch.empty_like(Y1)
    D.dualkv_gemm(0, A, B, Y1)
    D.dualkv_gemm(0, A, B, Y2)
    assert D.dualkv_last_device_error()[0] == 0
    assert torch.equal(Y1, Y2)
    rows = torch.arange(0, M, 97)
    assert _rel(Y1[rows], A[rows].double() @ B.double().T) <= 4e-3


@pytest.mark.parametrize("kind", [0, 1, 2])
def test_256_row_tiles_with_ragged_edges(kind):
    """M = 19000, N = 2056: 675 tiles of 256 x 256, so the 256-row kernel runs,
    with partial tiles at the M and N edges (and K not a multiple of 64)."""
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    M, N, K = 19000, 2056, 200
    if kind == 0:
        A, B = _bf16((M, K), 10), _bf16((N, K), 11)
        ref = A.double() @ B.double().T
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    elif kind == 1:
        A, B = _bf16((M, K), 12), _bf16((K, N), 13)
        ref = A.double() @ B.double()
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    else:
        A, B = _bf16((K, M), 14), _bf16((K, N), 15)
        ref = A.double().T @ B.double()
        Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    D.dualkv_gemm(kind, A.cuda(), B.cuda(), Y)
    Y2 = Y.clone()
    D.dualkv_gemm(kind, A.cuda(), B.cuda(), Y2)
    assert D.dualkv_last_device_error()[0] == 0
    assert torch.isfinite(Y.float()).all()
    assert torch.equal(Y, Y2)
    assert _rel(Y, ref) <= (1e-5 if kind == 2 else 4e-3)
