"""The tcgen05 tensor-core pipeline of the prefill path, checked on its own.

awq_gemm_f16 runs the prefill kernel with an already dequantised fp16 W
loaded by TMA (no dequant stage): y = x . W + bias. It is compared with the
exact product of the same fp16 inputs (a float64 library matmul), within the
forward tolerance 1e-3 + 4e-3 |y|. Shapes cover one tile and one k-stage,
several tiles and stages, and ragged M, N and K edges. Structured inputs
(one-hot rows of x, one-hot columns of W) pin the row and column mapping of
the accumulator.
"""
import numpy as np
import pytest
import torch

import bit_weight_quantized_awq_gb300 as awq
from bit_weight_quantized_awq_gb300 import Status

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 4e-3


def gemm(x, W, bias=None):
    M, K = x.shape
    N = W.shape[1]
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device=x.device)
    st = awq.awq_gemm_f16(x.data_ptr(), W.data_ptr(), None if bias is None else bias.data_ptr(),
                          y.data_ptr(), M, K, N, torch.cuda.current_stream().cuda_stream)
    assert st == Status.OK, awq.awq_status_string(st)
    torch.cuda.synchronize()
    return y


def check(y, ref):
    y = y.double().cpu().numpy()
    ref = ref.cpu().numpy()
    bad = ~(np.abs(y - ref) <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{bad.sum()} of {bad.size} differ; first {np.argwhere(bad)[:4].tolist()}"


@pytest.mark.parametrize("M,K,N,bias", [
    (128, 64, 256, False),     # one tile, one stage
    (128, 1024, 256, True),    # one tile, 16 stages
    (384, 512, 768, False),    # several tiles both ways
    (200, 1040, 288, True),    # ragged M, N (9 x 32) and K (16 past a stage)
    (1, 64, 32, False),        # smallest
])
def test_gemm_f16_matches_exact_product(gpu, M, K, N, bias):
    g = torch.Generator().manual_seed(M + K + N)
    x = torch.randn((M, K), generator=g).half()
    W = (0.05 * torch.randn((K, N), generator=g)).half()
    b = (0.1 * torch.randn((N,), generator=g)).half() if bias else None
    y = gemm(x.cuda(), W.cuda(), None if b is None else b.cuda())
    ref = x.double() @ W.double()
    if b is not None:
        ref = ref + b.double()
    check(y, ref)


def test_gemm_f16_row_and_column_mapping(gpu):
    """x = identity rows picks W's rows; W = identity picks x's columns."""
    M = K = 128
    N = 256
    g = torch.Generator().manual_seed(5)
    W = torch.randn((K, N), generator=g).half()
    y = gemm(torch.eye(M, K).half().cuda(), W.cuda())
    assert torch.equal(y.cpu(), W[:M])
    x = torch.randn((M, K), generator=g).half()
    eye = torch.zeros((K, N)).half()
    eye[:, :K] = torch.eye(K).half()
    y = gemm(x.cuda(), eye.cuda())
    assert torch.equal(y[:, :K].cpu(), x)
    assert torch.count_nonzero(y[:, K:]) == 0


def test_gemm_f16_argument_rules(gpu):
    A, B = 0x10000, 0x20000
    assert awq.awq_gemm_f16(A, A, None, B, 4, 100, 256, None) == Status.ERR_INVALID_ARG  # K % 16
    assert awq.awq_gemm_f16(A, A, None, B, 4, 64, 40, None) == Status.ERR_INVALID_ARG    # N % 32
    assert awq.awq_gemm_f16(A + 2, A, None, B, 4, 64, 256, None) == Status.ERR_MISALIGNED
    assert awq.awq_gemm_f16(None, None, None, None, 0, 64, 256, None) == Status.OK


@pytest.mark.parametrize("M,K,N,bias", [
    (128, 8192, 512, True),    # 2 tiles split along k between 32 CTAs
    (300, 2048, 1056, False),  # ragged tiles, pieces of 8 k-stages
])
def test_gemm_f16_stream_k_tiles(gpu, M, K, N, bias):
    """Fewer tiles than SMs: the k-stages of each tile are split between
    CTAs and the partial sums added by whichever contributor finishes last;
    the result must not depend on which one that was."""
    g = torch.Generator().manual_seed(M + K + N + 1)
    x = torch.randn((M, K), generator=g).half()
    W = (0.05 * torch.randn((K, N), generator=g)).half()
    b = (0.1 * torch.randn((N,), generator=g)).half() if bias else None
    xc, Wc, bc = x.cuda(), W.cuda(), None if b is None else b.cuda()
    y = gemm(xc, Wc, bc)
    ref = x.double() @ W.double()
    if b is not None:
        ref = ref + b.double()
    check(y, ref)
    for _ in range(3):
        assert torch.equal(gemm(xc, Wc, bc).view(torch.int16), y.view(torch.int16))
