"""Split-K parity and determinism.

Skinny GEMM (M = 16, 32, 64; N = 4096; K = 16384; alpha = 1, beta = 1 with a
bf16 C) runs with the K loop split across CTAs and the FP32 partials reduced
in split order by a second kernel ("为什么 GEMM 是 CUDA 的必修课", 关键技术
item 5).  The reduction order is fixed, so repeated calls must give identical
bits.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import check_half, to_f64

pytestmark = pytest.mark.gpu


def _skinny(M, seed=4):
    A, B, C = synth.skinny(M, seed=seed)
    return A, B, C


@pytest.mark.parametrize("M", [16, 32, 64])
def test_skinny_full_config(M):
    N, K = 4096, 16384
    A, B, C = _skinny(M)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = C.cuda()
    swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, Cd, N, swg.BF16)
    assert swg.get_device_error() == 0
    rows = list(range(M)) if M == 16 else [0, 1, M // 2, M - 1]
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N, rows=rows)
    check_half(to_f64(Cd)[rows], yhat, f"skinny M={M}")


@pytest.mark.parametrize("M", [16, 64])
def test_skinny_bitwise_deterministic(M):
    N, K = 4096, 16384
    A, B, C = _skinny(M, seed=12)
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for _ in range(3):
        Cd = C.cuda()
        swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, Cd, N, swg.BF16)
        outs.append(Cd.cpu())
    assert swg.get_device_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("split_k", [1, 2, 3, 7, 16])
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_forced_splits_ragged(split_k, tA, tB):
    """Explicit split factors on a ragged shape; K blocks do not divide evenly."""
    M, N, K = 40, 600, 1000
    g = synth.generator(60 + split_k)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g)
    C = synth.normal((M, N), g)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    swg.gemm_ex(tA, tB, M, N, K, 0.5, Ad, A.shape[1], Bd, B.shape[1], 2.0, Cd, N, swg.BF16,
                split_k)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(tA, tB, M, N, K, 0.5, A, A.shape[1], B, B.shape[1], 2.0, C, N)
    check_half(to_f64(Cd), yhat, f"split_k={split_k} tA={tA} tB={tB}")


def test_split_f32_output_and_beta_zero_nan():
    M, N, K = 48, 4096, 8192
    A, B, _ = synth.gemm_bf16(M, N, K, seed=66)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    swg.gemm_ex(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 0.0, Cd, N, swg.BF16_F32OUT, 8)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, rows=[0, 17, 47])
    y = to_f64(Cd)[[0, 17, 47]]
    assert np.isfinite(to_f64(Cd)).all()
    scale = np.abs(yhat).max()
    assert np.abs(y - yhat).max() <= 1e-4 * np.sqrt(K) * scale


def test_split_and_unsplit_agree():
    M, N, K = 32, 2048, 4096
    A, B, C = synth.gemm_bf16(M, N, K, seed=70, c=True)
    Ad, Bd = A.cuda(), B.cuda()
    D1 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    D2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    swg.gemm_ex(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 0.0, D1, N, swg.BF16_F32OUT, 1)
    swg.gemm_ex(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 0.0, D2, N, swg.BF16_F32OUT, 9)
    torch.cuda.synchronize()
    d = (D1 - D2).abs().max().item()
    assert d <= 1e-4 * np.sqrt(K) * D1.abs().max().item()


@pytest.mark.parametrize("M", [1, 7, 16, 17, 33, 64])
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1)])
@pytest.mark.parametrize("split_k", [0, 4])
def test_few_rows_swapped_operands(M, tA, tB, split_k):
    """M <= 64 with a split K runs the transposed product (the large operand
    on the MMA's 128 rows); ragged N and K, beta != 0."""
    N, K = 520, 2056
    g = synth.generator(200 + M + 2 * tA + tB + split_k)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g)
    C = synth.normal((M, N), g)
    lda = ((A.shape[1] + 7) // 8) * 8
    from helpers import padded
    Ap = padded(A, lda, 7.0)
    Cd = torch.zeros((M, 528), dtype=torch.bfloat16)
    Cd[:, :N] = C
    Cd = Cd.cuda()
    swg.gemm_ex(tA, tB, M, N, K, 1.25, Ap.cuda(), lda, B.cuda(), B.shape[1], -0.5, Cd, 528,
                swg.BF16, split_k)
    assert swg.get_device_error() == 0
    out = Cd.cpu()
    assert torch.all(out[:, N:] == 0)
    yhat = oracle.gemm(tA, tB, M, N, K, 1.25, Ap, lda, B, B.shape[1], -0.5, C, N)
    check_half(to_f64(out[:, :N]), yhat, f"swapped M={M} tA={tA} tB={tB} split={split_k}")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_decode_gemv_shapes(M, tA, tB):
    """Decode-time GEMV: M = 1..8 rows against a 4096 x 4096 weight (about one
    FLOP per byte, "GEMM o Coração Matemático" §14), every output checked."""
    N = K = 4096
    g = synth.generator(300 + M + 2 * tA + tB)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g)
    lda = ((A.shape[1] + 7) // 8) * 8
    from helpers import padded
    Ap = padded(A, lda, 5.0)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    swg.gemm(tA, tB, M, N, K, 1.0, Ap.cuda(), lda, B.cuda(), B.shape[1], 0.0, D, N, swg.BF16)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(tA, tB, M, N, K, 1.0, Ap, lda, B, B.shape[1], 0.0)
    check_half(to_f64(D), yhat, f"gemv M={M} tA={tA} tB={tB}")
