"""8-bit (e4m3) GEMM and fused SwiGLU with per-tensor scales, against the
oracle on the same stored e4m3 values ("GEMM o Coração Matemático", §12.4 on
quantised operands; the SwiGLU page on the activation's share of the cost
growing with FP8).  A is stored M x K and B (or the interleaved weight)
N x K: both operands K-contiguous, as kind::f8f6f4 reads them here.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import Guarded, check_f32, check_half, to_f64

pytestmark = pytest.mark.gpu


def _e4m3(shape, g, std=1.0):
    return (torch.randn(*shape, generator=g) * std).to(torch.float8_e4m3fn)


@pytest.mark.parametrize("tile_mode", [None, "1cta", "2cta256"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 520, 272), (1000, 640, 1024),
                                   (1, 16, 16), (257, 129, 96)])
def test_fp8_gemm(monkeypatch, tile_mode, M, N, K):
    if tile_mode:
        monkeypatch.setenv("SWG_TILE_MODE", tile_mode)
    g = synth.generator(M + N + K)
    A = _e4m3((M, K), g)
    Bt = _e4m3((N, K), g)
    sa, sb = 0.5, 0.03
    lda = ldb = ((K + 15) // 16) * 16
    Ap = torch.zeros((M, lda), dtype=torch.float8_e4m3fn)
    Ap[:, :K] = A
    Bp = torch.zeros((N, ldb), dtype=torch.float8_e4m3fn)
    Bp[:, :K] = Bt
    C = synth.normal((M, N), g)
    ldc = ((N + 7) // 8) * 8
    Cp = torch.zeros((M, ldc), dtype=torch.bfloat16)
    Cp[:, :N] = C
    Cg = Guarded(M, N, torch.bfloat16, init=C, ld=ldc)
    swg.gemm(0, 1, M, N, K, 1.5 * sa * sb, Ap.cuda(), lda, Bp.cuda(), ldb, 0.5, Cg.view, ldc,
             swg.E4M3_BF16OUT)
    assert swg.get_device_error() == 0
    out = Cg.cpu(f"fp8 gemm {M}x{N}x{K}")
    yhat = oracle.gemm(0, 1, M, N, K, 1.5 * sa * sb, Ap, lda, Bp, ldb, 0.5, Cp, ldc,
                       in_type="e4m3", c_type="bf16")
    check_half(to_f64(out), yhat, f"fp8 gemm {tile_mode} {M}x{N}x{K}")


def test_fp8_gemm_f32_out():
    M, N, K = 256, 384, 512
    g = synth.generator(77)
    A, Bt = _e4m3((M, K), g), _e4m3((N, K), g)
    D = Guarded(M, N, torch.float32)
    swg.gemm(0, 1, M, N, K, 0.25, A.cuda(), K, Bt.cuda(), K, 0.0, D.view, D.ld, swg.E4M3_F32OUT)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(0, 1, M, N, K, 0.25, A, K, Bt, K, 0.0, in_type="e4m3")
    check_f32(to_f64(D.cpu("fp8 f32 out")), yhat, K, "fp8 f32 out")


def test_fp8_square_8192_sampled():
    M = N = K = 8192
    g = synth.generator(1)
    A, Bt = _e4m3((M, K), g), _e4m3((N, K), g)
    D = Guarded(M, N, torch.bfloat16, ld=N)
    swg.gemm(0, 1, M, N, K, 1.0 / 64, A.cuda(), K, Bt.cuda(), K, 0.0, D.view, N,
             swg.E4M3_BF16OUT)
    assert swg.get_device_error() == 0
    out = D.cpu("fp8 8192^3")
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(8192)
    rows = sorted({0, 127, 128, 255, 256, 4097, M - 257, M - 256, M - 1,
                   *rng.integers(0, M, 4).tolist()})
    yhat = oracle.gemm(0, 1, M, N, K, 1.0 / 64, A, K, Bt, K, 0.0, in_type="e4m3", rows=rows)
    check_half(to_f64(out)[rows], yhat, "fp8 8192^3")


def test_fp8_layout_rules():
    P = 0x10000
    lib = swg.load()
    # only op(A) = A, op(B) = B^T; split-K only for M <= 64 (rejected before
    # any CUDA call, so the fake pointers are never used)
    assert lib.gemm_ex(0, 0, 16, 16, 16, 1.0, P, 16, P, 16, 0.0, P, 16, swg.E4M3_BF16OUT, 0, None) == 3
    assert lib.gemm_ex(1, 1, 16, 16, 16, 1.0, P, 16, P, 16, 0.0, P, 16, swg.E4M3_BF16OUT, 0, None) == 3
    assert lib.gemm_ex(0, 1, 65, 16, 16, 1.0, P, 16, P, 16, 0.0, P, 16, swg.E4M3_BF16OUT, 4, None) == 3
    assert lib.gemm_ex(0, 1, 16, 16, 24, 1.0, P, 24, P, 24, 0.0, P, 16, swg.E4M3_BF16OUT, 0, None) == 2


@pytest.mark.parametrize("tile_mode", [None, "1cta", "2cta256"])
@pytest.mark.parametrize("M,K,N", [(128, 128, 128), (300, 256, 520), (640, 896, 4864)])
def test_fp8_swiglu(monkeypatch, tile_mode, M, K, N):
    if tile_mode:
        monkeypatch.setenv("SWG_TILE_MODE", tile_mode)
    A, W1, W2, sw = synth.swiglu_e4m3(M, K, N, seed=M + K + N, w_std=0.05)
    Wt = torch.from_numpy(oracle.interleave_t8(W1, W2, K, N)).view(torch.float8_e4m3fn)
    Y = Guarded(M, N, torch.bfloat16, fill=9.0, ld=N)
    swg.swiglu_mlp_fp8(A.cuda(), Wt.cuda(), Y.view, M, N, K, sw)
    assert swg.get_device_error() == 0
    rows = None if M <= 300 else [0, 127, 128, 255, 256, 383, 384, 511, 512, M - 1]
    yhat = oracle.swiglu_typed(A, W1, W2, M, N, K, in_type="e4m3", scale=sw, rows=rows)
    out = to_f64(Y.cpu(f"fp8 swiglu {M}x{K}x{N}"))
    y = out if rows is None else out[rows]
    check_half(y, yhat, f"fp8 swiglu {tile_mode} {M}x{K}x{N}")


def test_fp8_swiglu_8b_sampled():
    M, K, N = 2048, 4096, 14336
    A, W1, W2, sw = synth.swiglu_e4m3(M, K, N, seed=3)
    Wt = torch.from_numpy(oracle.interleave_t8(W1, W2, K, N)).view(torch.float8_e4m3fn)
    Y = Guarded(M, N, torch.bfloat16, ld=N)
    swg.swiglu_mlp_fp8(A.cuda(), Wt.cuda(), Y.view, M, N, K, sw)
    assert swg.get_device_error() == 0
    rng = np.random.default_rng(2049)
    rows = sorted({0, 127, 128, 255, 256, M // 2, M - 257, M - 256, M - 1,
                   *rng.integers(0, M, 4).tolist()})
    yhat = oracle.swiglu_typed(A, W1, W2, M, N, K, in_type="e4m3", scale=sw, rows=rows)
    check_half(to_f64(Y.cpu("fp8 swiglu 8B"))[rows], yhat, "fp8 swiglu 8B")


@pytest.mark.parametrize("M", [1, 7, 16, 33, 64])
@pytest.mark.parametrize("split_k", [0, 3])
def test_fp8_few_rows_split_k(M, split_k):
    """Few rows (decode): the transposed product with the K loop split and the
    partials reduced in split order; ragged N, beta != 0, bf16 output."""
    N, K = 520, 4096
    g = synth.generator(1300 + M + split_k)
    A = _e4m3((M, K), g)
    Bt = _e4m3((N, K), g)
    C = synth.normal((M, N), g)
    ldc = 528
    Cg = Guarded(M, N, torch.bfloat16, init=C, ld=ldc)
    swg.gemm_ex(0, 1, M, N, K, 1.0 / 32, A.cuda(), K, Bt.cuda(), K, 0.5, Cg.view, ldc,
                swg.E4M3_BF16OUT, split_k)
    assert swg.get_device_error() == 0
    out = Cg.cpu(f"fp8 few rows M={M}")
    yhat = oracle.gemm(0, 1, M, N, K, 1.0 / 32, A, K, Bt, K, 0.5, C, N, in_type="e4m3")
    check_half(to_f64(out), yhat, f"fp8 few rows M={M} split={split_k}")


def test_fp8_decode_gemv_f32_out_deterministic():
    """M = 1 against a 4096 x 4096 e4m3 weight, FP32 output: repeated calls give
    identical bits (fixed reduction order) and match the oracle."""
    M, N, K = 1, 4096, 4096
    g = synth.generator(1310)
    A = _e4m3((M, K), g)
    Bt = _e4m3((N, K), g, std=0.5)
    Ad, Bd = A.cuda(), Bt.cuda()
    outs = []
    for _ in range(3):
        D = torch.empty((M, N), dtype=torch.float32, device="cuda")
        swg.gemm(0, 1, M, N, K, 0.25, Ad, K, Bd, K, 0.0, D, N, swg.E4M3_F32OUT)
        outs.append(D.cpu())
    assert swg.get_device_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    yhat = oracle.gemm(0, 1, M, N, K, 0.25, A, K, Bt, K, 0.0, in_type="e4m3", c_type="f32")
    check_f32(to_f64(outs[0]), yhat, K, "fp8 decode f32")
