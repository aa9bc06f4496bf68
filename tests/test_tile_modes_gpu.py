"""Both tile shapes of the tcgen05 kernels against the oracle.

The library picks, per call, single-CTA 128-row tiles or CTA-pair 256-row
tiles (two CTAs of a cluster sharing one cta_group::2 MMA, each holding half
of B).  SWG_TILE_MODE forces one or the other so both are checked on the same
ragged shapes, all four op combinations, and the fused SwiGLU epilogue.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import Guarded, check_f32, check_half, padded, round_up, to_f64

pytestmark = pytest.mark.gpu

MODES = ["1cta", "2cta128", "2cta256"]


@pytest.fixture
def tile_mode(request, monkeypatch):
    monkeypatch.setenv("SWG_TILE_MODE", request.param)
    return request.param


@pytest.mark.parametrize("tile_mode", MODES, indirect=True)
@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("shape", [(256, 256, 128), (300, 520, 200), (129, 392, 72),
                                   (1000, 640, 1024), (64, 256, 64)])
def test_gemm_tile_modes(tile_mode, tA, tB, shape):
    M, N, K = shape
    g = synth.generator(M * 7 + N * 3 + K + 11 * tA + 13 * tB)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g)
    C = synth.normal((M, N), g)
    lda, ldb, ldc = round_up(A.shape[1], 8), round_up(B.shape[1], 8), round_up(N, 8)
    Ap, Bp, Cp = padded(A, lda, 2.0), padded(B, ldb, 2.0), padded(C, ldc, 4.0)
    Cg = Guarded(M, N, torch.bfloat16, init=C, ld=ldc)
    swg.gemm(tA, tB, M, N, K, 0.5, Ap.cuda(), lda, Bp.cuda(), ldb, 1.0, Cg.view, ldc, swg.BF16)
    assert swg.get_device_error() == 0
    out = Cg.cpu(f"{tile_mode} {shape}")
    yhat = oracle.gemm(tA, tB, M, N, K, 0.5, Ap, lda, Bp, ldb, 1.0, Cp, ldc)
    check_half(to_f64(out), yhat, f"{tile_mode} {shape} tA={tA} tB={tB}")


@pytest.mark.parametrize("tile_mode", MODES, indirect=True)
@pytest.mark.parametrize("M,K,N", [(256, 256, 128), (300, 136, 520), (640, 896, 1216)])
def test_swiglu_tile_modes(tile_mode, M, K, N):
    A, W1, W2 = synth.swiglu(M, K, N, seed=M + K, w_std=0.08)
    Wf = torch.from_numpy(oracle.interleave(W1, W2, K, N).view(np.int16)).view(torch.bfloat16)
    Y = Guarded(M, N, torch.bfloat16, ld=N)
    swg.swiglu_mlp(A.cuda(), Wf.cuda(), Y.view, M, N, K)
    assert swg.get_device_error() == 0
    check_half(to_f64(Y.cpu(f"{tile_mode} swiglu")), oracle.swiglu(A, W1, W2, M, N, K),
               f"{tile_mode} swiglu {M}x{K}x{N}")


@pytest.mark.parametrize("tile_mode", ["1cta", "2cta256"], indirect=True)
def test_square_4096_tile_modes(tile_mode):
    M = N = K = 4096
    A, B, _ = synth.gemm_bf16(M, N, K, 0, 0, seed=1)
    D = Guarded(M, N, torch.bfloat16, ld=N)
    swg.gemm(0, 0, M, N, K, 1.0, A.cuda(), K, B.cuda(), N, 0.0, D.view, N, swg.BF16)
    assert swg.get_device_error() == 0
    rows = [0, 127, 128, 255, 256, 2049, M - 257, M - 256, M - 1]
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, rows=rows)
    check_half(to_f64(D.cpu(f"{tile_mode} 4096^3"))[rows], yhat, f"{tile_mode} 4096^3")


@pytest.mark.parametrize("tile_mode", ["1cta", "2cta128", "2cta256"], indirect=True)
@pytest.mark.parametrize("split_k", [2, 3])
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1), (0, 1)])
def test_split_k_both_tile_shapes(tile_mode, split_k, tA, tB):
    """Split-K partials from single-CTA and CTA-pair tiles (M > 64, so the
    operands are not swapped), reduced in split order."""
    M, N, K = 300, 520, 1000
    g = synth.generator(400 + split_k + 3 * tA + tB)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g)
    C = synth.normal((M, N), g)
    lda, ldb = round_up(A.shape[1], 8), round_up(B.shape[1], 8)
    Ap, Bp = padded(A, lda, 2.0), padded(B, ldb, 2.0)
    Cg = Guarded(M, N, torch.bfloat16, init=C)
    swg.gemm_ex(tA, tB, M, N, K, 0.75, Ap.cuda(), lda, Bp.cuda(), ldb, 0.5, Cg.view, Cg.ld,
                swg.BF16, split_k)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(tA, tB, M, N, K, 0.75, Ap, lda, Bp, ldb, 0.5, C, N)
    check_half(to_f64(Cg.cpu(f"{tile_mode} split")), yhat,
               f"{tile_mode} split={split_k} tA={tA} tB={tB}")


@pytest.mark.parametrize("tile_mode", MODES, indirect=True)
@pytest.mark.parametrize("code", ["BF16", "BF16_F32OUT"])
@pytest.mark.parametrize("shape", [(300, 520, 200), (129, 392, 72), (1000, 648, 1024),
                                   (17, 136, 64), (300, 517, 200), (260, 130, 96)])
def test_beta_zero_edges_and_padding(tile_mode, code, shape):
    """beta = 0: each CTA's last tile is staged in shared memory and written
    with TMA stores clipped at the output's bounds (rows ending mid-granule,
    N * size not a multiple of 16 bytes, keep the direct stores).  Ragged M
    and N with a padded ldc: every output element matches the oracle and no
    byte of the padding columns changes."""
    M, N, K = shape
    dt = getattr(swg, code)
    g = synth.generator(900 + M + N + K + dt)
    A = synth.normal((M, K), g)
    B = synth.normal((K, N), g)
    out_t = torch.float32 if dt == swg.BF16_F32OUT else torch.bfloat16
    ldb = round_up(N, 8)
    Bp = padded(B, ldb, 3.0)
    ldc = round_up(N + 24, 8)
    Dg = Guarded(M, N, out_t, fill=7.0, ld=ldc)
    swg.gemm(0, 0, M, N, K, 1.0, A.cuda(), K, Bp.cuda(), ldb, 0.0, Dg.view, ldc, dt)
    assert swg.get_device_error() == 0
    out = Dg.cpu(f"{tile_mode} {shape} staged stores")
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, Bp, ldb, 0.0)
    if dt == swg.BF16_F32OUT:
        check_f32(to_f64(out), yhat, K, f"{tile_mode} {shape} f32 out")
    else:
        check_half(to_f64(out), yhat, f"{tile_mode} {shape} bf16 out")
