"""Fused SwiGLU parity: Y = SiLU(A W1) (.) (A W2) as one GEMM over the
interleaved W_fused with the pair-multiply epilogue ("Sobreposição de Ativação
em Nível de Tile para Inferência Eficiente de LLM", Metodologia, Kernel-2),
against the oracle computed from SEPARATE W1 and W2.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import Guarded, check_half, to_f64

pytestmark = pytest.mark.gpu


def _fused_weight(W1, W2, K, N):
    """W_fused from the oracle's interleave (not from the CUDA path)."""
    Wf = oracle.interleave(W1, W2, K, N)
    return torch.from_numpy(Wf.view(np.int16)).view(torch.bfloat16)


def run(M, K, N, seed, rows=None, w_std=0.02):
    A, W1, W2 = synth.swiglu(M, K, N, seed=seed, w_std=w_std)
    Wf = _fused_weight(W1, W2, K, N)
    # Y's row stride is N by contract: guard rows above and below it
    Y = Guarded(M, N, torch.bfloat16, fill=9.0, ld=N)
    swg.swiglu_mlp(A.cuda(), Wf.cuda(), Y.view, M, N, K)
    assert swg.get_device_error() == 0
    yhat = oracle.swiglu(A, W1, W2, M, N, K, rows=rows)
    y = to_f64(Y.cpu(f"swiglu {M}x{K}x{N}"))
    if rows is not None:
        y = y[np.asarray(rows)]
    return y, yhat


@pytest.mark.parametrize("M,K,N", [(128, 64, 128), (1, 8, 8), (100, 200, 48), (300, 136, 520),
                                   (129, 72, 264), (256, 512, 1024)])
def test_swiglu_small_shapes(M, K, N):
    y, yhat = run(M, K, N, seed=M + K + N, w_std=0.1)
    check_half(y, yhat, f"swiglu {M}x{K}x{N}")


@pytest.mark.parametrize("M", [128, 512, 2048])
def test_swiglu_small_model_shape(M):
    """A [M x 896] ~ N(0,1), W1, W2 [896 x 4864] ~ N(0, 0.02); every row up
    to M = 512, at M = 2048 the tile and pair-tile edges plus random rows."""
    rng = np.random.default_rng(M)
    rows = None if M <= 512 else sorted(
        {0, 127, 128, 255, 256, 511, 512, 1023, 1024, M - 257, M - 256, M - 129, M - 128,
         M - 1, *rng.integers(0, M, 8).tolist()})
    y, yhat = run(M, 896, 4864, seed=3, rows=rows)
    check_half(y, yhat, f"small-model M={M}")


@pytest.mark.parametrize("M", [512, 2048, 8192])
def test_swiglu_8b_shape_sampled(M):
    """A [M x 4096] ~ N(0,1), W1, W2 [4096 x 14336] ~ N(0, 0.02); sampled rows:
    the first and last, both sides of the 128-row tile and 256-row pair-tile
    boundaries, the middle, the last full pair tile, and random rows."""
    rng = np.random.default_rng(M + 1)
    rows = sorted({0, 127, 128, 255, 256, M // 2, M - 257, M - 256, M - 1,
                   *rng.integers(0, M, 4).tolist()})
    y, yhat = run(M, 4096, 14336, seed=3, rows=rows)
    check_half(y, yhat, f"8B M={M}")


def test_interleave_kernel_bitwise():
    K, N = 96, 4864
    _, W1, W2 = synth.swiglu(1, K, N, seed=77)
    Wf = swg.interleave_weights(W1.cuda(), W2.cuda())
    torch.cuda.synchronize()
    want = oracle.interleave(W1, W2, K, N)
    assert np.array_equal(Wf.cpu().view(torch.int16).numpy().view(np.uint16), want)


def test_fused_equals_two_gemms_plus_elementwise():
    """The fused kernel against the unfused data flow: two FP32-output GEMMs
    (Gate, Up) from the same library, then SiLU(Gate) * Up in FP64 on the
    host."""
    M, K, N = 384, 896, 640
    A, W1, W2 = synth.swiglu(M, K, N, seed=88, w_std=0.05)
    Ad = A.cuda()
    G = Guarded(M, N, torch.float32)
    U = Guarded(M, N, torch.float32)
    swg.gemm(0, 0, M, N, K, 1.0, Ad, K, W1.cuda(), N, 0.0, G.view, G.ld, swg.BF16_F32OUT)
    swg.gemm(0, 0, M, N, K, 1.0, Ad, K, W2.cuda(), N, 0.0, U.view, U.ld, swg.BF16_F32OUT)
    Y = Guarded(M, N, torch.bfloat16, ld=N)
    swg.swiglu_mlp(Ad, _fused_weight(W1, W2, K, N).cuda(), Y.view, M, N, K)
    torch.cuda.synchronize()
    g, u = to_f64(G.cpu("Gate")), to_f64(U.cpu("Up"))
    unfused = g / (1.0 + np.exp(-g)) * u
    check_half(to_f64(Y.cpu("fused")), unfused, "fused vs two GEMMs")


def test_swiglu_k_zero_gives_zero():
    M, N = 64, 64
    Y = Guarded(M, N, torch.bfloat16, fill=3.0, ld=N)
    swg.swiglu_mlp(0, 0, Y.view, M, N, 0)
    torch.cuda.synchronize()
    assert torch.all(Y.cpu("K = 0") == 0)


def test_swiglu_large_magnitudes_finite():
    """Gate values far into both SiLU tails: outputs stay finite and match."""
    M, K, N = 128, 64, 256
    y, yhat = run(M, K, N, seed=91, w_std=8.0)
    check_half(y, yhat, "large gate magnitudes")


def test_swiglu_tails_keep_relative_accuracy():
    """Gates of standard deviation 8 reach |g| of several hundred.  SiLU is
    computed as x / (1 + e^-x), which keeps its relative accuracy in the
    negative tail (a form through 1 + tanh(x/2) cancels to zero there): no
    output may differ from the oracle by more than 1% relative (the measure
    "Sobreposição de Ativação em Nível de Tile para Inferência Eficiente de
    LLM" reports for its fused kernels)."""
    M, K, N = 128, 64, 256
    y, yhat = run(M, K, N, seed=91, w_std=8.0)
    stats = check_half(y, yhat, "tails")
    assert stats["frac_rel_gt_1pct"] == 0.0, stats
    assert stats["max_rel"] < 1e-2, stats


@pytest.mark.parametrize("tile_mode", ["1cta", "2cta256", None])
@pytest.mark.parametrize("M,K,N", [(128, 64, 128), (300, 136, 520), (1, 8, 8), (640, 896, 4864)])
def test_swiglu_separate_weights(monkeypatch, tile_mode, M, K, N):
    """swiglu_mlp_dual: Gate from W1 and Up from W2 in one accumulator, no
    interleaved copy; against the oracle from the same separate weights."""
    if tile_mode:
        monkeypatch.setenv("SWG_TILE_MODE", tile_mode)
    A, W1, W2 = synth.swiglu(M, K, N, seed=M + 2 * N + K, w_std=0.08)
    Y = Guarded(M, N, torch.bfloat16, fill=9.0, ld=N)
    swg.swiglu_mlp_dual(A.cuda(), W1.cuda(), W2.cuda(), Y.view, M, N, K)
    assert swg.get_device_error() == 0
    rows = None if M <= 300 else [0, 127, 128, 255, 256, 383, 384, 511, 512, M - 1]
    yhat = oracle.swiglu(A, W1, W2, M, N, K, rows=rows)
    out = to_f64(Y.cpu(f"dual {tile_mode} {M}x{K}x{N}"))
    y = out if rows is None else out[rows]
    check_half(y, yhat, f"dual {tile_mode} {M}x{K}x{N}")


def test_swiglu_separate_weights_8b_sampled():
    M, K, N = 2048, 4096, 14336
    A, W1, W2 = synth.swiglu(M, K, N, seed=3)
    Y = Guarded(M, N, torch.bfloat16, ld=N)
    swg.swiglu_mlp_dual(A.cuda(), W1.cuda(), W2.cuda(), Y.view, M, N, K)
    assert swg.get_device_error() == 0
    rng = np.random.default_rng(17)
    rows = sorted({0, 127, 128, 255, 256, M // 2, M - 257, M - 256, M - 1,
                   *rng.integers(0, M, 4).tolist()})
    check_half(to_f64(Y.cpu("dual 8B"))[rows], oracle.swiglu(A, W1, W2, M, N, K, rows=rows),
               "dual 8B")
