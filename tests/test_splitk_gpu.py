"""Split-K parity and determinism.

Skinny GEMM (M = 16, 32, 64; N = 4096; K = 16384; alpha = 1, beta = 1 with a
bf16 C) runs with the K loop split across CTAs and the FP32 partials reduced
in split order by a second kernel ("为什么 GEMM 是 CUDA 的必修课", 关键技术
item 5).  The reduction order is fixed, so repeated calls must give identical
bits.

Every output sits inside guard bands (rows above and below, columns past N),
and the split-K workspaces are created with guard bands of their own
(SWG_TEST_WS_GUARD=1, on a stream of the test's own so that its workspace is
made under the switch); both must be untouched after the calls.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import Guarded, check_f32, check_half, padded, to_f64

pytestmark = pytest.mark.gpu


def _skinny(M, seed=4):
    A, B, C = synth.skinny(M, seed=seed)
    return A, B, C


@pytest.fixture
def guarded_ws(monkeypatch):
    """A fresh stream whose split-K workspace is made with guard bands; the
    guards are checked after the test body."""
    monkeypatch.setenv("SWG_TEST_WS_GUARD", "1")
    s = torch.cuda.Stream()
    yield s
    s.synchronize()
    assert swg.debug_workspace_guards(s) == 0


@pytest.mark.parametrize("M", [16, 32, 64])
def test_skinny_full_config(M, guarded_ws):
    """The skinny benchmark shapes (ldc = N, as timed), every output row."""
    N, K = 4096, 16384
    A, B, C = _skinny(M)
    Ad, Bd = A.cuda(), B.cuda()
    Cg = Guarded(M, N, torch.bfloat16, init=C, ld=N)
    swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, Cg.view, N, swg.BF16, stream=guarded_ws)
    assert swg.get_device_error(guarded_ws) == 0
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N)
    check_half(to_f64(Cg.cpu(f"skinny M={M}")), yhat, f"skinny M={M}")


@pytest.mark.parametrize("M", [16, 64])
def test_skinny_bitwise_deterministic(M):
    N, K = 4096, 16384
    A, B, C = _skinny(M, seed=12)
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for _ in range(3):
        Cg = Guarded(M, N, torch.bfloat16, init=C)
        swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, Cg.view, Cg.ld, swg.BF16)
        outs.append(Cg.cpu("repeat"))
    assert swg.get_device_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("split_k", [1, 2, 3, 7, 16])
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_forced_splits_ragged(split_k, tA, tB, guarded_ws):
    """Explicit split factors on a ragged shape; K blocks do not divide evenly."""
    M, N, K = 40, 600, 1000
    g = synth.generator(60 + split_k)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g)
    C = synth.normal((M, N), g)
    Ad, Bd = A.cuda(), B.cuda()
    Cg = Guarded(M, N, torch.bfloat16, init=C)
    swg.gemm_ex(tA, tB, M, N, K, 0.5, Ad, A.shape[1], Bd, B.shape[1], 2.0, Cg.view, Cg.ld,
                swg.BF16, split_k, stream=guarded_ws)
    assert swg.get_device_error(guarded_ws) == 0
    yhat = oracle.gemm(tA, tB, M, N, K, 0.5, A, A.shape[1], B, B.shape[1], 2.0, C, N)
    check_half(to_f64(Cg.cpu("forced split")), yhat, f"split_k={split_k} tA={tA} tB={tB}")


@pytest.mark.parametrize("split_k", [2, 5])
@pytest.mark.parametrize("M,N", [(300, 520), (129, 264), (640, 384)])
def test_forced_splits_unswapped_tiles(split_k, M, N, guarded_ws):
    """M > 64 with a forced split: the 128- or 256-row split-K tiles whose
    last partial tile leaves through a 3-D TMA store into the workspace."""
    K = 1224
    g = synth.generator(80 + M + split_k)
    A = synth.normal((M, K), g)
    B = synth.normal((K, N), g)
    C = synth.normal((M, N), g)
    Cg = Guarded(M, N, torch.bfloat16, init=C)
    swg.gemm_ex(0, 0, M, N, K, 1.0, A.cuda(), K, B.cuda(), N, 0.5, Cg.view, Cg.ld, swg.BF16,
                split_k, stream=guarded_ws)
    assert swg.get_device_error(guarded_ws) == 0
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.5, C, N)
    check_half(to_f64(Cg.cpu("unswapped split")), yhat, f"split_k={split_k} {M}x{N}")


def test_split_f32_output_and_beta_zero_nan():
    M, N, K = 48, 4096, 8192
    A, B, _ = synth.gemm_bf16(M, N, K, seed=66)
    Ad, Bd = A.cuda(), B.cuda()
    Cg = Guarded(M, N, torch.float32, fill=float("nan"))
    swg.gemm_ex(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 0.0, Cg.view, Cg.ld, swg.BF16_F32OUT, 8)
    assert swg.get_device_error() == 0
    out = to_f64(Cg.cpu("f32 split"))
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, rows=[0, 17, 47])
    y = out[[0, 17, 47]]
    assert np.isfinite(out).all()
    scale = np.abs(yhat).max()
    assert np.abs(y - yhat).max() <= 1e-4 * np.sqrt(K) * scale


def test_split_and_unsplit_agree():
    M, N, K = 32, 2048, 4096
    A, B, C = synth.gemm_bf16(M, N, K, seed=70, c=True)
    Ad, Bd = A.cuda(), B.cuda()
    G1 = Guarded(M, N, torch.float32)
    G2 = Guarded(M, N, torch.float32)
    swg.gemm_ex(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 0.0, G1.view, G1.ld, swg.BF16_F32OUT, 1)
    swg.gemm_ex(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 0.0, G2.view, G2.ld, swg.BF16_F32OUT, 9)
    torch.cuda.synchronize()
    D1, D2 = G1.cpu("unsplit"), G2.cpu("split 9")
    d = (D1 - D2).abs().max().item()
    assert d <= 1e-4 * np.sqrt(K) * D1.abs().max().item()


@pytest.mark.parametrize("M", [1, 7, 16, 17, 33, 64])
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1)])
@pytest.mark.parametrize("split_k", [0, 4])
def test_few_rows_swapped_operands(M, tA, tB, split_k, guarded_ws):
    """M <= 64 with a split K runs the transposed product (the large operand
    on the MMA's 128 rows); ragged N and K, beta != 0."""
    N, K = 520, 2056
    g = synth.generator(200 + M + 2 * tA + tB + split_k)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g)
    C = synth.normal((M, N), g)
    lda = ((A.shape[1] + 7) // 8) * 8
    Ap = padded(A, lda, 7.0)
    Cg = Guarded(M, N, torch.bfloat16, init=C, ld=528)
    swg.gemm_ex(tA, tB, M, N, K, 1.25, Ap.cuda(), lda, B.cuda(), B.shape[1], -0.5, Cg.view, 528,
                swg.BF16, split_k, stream=guarded_ws)
    assert swg.get_device_error(guarded_ws) == 0
    out = Cg.cpu(f"swapped M={M}")
    yhat = oracle.gemm(tA, tB, M, N, K, 1.25, Ap, lda, B, B.shape[1], -0.5, C, N)
    check_half(to_f64(out), yhat, f"swapped M={M} tA={tA} tB={tB} split={split_k}")


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
    Ap = padded(A, lda, 5.0)
    D = Guarded(M, N, torch.bfloat16, ld=N)
    swg.gemm(tA, tB, M, N, K, 1.0, Ap.cuda(), lda, B.cuda(), B.shape[1], 0.0, D.view, N, swg.BF16)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(tA, tB, M, N, K, 1.0, Ap, lda, B, B.shape[1], 0.0)
    check_half(to_f64(D.cpu("decode")), yhat, f"gemv M={M} tA={tA} tB={tB}")
