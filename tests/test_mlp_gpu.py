"""Full gated MLP through the C ABI against the oracle:
Out = (SiLU(A W1) (.) (A W2)) W_down + beta * Out ("GEMM o Coração
Matemático", §13.3, with the gated activation of the SwiGLU page).

The product stores the gated activation Y in bf16 between its two GEMMs, a
step of its own contract; the oracle takes that step too (its exact Y rounded
once to bf16, round-to-nearest-even) before its down projection.  Y and Out
are then both checked with the plain bf16 bound.  Y and Out sit inside guard
bands (rows above and below; Out's row stride is fixed by the call).
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import Guarded, check_half, to_f64

pytestmark = pytest.mark.gpu


def _weights(K, N, seed, w_std):
    A_, W1, W2 = synth.swiglu(1, K, N, seed=seed, w_std=w_std)
    g = synth.generator(seed + 1)
    Wd = synth.normal((N, K), g, std=w_std)
    Wf = torch.from_numpy(oracle.interleave(W1, W2, K, N).view(np.int16)).view(torch.bfloat16)
    return W1, W2, Wd, Wf


@pytest.mark.parametrize("M,K,N,beta", [(128, 64, 128, 0.0), (300, 136, 520, 1.0),
                                        (64, 256, 1024, 0.0), (640, 896, 4864, 1.0)])
def test_mlp_small(M, K, N, beta):
    W1, W2, Wd, Wf = _weights(K, N, seed=M + N, w_std=0.05)
    A = synth.normal((M, K), synth.generator(M))
    R = synth.normal((M, K), synth.generator(M + 7))
    Y = Guarded(M, N, torch.bfloat16, ld=N)
    Out = Guarded(M, K, torch.bfloat16, init=R, ld=K)
    swg.swiglu_mlp_forward(A.cuda(), Wf.cuda(), Wd.cuda(), Y.view, Out.view, M, N, K, beta)
    assert swg.get_device_error() == 0
    rows = None if M <= 300 else [0, 1, 127, 128, 255, 256, 511, 512, M - 1]
    y_all, out_all = to_f64(Y.cpu("Y")), to_f64(Out.cpu("Out"))
    check_half(y_all if rows is None else y_all[rows],
               oracle.swiglu(A, W1, W2, M, N, K, rows=rows), "Y")
    yhat = oracle.mlp(A, W1, W2, Wd, M, N, K, beta=beta, Out_old=R, rows=rows, round_y=True)
    check_half(out_all if rows is None else out_all[rows], yhat,
               f"mlp {M}x{K}x{N} beta={beta}")


def test_mlp_8b_shape_sampled():
    """A [512 x 4096], W1, W2 [4096 x 14336], W_down [14336 x 4096], residual."""
    M, K, N = 512, 4096, 14336
    W1, W2, Wd, Wf = _weights(K, N, seed=3, w_std=0.02)
    A = synth.normal((M, K), synth.generator(9))
    R = synth.normal((M, K), synth.generator(10))
    Y = Guarded(M, N, torch.bfloat16, ld=N)
    Out = Guarded(M, K, torch.bfloat16, init=R, ld=K)
    swg.swiglu_mlp_forward(A.cuda(), Wf.cuda(), Wd.cuda(), Y.view, Out.view, M, N, K, 1.0)
    assert swg.get_device_error() == 0
    rows = [0, 127, 128, 255, 256, 383, M - 2, M - 1]
    y_all, out_all = to_f64(Y.cpu("Y 8B")), to_f64(Out.cpu("Out 8B"))
    check_half(y_all[rows], oracle.swiglu(A, W1, W2, M, N, K, rows=rows), "Y 8B")
    yhat = oracle.mlp(A, W1, W2, Wd, M, N, K, beta=1.0, Out_old=R, rows=rows, round_y=True)
    check_half(out_all[rows], yhat, "mlp 8B")


def test_mlp_rejects_before_launch():
    before = swg.launch_count()
    Y = torch.empty((8, 8), dtype=torch.bfloat16, device="cuda")
    Out = torch.empty((8, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(swg.SwgError) as e:
        swg.swiglu_mlp_forward(Y, Y, Y, Y, Out, 8, 12, 8)     # N % 8 != 0
    assert e.value.status == 2
    assert swg.launch_count() == before


@pytest.mark.parametrize("M,K,N", [(1, 896, 4864), (2, 136, 520), (1, 4096, 14336)])
def test_mlp_decode_rows(M, K, N):
    """Decode: one or two rows through the whole MLP, two launches (the
    one-or-two-rows kernel for the SwiGLU and again for the down projection,
    beta = 1 residual), every output against the oracle."""
    W1, W2, Wd, Wf = _weights(K, N, seed=40 + M + K, w_std=0.02)
    A = synth.normal((M, K), synth.generator(41 + M))
    R = synth.normal((M, K), synth.generator(42 + M))
    Y = Guarded(M, N, torch.bfloat16, ld=N)
    Out = Guarded(M, K, torch.bfloat16, init=R, ld=K)
    before = swg.launch_count()
    swg.swiglu_mlp_forward(A.cuda(), Wf.cuda(), Wd.cuda(), Y.view, Out.view, M, N, K, 1.0)
    assert swg.launch_count() - before == 2
    assert swg.get_device_error() == 0
    check_half(to_f64(Y.cpu("Y decode")), oracle.swiglu(A, W1, W2, M, N, K), "Y")
    yhat = oracle.mlp(A, W1, W2, Wd, M, N, K, beta=1.0, Out_old=R, round_y=True)
    check_half(to_f64(Out.cpu("Out decode")), yhat, f"mlp decode {M}x{K}x{N}")
