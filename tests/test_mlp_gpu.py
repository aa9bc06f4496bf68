"""Full gated MLP through the C ABI against the oracle:
Out = (SiLU(A W1) (.) (A W2)) W_down + beta * Out ("GEMM o Coração
Matemático", §13.3, with the gated activation of the SwiGLU page).

The product stores the gated activation Y in bf16 before the down projection;
the oracle keeps it in double.  Y itself is checked with the bf16 bound; Out
with that bound plus the propagated rounding of Y, 2^-8 * sum_n |Y_n| |W_down|.
"""


def _prop_bound(A, W1, W2, Wd, M, N, K, rows):
    Y = oracle.swiglu(A, W1, W2, M, N, K, rows=rows)
    return 2.0 ** -8 * (np.abs(Y) @ np.abs(Wd.to(torch.float64).numpy()))
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import check_half, check_two_stage, to_f64

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
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Out = R.cuda()
    swg.swiglu_mlp_forward(A.cuda(), Wf.cuda(), Wd.cuda(), Y, Out, M, N, K, beta)
    assert swg.get_device_error() == 0
    rows = None if M <= 300 else [0, 1, 255, 256, M - 1]
    check_half(to_f64(Y) if rows is None else to_f64(Y)[rows],
               oracle.swiglu(A, W1, W2, M, N, K, rows=rows), "Y")
    yhat = oracle.mlp(A, W1, W2, Wd, M, N, K, beta=beta, Out_old=R, rows=rows)
    out = to_f64(Out) if rows is None else to_f64(Out)[rows]
    check_two_stage(out, yhat, _prop_bound(A, W1, W2, Wd, M, N, K, rows),
                    f"mlp {M}x{K}x{N} beta={beta}")


def test_mlp_8b_shape_sampled():
    """A [512 x 4096], W1, W2 [4096 x 14336], W_down [14336 x 4096], residual."""
    M, K, N = 512, 4096, 14336
    W1, W2, Wd, Wf = _weights(K, N, seed=3, w_std=0.02)
    A = synth.normal((M, K), synth.generator(9))
    R = synth.normal((M, K), synth.generator(10))
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Out = R.cuda()
    swg.swiglu_mlp_forward(A.cuda(), Wf.cuda(), Wd.cuda(), Y, Out, M, N, K, 1.0)
    assert swg.get_device_error() == 0
    rows = [0, 255, 256, M - 1]
    yhat = oracle.mlp(A, W1, W2, Wd, M, N, K, beta=1.0, Out_old=R, rows=rows)
    check_two_stage(to_f64(Out)[rows], yhat, _prop_bound(A, W1, W2, Wd, M, N, K, rows),
                    "mlp 8B")


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
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Out = R.cuda()
    before = swg.launch_count()
    swg.swiglu_mlp_forward(A.cuda(), Wf.cuda(), Wd.cuda(), Y, Out, M, N, K, 1.0)
    assert swg.launch_count() - before == 2
    assert swg.get_device_error() == 0
    check_half(to_f64(Y), oracle.swiglu(A, W1, W2, M, N, K), "Y")
    yhat = oracle.mlp(A, W1, W2, Wd, M, N, K, beta=1.0, Out_old=R)
    check_two_stage(to_f64(Out), yhat, _prop_bound(A, W1, W2, Wd, M, N, K, None),
                    f"mlp decode {M}x{K}x{N}")
