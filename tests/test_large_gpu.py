"""Outputs with more than 2^31 elements.

Element offsets in the epilogues (row * ld + column), the TMA store
coordinates and the split-K workspace index are 64-bit; these calls write
outputs of 2.4e9 elements (4.8 GB in bf16) with a short K, so they are cheap
to compute, and check rows and columns near the far end against the oracle.
"""
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import check_half, to_f64

pytestmark = pytest.mark.gpu

M, N = 40000, 60000            # M * N = 2.4e9 > 2^31; neither a tile multiple
ROWS = [0, 12345, 26843, 39999]
COLS = [0, 1, 35791, 59743, 59999]


def _free_gb():
    free, _ = torch.cuda.mem_get_info()
    return free / 2 ** 30


def test_gemm_output_beyond_2_31_elements():
    if _free_gb() < 12:
        pytest.skip("needs about 12 GB of free device memory")
    K = 136
    g = synth.generator(1200)
    A = synth.normal((M, K), g)
    B = synth.normal((K, N), g)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    swg.gemm(0, 0, M, N, K, 1.0, A.cuda(), K, B.cuda(), N, 0.0, D, N, swg.BF16)
    assert swg.get_device_error() == 0
    y = to_f64(D[ROWS][:, COLS])
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, rows=ROWS, cols=COLS)
    check_half(y, yhat, "gemm 40000 x 60000")
    del D
    torch.cuda.empty_cache()


def test_swiglu_output_beyond_2_31_elements():
    if _free_gb() < 12:
        pytest.skip("needs about 12 GB of free device memory")
    K = 64
    A, W1, W2 = synth.swiglu(M, K, N, seed=1201, w_std=0.1)
    Wf = swg.interleave_weights(W1.cuda(), W2.cuda())
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    swg.swiglu_mlp(A.cuda(), Wf, Y, M, N, K)
    assert swg.get_device_error() == 0
    y = to_f64(Y[ROWS][:, COLS])
    full = oracle.swiglu(A, W1, W2, M, N, K, rows=ROWS)
    check_half(y, full[:, COLS], "swiglu 40000 x 60000")
    del Y, Wf
    torch.cuda.empty_cache()


def test_split_k_workspace_beyond_2_31_bytes():
    """A forced split over a wide output: the partials span more than 2^31
    bytes of workspace (8 x 64 x 1.2e6 x 4 B = 2.5 GB)."""
    if _free_gb() < 8:
        pytest.skip("needs about 8 GB of free device memory")
    Ms, Ns, K = 64, 1_200_000, 512
    g = synth.generator(1202)
    A = synth.normal((Ms, K), g)
    B = synth.normal((K, Ns), g, std=0.05)
    D = torch.empty((Ms, Ns), dtype=torch.bfloat16, device="cuda")
    swg.gemm_ex(0, 0, Ms, Ns, K, 1.0, A.cuda(), K, B.cuda(), Ns, 0.0, D, Ns, swg.BF16, 8)
    assert swg.get_device_error() == 0
    rows, cols = [0, 63], [0, 600_001, 1_199_999]
    y = to_f64(D[rows][:, cols])
    yhat = oracle.gemm(0, 0, Ms, Ns, K, 1.0, A, K, B, Ns, 0.0, rows=rows, cols=cols)
    check_half(y, yhat, "split-K 64 x 1.2e6")
    del D
    torch.cuda.empty_cache()
