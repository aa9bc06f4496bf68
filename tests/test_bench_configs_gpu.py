"""Every workload bench.py times, checked against the oracle exactly as it is
timed: the same seeded inputs, the same call (shapes, strides, alpha, beta,
dtype, split) on the same stream, built by bench.build_case itself.  Outputs
are compared element by element on sampled rows (all rows up to 16) with the
bounds of the other parity tests: |y - yhat| <= 1e-2 + 1e-2 |yhat| for 16-bit
outputs, 1e-4 sqrt(K) max|yhat| for FP32 outputs."""
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import swiglu_mlp_gb300 as swg  # noqa: E402
import synth  # noqa: E402
from helpers import check_f32, check_half, to_f64  # noqa: E402

pytestmark = pytest.mark.gpu

CASES = bench.component_cases()


def _rows(M: int, seed: int):
    """All rows up to 16; otherwise both edges of the 128-row tiles and the
    256-row pair tiles near the start, the middle and the end, plus four
    seeded random rows."""
    if M <= 16:
        return list(range(M))
    rng = np.random.default_rng(seed)
    picks = {0, 1, 127, 128, 255, 256, M // 2, M - 257, M - 256, M - 129, M - 128, M - 1,
             *rng.integers(0, M, 4).tolist()}
    return sorted(r for r in picks if 0 <= r < M)


@pytest.mark.parametrize("name,kind,M,K,N", CASES, ids=[c[0] for c in CASES])
def test_timed_workload_matches_oracle(name, kind, M, K, N):
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    keep = {}
    fn, reset, _, _ = bench.build_case(kind, M, K, N, dev, stream, keep=keep)
    if reset:
        reset()
    fn()
    torch.cuda.synchronize(dev)
    assert swg.get_device_error() == 0
    rows = _rows(M, seed=len(name) * 1000 + M)
    out = to_f64(keep["out"].cpu())[rows]

    if kind in ("swiglu", "dual"):
        yhat = oracle.swiglu(keep["A"], keep["W1"], keep["W2"], M, N, K, rows=rows)
        check_half(out, yhat, name)
    elif kind == "fp8swiglu":
        yhat = oracle.swiglu_typed(keep["A"], keep["W1"], keep["W2"], M, N, K, in_type="e4m3",
                                   scale=keep["scale"], rows=rows)
        check_half(out, yhat, name)
    elif kind in ("skinny", "skinny_noalloc", "skinny_ws4"):
        # D = A B + C, beta = 1, bf16 output
        yhat = oracle.gemm(0, 0, M, N, K, 1.0, keep["A"], K, keep["B"], N, 1.0, keep["C"], N,
                           rows=rows)
        check_half(out, yhat, name)
    elif kind == "gemv":
        yhat = oracle.gemm(0, 0, M, N, K, 1.0, keep["A"], K, keep["B"], N, 0.0, rows=rows)
        check_half(out, yhat, name)
    elif kind == "fp8gemm":
        yhat = oracle.gemm(0, 1, M, N, K, 1.0 / 64, keep["A"], K, keep["Bt"], K, 0.0,
                           in_type="e4m3", rows=rows)
        check_half(out, yhat, name)
    elif kind == "mlp":
        # Out = Y W_down + Out_old, Y rounded to bf16 as the product stores it
        yhat = oracle.mlp(keep["A"], keep["W1"], keep["W2"], keep["Wd"], M, N, K, beta=1.0,
                          Out_old=keep["R"], rows=rows, round_y=True)
        check_half(out, yhat, name)
        y = to_f64(keep["Y"].cpu())[rows]
        check_half(y, oracle.swiglu(keep["A"], keep["W1"], keep["W2"], M, N, K, rows=rows),
                   name + " Y")
    elif kind == "gemm_f16_small":
        # D = 1.5 A B + 0.5 C: fp16 inputs, FP32 C and D
        yhat = oracle.gemm(0, 0, M, N, K, 1.5, keep["A"], K, keep["B"], N, 0.5, keep["C"], N,
                           in_type="f16", c_type="f32", rows=rows)
        check_f32(out, yhat, K, name)
    elif kind.startswith("gemm_"):
        tA, tB = keep["trans"]
        A, B = keep["A"], keep["B"]
        yhat = oracle.gemm(tA, tB, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 0.0, rows=rows)
        check_half(out, yhat, name)
    else:
        raise AssertionError(f"no check for workload kind {kind}")
    del fn, reset, keep
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tA,tB", bench.TRANS)
def test_headline_step_matches_oracle(tA, tB):
    """The timed step: one 8192^3 bf16 GEMM per op combination on the same
    stored A and B (seed 1), alpha = 1, beta = 0, leading dimensions 8192."""
    S = bench.SIZE
    A, B, _ = synth.gemm_bf16(S, S, S, 0, 0, seed=1)
    D = torch.empty((S, S), dtype=torch.bfloat16, device="cuda")
    swg.gemm(tA, tB, S, S, S, 1.0, A.cuda(), S, B.cuda(), S, 0.0, D, S, swg.BF16)
    torch.cuda.synchronize()
    assert swg.get_device_error() == 0
    rows = _rows(S, seed=10 * tA + tB)
    yhat = oracle.gemm(tA, tB, S, S, S, 1.0, A, S, B, S, 0.0, rows=rows)
    check_half(to_f64(D.cpu())[rows], yhat, f"headline {tA}{tB}")
