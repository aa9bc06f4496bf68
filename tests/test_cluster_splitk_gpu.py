"""Few rows with an automatic split: the K ranges of a tile run as one
thread-block cluster whose CTAs sum their FP32 partials over distributed
shared memory in rank order ("为什么 GEMM 是 CUDA 的必修课", 关键技术 item 5:
split K when M and N are too small to fill the GPU, then reduce).  One launch,
no workspace.

Decode shapes ("GEMM o Coração Matemático" §14: a few rows against a
4096 x 4096 weight) with 3..64 rows, every op combination, every output
checked against the FP64 oracle; ragged N and K; clusters of 4, 2 and 1; FP32
output with a NaN-filled C at beta = 0; e4m3 operands; the same products
through the workspace path (SWG_CLUSTER_SPLITK=0) within the same tolerance;
bit-identical repeats.  Every output sits inside guard bands.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import Guarded, check_f32, check_half, padded, to_f64

pytestmark = pytest.mark.gpu


def _inputs(tA, tB, M, N, K, seed, lda_pad=8):
    g = synth.generator(seed)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g)
    C = synth.normal((M, N), g)
    lda = ((A.shape[1] + lda_pad - 1) // lda_pad) * lda_pad
    return padded(A, lda, 3.0), lda, B, C


@pytest.mark.parametrize("M", [3, 4, 7, 8, 16, 33, 64])
@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_decode_rows_every_output(M, tA, tB):
    """M x 4096 x 4096, beta = 0.5: 32 tiles of 128 output columns, four K
    ranges per cluster."""
    N = K = 4096
    Ap, lda, B, C = _inputs(tA, tB, M, N, K, seed=400 + M + 2 * tA + tB)
    D = Guarded(M, N, torch.bfloat16, init=C)
    swg.gemm(tA, tB, M, N, K, 1.0, Ap.cuda(), lda, B.cuda(), B.shape[1], 0.5, D.view, D.ld,
             swg.BF16)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(tA, tB, M, N, K, 1.0, Ap, lda, B, B.shape[1], 0.5, C, N)
    check_half(to_f64(D.cpu(f"decode M={M}")), yhat, f"cluster decode M={M} tA={tA} tB={tB}")


@pytest.mark.parametrize("M,N,K", [(33, 4000, 3000),     # 32 tiles, 4 ranges, ragged N, K
                                   (16, 8192, 2048),     # 64 tiles, 2 ranges
                                   (5, 6000, 1000),      # 47 tiles, 2 ranges, ragged N
                                   (64, 3968, 16384)])   # 31 tiles, 4 ranges
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1)])
def test_cluster_sizes_and_ragged_edges(M, N, K, tA, tB):
    Ap, lda, B, C = _inputs(tA, tB, M, N, K, seed=500 + M + N % 97)
    D = Guarded(M, N, torch.bfloat16, init=C)
    swg.gemm(tA, tB, M, N, K, 0.75, Ap.cuda(), lda, B.cuda(), B.shape[1], -1.0, D.view, D.ld,
             swg.BF16)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(tA, tB, M, N, K, 0.75, Ap, lda, B, B.shape[1], -1.0, C, N)
    check_half(to_f64(D.cpu(f"cluster {M}x{N}x{K}")), yhat, f"cluster {M}x{N}x{K} tA={tA}")


def test_f32_output_beta_zero_ignores_nan_c():
    M, N, K = 48, 4096, 8192
    A, B, _ = synth.gemm_bf16(M, N, K, seed=66)
    D = Guarded(M, N, torch.float32, fill=float("nan"))
    swg.gemm(0, 0, M, N, K, 1.0, A.cuda(), K, B.cuda(), N, 0.0, D.view, D.ld, swg.BF16_F32OUT)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0)
    check_f32(to_f64(D.cpu("cluster f32")), yhat, K, "cluster f32 out")


def test_e4m3_few_rows():
    M, N, K = 16, 4096, 4096
    g = synth.generator(77)
    A = torch.randn(M, K, generator=g).to(torch.float8_e4m3fn)
    Bt = (torch.randn(N, K, generator=g) * 0.5).to(torch.float8_e4m3fn)
    C = synth.normal((M, N), g)
    D = Guarded(M, N, torch.bfloat16, init=C)
    swg.gemm(0, 1, M, N, K, 1.0 / 16, A.cuda(), K, Bt.cuda(), K, 1.0, D.view, D.ld,
             swg.E4M3_BF16OUT)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(0, 1, M, N, K, 1.0 / 16, A, K, Bt, K, 1.0, C, N, in_type="e4m3")
    check_half(to_f64(D.cpu("cluster e4m3")), yhat, "cluster e4m3")


@pytest.mark.parametrize("M", [16, 64])
def test_matches_workspace_path_and_repeats(monkeypatch, M):
    """The skinny shape through the cluster reduction and through the
    workspace reduction: both within tolerance of the oracle, and the cluster
    path bit-identical over repeated calls."""
    N, K = 4096, 16384
    A, B, C = synth.skinny(M, seed=9)
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for flag in ("1", "1", "0"):
        monkeypatch.setenv("SWG_CLUSTER_SPLITK", flag)
        D = Guarded(M, N, torch.bfloat16, init=C, ld=N)
        swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, D.view, N, swg.BF16)
        outs.append(D.cpu(f"cluster={flag}"))
    assert swg.get_device_error() == 0
    assert torch.equal(outs[0], outs[1])
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N)
    check_half(to_f64(outs[0]), yhat, f"cluster M={M}")
    check_half(to_f64(outs[2]), yhat, f"workspace M={M}")


def test_graph_capture_without_warm_up():
    """No workspace: the first call of a shape can be captured directly."""
    M, N, K = 8, 4096, 4096
    A, B, C = synth.gemm_bf16(M, N, K, seed=81, c=True)
    Ad, Bd = A.cuda(), B.cuda()
    D = Guarded(M, N, torch.bfloat16, init=C)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        swg.gemm(0, 0, M, N, K, 2.0, Ad, K, Bd, N, 0.0, D.view, D.ld, swg.BF16, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(0, 0, M, N, K, 2.0, A, K, B, N, 0.0)
    check_half(to_f64(D.cpu("graph")), yhat, "cluster graph replay")


# ---------------------------------------------------------------- M > 64
# With more rows an automatic split runs 128 x 256 tiles whose K ranges form
# one cluster of 2 or 4 CTAs; the partials are exchanged in the consumed
# pipeline stages and each rank stores alpha * sum + beta * C for its share of
# the tile's columns.

@pytest.mark.parametrize("M,N,K", [(2048, 896, 4864),      # the small MLP's down projection, 2 ranks
                                   (1024, 1024, 8192),     # 32 tiles, 4 ranks
                                   (600, 1200, 4000)])     # ragged M, N and K, 4 ranks
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_tiles_with_cluster_split_every_output(M, N, K, tA, tB):
    g = synth.generator(600 + M + 2 * tA + tB)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g, std=0.05)
    C = synth.normal((M, N), g)
    D = Guarded(M, N, torch.bfloat16, init=C)
    swg.gemm(tA, tB, M, N, K, 1.0, A.cuda(), A.shape[1], B.cuda(), B.shape[1], 1.0, D.view, D.ld,
             swg.BF16)
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(tA, tB, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 1.0, C, N)
    check_half(to_f64(D.cpu(f"cluster tiles {M}x{N}x{K}")), yhat,
               f"cluster tiles {M}x{N}x{K} tA={tA} tB={tB}")


def test_tiles_with_cluster_split_f32_out_nan_c():
    M, N, K = 1024, 1024, 8192
    A, B, _ = synth.gemm_bf16(M, N, K, seed=67)
    D = Guarded(M, N, torch.float32, fill=float("nan"))
    swg.gemm(0, 0, M, N, K, 0.5, A.cuda(), K, B.cuda(), N, 0.0, D.view, D.ld, swg.BF16_F32OUT)
    assert swg.get_device_error() == 0
    rows = sorted({0, 127, 128, 511, 512, M - 1})
    yhat = oracle.gemm(0, 0, M, N, K, 0.5, A, K, B, N, 0.0, rows=rows)
    out = to_f64(D.cpu("cluster tiles f32"))
    assert np.isfinite(out).all()
    check_f32(out[rows], yhat, K, "cluster tiles f32 out")


def test_tiles_with_cluster_split_match_workspace_and_repeat(monkeypatch):
    M, N, K = 2048, 896, 4864
    A, B, C = synth.gemm_bf16(M, N, K, seed=68, c=True)
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for flag in ("1", "1", "0"):
        monkeypatch.setenv("SWG_CLUSTER_SPLITK", flag)
        D = Guarded(M, N, torch.bfloat16, init=C, ld=N)
        swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, D.view, N, swg.BF16)
        outs.append(D.cpu(f"cluster={flag}"))
    assert swg.get_device_error() == 0
    assert torch.equal(outs[0], outs[1])
    rows = sorted({0, 127, 128, 1023, 1024, M - 1})
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N, rows=rows)
    check_half(to_f64(outs[0])[rows], yhat, "cluster tiles")
    check_half(to_f64(outs[2])[rows], yhat, "workspace tiles")


# Ragged edges of the 128 x 256 cluster tiles: M past the last full 128-row
# block, N past the last full 256-column block (a rank's share cut short), K
# not a multiple of the two ranges.
@pytest.mark.parametrize("M,N,K", [(2000, 904, 4000),      # 64 tiles x 2 ranks
                                   (1800, 1000, 3000)])    # 60 tiles x 2 ranks
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_cluster_tiles_ragged_every_output(M, N, K, tA, tB):
    g = synth.generator(700 + M + 2 * tA + tB)
    A = synth.normal(synth.stored_shape(tA, M, K), g)
    B = synth.normal(synth.stored_shape(tB, K, N), g, std=0.05)
    C = synth.normal((M, N), g)
    D = Guarded(M, N, torch.bfloat16, init=C)
    n0 = swg.launch_count()
    swg.gemm(tA, tB, M, N, K, 1.0, A.cuda(), A.shape[1], B.cuda(), B.shape[1], 1.0, D.view, D.ld,
             swg.BF16)
    assert swg.launch_count() - n0 == 1
    assert swg.get_device_error() == 0
    yhat = oracle.gemm(tA, tB, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 1.0, C, N)
    check_half(to_f64(D.cpu(f"cluster tiles {M}x{N}x{K}")), yhat,
               f"cluster tiles {M}x{N}x{K} tA={tA} tB={tB}")


def test_cluster_tiles_two_ranks_f32_out_nan_c():
    M, N, K = 2048, 896, 4864
    A, B, _ = synth.gemm_bf16(M, N, K, seed=69)
    D = Guarded(M, N, torch.float32, fill=float("nan"))
    swg.gemm(0, 0, M, N, K, 0.5, A.cuda(), K, B.cuda(), N, 0.0, D.view, D.ld, swg.BF16_F32OUT)
    assert swg.get_device_error() == 0
    rows = sorted({0, 127, 128, 255, 256, 1023, 1024, M - 129, M - 128, M - 1})
    yhat = oracle.gemm(0, 0, M, N, K, 0.5, A, K, B, N, 0.0, rows=rows)
    out = to_f64(D.cpu("cluster tiles f32, two ranks"))
    assert np.isfinite(out).all()
    check_f32(out[rows], yhat, K, "cluster tiles f32 out, two ranks")
