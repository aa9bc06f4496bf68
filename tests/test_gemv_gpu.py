"""Few-rows product (M <= 2) on the FP32 pipes: one launch, B streamed through
shared memory by TMA, the K ranges of a block of output columns reduced
inside a thread-block cluster in rank order.

gemm / gemm_ex with split_k = 0 take this path for 16-bit and e4m3 inputs when
M <= 2 and K fits in 8 ranges of the op(A) slice a CTA stages (8192 / rows
elements); more rows, larger K and explicit split_k keep the tensor-core path.  Every output is checked against the FP64 oracle ("GEMM o Coração
Matemático", §1: D_ij = alpha sum_p op(A)_ip op(B)_pj + beta C_ij).  Storage
padding carries a large fill value, so a read past a row shows in the result.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import Guarded, check_f32, check_half, padded, round_up, to_f64

pytestmark = pytest.mark.gpu


def _operands(seed, tA, tB, M, N, K, dtype=torch.bfloat16, fill=9.0):
    g = synth.generator(seed)
    A = synth.normal(synth.stored_shape(tA, M, K), g, dtype=dtype)
    B = synth.normal(synth.stored_shape(tB, K, N), g, dtype=dtype)
    lda, ldb = round_up(A.shape[1], 8), round_up(B.shape[1], 8)
    return padded(A, lda, fill), lda, padded(B, ldb, fill), ldb


def _run(tA, tB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, split_k=0):
    """C (M x ldc on the host) goes to the device inside guard bands: rows
    above and below, and its columns past N.  Returns C with the first N
    columns replaced by the result (after checking every guard) and the
    number of kernel launches."""
    N_out = min(N, C.shape[1])
    Cg = Guarded(M, N_out, C.dtype, init=C[:, :N_out], ld=ldc)
    before = swg.launch_count()
    swg.gemm_ex(tA, tB, M, N, K, alpha, A.cuda(), lda, B.cuda(), ldb, beta, Cg.view, ldc, dtype,
                split_k)
    launches = swg.launch_count() - before
    assert swg.get_device_error() == 0
    out = C.clone()
    out[:, :N_out] = Cg.cpu(f"gemv {M}x{N}x{K}")
    return out, launches


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("N,K", [(7, 9), (33, 1000), (600, 2056), (520, 4100)])
def test_ragged_shapes_all_outputs(M, tA, tB, N, K):
    """Ragged N (not a multiple of the column block or of 8) and K (not a
    multiple of 8 or of the range), beta != 0 with a bf16 C; one launch for
    M <= 2 (M = 3, 4 take the tensor-core path, checked the same way)."""
    A, lda, B, ldb = _operands(400 + M + 2 * tA + tB + N, tA, tB, M, N, K)
    ldc = round_up(N, 8)
    C = padded(synth.normal((M, N), synth.generator(401 + N)), ldc, 3.0)
    out, launches = _run(tA, tB, M, N, K, 0.75, A, lda, B, ldb, -1.5, C, ldc, swg.BF16)
    if M <= 2:
        assert launches == 1
    assert torch.equal(out[:, N:], C[:, N:])          # padding of C untouched
    yhat = oracle.gemm(tA, tB, M, N, K, 0.75, A, lda, B, ldb, -1.5, C, ldc)
    check_half(to_f64(out[:, :N]), yhat, f"gemv M={M} tA={tA} tB={tB} N={N} K={K}")


@pytest.mark.parametrize("dtype,in_t,out_t", [
    (swg.F16, torch.float16, torch.float16),
    (swg.F16_F32OUT, torch.float16, torch.float32),
    (swg.BF16_F32OUT, torch.bfloat16, torch.float32),
])
@pytest.mark.parametrize("tB", [0, 1])
def test_output_types(dtype, in_t, out_t, tB):
    M, N, K = 2, 1000, 3000
    A, lda, B, ldb = _operands(420 + dtype + tB, 0, tB, M, N, K, dtype=in_t)
    C = synth.normal((M, N), synth.generator(421), dtype=out_t)
    out, launches = _run(0, tB, M, N, K, 1.0, A, lda, B, ldb, 0.5, C, N, dtype)
    assert launches == 1
    in_name = "f16" if in_t == torch.float16 else "bf16"
    c_name = "f32" if out_t == torch.float32 else in_name
    yhat = oracle.gemm(0, tB, M, N, K, 1.0, A, lda, B, ldb, 0.5, C, N, in_type=in_name,
                       c_type=c_name)
    if out_t == torch.float32:
        check_f32(to_f64(out), yhat, K, f"gemv dtype={dtype}")
    else:
        check_half(to_f64(out), yhat, f"gemv dtype={dtype}")


def test_beta_zero_ignores_nan_in_c():
    M, N, K = 2, 4096, 4096
    A, lda, B, ldb = _operands(430, 0, 1, M, N, K)
    C = torch.full((M, N), float("nan"), dtype=torch.float32)
    out, _ = _run(0, 1, M, N, K, 1.0, A, lda, B, ldb, 0.0, C, N, swg.BF16_F32OUT)
    assert torch.isfinite(out).all()
    yhat = oracle.gemm(0, 1, M, N, K, 1.0, A, lda, B, ldb, 0.0)
    check_f32(to_f64(out), yhat, K, "gemv beta=0")


@pytest.mark.parametrize("M,K", [(1, 65536), (2, 32768)])
@pytest.mark.parametrize("tB", [0, 1])
def test_longest_k_eight_ranges(M, K, tB):
    """K at the path's limit: 8 ranges of 8192 / rows elements each."""
    N = 264
    A, lda, B, ldb = _operands(440 + M + tB, 0, tB, M, N, K)
    C = torch.zeros((M, N), dtype=torch.float32)
    out, launches = _run(0, tB, M, N, K, 1.0, A, lda, B, ldb, 0.0, C, N, swg.BF16_F32OUT)
    assert launches == 1
    yhat = oracle.gemm(0, tB, M, N, K, 1.0, A, lda, B, ldb, 0.0)
    check_f32(to_f64(out), yhat, K, f"gemv M={M} K={K}")


def test_beyond_the_limit_takes_the_tensor_path():
    """K one 8-element group past 8 ranges: the split-K tensor-core path
    (a GEMM and its reduction, two launches) gives the same answer."""
    M, N, K = 2, 264, 32776
    A, lda, B, ldb = _operands(450, 0, 0, M, N, K)
    C = torch.zeros((M, N), dtype=torch.float32)
    out, launches = _run(0, 0, M, N, K, 1.0, A, lda, B, ldb, 0.0, C, N, swg.BF16_F32OUT)
    assert launches == 2
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, lda, B, ldb, 0.0)
    check_f32(to_f64(out), yhat, K, "tensor path")


def test_bitwise_deterministic():
    M, N, K = 2, 4096, 4096
    A, lda, B, ldb = _operands(460, 0, 1, M, N, K)
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for _ in range(3):
        D = Guarded(M, N, torch.float32)
        swg.gemm(0, 1, M, N, K, 1.0, Ad, lda, Bd, ldb, 0.0, D.view, D.ld, swg.BF16_F32OUT)
        outs.append(D.cpu("repeat"))
    assert swg.get_device_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("tB", [0, 1])
def test_agrees_with_tensor_path(tB):
    """The same call through the FP32-pipe kernel (split_k = 0) and through
    the tensor-core split-K path (split_k = 4): both within the FP32-output
    bound of the oracle, and of each other."""
    M, N, K = 1, 4096, 4096
    A, lda, B, ldb = _operands(470 + tB, 0, tB, M, N, K)
    C = torch.zeros((M, N), dtype=torch.float32)
    d0, n0 = _run(0, tB, M, N, K, 1.0, A, lda, B, ldb, 0.0, C, N, swg.BF16_F32OUT, 0)
    d4, n4 = _run(0, tB, M, N, K, 1.0, A, lda, B, ldb, 0.0, C, N, swg.BF16_F32OUT, 4)
    assert (n0, n4) == (1, 2)
    yhat = oracle.gemm(0, tB, M, N, K, 1.0, A, lda, B, ldb, 0.0)
    check_f32(to_f64(d0), yhat, K, "gemv")
    check_f32(to_f64(d4), yhat, K, "split-K")
    scale = float(np.abs(yhat).max())
    assert float((d0 - d4).abs().max()) <= 2e-4 * np.sqrt(K) * scale


def test_switch_off_takes_the_tensor_path(monkeypatch):
    M, N, K = 1, 4096, 4096
    A, lda, B, ldb = _operands(480, 0, 1, M, N, K)
    C = torch.zeros((M, N), dtype=torch.bfloat16)
    monkeypatch.setenv("SWG_GEMV", "0")
    out, launches = _run(0, 1, M, N, K, 1.0, A, lda, B, ldb, 0.0, C, N, swg.BF16)
    # the tensor-core few-rows path: K ranges reduced inside a cluster
    assert launches == 1
    yhat = oracle.gemm(0, 1, M, N, K, 1.0, A, lda, B, ldb, 0.0)
    check_half(to_f64(out), yhat, "SWG_GEMV=0")


def test_graph_capture_without_warm_up():
    """The path needs no workspace, so its first call on a fresh stream can be
    captured into a CUDA graph; replays recompute from the current inputs."""
    M, N, K = 1, 2048, 4096
    A, lda, B, ldb = _operands(490, 0, 1, M, N, K)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            swg.gemm(0, 1, M, N, K, 1.0, Ad, lda, Bd, ldb, 0.0, D, N, swg.BF16,
                     stream=s.cuda_stream)
    for scale in (1.0, -2.0):
        Ad.copy_((A.float() * scale).to(torch.bfloat16).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert swg.get_device_error() == 0
        A_now = Ad.cpu()
        yhat = oracle.gemm(0, 1, M, N, K, 1.0, A_now, lda, B, ldb, 0.0)
        check_half(to_f64(D.cpu()), yhat, f"graph replay scale={scale}")


def test_chained_calls_on_one_stream():
    """y1 = x W1^T, then y2 = y1 W2^T reading y1 (programmatic dependent
    launch: the second kernel waits for the first one's writes)."""
    K1, N1, N2 = 4096, 2048, 1024
    g = synth.generator(495)
    x = synth.normal((1, K1), g)
    W1 = synth.normal((N1, K1), g, std=0.02)
    W2 = synth.normal((N2, N1), g, std=0.02)
    y1 = torch.empty((1, N1), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((1, N2), dtype=torch.bfloat16, device="cuda")
    xd, W1d, W2d = x.cuda(), W1.cuda(), W2.cuda()
    for _ in range(3):
        swg.gemm(0, 1, 1, N1, K1, 1.0, xd, K1, W1d, K1, 0.0, y1, N1, swg.BF16)
        swg.gemm(0, 1, 1, N2, N1, 1.0, y1, N1, W2d, N1, 0.0, y2, N2, swg.BF16)
    assert swg.get_device_error() == 0
    y1_host = y1.cpu()
    check_half(to_f64(y1_host), oracle.gemm(0, 1, 1, N1, K1, 1.0, x, K1, W1, K1, 0.0), "y1")
    check_half(to_f64(y2.cpu()), oracle.gemm(0, 1, 1, N2, N1, 1.0, y1_host, N1, W2, N1, 0.0),
               "y2")


def _e4m3_padded(rows, cols, ld, g, std=1.0, fill=256.0):
    """rows x ld e4m3 storage (values exact in e4m3) holding N(0, std) values
    rounded to e4m3 in its first cols columns and `fill` after them."""
    t = torch.full((rows, ld), fill, dtype=torch.float32)
    t[:, :cols] = (torch.randn(rows, cols, generator=g) * std).to(torch.float8_e4m3fn).float()
    return t.to(torch.float8_e4m3fn)


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", [(7, 16), (520, 1000), (600, 4100)])
def test_e4m3_weights_ragged(M, N, K):
    """8-bit operands (A stored M x K, B stored N x K, the e4m3 contract): the
    same one-launch kernel with 64-row boxes; per-tensor scales folded into
    alpha; ragged N and K, beta != 0 with a bf16 C."""
    g = synth.generator(500 + M + N)
    ld = round_up(K, 16)
    A = _e4m3_padded(M, K, ld, g)
    B = _e4m3_padded(N, K, ld, g, std=0.5)
    ldc = round_up(N, 8)
    C = padded(synth.normal((M, N), g), ldc, 3.0)
    out, launches = _run(0, 1, M, N, K, 1.0 / 32, A, ld, B, ld, 0.5, C, ldc, swg.E4M3_BF16OUT)
    assert launches == 1
    assert torch.equal(out[:, N:], C[:, N:])
    yhat = oracle.gemm(0, 1, M, N, K, 1.0 / 32, A, ld, B, ld, 0.5, C, ldc, in_type="e4m3")
    check_half(to_f64(out[:, :N]), yhat, f"e4m3 gemv M={M} N={N} K={K}")


@pytest.mark.parametrize("M,K", [(1, 65536), (2, 32768)])
def test_e4m3_longest_k(M, K):
    N = 200
    g = synth.generator(510 + M)
    A = _e4m3_padded(M, K, K, g)
    B = _e4m3_padded(N, K, K, g, std=0.25)
    C = torch.zeros((M, N), dtype=torch.float32)
    out, launches = _run(0, 1, M, N, K, 0.5, A, K, B, K, 0.0, C, N, swg.E4M3_F32OUT)
    assert launches == 1
    yhat = oracle.gemm(0, 1, M, N, K, 0.5, A, K, B, K, 0.0, in_type="e4m3", c_type="f32")
    check_f32(to_f64(out), yhat, K, f"e4m3 gemv M={M} K={K}")


def test_e4m3_switch_off_agrees(monkeypatch):
    """The same e4m3 decode through the tensor-core few-rows path
    (SWG_GEMV=0; K ranges reduced inside a cluster, one launch): both within
    the FP32-output bound of the oracle."""
    M, N, K = 1, 4096, 4096
    g = synth.generator(520)
    A = _e4m3_padded(M, K, K, g)
    B = _e4m3_padded(N, K, K, g, std=0.5)
    C = torch.zeros((M, N), dtype=torch.float32)
    d_on, n_on = _run(0, 1, M, N, K, 0.25, A, K, B, K, 0.0, C, N, swg.E4M3_F32OUT)
    monkeypatch.setenv("SWG_GEMV", "0")
    d_off, n_off = _run(0, 1, M, N, K, 0.25, A, K, B, K, 0.0, C, N, swg.E4M3_F32OUT)
    assert (n_on, n_off) == (1, 1)
    yhat = oracle.gemm(0, 1, M, N, K, 0.25, A, K, B, K, 0.0, in_type="e4m3", c_type="f32")
    check_f32(to_f64(d_on), yhat, K, "e4m3 gemv")
    check_f32(to_f64(d_off), yhat, K, "e4m3 split-K")


def _swiglu_fused(W1, W2, K, N):
    """W_fused from the oracle's interleave (not from the CUDA path)."""
    Wf = oracle.interleave(W1, W2, K, N)
    return torch.from_numpy(Wf.view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("K,N", [(8, 8), (136, 520), (1000, 264), (896, 4864), (4096, 14336)])
def test_swiglu_decode_rows(M, K, N):
    """swiglu_mlp with one or two rows: one launch of the same kernel over the
    interleaved W_fused, SiLU(Gate) * Up formed per column pair in its final
    reduction ("Sobreposição de Ativação em Nível de Tile para Inferência
    Eficiente de LLM", Metodologia); checked against the oracle from separate
    W1 and W2, every output."""
    A, W1, W2 = synth.swiglu(M, K, N, seed=600 + M + K, w_std=0.02 if K >= 896 else 0.1)
    Wf = _swiglu_fused(W1, W2, K, N)
    Y = Guarded(M, N, torch.bfloat16, fill=9.0, ld=N)
    before = swg.launch_count()
    swg.swiglu_mlp(A.cuda(), Wf.cuda(), Y.view, M, N, K)
    assert swg.launch_count() - before == 1
    assert swg.get_device_error() == 0
    yhat = oracle.swiglu(A, W1, W2, M, N, K)
    check_half(to_f64(Y.cpu("swiglu decode")), yhat, f"swiglu decode M={M} K={K} N={N}")


def test_swiglu_decode_agrees_with_tensor_path(monkeypatch):
    M, K, N = 1, 896, 4864
    A, W1, W2 = synth.swiglu(M, K, N, seed=610)
    Wf = _swiglu_fused(W1, W2, K, N).cuda()
    Ad = A.cuda()
    Y1 = Guarded(M, N, torch.bfloat16, ld=N)
    Y2 = Guarded(M, N, torch.bfloat16, ld=N)
    swg.swiglu_mlp(Ad, Wf, Y1.view, M, N, K)
    monkeypatch.setenv("SWG_GEMV", "0")
    swg.swiglu_mlp(Ad, Wf, Y2.view, M, N, K)
    assert swg.get_device_error() == 0
    yhat = oracle.swiglu(A, W1, W2, M, N, K)
    check_half(to_f64(Y1.cpu("one-launch")), yhat, "swiglu decode, one-launch kernel")
    check_half(to_f64(Y2.cpu("tensor path")), yhat, "swiglu decode, tensor-core path")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("K,N", [(16, 8), (256, 520), (4096, 14336)])
def test_fp8_swiglu_decode_rows(M, K, N):
    """swiglu_mlp_fp8 with one or two rows: the e4m3 kernel over the
    transposed interleaved weight [2N x K] (64-row boxes), the per-tensor
    scale applied to Gate and Up before SiLU; every output against the
    oracle on the same e4m3 values."""
    A, W1, W2, sw = synth.swiglu_e4m3(M, K, N, seed=620 + M + K, w_std=0.05)
    Wt = torch.from_numpy(oracle.interleave_t8(W1, W2, K, N)).view(torch.float8_e4m3fn)
    Y = Guarded(M, N, torch.bfloat16, fill=9.0, ld=N)
    before = swg.launch_count()
    swg.swiglu_mlp_fp8(A.cuda(), Wt.cuda(), Y.view, M, N, K, sw)
    assert swg.launch_count() - before == 1
    assert swg.get_device_error() == 0
    yhat = oracle.swiglu_typed(A, W1, W2, M, N, K, in_type="e4m3", scale=sw)
    check_half(to_f64(Y.cpu("fp8 decode")), yhat, f"fp8 swiglu decode M={M} K={K} N={N}")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("K,N", [(8, 8), (136, 520), (1000, 200), (4096, 14336)])
def test_swiglu_dual_decode_rows(M, K, N):
    """swiglu_mlp_dual (separate W1, W2, no interleaved copy) with one or two
    rows: one launch; each stage holds a 64-column box of W1 beside the same
    columns of W2, and column j pairs with column 64 + j in the final
    reduction.  Every output against the oracle."""
    A, W1, W2 = synth.swiglu(M, K, N, seed=630 + M + K, w_std=0.02 if K >= 896 else 0.1)
    Y = Guarded(M, N, torch.bfloat16, fill=9.0, ld=N)
    before = swg.launch_count()
    swg.swiglu_mlp_dual(A.cuda(), W1.cuda(), W2.cuda(), Y.view, M, N, K)
    assert swg.launch_count() - before == 1
    assert swg.get_device_error() == 0
    yhat = oracle.swiglu(A, W1, W2, M, N, K)
    check_half(to_f64(Y.cpu("dual decode")), yhat, f"swiglu dual decode M={M} K={K} N={N}")
