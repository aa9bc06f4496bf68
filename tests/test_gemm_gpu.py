"""GEMM parity: the CUDA path (through the C ABI) against the FP64 oracle.

D = alpha op(A) op(B) + beta C ("GEMM o Coração Matemático", §1), all four
op combinations, every storage type, ragged tails, padded row strides, the
beta = 0 / K = 0 special cases, the 256^3 fp16 case in full, and sampled
rows of the square 4096 / 8192 bf16 cases in the launch configuration the
benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import Guarded, check_f32, check_half, padded, round_up, to_f64

pytestmark = pytest.mark.gpu

DT = {  # code -> (input torch dtype, output torch dtype, oracle in, oracle out)
    swg.F16_F32OUT: (torch.float16, torch.float32, "f16", "f32"),
    swg.BF16: (torch.bfloat16, torch.bfloat16, "bf16", "bf16"),
    swg.F16: (torch.float16, torch.float16, "f16", "f16"),
    swg.BF16_F32OUT: (torch.bfloat16, torch.float32, "bf16", "f32"),
}


def run_case(M, N, K, tA, tB, code, alpha, beta, seed, pad=(0, 0, 0), c_fill=None,
             split_k=None, rows=None):
    """Runs one GEMM on the GPU and on the oracle; returns (y, yhat)."""
    tin, tout, oin, oout = DT[code]
    g = synth.generator(seed)
    A = synth.normal(synth.stored_shape(tA, M, K), g, dtype=tin)
    B = synth.normal(synth.stored_shape(tB, K, N), g, dtype=tin)
    C = synth.normal((M, N), g, dtype=tout)
    esz_out = 4 if tout == torch.float32 else 2
    lda = round_up(A.shape[1], 8) + pad[0]
    ldb = round_up(B.shape[1], 8) + pad[1]
    ldc = round_up(N, 16 // esz_out) + pad[2]
    Ap, Bp = padded(A, lda, 3.0), padded(B, ldb, 3.0)
    Cp = padded(C, ldc, 5.0)
    if c_fill is not None:
        Cp.fill_(c_fill)
    # C inside guard bands: rows above and below, and its padding columns
    Cg = Guarded(M, N, tout, init=Cp[:, :N], ld=ldc)
    Ad, Bd = Ap.cuda(), Bp.cuda()
    if split_k is None:
        swg.gemm(tA, tB, M, N, K, alpha, Ad, lda, Bd, ldb, beta, Cg.view, ldc, code)
    else:
        swg.gemm_ex(tA, tB, M, N, K, alpha, Ad, lda, Bd, ldb, beta, Cg.view, ldc, code, split_k)
    assert swg.get_device_error() == 0
    y = to_f64(Cg.cpu(f"gemm {M}x{N}x{K} tA={tA} tB={tB} code={code}"))
    yhat = oracle.gemm(tA, tB, M, N, K, alpha, Ap, lda, Bp, ldb, beta, Cp, ldc,
                       in_type=oin, c_type=oout, rows=rows)
    if rows is not None:
        y = y[np.asarray(rows)]
    return y, yhat


def check(y, yhat, code, K, what):
    if DT[code][1] == torch.float32:
        return check_f32(y, yhat, K, what)
    return check_half(y, yhat, what)


def test_config_f16_256_cubed_full():
    """FP16 in, FP32 out: C = 1.5 A B + 0.5 C, 256^3, U(-1,1) inputs, seed 0."""
    M = N = K = 256
    A, B, C = synth.gemm_f16_small(seed=0)
    Ad, Bd = A.cuda(), B.cuda()
    for ld in (N, N + 32):                  # the benchmark's ldc = N, and a guarded pad
        Cg = Guarded(M, N, torch.float32, init=C, ld=ld)
        swg.gemm(0, 0, M, N, K, 1.5, Ad, K, Bd, N, 0.5, Cg.view, ld, swg.F16_F32OUT)
        assert swg.get_device_error() == 0
        yhat = oracle.gemm(0, 0, M, N, K, 1.5, A, K, B, N, 0.5, C, N, in_type="f16",
                           c_type="f32")
        check_f32(to_f64(Cg.cpu("f16 256^3")), yhat, K, f"f16 256^3 ldc={ld}")


@pytest.mark.parametrize("tA", [0, 1])
@pytest.mark.parametrize("tB", [0, 1])
@pytest.mark.parametrize("shape", [(128, 256, 64), (256, 512, 320), (300, 520, 200),
                                   (129, 257, 72), (1, 8, 8), (7, 13, 5), (640, 384, 1000)])
def test_bf16_all_ops(tA, tB, shape):
    M, N, K = shape
    y, yhat = run_case(M, N, K, tA, tB, swg.BF16, 1.0, 0.0, seed=100 + M + N + K + tA * 2 + tB)
    check_half(y, yhat, f"bf16 {shape} tA={tA} tB={tB}")


@pytest.mark.parametrize("code", [swg.F16_F32OUT, swg.F16, swg.BF16_F32OUT])
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_other_dtypes(code, tA, tB):
    M, N, K = 200, 264, 136
    y, yhat = run_case(M, N, K, tA, tB, code, 0.75, 0.0, seed=7 + code * 4 + tA * 2 + tB)
    check(y, yhat, code, K, f"code={code} tA={tA} tB={tB}")


@pytest.mark.parametrize("code", [swg.BF16, swg.F16_F32OUT, swg.F16])
def test_beta_nonzero_and_padding(code):
    M, N, K = 190, 300, 256
    y, yhat = run_case(M, N, K, 0, 0, code, 1.5, -0.5, seed=31, pad=(8, 16, 8))
    check(y, yhat, code, K, f"beta code={code}")


def test_beta_zero_ignores_nan_c():
    M, N, K = 160, 272, 96
    y, yhat = run_case(M, N, K, 0, 1, swg.BF16, 1.0, 0.0, seed=5, c_fill=float("nan"))
    check_half(y, yhat, "beta=0 NaN C")


@pytest.mark.parametrize("code", [swg.BF16, swg.F16_F32OUT])
def test_k_zero_scales_c(code):
    M, N = 70, 40
    for beta in (0.0, 2.0):
        y, yhat = run_case(M, N, 0, 0, 0, code, 1.0, beta, seed=9)
        check(y, yhat, code, 1, f"K=0 beta={beta}")


def test_m_or_n_zero_is_noop():
    C = torch.full((4, 8), 7.0, dtype=torch.bfloat16, device="cuda")
    before = swg.launch_count()
    swg.gemm(0, 0, 0, 8, 16, 1.0, 0, 16, 0, 8, 0.0, C, 8, swg.BF16)
    swg.gemm(0, 0, 4, 0, 16, 1.0, 0, 16, 0, 8, 0.0, C, 8, swg.BF16)
    assert swg.launch_count() == before
    assert torch.all(C == 7.0)


def test_identity_product_exact():
    """A I = A exactly: every output is one bf16 value times 1."""
    M, K = 300, 256
    g = synth.generator(41)
    A = synth.normal((M, K), g).cuda()
    eye = torch.eye(K, dtype=torch.bfloat16, device="cuda")
    D = Guarded(M, K, torch.bfloat16)
    swg.gemm(0, 0, M, K, K, 1.0, A, K, eye, K, 0.0, D.view, D.ld, swg.BF16)
    torch.cuda.synchronize()
    assert torch.equal(D.cpu("A I"), A.cpu())


def test_transpose_identity_gpu():
    """(A B)^T = B^T A^T: computing D^T with both operands transposed gives the
    transpose of D (to within rounding of the same FP32 sums)."""
    M, N, K = 256, 384, 512
    A, B, _ = synth.gemm_bf16(M, N, K, seed=43)
    Ad, Bd = A.cuda(), B.cuda()
    D = Guarded(M, N, torch.float32)
    Dt = Guarded(N, M, torch.float32)
    swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 0.0, D.view, D.ld, swg.BF16_F32OUT)
    swg.gemm(1, 1, N, M, K, 1.0, Bd, N, Ad, K, 0.0, Dt.view, Dt.ld, swg.BF16_F32OUT)
    torch.cuda.synchronize()
    yhat = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0)
    check_f32(to_f64(D.cpu("D")), yhat, K, "D")
    check_f32(to_f64(Dt.cpu("D^T")).T, yhat, K, "D^T")


def test_alpha_linearity_power_of_two_exact():
    M, N, K = 256, 256, 192
    A, B, _ = synth.gemm_bf16(M, N, K, seed=47)
    Ad, Bd = A.cuda(), B.cuda()
    D1 = Guarded(M, N, torch.float32)
    D4 = Guarded(M, N, torch.float32)
    swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 0.0, D1.view, D1.ld, swg.BF16_F32OUT)
    swg.gemm(0, 0, M, N, K, 4.0, Ad, K, Bd, N, 0.0, D4.view, D4.ld, swg.BF16_F32OUT)
    torch.cuda.synchronize()
    assert torch.equal(D4.cpu("alpha 4"), 4.0 * D1.cpu("alpha 1"))


# alpha = 0 and alpha < 0 on every path a product can take: 128 x 256 pair
# tiles, the few-rows cluster kernel, the 128 x 256 cluster tiles, the explicit
# split with its reduction kernel, and the one-row FP32-pipe kernel.
_ALPHA_SHAPES = [(300, 264, 200, 0), (16, 4096, 4096, 0), (2048, 896, 4864, 0),
                 (200, 1024, 2048, 3), (1, 520, 1000, 0)]


@pytest.mark.parametrize("M,N,K,split", _ALPHA_SHAPES)
def test_alpha_zero_gives_beta_c_exactly(M, N, K, split):
    """With finite operands and alpha = 0 every product is scaled to zero, so
    D = beta * C with one rounding; beta = 1/2 halves a bf16 value exactly."""
    A, B, C = synth.gemm_bf16(M, N, K, seed=M + N, c=True)
    D = Guarded(M, N, torch.bfloat16, init=C)
    swg.gemm_ex(0, 0, M, N, K, 0.0, A.cuda(), K, B.cuda(), N, 0.5, D.view, D.ld, swg.BF16, split)
    assert swg.get_device_error() == 0
    assert torch.equal(D.cpu("alpha 0"), (0.5 * C.float()).to(torch.bfloat16))


@pytest.mark.parametrize("M,N,K,split", _ALPHA_SHAPES)
def test_negative_alpha(M, N, K, split):
    A, B, C = synth.gemm_bf16(M, N, K, seed=2 * M + N, c=True)
    D = Guarded(M, N, torch.bfloat16, init=C)
    swg.gemm_ex(0, 0, M, N, K, -0.75, A.cuda(), K, B.cuda(), N, 1.0, D.view, D.ld, swg.BF16,
                split)
    assert swg.get_device_error() == 0
    rows = None if M <= 300 else [0, 1, 127, 128, 255, 256, M // 2, M - 1]
    yhat = oracle.gemm(0, 0, M, N, K, -0.75, A, K, B, N, 1.0, C, N, rows=rows)
    out = to_f64(D.cpu("alpha < 0"))
    check_half(out if rows is None else out[rows], yhat, f"alpha -0.75 {M}x{N}x{K}")


def test_beta_one_accumulates_twice():
    """gemm with beta = 1 run twice over the same C adds A B twice."""
    M, N, K = 128, 256, 128
    A, B, _ = synth.gemm_bf16(M, N, K, seed=53, dist="ints")
    Ad, Bd = A.cuda(), B.cuda()
    C = Guarded(M, N, torch.float32, fill=0.0)
    swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, C.view, C.ld, swg.BF16_F32OUT)
    swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, C.view, C.ld, swg.BF16_F32OUT)
    torch.cuda.synchronize()
    AB = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0)
    assert np.array_equal(to_f64(C.cpu("beta 1")), 2 * AB)   # small integers: exact


@pytest.mark.parametrize("size", [4096, 8192])
@pytest.mark.parametrize("tA", [0, 1])
@pytest.mark.parametrize("tB", [0, 1])
def test_square_bf16_sampled(size, tA, tB):
    """The benchmark's square bf16 cases, alpha = 1, beta = 0 (ldc = N, as
    the benchmark calls it): every output finite, sampled rows (first, last,
    the 128-row tile and 256-row pair-tile edges, the middle, random) equal
    to the oracle within tolerance, guard rows above and below untouched."""
    M = N = K = size
    A, B, _ = synth.gemm_bf16(M, N, K, tA, tB, seed=1)
    Ad, Bd = A.cuda(), B.cuda()
    D = Guarded(M, N, torch.bfloat16, ld=N)
    swg.gemm(tA, tB, M, N, K, 1.0, Ad, A.shape[1], Bd, B.shape[1], 0.0, D.view, N, swg.BF16)
    assert swg.get_device_error() == 0
    out = D.cpu(f"{size}^3")
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(size + tA * 2 + tB)
    rows = sorted({0, 127, 128, 255, 256, M // 2, M - 257, M - 256, M - 1,
                   *rng.integers(0, M, 4).tolist()})
    yhat = oracle.gemm(tA, tB, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 0.0, rows=rows)
    check_half(to_f64(out)[rows], yhat, f"{size}^3 tA={tA} tB={tB}")


def test_default_stream_is_torch_current_stream():
    """Calls without a stream go on torch's current stream of the current
    device, also inside a `torch.cuda.stream` context."""
    s = torch.cuda.Stream()
    assert swg._stream(None) == torch.cuda.current_stream().cuda_stream
    with torch.cuda.stream(s):
        assert swg._stream(None) == s.cuda_stream
        A = torch.ones((128, 64), dtype=torch.bfloat16, device="cuda")
        D = torch.empty((128, 128), dtype=torch.bfloat16, device="cuda")
        swg.gemm(0, 0, 128, 128, 64, 1.0, A, 64, A.t().contiguous(), 128, 0.0, D, 128, swg.BF16)
    s.synchronize()
    assert torch.all(D == 64.0)
    assert swg._stream(None) == torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("shape", [(512, 768, 640), (256, 128, 1000), (384, 448, 72), (1024, 2048, 512)])
def test_mn_major_3d_boxes_match_2d(monkeypatch, tA, tB, shape):
    """An MN-major operand whose MN extent is a multiple of 64 is loaded with
    one 3-D TMA box per stage instead of one 2-D box per 64-wide atom; the
    stage contents, and so the outputs, must be identical (SWG_MN_3D=0 keeps
    the 2-D boxes)."""
    M, N, K = shape
    g = synth.generator(900 + M + N + K + 2 * tA + tB)
    A = synth.normal(synth.stored_shape(tA, M, K), g).cuda()
    B = synth.normal(synth.stored_shape(tB, K, N), g).cuda()
    C = synth.normal((M, N), g).cuda()
    out = []
    for flag in ("1", "0"):
        monkeypatch.setenv("SWG_MN_3D", flag)
        D = Guarded(M, N, torch.bfloat16, init=C)
        swg.gemm(tA, tB, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 0.5, D.view, D.ld, swg.BF16)
        out.append(D.cpu(f"3-D boxes={flag}"))
    assert swg.get_device_error() == 0
    assert torch.equal(out[0], out[1])
    yhat = oracle.gemm(tA, tB, M, N, K, 1.0, A.cpu(), A.shape[1], B.cpu(), B.shape[1], 0.5,
                       C.cpu(), N)
    check_half(to_f64(out[0]), yhat, f"3-D boxes {shape} tA={tA} tB={tB}")


@pytest.mark.parametrize("M,K,N", [(512, 896, 4864), (128, 512, 640)])
def test_swiglu_3d_weight_boxes_match_2d(monkeypatch, M, K, N):
    A, W1, W2 = synth.swiglu(M, K, N, seed=910 + M)
    Ad = A.cuda()
    Wf = swg.interleave_weights(W1.cuda(), W2.cuda())
    out = []
    for flag in ("1", "0"):
        monkeypatch.setenv("SWG_MN_3D", flag)
        Y = Guarded(M, N, torch.bfloat16, ld=N)
        swg.swiglu_mlp(Ad, Wf, Y.view, M, N, K)
        out.append(Y.cpu(f"swiglu 3-D boxes={flag}"))
    assert swg.get_device_error() == 0
    assert torch.equal(out[0], out[1])
    rows = sorted(r for r in {0, 127, 128, 255, 256, M - 1} if r < M)
    yhat = oracle.swiglu(A, W1, W2, M, N, K, rows=rows)
    check_half(to_f64(out[0])[rows], yhat, f"swiglu 3-D boxes M={M}")


@pytest.mark.parametrize("M", [16, 64])
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 0), (1, 1)])
def test_few_rows_3d_boxes_match_2d(monkeypatch, M, tA, tB):
    """The few-rows split-K path (transposed product) with MN-major operands
    in 3-D boxes gives the same bits as with 2-D boxes."""
    N, K = 1024, 4096
    g = synth.generator(920 + M + 2 * tA + tB)
    A = synth.normal(synth.stored_shape(tA, M, K), g).cuda()
    B = synth.normal(synth.stored_shape(tB, K, N), g).cuda()
    C = synth.normal((M, N), g).cuda()
    out = []
    for flag in ("1", "0"):
        monkeypatch.setenv("SWG_MN_3D", flag)
        D = Guarded(M, N, torch.bfloat16, init=C)
        swg.gemm(tA, tB, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 1.0, D.view, D.ld, swg.BF16)
        out.append(D.cpu(f"few rows 3-D boxes={flag}"))
    assert swg.get_device_error() == 0
    assert torch.equal(out[0], out[1])
    yhat = oracle.gemm(tA, tB, M, N, K, 1.0, A.cpu(), A.shape[1], B.cpu(), B.shape[1], 1.0,
                       C.cpu(), N)
    check_half(to_f64(out[0]), yhat, f"few rows 3-D M={M} tA={tA} tB={tB}")


@pytest.mark.parametrize("M", [128, 512])
def test_swiglu_dual_3d_boxes_match_2d(monkeypatch, M):
    K, N = 640, 1536
    A, W1, W2 = synth.swiglu(M, K, N, seed=930 + M)
    Ad, W1d, W2d = A.cuda(), W1.cuda(), W2.cuda()
    out = []
    for flag in ("1", "0"):
        monkeypatch.setenv("SWG_MN_3D", flag)
        Y = Guarded(M, N, torch.bfloat16, ld=N)
        swg.swiglu_mlp_dual(Ad, W1d, W2d, Y.view, M, N, K)
        out.append(Y.cpu(f"dual 3-D boxes={flag}"))
    assert swg.get_device_error() == 0
    assert torch.equal(out[0], out[1])
    yhat = oracle.swiglu(A, W1, W2, M, N, K)
    check_half(to_f64(out[0]), yhat, f"dual 3-D M={M}")
