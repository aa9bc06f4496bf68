"""Pins for the FP64 oracle, each fixed by something other than the oracle.

* the worked example printed on "GEMM o Coração Matemático", §1 (value 17)
  and its outer-product restatement in §2.1;
* exact brute force with Python integers / fractions on tiny shapes, for all
  four op combinations, padded row strides and several alpha, beta;
* algebraic identities: (AB)^T = B^T A^T, A I = A, alpha linearity, beta = 0
  never reading C, beta = 1 accumulation;
* closed forms of SiLU (odd part, minimum through Lambert W, sigmoid(ln 3));
* the storage decoders against numpy (binary16) and torch (bfloat16) on every
  16-bit pattern;
* the Kernel-2 column interleave on a hand-written example ("Sobreposição de
  Ativação em Nível de Tile ...", Metodologia, Kernel-2: even columns Gate,
  odd columns Up).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.txt")


def _read_golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            vals[key] = [int(x) for x in rest]
    return vals


def _stored(trans, mat):
    """Row-major storage of a Python list-of-lists for op = N / T."""
    m = np.array(mat, dtype=np.float32)
    return np.ascontiguousarray(m.T if trans else m)


def test_worked_example_value_17():
    g = _read_golden()
    M, K, N = g["M"][0], g["K"][0], g["N"][0]
    A = np.array(g["A"], dtype=np.float32).reshape(M, K)
    B = np.array(g["B"], dtype=np.float32).reshape(K, N)
    C = np.array(g["C_old"], dtype=np.float32).reshape(M, N)
    # §2: row-major storage puts A_{1,1} at position 4.
    assert A.reshape(-1)[g["A11_position"][0]] == g["A11_value"][0]
    for tA in (0, 1):
        for tB in (0, 1):
            a = _stored(tA, A)
            b = _stored(tB, B)
            D = oracle.gemm(tA, tB, M, N, K, g["alpha"][0], a, a.shape[1], b,
                            b.shape[1], g["beta"][0], C, N, in_type="f32",
                            c_type="f32")
            assert D[0, 0] == g["D00"][0]


def test_worked_example_all_elements_and_outer_product():
    """The other three elements are not printed; they follow from the printed
    data with Python integers, both as row-by-column dot products (§1) and as
    the sum of outer products a_p b_p^T (§2.1)."""
    g = _read_golden()
    M, K, N = g["M"][0], g["K"][0], g["N"][0]
    A = [g["A"][i * K:(i + 1) * K] for i in range(M)]
    B = [g["B"][p * N:(p + 1) * N] for p in range(K)]
    Cold = [g["C_old"][i * N:(i + 1) * N] for i in range(M)]
    dot = [[sum(A[i][p] * B[p][j] for p in range(K)) for j in range(N)] for i in range(M)]
    outer = [[0] * N for _ in range(M)]
    for p in range(K):
        col = [A[i][p] for i in range(M)]
        row = B[p]
        for i in range(M):
            for j in range(N):
                outer[i][j] += col[i] * row[j]
    assert dot == outer
    alpha, beta = g["alpha"][0], g["beta"][0]
    want = [[alpha * dot[i][j] + beta * Cold[i][j] for j in range(N)] for i in range(M)]
    D = oracle.gemm(0, 0, M, N, K, alpha, np.array(A, np.float32), K,
                    np.array(B, np.float32), N, beta, np.array(Cold, np.float32), N,
                    in_type="f32", c_type="f32")
    assert D.tolist() == want
    D0 = oracle.gemm(0, 0, M, N, K, 1.0, np.array(A, np.float32), K,
                     np.array(B, np.float32), N, 0.0, in_type="f32", c_type="f32")
    assert D0.tolist() == outer


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _exact(t):
    """Exact Fraction values of a half-precision torch tensor."""
    return [[Fraction(float(v)) for v in row] for row in t.to(torch.float64).tolist()]


def _pad(t, ld):
    """Stored matrix with row stride ld >= cols; padding filled with a large
    value so a wrong stride shows up."""
    rows, cols = t.shape
    out = torch.full((rows, ld), 1000.0, dtype=t.dtype)
    out[:, :cols] = t
    return out


@pytest.mark.parametrize("dtype,kind", [(torch.bfloat16, "bf16"), (torch.float16, "f16")])
@pytest.mark.parametrize("tA", [0, 1])
@pytest.mark.parametrize("tB", [0, 1])
@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (7, 4, 9), (16, 17, 33)])
def test_bruteforce_exact(dtype, kind, tA, tB, shape):
    M, N, K = shape
    g = synth.generator(M * 1000 + N * 100 + K + 7 * tA + 13 * tB + (50 if kind == "f16" else 0))
    A = synth.small_ints(synth.stored_shape(tA, M, K), g, dtype=dtype)
    B = synth.small_ints(synth.stored_shape(tB, K, N), g, dtype=dtype)
    C = synth.small_ints((M, N), g, dtype=torch.float32)
    opA = _exact(A.T if tA else A)
    opB = _exact(B.T if tB else B)
    Cx = _exact(C)
    lda, ldb, ldc = A.shape[1] + 3, B.shape[1] + 5, N + 2
    Ap, Bp, Cp = _pad(A, lda), _pad(B, ldb), _pad(C, ldc)
    for alpha, beta in [(1.0, 0.0), (2.0, 1.0), (-0.5, -2.0), (0.25, 0.5)]:
        D = oracle.gemm(tA, tB, M, N, K, alpha, _bits(Ap), lda, _bits(Bp), ldb,
                        beta, Cp.numpy(), ldc, in_type=kind, c_type="f32")
        for i in range(M):
            for j in range(N):
                s = sum(opA[i][p] * opB[p][j] for p in range(K))
                want = Fraction(alpha) * s + Fraction(beta) * Cx[i][j]
                assert Fraction(D[i, j]) == want, (i, j, alpha, beta)


@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1)])
def test_rows_and_cols_subsets_match_full(tA, tB):
    M, N, K = 9, 6, 11
    A, B, C = synth.gemm_bf16(M, N, K, tA, tB, seed=7, c=True)
    lda, ldb = A.shape[1], B.shape[1]
    full = oracle.gemm(tA, tB, M, N, K, 1.5, A, lda, B, ldb, -1.0, C, N)
    part = oracle.gemm(tA, tB, M, N, K, 1.5, A, lda, B, ldb, -1.0, C, N, rows=[5, 2, 8])
    assert np.array_equal(part, full[[5, 2, 8]])
    sub = oracle.gemm(tA, tB, M, N, K, 1.5, A, lda, B, ldb, -1.0, C, N, rows=[5, 2, 8],
                      cols=[4, 0, 5])
    assert np.array_equal(sub, full[np.ix_([5, 2, 8], [4, 0, 5])])
    A2, W1, W2 = synth.swiglu(M, K, N, seed=8)
    yf = oracle.swiglu(A2, W1, W2, M, N, K)
    assert np.array_equal(oracle.swiglu(A2, W1, W2, M, N, K, rows=[1, 3], cols=[5, 1]),
                          yf[np.ix_([1, 3], [5, 1])])


def test_transpose_identity():
    """(AB)^T = B^T A^T: computing D^T with both operands transposed uses the
    same products in the same order, so it agrees bit for bit."""
    M, N, K = 13, 9, 40
    A, B, _ = synth.gemm_bf16(M, N, K, seed=11)
    D = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0)
    # op(A') = B^T with A' = B stored K x N; op(B') = A^T with B' = A stored M x K.
    Dt = oracle.gemm(1, 1, N, M, K, 1.0, B, N, A, K, 0.0)
    assert np.array_equal(Dt, D.T)


def test_identity_matrix():
    M, K = 12, 20
    g = synth.generator(5)
    A = synth.normal((M, K), g)
    eye = torch.eye(K, dtype=torch.bfloat16)
    D = oracle.gemm(0, 0, M, K, K, 1.0, A, K, eye, K, 0.0)
    assert np.array_equal(D, A.to(torch.float64).numpy())
    # I A^T stored as A: op(B) = A^T, so D = I * A^T = A^T.
    eyeM = torch.eye(K, dtype=torch.bfloat16)
    D2 = oracle.gemm(0, 1, K, M, K, 1.0, eyeM, K, A, K, 0.0)
    assert np.array_equal(D2, A.to(torch.float64).numpy().T)


def test_alpha_linearity_and_beta_zero_ignores_nan():
    M, N, K = 10, 7, 33
    A, B, _ = synth.gemm_bf16(M, N, K, seed=13)
    C = torch.full((M, N), float("nan"), dtype=torch.float32)
    D1 = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, C, N, c_type="f32")
    assert np.isfinite(D1).all()
    D4 = oracle.gemm(0, 0, M, N, K, 4.0, A, K, B, N, 0.0, C, N, c_type="f32")
    assert np.array_equal(D4, 4.0 * D1)          # power of two: exact
    D3 = oracle.gemm(0, 0, M, N, K, 0.3, A, K, B, N, 0.0)
    np.testing.assert_allclose(D3, 0.3 * D1, rtol=1e-15, atol=0)
    # beta != 0 with NaN in C must propagate (C is read).
    Dn = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N, c_type="f32")
    assert np.isnan(Dn).all()


def test_beta_one_accumulates():
    """beta = 1 turns GEMM into an accumulator (§1): gemm(C = A B) with
    beta = 1 gives 2 A B, exact for small integers."""
    M, N, K = 8, 8, 16
    A, B, _ = synth.gemm_bf16(M, N, K, seed=17, dist="ints")
    AB = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0)
    C = torch.from_numpy(AB.astype(np.float32))
    D = oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N, c_type="f32")
    assert np.array_equal(D, 2 * AB)


def test_silu_closed_forms():
    scipy_special = pytest.importorskip("scipy.special")
    assert oracle.silu(0.0) == 0.0
    # sigmoid(ln 3) = 3/4, so SiLU(ln 3) = 0.75 ln 3.
    assert oracle.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    # SiLU(x) - SiLU(-x) = x (x * (sigma(x) + sigma(-x) - 1) = 0 ... odd part is x/2 * 2).
    for x in (1e-3, 0.5, 1.0, 2.5, 7.0, 30.0):
        assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, rel=1e-14)
    # Asymptotes: SiLU(x)/x -> 1 as x -> +inf, SiLU(x) -> 0- as x -> -inf.
    assert oracle.silu(40.0) / 40.0 == pytest.approx(1.0, abs=1e-15)
    assert -1e-15 < oracle.silu(-40.0) < 0.0
    assert oracle.silu(-1000.0) == 0.0 and math.copysign(1, oracle.silu(-1000.0)) < 0
    # Minimum: SiLU'(x) = 0 at x* = -(1 + W0(1/e)), value -W0(1/e).
    w = float(scipy_special.lambertw(math.exp(-1.0)).real)
    xs = -(1.0 + w)
    assert oracle.silu(xs) == pytest.approx(-w, rel=1e-14)
    for d in (1e-3, -1e-3):
        assert oracle.silu(xs + d) > oracle.silu(xs)


def test_f16_decoder_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_all_patterns():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b) & 0xFFFF) for b in bits.tolist()])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_interleave_hand_example():
    W1 = torch.tensor([[1, 2], [3, 4]], dtype=torch.bfloat16)
    W2 = torch.tensor([[5, 6], [7, 8]], dtype=torch.bfloat16)
    Wf = oracle.interleave(W1, W2, 2, 2)
    got = torch.from_numpy(Wf.view(np.int16)).view(torch.bfloat16).to(torch.int64)
    assert got.tolist() == [[1, 5, 2, 6], [3, 7, 4, 8]]


def test_swiglu_odd_part_pins_gate_side():
    """With one-hot rows of A, G and U are single weights.  SiLU(g)u -
    SiLU(-g)u = g u exactly in real arithmetic; that fails if SiLU were put on
    the Up side, left out, or replaced by the sigmoid."""
    K, N = 4, 6
    gvals = [0.5, 1.0, 2.0, 3.0, -1.5, 0.25]
    uvals = [1.0, 2.0, -0.5, 4.0, 1.0, -3.0]
    W1 = torch.zeros((K, N), dtype=torch.bfloat16)
    W2 = torch.zeros((K, N), dtype=torch.bfloat16)
    W1[0] = torch.tensor(gvals)
    W1[1] = -torch.tensor(gvals)
    W2[0] = torch.tensor(uvals)
    W2[1] = torch.tensor(uvals)
    W1[2] = 0.0
    W2[2] = torch.tensor(uvals)
    A = torch.zeros((3, K), dtype=torch.bfloat16)
    A[0, 0] = 1
    A[1, 1] = 1
    A[2, 2] = 1
    Y = oracle.swiglu(A, W1, W2, 3, N, K)
    for n in range(N):
        assert Y[0, n] - Y[1, n] == pytest.approx(gvals[n] * uvals[n], rel=1e-14)
        assert Y[2, n] == 0.0


def test_swiglu_bruteforce_integer_products():
    """Gate and Up sums checked with Python integers, then combined with the
    (separately pinned) scalar SiLU."""
    M, K, N = 5, 12, 7
    g = synth.generator(21)
    A = synth.small_ints((M, K), g, -3, 3)
    W1 = synth.small_ints((K, N), g, -2, 2)
    W2 = synth.small_ints((K, N), g, -2, 2)
    Ai, W1i, W2i = (t.to(torch.int64).tolist() for t in (A, W1, W2))
    Y = oracle.swiglu(A, W1, W2, M, N, K)
    for i in range(M):
        for n in range(N):
            gs = sum(Ai[i][p] * W1i[p][n] for p in range(K))
            us = sum(Ai[i][p] * W2i[p][n] for p in range(K))
            assert Y[i, n] == oracle.silu(gs) * us


def test_swiglu_equals_two_gemms_plus_elementwise():
    M, K, N = 6, 40, 10
    A, W1, W2 = synth.swiglu(M, K, N, seed=23)
    G = oracle.gemm(0, 0, M, N, K, 1.0, A, K, W1, N, 0.0)
    U = oracle.gemm(0, 0, M, N, K, 1.0, A, K, W2, N, 0.0)
    want = np.vectorize(oracle.silu)(G) * U
    assert np.array_equal(oracle.swiglu(A, W1, W2, M, N, K), want)
    # and through the interleaved weight read as Gate / Up column pairs
    Wf = oracle.interleave(W1, W2, K, N)
    assert np.array_equal(Wf[:, 0::2], W1.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(Wf[:, 1::2], W2.view(torch.int16).numpy().view(np.uint16))


def test_mlp_identity_down_projection_and_residual():
    """With W_down = I (N = K) the MLP returns the gated activation itself, and
    beta = 1 adds the residual; both exact in double."""
    M, K = 6, 16
    A, W1, W2 = synth.swiglu(M, K, K, seed=31, w_std=0.2)
    eye = torch.eye(K, dtype=torch.bfloat16)
    Y = oracle.swiglu(A, W1, W2, M, K, K)
    assert np.array_equal(oracle.mlp(A, W1, W2, eye, M, K, K), Y)
    R = synth.small_ints((M, K), synth.generator(32), -3, 3)
    got = oracle.mlp(A, W1, W2, eye, M, K, K, beta=1.0, Out_old=R)
    assert np.array_equal(got, Y + R.to(torch.float64).numpy())


def test_mlp_down_projection_bruteforce():
    """The down projection of the (pinned) gated activation, checked element
    by element with Python floats summed in the same order; scaling W_down by
    2 doubles the output exactly."""
    M, N, K = 4, 10, 6
    A, W1, W2 = synth.swiglu(M, K, N, seed=33, w_std=0.3)
    Wd = synth.small_ints((N, K), synth.generator(34), -2, 2)
    Y = oracle.swiglu(A, W1, W2, M, N, K)
    Wdf = Wd.to(torch.float64).tolist()
    out = oracle.mlp(A, W1, W2, Wd, M, N, K)
    for i in range(M):
        for k in range(K):
            s = 0.0
            for n in range(N):
                s += Y[i, n] * Wdf[n][k]
            assert out[i, k] == s
    assert np.array_equal(oracle.mlp(A, W1, W2, (2 * Wd).to(torch.bfloat16), M, N, K), 2 * out)



def test_round_bf16_matches_torch_on_binary32_values():
    """round_bf16 against torch's binary32 -> bfloat16 conversion (round to
    nearest, ties to even), on values exactly representable in binary32, so
    that conversion rounds them once: random bit patterns over the whole range
    (normal, subnormal, near overflow) and patterns whose dropped half is
    exactly a tie or one unit either side of it."""
    rng = np.random.default_rng(5)
    hi = rng.integers(0, 2 ** 16, 20000, dtype=np.uint64)
    lows = [rng.integers(0, 2 ** 16, 20000, dtype=np.uint64)] + [
        np.full(20000, v, dtype=np.uint64) for v in (0x8000, 0x7FFF, 0x8001, 0x0000)]
    for lo in lows:
        f = ((hi << 16) | lo).astype(np.uint32).view(np.float32)
        f = f[np.isfinite(f)]
        ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float64).numpy()
        got = np.array([oracle.round_bf16(float(x)) for x in f])
        assert np.array_equal(got, ref)


def test_round_bf16_hand_cases():
    """Ties go to the even neighbour; the exact value is rounded once (a value
    just above a tie goes up, where rounding through binary32 first would
    land on the tie and go down); every bfloat16 value is unchanged; the
    overflow and subnormal ends."""
    assert oracle.round_bf16(1 + 2 ** -8) == 1.0
    assert oracle.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6
    assert oracle.round_bf16(-(1 + 2 ** -8)) == -1.0
    assert oracle.round_bf16(1 + 2 ** -8 + 2 ** -40) == 1 + 2 ** -7
    big = (2 - 2 ** -7) * 2.0 ** 127                   # largest finite bfloat16
    assert oracle.round_bf16(big) == big
    assert oracle.round_bf16((2 - 2 ** -8 - 2 ** -30) * 2.0 ** 127) == big
    assert oracle.round_bf16((2 - 2 ** -8) * 2.0 ** 127) == float("inf")   # tie: even is 2^128
    assert oracle.round_bf16(-1e39) == float("-inf")
    assert oracle.round_bf16(2.0 ** -134) == 0.0                          # tie with 0
    assert oracle.round_bf16(3 * 2.0 ** -134) == 2.0 ** -132              # tie, even side
    assert oracle.round_bf16(2.0 ** -133) == 2.0 ** -133
    assert np.isnan(oracle.round_bf16(float("nan")))
    for b in range(0, 1 << 16, 7):
        v = oracle.bf16_to_f64(b)
        if np.isfinite(v):
            assert oracle.round_bf16(v) == v


def test_mlp_with_bf16_activation():
    """round_y: W_down = I returns the gated activation rounded to bfloat16
    element by element, and the down projection of a general W_down is the
    in-order sum over the rounded activation."""
    M, K = 5, 16
    A, W1, W2 = synth.swiglu(M, K, K, seed=35, w_std=0.2)
    eye = torch.eye(K, dtype=torch.bfloat16)
    Y = oracle.swiglu(A, W1, W2, M, K, K)
    Yr = np.vectorize(oracle.round_bf16)(Y)
    assert not np.array_equal(Yr, Y)
    assert np.array_equal(oracle.mlp(A, W1, W2, eye, M, K, K, round_y=True), Yr)
    N = 10
    A, W1, W2 = synth.swiglu(M, K, N, seed=36, w_std=0.3)
    Wd = synth.small_ints((N, K), synth.generator(37), -2, 2)
    Yr = np.vectorize(oracle.round_bf16)(oracle.swiglu(A, W1, W2, M, N, K))
    Wdf = Wd.to(torch.float64).tolist()
    out = oracle.mlp(A, W1, W2, Wd, M, N, K, round_y=True)
    for i in range(M):
        for k in range(K):
            s = 0.0
            for n in range(N):
                s += Yr[i, n] * Wdf[n][k]
            assert out[i, k] == s


def test_e4m3_decoder_all_patterns():
    bits = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = bits.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(int(b)) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_to_f64(0x7E) == 448.0          # largest finite value


@pytest.mark.parametrize("shape", [(3, 5, 7), (9, 16, 33)])
def test_e4m3_gemm_bruteforce_exact(shape):
    """Small integers are exact in e4m3 (|x| <= 16) and in every partial sum."""
    M, N, K = shape
    g = synth.generator(M + N + K + 500)
    A = synth.small_ints((M, K), g, -6, 6, dtype=torch.float32).to(torch.float8_e4m3fn)
    Bt = synth.small_ints((N, K), g, -6, 6, dtype=torch.float32).to(torch.float8_e4m3fn)
    Ai = A.to(torch.float64).tolist()
    Bi = Bt.to(torch.float64).tolist()
    D = oracle.gemm(0, 1, M, N, K, 0.5, A, K, Bt, K, 0.0, in_type="e4m3")
    for i in range(M):
        for j in range(N):
            assert D[i, j] == 0.5 * sum(Ai[i][p] * Bi[j][p] for p in range(K))


def test_swiglu_typed_matches_swiglu_and_scales():
    M, K, N = 5, 24, 7
    A, W1, W2 = synth.swiglu(M, K, N, seed=41, w_std=0.2)
    ref = oracle.swiglu(A, W1, W2, M, N, K)
    assert np.array_equal(oracle.swiglu_typed(A, W1, W2, M, N, K, in_type="bf16", scale=1.0), ref)
    # scale s on both products: SiLU(s g) s u; with s = 2 and W halved it is unchanged
    W1h = (W1.to(torch.float32) / 2).to(torch.bfloat16)
    W2h = (W2.to(torch.float32) / 2).to(torch.bfloat16)
    got = oracle.swiglu_typed(A, W1h, W2h, M, N, K, in_type="bf16", scale=2.0)
    assert np.allclose(got, ref, rtol=1e-15, atol=1e-15)


def test_interleave_t8_hand_example():
    W1 = torch.tensor([[1, 2], [3, 4]], dtype=torch.float32).to(torch.float8_e4m3fn)
    W2 = torch.tensor([[5, 6], [7, 8]], dtype=torch.float32).to(torch.float8_e4m3fn)
    Wt = oracle.interleave_t8(W1, W2, 2, 2)
    got = torch.from_numpy(Wt).view(torch.float8_e4m3fn).to(torch.int64).tolist()
    # rows: W1 col 0, W2 col 0, W1 col 1, W2 col 1
    assert got == [[1, 3], [5, 7], [2, 4], [6, 8]]
