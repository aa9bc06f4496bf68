/*
 * oracle.c — plain FP64 CPU oracle for the GEMM and fused-SwiGLU hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or helper with the CUDA
 * library under swiglu_mlp_gb300/.
 *
 * What it computes (sources, by page title and section):
 *
 *   GEMM   D[i][j] = alpha * sum_p opA(i,p) * opB(p,j) + beta * C_old[i][j]
 *          "GEMM o Coração Matemático", §1 (the BLAS GEMM statement and its
 *          element-wise form; op(X) is X or its transpose) and §2 (row-major
 *          linearisation, position i*N + j).  The sum over p runs in ascending
 *          order, one element at a time, in double precision.
 *          When beta == 0, C is not read at all (§2.1, the ikj kernel fills C
 *          with zeros instead of scaling it), so NaN in C cannot leak out.
 *
 *   SwiGLU Y = SiLU(A*W1) (.) (A*W2), with SiLU(x) = x * sigmoid(x)
 *          = x / (1 + exp(-x))
 *          "Sobreposição de Ativação em Nível de Tile para Inferência
 *          Eficiente de LLM", Definição do Problema (the gated MLP) and
 *          Metodologia, Kernel-2 (SiLU applied to the Gate column, multiplied
 *          by the Up column).  The oracle takes W1 and W2 SEPARATELY, so the
 *          column interleave used by the product is checked independently.
 *
 *   Interleave  W_fused[k][2n] = W1[k][n], W_fused[k][2n+1] = W2[k][n]
 *          Same page, Metodologia, Kernel-2 (even columns Gate, odd Up).
 *
 * Inputs arrive as the stored, already-rounded values: IEEE binary16 bits,
 * bfloat16 bits, or binary32.  Each is widened to double exactly (every
 * binary16, bfloat16 and binary32 value is a double).  Outputs are double and
 * are NOT rounded to the product's output type.
 *
 * Speed comes only from splitting rows across threads and from visiting
 * (p, j) in the ikj order ("GEMM o Coração Matemático", §2.1), which keeps the
 * per-element summation order p = 0, 1, ..., K-1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2, ORC_E4M3 = 3 };

/* ---- exact widening of the stored formats ---------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)            /* zero or subnormal: f * 2^-24 */
        v = ldexp((double)f, -24);
    else if (e == 31)      /* infinity or NaN */
        v = f ? NAN : INFINITY;
    else                   /* normal: (1024 + f) * 2^(e - 15 - 10) */
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32: 1 sign, 8 exponent bits
 * (bias 127), 7 fraction bits.  Decoded from the fields, not by a bit cast. */
double orc_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)            /* zero or subnormal: f * 2^-133 */
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else                   /* (128 + f) * 2^(e - 127 - 7) */
        v = ldexp((double)(128 + f), e - 134);
    return sign ? -v : v;
}

/* e4m3: 1 sign, 4 exponent bits (bias 7), 3 fraction bits; no infinities,
 * exponent and fraction all ones is NaN, so the largest value is
 * 1.75 * 2^8 = 448.  The field layout is the E4M3 encoding of the OCP 8-bit
 * floating-point format (the one torch's float8_e4m3fn implements, against
 * which this decoder is pinned on all 256 patterns); the pages define no
 * 8-bit layout -- "GEMM o Coração Matemático", §12.4 covers only quantised
 * operands with a scale. */
double orc_e4m3_to_f64(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int f = b & 0x7;
    double v;
    if (e == 0)                    /* zero or subnormal: f * 2^-9 */
        v = ldexp((double)f, -9);
    else if (e == 15 && f == 7)
        v = NAN;
    else                           /* (8 + f) * 2^(e - 7 - 3) */
        v = ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

static double load_elem(const void *base, int64_t idx, int type)
{
    switch (type) {
    case ORC_F16:  return orc_f16_to_f64(((const uint16_t *)base)[idx]);
    case ORC_BF16: return orc_bf16_to_f64(((const uint16_t *)base)[idx]);
    case ORC_E4M3: return orc_e4m3_to_f64(((const uint8_t *)base)[idx]);
    default:       return (double)((const float *)base)[idx];
    }
}

/* SiLU(x) = x * sigmoid(x) = x / (1 + e^-x). */
double orc_silu(double x)
{
    return x / (1.0 + exp(-x));
}

/* ---- GEMM ------------------------------------------------------------ */

typedef struct {
    int transA, transB;
    int64_t M, N, K;
    double alpha, beta;
    const void *A; int64_t lda; int a_type;
    const double *opB;            /* op(B) widened, K x N, row-major */
    const void *C; int64_t ldc; int c_type;
    const int64_t *rows; int64_t n_rows;
    const int64_t *cols;          /* output column j of D is column cols[j] (NULL: j) */
    double *D;                    /* n_rows x N, N = number of computed columns */
    int64_t r_begin, r_end;
} gemm_job;

/* opA(i,p): row-major A is M x K (op = N) or K x M (op = T), row stride lda. */
static double opA_at(const gemm_job *g, int64_t i, int64_t p)
{
    int64_t idx = g->transA ? p * g->lda + i : i * g->lda + p;
    return load_elem(g->A, idx, g->a_type);
}

static void *gemm_rows(void *arg)
{
    gemm_job *g = (gemm_job *)arg;
    const int64_t N = g->N, K = g->K;
    double *arow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (int64_t r = g->r_begin; r < g->r_end; ++r) {
        int64_t i = g->rows ? g->rows[r] : r;
        double *acc = g->D + r * N;
        for (int64_t j = 0; j < N; ++j)
            acc[j] = 0.0;
        for (int64_t p = 0; p < K; ++p)
            arow[p] = opA_at(g, i, p);
        /* ikj: acc[j] += a_ip * b_pj for p = 0..K-1; each acc[j] still sums
         * its K products in ascending p. */
        for (int64_t p = 0; p < K; ++p) {
            const double a = arow[p];
            const double *brow = g->opB + p * N;
            for (int64_t j = 0; j < N; ++j)
                acc[j] += a * brow[j];
        }
        for (int64_t j = 0; j < N; ++j) {
            int64_t col = g->cols ? g->cols[j] : j;
            double y = g->alpha * acc[j];
            if (g->beta != 0.0)
                y += g->beta * load_elem(g->C, i * g->ldc + col, g->c_type);
            acc[j] = y;
        }
    }
    free(arow);
    return NULL;
}

static int pick_threads(int n_threads, int64_t n_rows)
{
    if (n_threads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = c > 0 ? (int)c : 1;
    }
    if (n_threads > 256) n_threads = 256;
    if ((int64_t)n_threads > n_rows) n_threads = (int)(n_rows > 0 ? n_rows : 1);
    return n_threads;
}

/* Widen the selected columns of op(B) into a dense K x N double matrix:
 * opB(p,c) = B[p*ldb + c] (op = N, B stored K x N) or B[c*ldb + p] (op = T,
 * B stored N x K), with c = cols[j] (or j when cols is NULL). */
static double *widen_opB(int transB, int64_t N, int64_t K, const void *B,
                         int64_t ldb, int b_type, const int64_t *cols)
{
    double *opB = (double *)malloc(sizeof(double) * (size_t)(K * N > 0 ? K * N : 1));
    if (!opB) return NULL;
    for (int64_t p = 0; p < K; ++p)
        for (int64_t j = 0; j < N; ++j) {
            int64_t c = cols ? cols[j] : j;
            opB[p * N + j] = load_elem(B, transB ? c * ldb + p : p * ldb + c, b_type);
        }
    return opB;
}

/* Computes D at rows[0..n_rows) x cols[0..n_cols) (all rows 0..M-1 when rows
 * == NULL, and then n_rows must equal M; all columns when cols == NULL, and
 * then n_cols must equal N).  D is n_rows x n_cols doubles, row-major.  Each
 * element is the same sum whichever rows and columns are requested.  Returns
 * 0 on success, -1 on bad arguments or allocation failure. */
int orc_gemm(int transA, int transB, int64_t M, int64_t N, int64_t K,
             double alpha, const void *A, int64_t lda, int a_type,
             const void *B, int64_t ldb, int b_type, double beta,
             const void *C, int64_t ldc, int c_type,
             const int64_t *rows, int64_t n_rows, const int64_t *cols,
             int64_t n_cols, double *D, int n_threads)
{
    if (M < 0 || N < 0 || K < 0 || n_rows < 0 || n_cols < 0 || !D) return -1;
    if (!rows && n_rows != M) return -1;
    if (!cols && n_cols != N) return -1;
    N = n_cols;
    if (n_rows == 0 || N == 0) return 0;
    double *opB = widen_opB(transB, N, K, B, ldb, b_type, cols);
    if (!opB) return -1;
    int T = pick_threads(n_threads, n_rows);
    pthread_t th[256];
    gemm_job jobs[256];
    for (int t = 0; t < T; ++t) {
        gemm_job *g = &jobs[t];
        g->transA = transA; g->transB = transB;
        g->M = M; g->N = N; g->K = K;
        g->alpha = alpha; g->beta = beta;
        g->A = A; g->lda = lda; g->a_type = a_type;
        g->opB = opB;
        g->C = C; g->ldc = ldc; g->c_type = c_type;
        g->rows = rows; g->n_rows = n_rows; g->cols = cols; g->D = D;
        g->r_begin = n_rows * t / T;
        g->r_end = n_rows * (t + 1) / T;
        pthread_create(&th[t], NULL, gemm_rows, g);
    }
    for (int t = 0; t < T; ++t)
        pthread_join(th[t], NULL);
    free(opB);
    return 0;
}

/* ---- SwiGLU ---------------------------------------------------------- */

/* Y[i][n] = SiLU(G[i][n]) * U[i][n] with G = A*W1, U = A*W2; A is M x K
 * bfloat16 (row stride lda), W1 and W2 are K x N bfloat16 (row stride ldw).
 * Both products come from orc_gemm with alpha = 1, beta = 0. */
int orc_swiglu(const uint16_t *A, int64_t lda, const uint16_t *W1,
               const uint16_t *W2, int64_t ldw, int64_t M, int64_t N,
               int64_t K, const int64_t *rows, int64_t n_rows,
               const int64_t *cols, int64_t n_cols, double *Y, int n_threads)
{
    if (!rows && n_rows != M) return -1;
    if (!cols && n_cols != N) return -1;
    if (n_rows == 0 || n_cols == 0) return 0;
    double *G = (double *)malloc(sizeof(double) * (size_t)(n_rows * n_cols));
    double *U = (double *)malloc(sizeof(double) * (size_t)(n_rows * n_cols));
    int rc = (G && U) ? 0 : -1;
    if (rc == 0)
        rc = orc_gemm(0, 0, M, N, K, 1.0, A, lda, ORC_BF16, W1, ldw, ORC_BF16,
                      0.0, NULL, 0, ORC_BF16, rows, n_rows, cols, n_cols, G,
                      n_threads);
    if (rc == 0)
        rc = orc_gemm(0, 0, M, N, K, 1.0, A, lda, ORC_BF16, W2, ldw, ORC_BF16,
                      0.0, NULL, 0, ORC_BF16, rows, n_rows, cols, n_cols, U,
                      n_threads);
    if (rc == 0)
        for (int64_t e = 0; e < n_rows * n_cols; ++e)
            Y[e] = orc_silu(G[e]) * U[e];
    free(G);
    free(U);
    return rc;
}

/* W_fused (K x 2N, row stride 2N) from W1, W2 (K x N, row stride N):
 * column 2n is W1's column n (Gate), column 2n+1 is W2's column n (Up). */
void orc_interleave(const uint16_t *W1, const uint16_t *W2, uint16_t *Wf,
                    int64_t K, int64_t N)
{
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            Wf[k * 2 * N + 2 * n] = W1[k * N + n];
            Wf[k * 2 * N + 2 * n + 1] = W2[k * N + n];
        }
}

int orc_num_cores(void)
{
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

/* ---- rounding to bfloat16 -------------------------------------------- */

/* x rounded to the nearest bfloat16 value, ties to the one whose last
 * fraction bit is 0 (IEEE round-to-nearest-even), directly from the double
 * (one rounding).  bfloat16 keeps 8 significant bits (1 implicit + 7 stored)
 * over binary32's exponent range: normal values from 2^-126, subnormals in
 * steps of 2^-133, largest finite (2 - 2^-7) * 2^127; larger magnitudes after
 * rounding become infinities.  Used where the product stores an intermediate
 * in bfloat16 (the gated activation between the MLP's two GEMMs). */
double orc_round_bf16(double x)
{
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    int e;
    (void)frexp(x, &e);                  /* |x| = m * 2^e, 0.5 <= m < 1 */
    int q = e - 8;                       /* 8 significant bits: step 2^(e-8) */
    if (q < -133) q = -133;              /* subnormal range: fixed step 2^-133 */
    double r = ldexp(nearbyint(ldexp(x, -q)), q);   /* default mode: ties to even */
    if (fabs(r) >= ldexp(1.0, 128)) r = x > 0 ? INFINITY : -INFINITY;
    return r;
}

/* ---- full gated MLP -------------------------------------------------- */

/* Out = Y * W_down + beta * Out_old with Y = SiLU(A W1) (.) (A W2).  The FFN
 * of "GEMM o Coração Matemático", §13.3 (two GEMMs around an activation),
 * with the gated activation of "Sobreposição de Ativação em Nível de Tile
 * ...", Definição do Problema.  A: M x K bf16, W1/W2: K x N bf16, W_down:
 * N x K bf16, Out_old: M x K bf16 (read only when beta != 0).  Out: n_rows x K
 * doubles for rows[] (all when rows == NULL).  round_y == 0 keeps Y in
 * double; round_y == 1 rounds each exact Y to bfloat16 (orc_round_bf16)
 * before the down projection, as a product that stores Y in bfloat16 between
 * the two GEMMs does. */
int orc_mlp(const uint16_t *A, const uint16_t *W1, const uint16_t *W2,
            const uint16_t *Wd, const uint16_t *Out_old, double beta, int64_t M,
            int64_t N, int64_t K, const int64_t *rows, int64_t n_rows,
            double *Out, int n_threads, int round_y)
{
    if (!rows && n_rows != M) return -1;
    if (n_rows == 0 || K == 0) return 0;
    double *Y = (double *)malloc(sizeof(double) * (size_t)(n_rows * (N > 0 ? N : 1)));
    if (!Y) return -1;
    int rc = orc_swiglu(A, K, W1, W2, N, M, N, K, rows, n_rows, NULL, N, Y, n_threads);
    if (rc == 0 && round_y)
        for (int64_t e = 0; e < n_rows * N; ++e)
            Y[e] = orc_round_bf16(Y[e]);
    if (rc == 0) {
        for (int64_t r = 0; r < n_rows; ++r) {
            const int64_t i = rows ? rows[r] : r;
            double *o = Out + r * K;
            for (int64_t k = 0; k < K; ++k)
                o[k] = 0.0;
            for (int64_t n = 0; n < N; ++n) {        /* ascending n for each o[k] */
                const double y = Y[r * N + n];
                for (int64_t k = 0; k < K; ++k)
                    o[k] += y * orc_bf16_to_f64(Wd[n * K + k]);
            }
            if (beta != 0.0)
                for (int64_t k = 0; k < K; ++k)
                    o[k] += beta * orc_bf16_to_f64(Out_old[i * K + k]);
        }
    }
    free(Y);
    return rc;
}

/* ---- quantised SwiGLU -------------------------------------------------- */

/* Y = SiLU(scale * G) * (scale * U), G = A W1, U = A W2, for A (M x K, row
 * stride K) and W1, W2 (K x N, row stride N) of storage type `type`; scale is
 * the product of the per-tensor dequantisation scales of A and W.  The same
 * SwiGLU as orc_swiglu, on quantised operands ("GEMM o Coração Matemático",
 * §12.4). */
int orc_swiglu_typed(const void *A, const void *W1, const void *W2, int type,
                     double scale, int64_t M, int64_t N, int64_t K,
                     const int64_t *rows, int64_t n_rows, const int64_t *cols,
                     int64_t n_cols, double *Y, int n_threads)
{
    if (!rows && n_rows != M) return -1;
    if (!cols && n_cols != N) return -1;
    if (n_rows == 0 || n_cols == 0) return 0;
    double *G = (double *)malloc(sizeof(double) * (size_t)(n_rows * n_cols));
    double *U = (double *)malloc(sizeof(double) * (size_t)(n_rows * n_cols));
    int rc = (G && U) ? 0 : -1;
    if (rc == 0)
        rc = orc_gemm(0, 0, M, N, K, 1.0, A, K, type, W1, N, type, 0.0, NULL, 0,
                      type, rows, n_rows, cols, n_cols, G, n_threads);
    if (rc == 0)
        rc = orc_gemm(0, 0, M, N, K, 1.0, A, K, type, W2, N, type, 0.0, NULL, 0,
                      type, rows, n_rows, cols, n_cols, U, n_threads);
    if (rc == 0)
        for (int64_t e = 0; e < n_rows * n_cols; ++e)
            Y[e] = orc_silu(scale * G[e]) * (scale * U[e]);
    free(G);
    free(U);
    return rc;
}

/* Transposed interleave for 8-bit weights: Wt (2N x K, row stride K) with
 * row 2n = W1 column n (Gate) and row 2n+1 = W2 column n (Up), from W1, W2
 * (K x N, row stride N).  Same column order as orc_interleave. */
void orc_interleave_t8(const uint8_t *W1, const uint8_t *W2, uint8_t *Wt,
                       int64_t K, int64_t N)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            Wt[(2 * n) * K + k] = W1[k * N + n];
            Wt[(2 * n + 1) * K + k] = W2[k * N + n];
        }
}
