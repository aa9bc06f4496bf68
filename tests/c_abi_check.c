/*
 * c_abi_check.c — the C ABI used from plain C: device memory from cudaMalloc,
 * no Python and no torch.  Calls gemm (CTA-pair tiles), gemm_ex with a forced
 * split-K, and swiglu_mlp on the default stream, and checks the results
 * against brute-force host sums.
 *
 * GEMM inputs are small integers, so every product and every partial sum is
 * exact in FP32 accumulation (split or not), and the only rounding is the
 * final one to bf16: the device result must equal the host sum rounded to
 * nearest-even in bf16, bit for bit.  The SwiGLU check compares against
 * SiLU(g) * u in double with the bf16 tolerance 1e-2 + 1e-2 |y|.
 *
 * Build and run (done by tests/test_c_abi_gpu.py):
 *   nvcc -I include tests/c_abi_check.c -o c_abi_check \
 *        -L swiglu_mlp_gb300 -lswiglu_mlp -Xlinker -rpath=<dir of the library>
 * Exit status 0 on success; the first mismatch is printed otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "swiglu_mlp.h"

/* float -> bf16, round to nearest, ties to even (finite values only). */
static uint16_t f2bf(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf2f(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Small integer in [-span, span] from a hash of (i, k, salt). */
static float hval(int64_t i, int64_t k, uint32_t salt, int span)
{
    uint32_t h = (uint32_t)i * 0x9E3779B1u ^ (uint32_t)k * 0x85EBCA77u ^ salt;
    h ^= h >> 15;
    h *= 0x2C1B3C6Du;
    h ^= h >> 12;
    return (float)((int)(h % (uint32_t)(2 * span + 1)) - span);
}

static int check_cuda(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

static int check_swg(int rc, const char *what)
{
    if (rc != SWG_OK) {
        fprintf(stderr, "%s: %s (CUDA error %d: %s)\n", what, swg_status_string(rc),
                swg_last_cuda_error(), swg_cuda_error_name(swg_last_cuda_error()));
        return 1;
    }
    return 0;
}

/* D = A B (bf16 in and out) for M x N x K through gemm_ex with split_k;
 * A in [-4, 4] and B in [-3, 3], hashed integers. */
static int gemm_case(int64_t M, int64_t N, int64_t K, int split_k)
{
    const size_t na = (size_t)M * K, nb = (size_t)K * N, nd = (size_t)M * N;
    uint16_t *ha = malloc(na * 2), *hb = malloc(nb * 2), *hd = malloc(nd * 2);
    float *fa = malloc(na * 4), *fb = malloc(nb * 4);
    int bad = 0;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) {
            fa[i * K + k] = hval(i, k, 1u, 4);
            ha[i * K + k] = f2bf(fa[i * K + k]);
        }
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j) {
            fb[k * N + j] = hval(k, j, 2u, 3);
            hb[k * N + j] = f2bf(fb[k * N + j]);
        }
    void *da = NULL, *db = NULL, *dd = NULL;
    bad |= check_cuda(cudaMalloc(&da, na * 2), "cudaMalloc A");
    bad |= check_cuda(cudaMalloc(&db, nb * 2), "cudaMalloc B");
    bad |= check_cuda(cudaMalloc(&dd, nd * 2), "cudaMalloc D");
    if (!bad) {
        bad |= check_cuda(cudaMemcpy(da, ha, na * 2, cudaMemcpyHostToDevice), "copy A");
        bad |= check_cuda(cudaMemcpy(db, hb, nb * 2, cudaMemcpyHostToDevice), "copy B");
        bad |= check_swg(gemm_ex(SWG_OP_N, SWG_OP_N, M, N, K, 1.0f, da, K, db, N, 0.0f, dd, N,
                                 SWG_BF16, split_k, NULL),
                         "gemm_ex");
        bad |= check_cuda(cudaMemcpy(hd, dd, nd * 2, cudaMemcpyDeviceToHost), "copy D");
        bad |= check_swg(swg_get_device_error(NULL), "device error word");
    }
    for (int64_t i = 0; i < M && !bad; ++i)
        for (int64_t j = 0; j < N && !bad; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += (double)fa[i * K + k] * fb[k * N + j];
            const float got = bf2f(hd[i * N + j]);
            if (hd[i * N + j] != f2bf((float)s)) {
                fprintf(stderr, "gemm %lldx%lldx%lld split %d: D[%lld][%lld] = %g, expected %g\n",
                        (long long)M, (long long)N, (long long)K, split_k, (long long)i,
                        (long long)j, got, s);
                bad = 1;
            }
        }
    cudaFree(da);
    cudaFree(db);
    cudaFree(dd);
    free(ha);
    free(hb);
    free(hd);
    free(fa);
    free(fb);
    return bad;
}

/* Y = SiLU(A W1) * (A W2) through the interleaved weight; A in
 * {-1/4, 0, 1/4}, W1 and W2 multiples of 1/32 in [-1/8, 1/8] (exact in
 * bf16). */
static int swiglu_case(int64_t M, int64_t N, int64_t K)
{
    const size_t na = (size_t)M * K, nw = (size_t)K * 2 * N, ny = (size_t)M * N;
    uint16_t *ha = malloc(na * 2), *hw = malloc(nw * 2), *hy = malloc(ny * 2);
    int bad = 0;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) ha[i * K + k] = f2bf(hval(i, k, 3u, 1) / 4.0f);
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            hw[k * 2 * N + 2 * n] = f2bf(hval(k, n, 4u, 4) / 32.0f);
            hw[k * 2 * N + 2 * n + 1] = f2bf(hval(k, n, 5u, 4) / 32.0f);
        }
    void *da = NULL, *dw = NULL, *dy = NULL;
    bad |= check_cuda(cudaMalloc(&da, na * 2), "cudaMalloc A");
    bad |= check_cuda(cudaMalloc(&dw, nw * 2), "cudaMalloc W_fused");
    bad |= check_cuda(cudaMalloc(&dy, ny * 2), "cudaMalloc Y");
    if (!bad) {
        bad |= check_cuda(cudaMemcpy(da, ha, na * 2, cudaMemcpyHostToDevice), "copy A");
        bad |= check_cuda(cudaMemcpy(dw, hw, nw * 2, cudaMemcpyHostToDevice), "copy W");
        bad |= check_swg(swiglu_mlp(da, dw, dy, M, N, K, NULL), "swiglu_mlp");
        bad |= check_cuda(cudaMemcpy(hy, dy, ny * 2, cudaMemcpyDeviceToHost), "copy Y");
        bad |= check_swg(swg_get_device_error(NULL), "device error word");
    }
    for (int64_t i = 0; i < M && !bad; ++i)
        for (int64_t n = 0; n < N && !bad; ++n) {
            double g = 0.0, u = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = bf2f(ha[i * K + k]);
                g += a * bf2f(hw[k * 2 * N + 2 * n]);
                u += a * bf2f(hw[k * 2 * N + 2 * n + 1]);
            }
            const double want = g / (1.0 + exp(-g)) * u;
            const double got = bf2f(hy[i * N + n]);
            if (fabs(got - want) > 1e-2 + 1e-2 * fabs(want)) {
                fprintf(stderr, "swiglu: Y[%lld][%lld] = %g, expected %g\n", (long long)i,
                        (long long)n, got, want);
                bad = 1;
            }
        }
    cudaFree(da);
    cudaFree(dw);
    cudaFree(dy);
    free(ha);
    free(hw);
    free(hy);
    return bad;
}

int main(void)
{
    int bad = 0;
    bad |= gemm_case(512, 768, 320, 0);     /* CTA-pair tiles */
    bad |= gemm_case(48, 600, 1000, 3);     /* few rows, forced split-K */
    bad |= swiglu_case(300, 520, 136);      /* ragged SwiGLU */
    swg_shutdown();
    if (!bad) printf("c_abi_check: ok (%llu launches)\n", (unsigned long long)swg_launch_count());
    return bad;
}
