/*
 * swiglu_mlp.h — C ABI of the GB300 (sm_103a) GEMM and fused-SwiGLU library.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Matrices are ROW-MAJOR: element (i, j) of a matrix with row stride ld
 *   sits at offset i*ld + j ("GEMM o Coração Matemático", §2, row-major
 *   linearisation).  ld counts elements, not bytes.
 * - op(X) is X (SWG_OP_N) or its transpose (SWG_OP_T) of the STORED row-major
 *   matrix ("GEMM o Coração Matemático", §1: reading a matrix as transposed
 *   needs no copy).
 * - All pointers except alpha/beta scalars are DEVICE pointers on the current
 *   CUDA device.  The caller owns every tensor; the library never frees them.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Calls are asynchronous: SWG_OK means the work was validated and enqueued.
 * - Every argument is validated BEFORE any CUDA call; a rejected call writes
 *   nothing and launches nothing.
 * - Accumulation is always FP32, in tensor memory; outputs are rounded once,
 *   round-to-nearest-even, at the store.
 * - There is no CPU fallback: an unsupported case returns an error.
 * - Device-side waits are bounded: a kernel that cannot make progress within
 *   about two seconds stops, records SWG_ERR_DEVICE_TIMEOUT in a device error
 *   word, and exits; read it with swg_get_device_error().
 */
#ifndef SWIGLU_MLP_H
#define SWIGLU_MLP_H

#include <stdint.h>

/* Exported with default visibility even when the library is built with
 * -fvisibility=hidden. */
#if defined(__GNUC__)
#define SWG_API __attribute__((visibility("default")))
#else
#define SWG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SWG_OK = 0,
    SWG_ERR_INVALID_ARG = 1,    /* negative size, null pointer, ld too small, bad enum */
    SWG_ERR_MISALIGNED = 2,     /* a pointer or row stride breaks the 16-byte rule */
    SWG_ERR_UNSUPPORTED = 3,    /* valid request this library does not implement */
    SWG_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
    SWG_ERR_NO_MEMORY = 5,      /* library workspace allocation failed */
    SWG_ERR_DEVICE_TIMEOUT = 6  /* a kernel gave up on a bounded wait */
} swg_status;

typedef enum { SWG_OP_N = 0, SWG_OP_T = 1 } swg_op;

/* Storage types.  A and B share one input type; C and D share one output type.
 * The e4m3 types quantise A and B to 8 bits, with per-tensor dequantisation
 * scales ("GEMM o Coração Matemático", §12.4: quantised operands with a
 * scale); the scales are applied by folding them into alpha
 * (alpha * scale_A * scale_B).  The 8-bit layout is E4M3 of the OCP 8-bit
 * floating-point format (as torch's float8_e4m3fn): 1 sign, 4 exponent bits
 * with bias 7, 3 fraction bits, no infinities, largest finite value 448.  They require
 * op(A) = A and op(B) = B^T, i.e. A stored M x K and B stored N x K (both
 * K-contiguous), and lda and ldb multiples of 16.  Split-K exists for them
 * only with M <= 64 (few rows, e.g. decode): such calls run the transposed
 * product with the K loop split, automatically or with split_k > 1, and
 * reduce the partials in split order (one or two rows with split_k = 0 run
 * the one-launch FP32-pipe kernel described under gemm); split_k > 1 with
 * M > 64 and other op combinations return SWG_ERR_UNSUPPORTED. */
typedef enum {
    SWG_F16_F32OUT = 0,   /* A, B binary16;  C, D binary32 */
    SWG_BF16 = 1,         /* A, B, C, D bfloat16            */
    SWG_F16 = 2,          /* A, B, C, D binary16            */
    SWG_BF16_F32OUT = 3,  /* A, B bfloat16;  C, D binary32  */
    SWG_E4M3_BF16OUT = 4, /* A, B e4m3;      C, D bfloat16  */
    SWG_E4M3_F32OUT = 5   /* A, B e4m3;      C, D binary32  */
} swg_dtype;

/*
 * gemm — D = alpha * op(A) * op(B) + beta * C, written in place over C.
 *
 * Defined by "GEMM o Coração Matemático", §1 (the BLAS GEMM statement, element
 * by element: D_ij = alpha * sum_p op(A)_ip op(B)_pj + beta * C_ij) and by
 * "为什么 GEMM 是 CUDA 的必修课" (the opening definition C = A B with 2K flops
 * per element).
 *
 *   transA, transB  SWG_OP_N or SWG_OP_T.
 *   M, N, K         op(A) is M x K, op(B) is K x N, C/D is M x N.  All >= 0.
 *                   M == 0 or N == 0: nothing to do, returns SWG_OK.
 *                   K == 0: D = beta * C (D = 0 when beta == 0).
 *   alpha, beta     host scalars.  When beta == 0, C is NOT read (so NaN or
 *                   garbage in C does not reach D).
 *   A, lda          stored M x K (op N) or K x M (op T); lda >= stored columns.
 *   B, ldb          stored K x N (op N) or N x K (op T); ldb >= stored columns.
 *   C, ldc          M x N, ldc >= N; read (when beta != 0) and overwritten.
 *   dtype           a swg_dtype.
 *   Alignment       A, B, C must be 16-byte aligned and lda, ldb, ldc times
 *                   the element size must be multiples of 16 bytes (tensor
 *                   memory accelerator rule); otherwise SWG_ERR_MISALIGNED.
 *   Sizes           M, N, K, lda, ldb, ldc <= 2^31 - 1, else SWG_ERR_UNSUPPORTED.
 *   Aliasing        A or B overlapping C is undefined.
 *   Split-K         chosen automatically when the output has too few tiles to
 *                   fill the GPU ("为什么 GEMM 是 CUDA 的必修课", 关键技术 item 5);
 *                   the partial sums are reduced in a fixed order, so repeated
 *                   calls give bit-identical results.
 *                   Few rows (M <= 64) with an automatic split: the K ranges
 *                   of each output tile run as one thread-block cluster of up
 *                   to 4 CTAs that sum their FP32 partials through shared
 *                   memory, in range order -- one kernel, no workspace --
 *                   when that occupies at least half of the SMs or splits K
 *                   as often as the workspace path would.  More rows with an
 *                   automatic split: the same over 128 x 256 tiles (2 or 4
 *                   ranks per tile) when all their clusters are resident at
 *                   once and fill at least half of the SMs.
 *                   SWG_CLUSTER_SPLITK=0 turns both off.
 *                   Otherwise the FP32 partials live
 *                   in a library-owned workspace, allocated (cudaMalloc) on
 *                   first use per (device, stream) and replaced by a larger
 *                   one when a larger split needs it; replaced workspaces stay
 *                   allocated (queued work or a captured graph may still use
 *                   them) until swg_shutdown() frees them all.  Two kernels are
 *                   launched: the GEMM and a dependent reduction.
 *   One or two rows M <= 2 with 16-bit or e4m3 A and B (decode of one or two
 *                   tokens), K <= 8 * 8192 / M and N <= 2^30: one kernel on the FP32 pipes
 *                   instead ("GEMM o Coração Matemático", §14: the product
 *                   streams op(B) once and is bound by memory).  Its K split
 *                   is summed inside the kernel, again in a fixed order; it
 *                   uses no workspace.  Setting the environment variable
 *                   SWG_GEMV=0 sends these calls to the tensor-core path.
 *   Graph capture   every call can be captured into a CUDA graph on a stream
 *                   once the same call (or one needing at least as much
 *                   workspace) has run on that stream; a call that would have
 *                   to allocate while its stream is capturing returns
 *                   SWG_ERR_UNSUPPORTED and launches nothing.  Calls of the
 *                   one-or-two-rows kernel and of the cluster-reduced split
 *                   need no earlier run.
 */
SWG_API int gemm(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
         const void *A, int64_t lda, const void *B, int64_t ldb, float beta,
         void *C, int64_t ldc, int dtype, void *stream);

/*
 * gemm_ex — gemm with an explicit split-K factor.
 *   split_k == 0  automatic choice (what gemm does, including the kernel for
 *                 one or two rows);
 *   split_k == 1  no split;
 *   split_k >= 2  split the K loop into at most min(split_k, 16) contiguous
 *                 ranges (fewer when K has fewer 64-wide blocks).
 * Every other argument and rule is that of gemm.
 */
SWG_API int gemm_ex(int transA, int transB, int64_t M, int64_t N, int64_t K,
            float alpha, const void *A, int64_t lda, const void *B,
            int64_t ldb, float beta, void *C, int64_t ldc, int dtype,
            int split_k, void *stream);

/*
 * swiglu_mlp — Y = SiLU(A * W1) (.) (A * W2) as ONE GEMM over the interleaved
 * weight W_fused, with SiLU(x) = x / (1 + e^-x).
 *
 * Defined by "Sobreposição de Ativação em Nível de Tile para Inferência
 * Eficiente de LLM": Definição do Problema (the SwiGLU MLP) and Metodologia,
 * Kernel-2 (one GEMM over W_fused in R^{K x 2N} whose even columns are Gate
 * and odd columns Up; the epilogue reads each column pair of the accumulator
 * and stores SiLU(gate) * up).  Gate and Up stay in tensor memory and
 * registers; neither is written to global memory.
 *
 *   A        bfloat16, M x K, row stride K.
 *   W_fused  bfloat16, K x 2N, row stride 2N: W_fused[k][2n] = W1[k][n],
 *            W_fused[k][2n+1] = W2[k][n] (see swiglu_interleave).
 *   Y        bfloat16, M x N, row stride N (written).
 *   Alignment  all three pointers 16-byte aligned, K % 8 == 0 and
 *            N % 8 == 0; otherwise SWG_ERR_MISALIGNED.
 *   M == 0 or N == 0: nothing to do.  K == 0: Y = SiLU(0) * 0 = 0.
 *   One or two rows (M <= 2, decode; K <= 8 * 8192 / M): one kernel on the
 *            FP32 pipes streams W_fused once and forms SiLU(gate) * up per
 *            column pair in its final, fixed-order reduction (the gemm
 *            kernel for one or two rows); SWG_GEMV=0 keeps the tensor-core
 *            tiles.
 *   At most 64 rows (decode of a few sequences): one 128 x 128 tile per
 *            128 columns of the 2N-space, its K range split over a
 *            thread-block cluster of up to 4 CTAs whose Gate and Up partials
 *            (first M rows) are summed through shared memory, in range
 *            order, before the pair-multiply (one kernel, no workspace), when
 *            the tiles leave at least half of the SMs free
 *            ("为什么 GEMM 是 CUDA 的必修课", 关键技术 item 5); otherwise, and
 *            with SWG_CLUSTER_SPLITK=0, the persistent tiles.
 */
SWG_API int swiglu_mlp(const void *A, const void *W_fused, void *Y, int64_t M,
               int64_t N, int64_t K, void *stream);

/*
 * swiglu_mlp_fp8 — Y = SiLU(s * A W1) (.) (s * A W2) with e4m3 A and weights,
 * s = scale_A * scale_W (per-tensor dequantisation scales), FP32
 * accumulation, bfloat16 Y.  Same operation and sources as swiglu_mlp; the
 * 8-bit form follows "GEMM o Coração Matemático", §12.4 (quantised operands
 * with a scale); the 8-bit layout is the OCP E4M3 format described at
 * swg_dtype.
 *
 *   A          e4m3, M x K, row stride K.
 *   W_fused_t  e4m3, 2N x K, row stride K: the TRANSPOSED interleaved weight,
 *              row 2n = W1 column n (Gate), row 2n+1 = W2 column n (Up)
 *              (8-bit operands are read K-contiguous).
 *   Y          bfloat16, M x N, row stride N (written).
 *   scale      s above; applied to Gate and Up before the SiLU.
 *   Alignment  pointers 16-byte aligned, K % 16 == 0, N % 8 == 0.
 *   One or two rows (M <= 2): the same one-kernel path as swiglu_mlp, reading
 *              W_fused_t in 256 x 64 byte boxes.
 */
SWG_API int swiglu_mlp_fp8(const void *A, const void *W_fused_t, void *Y,
                           int64_t M, int64_t N, int64_t K, float scale,
                           void *stream);

/*
 * swiglu_mlp_dual — the same Y = SiLU(A * W1) (.) (A * W2), computed directly
 * from SEPARATE W1 and W2 with no interleaved copy of the weights.
 *
 * Defined by "Sobreposição de Ativação em Nível de Tile para Inferência
 * Eficiente de LLM", Metodologia, Kernel-1 (Gate and Up from their own weight
 * matrices, SiLU on the Gate accumulator, the product formed in the
 * epilogue).  One kernel: each output tile's accumulator holds the Gate
 * columns in its first half and the matching Up columns in its second half,
 * and the epilogue stores SiLU(gate) * up; neither reaches memory.
 *
 *   A       bfloat16, M x K, row stride K.
 *   W1, W2  bfloat16, each K x N, row stride N.
 *   Y       bfloat16, M x N, row stride N (written).
 *   Alignment, sizes and the K == 0 case as for swiglu_mlp.
 *   One or two rows (M <= 2): the one-kernel path of swiglu_mlp, reading 64
 *           columns of W1 beside the same 64 columns of W2 per stage.
 */
SWG_API int swiglu_mlp_dual(const void *A, const void *W1, const void *W2,
                            void *Y, int64_t M, int64_t N, int64_t K,
                            void *stream);

/*
 * swiglu_mlp_forward — the whole gated MLP of a transformer block:
 *     Out = (SiLU(A * W1) (.) (A * W2)) * W_down + beta * Out
 * "GEMM o Coração Matemático", §13.3 (the feed-forward block as two GEMMs
 * around an activation) with the gated activation of "Sobreposição de
 * Ativação em Nível de Tile para Inferência Eficiente de LLM", Definição do
 * Problema.  beta = 1 adds a residual already held in Out.
 *
 *   A        bfloat16, M x K, row stride K (K = model width).
 *   W_fused  bfloat16, K x 2N, row stride 2N (interleaved Gate/Up, as for
 *            swiglu_mlp).
 *   W_down   bfloat16, N x K, row stride K.
 *   Y        bfloat16, M x N, row stride N: receives the gated activation
 *            (caller-owned; Gate and Up themselves never reach memory).
 *   Out      bfloat16, M x K, row stride K: read when beta != 0, written.
 *   Two kernels run on `stream`: swiglu_mlp's fused kernel, then gemm.
 *   Alignment: pointers 16-byte aligned, K % 8 == 0, N % 8 == 0, else
 *   SWG_ERR_MISALIGNED.  M == 0 or K == 0: nothing to do.  All arguments are
 *   checked before the first launch.
 */
SWG_API int swiglu_mlp_forward(const void *A, const void *W_fused,
                               const void *W_down, void *Y, void *Out,
                               int64_t M, int64_t N, int64_t K, float beta,
                               void *stream);

/*
 * swiglu_interleave — builds W_fused (K x 2N, row stride 2N) from W1 and W2
 * (each K x N, row stride N), bfloat16: column 2n <- W1 column n (Gate),
 * column 2n+1 <- W2 column n (Up).  Same page and section as swiglu_mlp.
 * A one-off weight-layout step, not part of the per-token hot path.
 * Pointers 16-byte aligned and N % 4 == 0, else SWG_ERR_MISALIGNED.
 */
SWG_API int swiglu_interleave(const void *W1, const void *W2, void *W_fused,
                      int64_t K, int64_t N, void *stream);

/*
 * gemm_splitk_noalloc — gemm_ex without any device allocation.  The pages
 * have no counterpart to this call.  It is for callers that cannot call
 * cudaMalloc once they are running: a host framework that has already
 * reserved nearly all device memory in its own pool (where a cudaMalloc
 * would fail, or fragment that pool), or a serving loop that forbids
 * cudaMalloc/cudaFree because either can synchronise the whole device.
 *
 * Same arguments, rules and results as gemm_ex: for every input it launches
 * the kernels gemm_ex would launch, with the same tiles, split count and
 * fixed-order reduction, so the two give bit-identical D.  The one
 * difference: a split-K call that keeps FP32 partial sums in global memory
 * keeps them in a fixed array of SWG_NOALLOC_SCRATCH_BYTES (plus two 64 KiB
 * guard bands) that is part of the library's device image, instead of a
 * workspace from cudaMalloc (few-row calls whose K ranges are reduced inside
 * a thread-block cluster keep none there).  The caller still passes A, B
 * and C.
 *
 *   Limit        a split needs splits * M * round_up(N, 4) * 4 bytes of
 *                partials; a call that would need more than
 *                SWG_NOALLOC_SCRATCH_BYTES returns SWG_ERR_UNSUPPORTED and
 *                launches nothing (pass a smaller split_k, or use gemm_ex).
 *   Allocation   none: no cudaMalloc, cudaFree or allocating library call.
 *   Residency    the array is device memory of the library's module.  With
 *                CUDA's default lazy module loading it is committed on a
 *                device the first time this library runs there (the first
 *                call of any of its entry points), and with
 *                CUDA_MODULE_LOADING=EAGER when the library is loaded; it
 *                stays until the process exits.  A caller about to reserve
 *                nearly all device memory should make one call on each
 *                device first.
 *   First call   on each device looks up the array's device address
 *                (cudaGetSymbolAddress) with that device current; make that
 *                first call before any stream capture.
 *   Sharing      all calls, on every stream, use the one array, and it keeps
 *                the last call's contents (each call writes every partial it
 *                reads, so nothing needs clearing).  Calls that overlap on the
 *                GPU race with each other: order them, e.g. on one stream.
 *   Reset        call swg_shutdown() before cudaDeviceReset(): it makes the
 *                next call look the address up again.
 */
#define SWG_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
SWG_API int gemm_splitk_noalloc(int transA, int transB, int64_t M, int64_t N,
                                int64_t K, float alpha, const void *A,
                                int64_t lda, const void *B, int64_t ldb,
                                float beta, void *C, int64_t ldc, int dtype,
                                int split_k, void *stream);

/*
 * swg_debug_workspace_guards — diagnostic for tests (no counterpart on the
 * pages).  With the environment variable SWG_TEST_WS_GUARD=1 set before a
 * workspace is created, every split-K workspace and the fixed array of
 * gemm_splitk_noalloc sit between 64 KiB guard bands of the byte 0xA5.  This
 * call synchronises `stream` and the current device, then stores in
 * *bad_bytes how many guard bytes of the current device's workspaces have
 * changed (0 when no kernel wrote outside its partials; workspaces made
 * without the variable are skipped).  SWG_ERR_INVALID_ARG for a null
 * bad_bytes, SWG_ERR_CUDA if a copy fails.
 */
SWG_API int swg_debug_workspace_guards(void *stream, int64_t *bad_bytes);

/* Human-readable name of a swg_status value (static string, never NULL). */
SWG_API const char *swg_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns SWG_OK when no kernel reported a problem since the last call,
 * SWG_ERR_DEVICE_TIMEOUT when a bounded wait ran out, SWG_ERR_CUDA when the
 * synchronisation itself failed.
 */
SWG_API int swg_get_device_error(void *stream);

/*
 * swg_selftest_wait_timeout — diagnostic: exercises the bounded-wait path the
 * pipeline kernels use, on purpose.  Launches one small kernel that waits, with
 * the kernels' own wait routine, on a barrier nothing ever completes; after
 * limit_ns (1 ns .. 1 s) it gives up, records SWG_ERR_DEVICE_TIMEOUT in the
 * device error word and exits, leaving the context usable.  The next
 * swg_get_device_error() on that stream returns SWG_ERR_DEVICE_TIMEOUT (and
 * clears it).  No counterpart on the pages: it tests this library's failure
 * reporting without faulting or hanging the GPU.
 */
SWG_API int swg_selftest_wait_timeout(int64_t limit_ns, void *stream);

/* Why the calling thread's most recent call returned SWG_ERR_CUDA: the CUDA
 * runtime error code (cudaError_t), or 10000 + the driver's CUresult when
 * encoding a tensor map failed; 0 if no call of this thread has failed that
 * way.  Thread-local; a later successful call does not clear it. */
SWG_API int swg_last_cuda_error(void);

/* Name of a code returned by swg_last_cuda_error (static storage). */
SWG_API const char *swg_cuda_error_name(int code);

/* Number of kernels this library has launched in this process (all devices). */
SWG_API uint64_t swg_launch_count(void);

/* Frees every library-owned workspace on every device, including replaced
 * ones, and forgets every cached per-device lookup (device addresses,
 * occupancy, kernel attributes), so it is also the call to make before
 * cudaDeviceReset().  Safe to call twice; later calls allocate and look up
 * afresh.  Call only when no library work is in flight and no captured graph
 * that used the workspaces will be replayed. */
SWG_API void swg_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* SWIGLU_MLP_H */
