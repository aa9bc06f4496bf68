// launch.h — internal interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "tc_gemm.cuh"

namespace swg {

// Launch set-up done once per kernel and device (the dynamic shared-memory
// opt-in).  swg_shutdown advances g_setup_epoch, so set-up cached before it is
// done again on the next launch -- after a cudaDeviceReset, which clears
// function attributes, it has to be.
extern std::atomic<unsigned> g_setup_epoch;

struct DeviceOnce {
    static constexpr int kDevices = 64;
    std::atomic<unsigned> done[kDevices] = {};      // epoch + 1 of the last set-up
    bool needed(int dev) const
    {
        return dev < 0 || dev >= kDevices || done[dev].load() != g_setup_epoch.load() + 1u;
    }
    void mark(int dev)
    {
        if (dev >= 0 && dev < kDevices) done[dev].store(g_setup_epoch.load() + 1u);
    }
};

// Launch the persistent tcgen05 kernel with the given epilogue.  `bn` is one
// of the tile widths the TU instantiates (anything else returns
// cudaErrorInvalidValue without launching); `pair` selects the CTA-pair
// (cta_group::2, 256-row tile) variant, for which `units` counts pairs.
// `tout`: output map of the staged last-tile stores, when p.tma_store is set.
cudaError_t launch_tc_store(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                            const TileParams &p, int units, cudaStream_t s,
                            const CUtensorMap *tout = nullptr);
cudaError_t launch_tc_swiglu(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                             const TileParams &p, int units, cudaStream_t s,
                             const CUtensorMap *tout = nullptr);
cudaError_t launch_tc_splitk(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                             const TileParams &p, int units, cudaStream_t s,
                             const CUtensorMap *tout = nullptr);

// GEMM tiles of 128 x 256 with the K range split over a cluster of p.splits
// (2 or 4) CTAs that reduce through shared memory (EPI_STORE_CL); `ctas` =
// tiles x splits.
cudaError_t launch_tc_store_cl(const CUtensorMap &ta, const CUtensorMap &tb, const TileParams &p,
                               int ctas, cudaStream_t s);
int max_active_clusters_store_cl(int csize, int sms);

// Split-K with swapped operands (the kernel computes the transposed product;
// `bn` 16, 32 or 64 is the width of the original rows it covers).
cudaError_t launch_tc_splitk_t(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                               const TileParams &p, int units, cudaStream_t s);

// The same product with the K ranges of a tile reduced inside a cluster of
// p.splits CTAs (1, 2 or 4; EPI_SPLITK_CL): one launch of `ctas` = tiles x
// splits CTAs, no workspace.  16-bit operands, and e4m3 (both K-major).
cudaError_t launch_tc_splitk_cl(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                                const TileParams &p, int ctas, cudaStream_t s);
cudaError_t launch_tc_splitk_cl_fp8(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                                    const TileParams &p, int ctas, cudaStream_t s);
// Resident clusters of `csize` CTAs of those kernels (0 if unknown).
int max_active_clusters_splitk_cl(int bn, int csize, int sms);
int max_active_clusters_splitk_cl_fp8(int bn, int csize, int sms);

// Fused SwiGLU over W_fused for at most 128 rows with the K ranges of each
// 128 x bn tile (bn = 128) reduced inside a cluster of p.splits CTAs
// (EPI_SWIGLU_CL); `ctas` = tiles x splits.
cudaError_t launch_tc_swiglu_cl(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                                const TileParams &p, int ctas, cudaStream_t s);
int max_active_clusters_swiglu_cl(int bn, int csize, int sms);

// SwiGLU from separate W1 (tw1) and W2 (tw2), each K x N; BN = 128 or 256
// (single CTA) or 256 (pair).
cudaError_t launch_tc_swiglu_dual(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tw1,
                                  const CUtensorMap &tw2, const TileParams &p, int units,
                                  cudaStream_t s);
int max_active_pairs_dual(int bn, int sms);

// 8-bit (e4m3) operands, kind::f8f6f4 MMAs, K-major A and B only.
cudaError_t launch_tc_store_fp8(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                                const TileParams &p, int units, cudaStream_t s,
                                const CUtensorMap *tout = nullptr);
cudaError_t launch_tc_swiglu_fp8(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                                 const TileParams &p, int units, cudaStream_t s,
                                 const CUtensorMap *tout = nullptr);
int max_active_pairs_fp8(int kind, int bn, int sms);   // kind 0 = GEMM, 1 = SwiGLU
// Swapped-operand split-K with e4m3 operands (both K-major), BN = 16, 32, 64.
cudaError_t launch_tc_splitk_t_fp8(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                                   const TileParams &p, int units, cudaStream_t s);

// Resident CTA pairs for the pair variants (0 if unknown or not instantiated).
int max_active_pairs_store(int bn, int sms);
int max_active_pairs_swiglu(int bn, int sms);
int max_active_pairs_splitk(int bn, int sms);

// In-order reduction of the split-K partials into D (alpha, beta, cast),
// launched as a programmatic dependent of the split-K GEMM on the same stream.
cudaError_t launch_splitk_reduce(const TileParams &p, int sms, cudaStream_t s);

// Few-rows product on the FP32 pipes (k_gemv.cu): D = alpha * op(A) op(B) +
// beta * C for M <= 2, one launch; B streams through shared memory by TMA in
// boxes (tensor map tmB: B stored N x K read as {K, N} in boxes of
// gemv_box_inner x gemv_box_outer, or B stored K x N read as {N, K}); the K
// ranges of a block of output columns are reduced inside a cluster.
// in_kind: 0 = binary16, 1 = bfloat16, 2 = e4m3 (B stored N x K only).
struct GemvArgs {
    const void *A;               // op(A) storage (elements of in_kind)
    long long lda;
    int a_t;                     // 1: A stored K x M (op T; 16-bit only)
    void *D;                     // output (also C when beta != 0)
    long long ldd;
    int M, N, K;
    int kr;                      // K elements per range, a multiple of gemv_k_per_stage
    int ranges;                  // K ranges = CTAs per cluster (1..8)
    int stages;                  // shared-memory ring depth (boxes of 16 KB)
    float alpha, beta;
    int out_kind;                // OutKind
    int *err;                    // device error word
    // 1: B is an interleaved SwiGLU weight (columns 2j, 2j + 1 = Gate, Up of
    // output j; N counts both) and D[m][j] = SiLU(alpha g) * (alpha u); no C.
    int swiglu;
};
constexpr int GV_MAX_SMEM = 232448;          // 227 KB, the per-CTA maximum
int gemv_cols_per_block(bool b_kn, int in_kind);   // output columns per cluster
int gemv_k_per_stage(bool b_kn);                   // K elements per box
int gemv_box_inner(bool b_kn);                     // box extent along the contiguous dimension
int gemv_box_outer(bool b_kn, int in_kind);
int gemv_smem_bytes(int mr, bool b_kn, int in_kind, int kr, int stages);
// mr: 1 or 2 (rows the kernel computes; M <= mr); b_kn: B stored K x N
// (op N); col_blocks: cdiv(N, gemv_cols_per_block(b_kn, in_kind)).
// tmB2 non-null: SwiGLU from two bf16 weights stored K x N, tmB = W1 (Gate)
// and tmB2 = W2 (Up), each read in boxes of 64 columns x 64 K rows; g.N is
// the output width and col_blocks = cdiv(N, 64).
cudaError_t launch_gemv(const CUtensorMap &tmB, const CUtensorMap *tmB2, const GemvArgs &g, int mr,
                        bool b_kn, int in_kind, int col_blocks, cudaStream_t s);

}  // namespace swg
