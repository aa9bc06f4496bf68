// launch.h — internal interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "tc_gemm.cuh"

namespace swg {

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

// Split-K with swapped operands (the kernel computes the transposed product;
// `bn` 16, 32 or 64 is the width of the original rows it covers).
cudaError_t launch_tc_splitk_t(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                               const TileParams &p, int units, cudaStream_t s);

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

}  // namespace swg
