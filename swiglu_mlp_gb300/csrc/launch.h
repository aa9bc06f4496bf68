// launch.h — internal interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "tc_gemm.cuh"

namespace swg {

// Shared-memory bytes the tcgen05 kernel needs for a given BN.
int tc_smem_bytes(int bn);

// Launches the persistent tcgen05 kernel with the given epilogue.  `bn` is one
// of the tile widths the TU instantiates; anything else returns
// cudaErrorInvalidValue without launching.
cudaError_t launch_tc_store(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                            const TileParams &p, int grid, cudaStream_t s);
cudaError_t launch_tc_swiglu(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                             const TileParams &p, int grid, cudaStream_t s);
cudaError_t launch_tc_splitk(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                             const TileParams &p, int grid, cudaStream_t s);

// In-order reduction of the split-K partials into D (alpha, beta, cast),
// launched as a programmatic dependent of the split-K GEMM on the same stream.
cudaError_t launch_splitk_reduce(const TileParams &p, int sms, cudaStream_t s);

}  // namespace swg
