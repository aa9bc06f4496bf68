// k_store.cu — instantiations of the tcgen05 GEMM with the alpha/beta/cast
// epilogue (D = alpha * acc + beta * C, "GEMM o Coração Matemático", §1).
#include "launch_impl.cuh"

namespace swg {
cudaError_t launch_tc_store(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                            const TileParams &p, int grid, cudaStream_t s)
{
    switch (bn) {
    case 64: return launch_tc_impl<64, EPI_STORE>(ta, tb, p, grid, s);
    case 128: return launch_tc_impl<128, EPI_STORE>(ta, tb, p, grid, s);
    case 256: return launch_tc_impl<256, EPI_STORE>(ta, tb, p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}
}  // namespace swg
