// k_swiglu.cu — instantiations of the tcgen05 GEMM with the SwiGLU
// pair-multiply epilogue over the interleaved weight ("Sobreposição de
// Ativação em Nível de Tile para Inferência Eficiente de LLM", Metodologia,
// Kernel-2).
#include "launch_impl.cuh"

namespace swg {
cudaError_t launch_tc_swiglu(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                             const TileParams &p, int grid, cudaStream_t s)
{
    switch (bn) {
    case 64: return launch_tc_impl<64, EPI_SWIGLU>(ta, tb, p, grid, s);
    case 128: return launch_tc_impl<128, EPI_SWIGLU>(ta, tb, p, grid, s);
    case 256: return launch_tc_impl<256, EPI_SWIGLU>(ta, tb, p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}
}  // namespace swg
