// k_swiglu.cu — instantiations of the tcgen05 GEMM with the SwiGLU
// pair-multiply epilogue over the interleaved weight ("Sobreposição de
// Ativação em Nível de Tile para Inferência Eficiente de LLM", Metodologia,
// Kernel-2).
#include "launch_impl.cuh"

namespace swg {
cudaError_t launch_tc_swiglu(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                             const TileParams &p, int units, cudaStream_t s)
{
    if (pair) {
        switch (bn) {
        case 128: return launch_tc_impl<128, EPI_SWIGLU, true>(ta, tb, p, units, s);
        case 256: return launch_tc_impl<256, EPI_SWIGLU, true>(ta, tb, p, units, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 64: return launch_tc_impl<64, EPI_SWIGLU, false>(ta, tb, p, units, s);
    case 128: return launch_tc_impl<128, EPI_SWIGLU, false>(ta, tb, p, units, s);
    case 256: return launch_tc_impl<256, EPI_SWIGLU, false>(ta, tb, p, units, s);
    default: return cudaErrorInvalidValue;
    }
}

int max_active_pairs_swiglu(int bn, int sms)
{
    switch (bn) {
    case 128: return max_active_pairs_impl<128, EPI_SWIGLU>(sms);
    case 256: return max_active_pairs_impl<256, EPI_SWIGLU>(sms);
    default: return 0;
    }
}
}  // namespace swg
