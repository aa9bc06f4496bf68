// k_swiglu.cu — instantiations of the tcgen05 GEMM with the SwiGLU
// epilogues ("Sobreposição de Ativação em Nível de Tile para Inferência
// Eficiente de LLM", Metodologia): over the interleaved weight (Kernel-2's
// pair-multiply) and over separate W1 and W2 (Kernel-1's separate weights,
// with Gate and Up in two column ranges of one accumulator).
#include "launch_impl.cuh"

namespace swg {
cudaError_t launch_tc_swiglu(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                             const TileParams &p, int units, cudaStream_t s,
                             const CUtensorMap *tout)
{
    if (pair) {
        switch (bn) {
        case 128: return launch_tc_impl<128, EPI_SWIGLU, true>(ta, tb, p, units, s, tout);
        case 256: return launch_tc_impl<256, EPI_SWIGLU, true>(ta, tb, p, units, s, tout);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 64: return launch_tc_impl<64, EPI_SWIGLU, false>(ta, tb, p, units, s, tout);
    case 128: return launch_tc_impl<128, EPI_SWIGLU, false>(ta, tb, p, units, s, tout);
    case 256: return launch_tc_impl<256, EPI_SWIGLU, false>(ta, tb, p, units, s, tout);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tc_swiglu_dual(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tw1,
                                  const CUtensorMap &tw2, const TileParams &p, int units,
                                  cudaStream_t s)
{
    if (pair) {
        switch (bn) {
        case 256: return launch_tc_impl<256, EPI_SWIGLU_DUAL, true>(ta, tw1, tw2, p, units, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 128: return launch_tc_impl<128, EPI_SWIGLU_DUAL, false>(ta, tw1, tw2, p, units, s);
    case 256: return launch_tc_impl<256, EPI_SWIGLU_DUAL, false>(ta, tw1, tw2, p, units, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tc_swiglu_cl(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                                const TileParams &p, int ctas, cudaStream_t s)
{
    if (bn != 128) return cudaErrorInvalidValue;
    return launch_tc_impl<128, EPI_SWIGLU_CL, false>(ta, tb, p, ctas, s);
}

int max_active_clusters_swiglu_cl(int bn, int csize, int sms)
{
    return bn == 128 ? max_active_clusters_impl<128, EPI_SWIGLU_CL>(sms, csize) : 0;
}

int max_active_pairs_dual(int bn, int sms)
{
    return bn == 256 ? max_active_pairs_impl<256, EPI_SWIGLU_DUAL>(sms) : 0;
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
