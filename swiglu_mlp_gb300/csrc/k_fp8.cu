// k_fp8.cu — instantiations of the tcgen05 GEMM with 8-bit (e4m3) operands
// and kind::f8f6f4 MMAs: the plain GEMM epilogue, the interleaved SwiGLU
// epilogue, and the swapped-operand split-K partials for few rows (decode).
// Per-tensor dequantisation scales arrive folded into alpha.
// Quantised operands with a scale: "GEMM o Coração Matemático", §12.4 (the
// 8-bit layout itself is the OCP E4M3 format, which the pages do not
// define); the SwiGLU page
// ("Sobreposição de Ativação ...", Definição do Problema) notes that FP8 /
// INT4 raise the relative cost of the memory-bound activation step.
#include "launch_impl.cuh"

namespace swg {
cudaError_t launch_tc_store_fp8(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                                const TileParams &p, int units, cudaStream_t s,
                                const CUtensorMap *tout)
{
    if (pair) {
        switch (bn) {
        case 256: return launch_tc_impl<256, EPI_STORE, true, true>(ta, tb, p, units, s, tout);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 128: return launch_tc_impl<128, EPI_STORE, false, true>(ta, tb, p, units, s, tout);
    case 256: return launch_tc_impl<256, EPI_STORE, false, true>(ta, tb, p, units, s, tout);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tc_swiglu_fp8(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                                 const TileParams &p, int units, cudaStream_t s,
                                 const CUtensorMap *tout)
{
    if (pair) {
        switch (bn) {
        case 256: return launch_tc_impl<256, EPI_SWIGLU, true, true>(ta, tb, p, units, s, tout);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 64: return launch_tc_impl<64, EPI_SWIGLU, false, true>(ta, tb, p, units, s, tout);
    case 128: return launch_tc_impl<128, EPI_SWIGLU, false, true>(ta, tb, p, units, s, tout);
    case 256: return launch_tc_impl<256, EPI_SWIGLU, false, true>(ta, tb, p, units, s, tout);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tc_splitk_t_fp8(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                                   const TileParams &p, int units, cudaStream_t s)
{
    switch (bn) {
    case 16: return launch_tc_impl<16, EPI_SPLITK_T, false, true>(ta, tb, p, units, s);
    case 32: return launch_tc_impl<32, EPI_SPLITK_T, false, true>(ta, tb, p, units, s);
    case 64: return launch_tc_impl<64, EPI_SPLITK_T, false, true>(ta, tb, p, units, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tc_splitk_cl_fp8(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                                    const TileParams &p, int ctas, cudaStream_t s)
{
    switch (bn) {
    case 16: return launch_tc_impl<16, EPI_SPLITK_CL, false, true>(ta, tb, p, ctas, s);
    case 32: return launch_tc_impl<32, EPI_SPLITK_CL, false, true>(ta, tb, p, ctas, s);
    case 64: return launch_tc_impl<64, EPI_SPLITK_CL, false, true>(ta, tb, p, ctas, s);
    default: return cudaErrorInvalidValue;
    }
}

int max_active_clusters_splitk_cl_fp8(int bn, int csize, int sms)
{
    switch (bn) {
    case 16: return max_active_clusters_impl<16, EPI_SPLITK_CL, true>(sms, csize);
    case 32: return max_active_clusters_impl<32, EPI_SPLITK_CL, true>(sms, csize);
    case 64: return max_active_clusters_impl<64, EPI_SPLITK_CL, true>(sms, csize);
    default: return 0;
    }
}

int max_active_pairs_fp8(int kind, int bn, int sms)
{
    if (bn != 256) return 0;
    return kind == 0 ? max_active_pairs_impl<256, EPI_STORE, true>(sms)
                     : max_active_pairs_impl<256, EPI_SWIGLU, true>(sms);
}
}  // namespace swg
