// k_store.cu — instantiations of the tcgen05 GEMM with the alpha/beta/cast
// epilogue (D = alpha * acc + beta * C, "GEMM o Coração Matemático", §1).
#include "launch_impl.cuh"

namespace swg {
cudaError_t launch_tc_store(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                            const TileParams &p, int units, cudaStream_t s,
                            const CUtensorMap *tout)
{
    if (pair) {
        switch (bn) {
        case 128: return launch_tc_impl<128, EPI_STORE, true>(ta, tb, p, units, s, tout);
        case 256: return launch_tc_impl<256, EPI_STORE, true>(ta, tb, p, units, s, tout);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 64: return launch_tc_impl<64, EPI_STORE, false>(ta, tb, p, units, s, tout);
    case 128: return launch_tc_impl<128, EPI_STORE, false>(ta, tb, p, units, s, tout);
    case 256: return launch_tc_impl<256, EPI_STORE, false>(ta, tb, p, units, s, tout);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tc_store_cl(const CUtensorMap &ta, const CUtensorMap &tb, const TileParams &p,
                               int ctas, cudaStream_t s)
{
    return launch_tc_impl<256, EPI_STORE_CL, false>(ta, tb, p, ctas, s);
}

int max_active_clusters_store_cl(int csize, int sms)
{
    return max_active_clusters_impl<256, EPI_STORE_CL>(sms, csize);
}

int max_active_pairs_store(int bn, int sms)
{
    switch (bn) {
    case 128: return max_active_pairs_impl<128, EPI_STORE>(sms);
    case 256: return max_active_pairs_impl<256, EPI_STORE>(sms);
    default: return 0;
    }
}
}  // namespace swg
