// k_splitk.cu — instantiations of the tcgen05 GEMM with the split-K epilogue
// (FP32 partials, last-arriving CTA reduces them in split order; split-K as in
// "为什么 GEMM 是 CUDA 的必修课", 关键技术 item 5).
#include "launch_impl.cuh"

namespace swg {
cudaError_t launch_tc_splitk(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                             const TileParams &p, int grid, cudaStream_t s)
{
    switch (bn) {
    case 128: return launch_tc_impl<128, EPI_SPLITK>(ta, tb, p, grid, s);
    case 256: return launch_tc_impl<256, EPI_SPLITK>(ta, tb, p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}
}  // namespace swg
