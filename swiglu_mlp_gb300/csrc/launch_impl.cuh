// launch_impl.cuh — launch helper shared by the kernel translation units.
#pragma once

#include <atomic>

#include "launch.h"

namespace swg {

// Opt the kernel into its dynamic shared memory once per device.
template <int BN, int EPI>
cudaError_t launch_tc_impl(const CUtensorMap &ta, const CUtensorMap &tb, const TileParams &p,
                           int grid, cudaStream_t s)
{
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    auto kernel = tc_gemm_kernel<BN, EPI>;
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<BN>::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    kernel<<<grid, NUM_THREADS, Cfg<BN>::SMEM_BYTES, s>>>(ta, tb, p);
    return cudaGetLastError();
}

}  // namespace swg
