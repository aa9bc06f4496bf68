// launch_impl.cuh — launch helper shared by the kernel translation units.
#pragma once

#include <atomic>

#include "launch.h"

namespace swg {

// Opts the kernel into its dynamic shared memory once per device and
// launches it.  `units` is the number of CTAs (1-CTA mode) or of CTA pairs
// (PAIR: launched as clusters of two).
template <int BN, int EPI, bool PAIR, bool FP8 = false>
cudaError_t launch_tc_impl(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tx,
                           const TileParams &p, int units, cudaStream_t s)
{
    using C = Cfg<BN, PAIR, EPI>;
    static DeviceOnce configured;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto kernel = tc_gemm_kernel<BN, EPI, PAIR, FP8>;
    if (configured.needed(dev)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.mark(dev);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    // Programmatic stream serialisation: this grid may be scheduled once the
    // kernel before it on the stream has triggered its dependents; it waits
    // for that kernel's completion (griddepcontrol.wait) after its set-up.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (PAIR) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        cfg.gridDim = dim3(2 * units);
    } else if (ClusterK<EPI>::value && p.splits > 1) {
        // one cluster of p.splits CTAs per tile; `units` = tiles x splits CTAs
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = p.splits;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        cfg.gridDim = dim3(units);
    } else {
        cfg.gridDim = dim3(units);
    }
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, tx, p);
}

// Kernels with one B operand: the third map slot carries the output map of
// the staged last-tile stores (p.tma_store), or B again when there is none.
template <int BN, int EPI, bool PAIR, bool FP8 = false>
cudaError_t launch_tc_impl(const CUtensorMap &ta, const CUtensorMap &tb, const TileParams &p,
                           int units, cudaStream_t s, const CUtensorMap *tout = nullptr)
{
    return launch_tc_impl<BN, EPI, PAIR, FP8>(ta, tb, tout ? *tout : tb, p, units, s);
}

// How many CTA pairs of this kernel can be resident at once (clusters of two
// need two free SMs in one GPC); 0 on error.
template <int BN, int EPI, bool FP8 = false>
int max_active_pairs_impl(int sms)
{
    using C = Cfg<BN, true, EPI>;
    auto kernel = tc_gemm_kernel<BN, EPI, true, FP8>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// How many clusters of `csize` single-CTA instances of this kernel can be
// resident at once (a cluster needs csize free SMs in one GPC); 0 on error.
template <int BN, int EPI, bool FP8 = false>
int max_active_clusters_impl(int sms, int csize)
{
    using C = Cfg<BN, false, EPI>;
    auto kernel = tc_gemm_kernel<BN, EPI, false, FP8>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csize * (sms / csize));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace swg
