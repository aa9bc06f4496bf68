// k_splitk.cu — split-K ("为什么 GEMM 是 CUDA 的必修课", 关键技术 item 5: split
// K across CTAs when M and N are too small to fill the GPU, then reduce the
// partial C).
//
// The tcgen05 kernel with EPI_SPLITK writes one FP32 partial per K range to
// the workspace ws[split][M][ld_ws].  splitk_reduce_kernel then forms
//   D[m][n] = alpha * (((p_0 + p_1) + p_2) + ... + p_{S-1}) + beta * C[m][n]
// in that fixed order, so the result is bit-identical from run to run.  It is
// launched with programmatic stream serialisation: its CTAs may be scheduled
// while the GEMM still runs and block in griddepcontrol.wait until the GEMM
// grid has completed and its writes are visible, which hides the launch gap.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch_impl.cuh"

namespace swg {

__global__ void __launch_bounds__(256)
    splitk_reduce_kernel(const float *__restrict__ ws, long long ld_ws, int splits, int M, int N,
                         float alpha, float beta, void *D, long long ldd, int out_kind)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // A GEMM queued behind this reduction may set up meanwhile; it waits for
    // this grid's completion before it touches global memory.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int quads = (N + 3) / 4;
    const long long total = (long long)M * quads;
    const long long split_stride = (long long)M * ld_ws;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i / quads);
        const int n = (int)(i - (long long)m * quads) * 4;
        const int cnt = (N - n) < 4 ? (N - n) : 4;
        const float *src = ws + (long long)m * ld_ws + n;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (cnt == 4) {
            float4 v[MAX_SPLITS];
#pragma unroll
            for (int s = 0; s < MAX_SPLITS; ++s)
                if (s < splits) v[s] = __ldcg(reinterpret_cast<const float4 *>(src + s * split_stride));
#pragma unroll
            for (int s = 0; s < MAX_SPLITS; ++s) {
                if (s < splits) {
                    acc[0] += v[s].x;
                    acc[1] += v[s].y;
                    acc[2] += v[s].z;
                    acc[3] += v[s].w;
                }
            }
        } else {
            for (int s = 0; s < splits; ++s) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (j < cnt) acc[j] += __ldcg(src + s * split_stride + j);
            }
        }
        const long long off = (long long)m * ldd + n;
        float out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) out[j] = alpha * acc[j];
        if (cnt == 4 && out_kind != OUT_F32) {
            // four 16-bit outputs: one 8-byte load of C (beta != 0), one store
            uint2 *dst = reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(D) + off);
            if (beta != 0.0f) {
                const uint2 c = *dst;
                uint32_t cw[2] = {c.x, c.y};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float lo, hi;
                    if (out_kind == OUT_F16) {
                        const __half2 c2 = *reinterpret_cast<const __half2 *>(&cw[h]);
                        lo = __low2float(c2);
                        hi = __high2float(c2);
                    } else {
                        const __nv_bfloat162 c2 = *reinterpret_cast<const __nv_bfloat162 *>(&cw[h]);
                        lo = __low2float(c2);
                        hi = __high2float(c2);
                    }
                    out[2 * h] += beta * lo;
                    out[2 * h + 1] += beta * hi;
                }
            }
            *dst = make_uint2(pack2(out[0], out[1], out_kind), pack2(out[2], out[3], out_kind));
        } else if (cnt == 4) {
            float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(D) + off);
            if (beta != 0.0f) {
                const float4 c = *dst;
                out[0] += beta * c.x;
                out[1] += beta * c.y;
                out[2] += beta * c.z;
                out[3] += beta * c.w;
            }
            *dst = make_float4(out[0], out[1], out[2], out[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < cnt) {
                    float v = out[j];
                    if (beta != 0.0f) v += beta * load_out(D, off + j, out_kind);
                    store_out(D, off + j, v, out_kind);
                }
            }
        }
    }
}

cudaError_t launch_tc_splitk(int bn, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
                             const TileParams &p, int units, cudaStream_t s,
                             const CUtensorMap *tout)
{
    if (pair) {
        switch (bn) {
        case 128: return launch_tc_impl<128, EPI_SPLITK, true>(ta, tb, p, units, s, tout);
        case 256: return launch_tc_impl<256, EPI_SPLITK, true>(ta, tb, p, units, s, tout);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 128: return launch_tc_impl<128, EPI_SPLITK, false>(ta, tb, p, units, s, tout);
    case 256: return launch_tc_impl<256, EPI_SPLITK, false>(ta, tb, p, units, s, tout);
    default: return cudaErrorInvalidValue;
    }
}

int max_active_pairs_splitk(int bn, int sms)
{
    switch (bn) {
    case 128: return max_active_pairs_impl<128, EPI_SPLITK>(sms);
    case 256: return max_active_pairs_impl<256, EPI_SPLITK>(sms);
    default: return 0;
    }
}

cudaError_t launch_tc_splitk_t(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                               const TileParams &p, int grid, cudaStream_t s)
{
    switch (bn) {
    case 16: return launch_tc_impl<16, EPI_SPLITK_T, false>(ta, tb, p, grid, s);
    case 32: return launch_tc_impl<32, EPI_SPLITK_T, false>(ta, tb, p, grid, s);
    case 64: return launch_tc_impl<64, EPI_SPLITK_T, false>(ta, tb, p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tc_splitk_cl(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                                const TileParams &p, int ctas, cudaStream_t s)
{
    switch (bn) {
    case 16: return launch_tc_impl<16, EPI_SPLITK_CL, false>(ta, tb, p, ctas, s);
    case 32: return launch_tc_impl<32, EPI_SPLITK_CL, false>(ta, tb, p, ctas, s);
    case 64: return launch_tc_impl<64, EPI_SPLITK_CL, false>(ta, tb, p, ctas, s);
    default: return cudaErrorInvalidValue;
    }
}

int max_active_clusters_splitk_cl(int bn, int csize, int sms)
{
    switch (bn) {
    case 16: return max_active_clusters_impl<16, EPI_SPLITK_CL>(sms, csize);
    case 32: return max_active_clusters_impl<32, EPI_SPLITK_CL>(sms, csize);
    case 64: return max_active_clusters_impl<64, EPI_SPLITK_CL>(sms, csize);
    default: return 0;
    }
}

cudaError_t launch_splitk_reduce(const TileParams &p, int sms, cudaStream_t s)
{
    const long long items = (long long)p.M * ((p.N + 3) / 4);
    long long blocks = (items + 255) / 256;
    const long long cap = (long long)sms * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, (const float *)p.ws, p.ld_ws, p.splits,
                              p.M, p.N, p.alpha, p.beta, p.D, p.ldd, p.out_kind);
}

}  // namespace swg
