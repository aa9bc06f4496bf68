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

// Four 16-bit or FP32 outputs of C/D as floats (beta != 0 only).
__device__ __forceinline__ void load_c4(const void *D, long long off, int out_kind, int cnt,
                                        float (&c)[4])
{
    if (cnt == 4 && out_kind == OUT_F32) {
        const float4 v = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(D) + off);
        c[0] = v.x;
        c[1] = v.y;
        c[2] = v.z;
        c[3] = v.w;
    } else if (cnt == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(D) + off);
        const uint32_t cw[2] = {w.x, w.y};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (out_kind == OUT_F16) {
                const __half2 c2 = *reinterpret_cast<const __half2 *>(&cw[h]);
                c[2 * h] = __low2float(c2);
                c[2 * h + 1] = __high2float(c2);
            } else {
                const __nv_bfloat162 c2 = *reinterpret_cast<const __nv_bfloat162 *>(&cw[h]);
                c[2 * h] = __low2float(c2);
                c[2 * h + 1] = __high2float(c2);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = j < cnt ? load_out(D, off + j, out_kind) : 0.0f;
    }
}

// Each thread owns Q groups of four outputs per round (i, i + stride, ..,
// i + (Q-1) stride) and issues every load of the round -- the S_MAX >=
// splits partials and, with beta != 0, C -- before the first add, so one
// memory round trip covers the round.
template <int S_MAX, int Q>
__global__ void __launch_bounds__(256, 2)
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
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i0 = blockIdx.x * (long long)blockDim.x + threadIdx.x; i0 < total;
         i0 += stride * Q) {
        float4 v[Q][S_MAX];
        float c[Q][4];
        long long off[Q];
        int cnt[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const long long i = i0 + q * stride;
            cnt[q] = 0;
            off[q] = 0;
            if (i >= total) continue;
            const int m = (int)(i / quads);
            const int n = (int)(i - (long long)m * quads) * 4;
            cnt[q] = (N - n) < 4 ? (N - n) : 4;
            off[q] = (long long)m * ldd + n;
            const float *src = ws + (long long)m * ld_ws + n;
            if (cnt[q] == 4) {
#pragma unroll
                for (int sp = 0; sp < S_MAX; ++sp)
                    if (sp < splits)
                        v[q][sp] = __ldcg(reinterpret_cast<const float4 *>(src + sp * split_stride));
            } else {
#pragma unroll
                for (int sp = 0; sp < S_MAX; ++sp) {
                    if (sp < splits) {
                        const float *sq = src + sp * split_stride;
                        v[q][sp] = make_float4(__ldcg(sq), cnt[q] > 1 ? __ldcg(sq + 1) : 0.0f,
                                               cnt[q] > 2 ? __ldcg(sq + 2) : 0.0f, 0.0f);
                    }
                }
            }
            if (beta != 0.0f) load_c4(D, off[q], out_kind, cnt[q], c[q]);
        }
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            if (cnt[q] == 0) continue;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int sp = 0; sp < S_MAX; ++sp) {
                if (sp < splits) {
                    acc[0] += v[q][sp].x;
                    acc[1] += v[q][sp].y;
                    acc[2] += v[q][sp].z;
                    acc[3] += v[q][sp].w;
                }
            }
            float out[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                out[j] = alpha * acc[j];
                if (beta != 0.0f) out[j] += beta * c[q][j];
            }
            if (cnt[q] == 4 && out_kind != OUT_F32) {
                *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(D) + off[q]) =
                    make_uint2(pack2(out[0], out[1], out_kind), pack2(out[2], out[3], out_kind));
            } else if (cnt[q] == 4) {
                *reinterpret_cast<float4 *>(reinterpret_cast<float *>(D) + off[q]) =
                    make_float4(out[0], out[1], out[2], out[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (j < cnt[q]) store_out(D, off[q] + j, out[j], out_kind);
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
    // Up to eight float4 partial loads in flight per thread (Q = 8 / S_MAX
    // groups per round), two CTAs per SM; the grid as before: one group per
    // thread up to four CTAs per SM, so a thread's groups fit in one round.
    const int smax = p.splits <= 2 ? 2 : p.splits <= 4 ? 4 : p.splits <= 8 ? 8 : 16;
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
    auto kernel = smax == 2   ? splitk_reduce_kernel<2, 4>
                  : smax == 4 ? splitk_reduce_kernel<4, 2>
                  : smax == 8 ? splitk_reduce_kernel<8, 1>
                              : splitk_reduce_kernel<16, 1>;
    return cudaLaunchKernelEx(&cfg, kernel, (const float *)p.ws, p.ld_ws, p.splits, p.M, p.N,
                              p.alpha, p.beta, p.D, p.ldd, p.out_kind);
}

}  // namespace swg
