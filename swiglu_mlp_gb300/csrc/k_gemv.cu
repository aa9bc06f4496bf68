// k_gemv.cu — the few-rows product (one or two rows of op(A): decode of one
// or two tokens) on the FP32 pipes, in one launch per call: GEMM (16-bit or
// e4m3 operands) and the SwiGLU MLP's gate/up product (interleaved W_fused,
// its transposed e4m3 form, or separate W1 and W2) with the pair-multiply
// SiLU(Gate) * Up in the final reduction.
//
// With M <= 2 every weight element is used at most twice, so the call costs
// the time to stream op(B) from HBM once ("GEMM o Coração Matemático", §14:
// about one FLOP per byte at M = 1), and a 128-row tensor-core tile would be
// at least 98% padding.  (With three or four rows the FP32 work per byte no
// longer hides under the stream; those calls stay on the tensor cores.)  The
// K loop is split across CTAs when the output has too few columns to fill the
// GPU ("为什么 GEMM 是 CUDA 的必修课", 关键技术 item 5); here the S K ranges
// of one block of output columns run as ONE thread-block cluster, and CTA 0
// of the cluster sums the S partial blocks, read from the other CTAs' shared
// memory in rank order.  The result is bit-identical from run to run, and
// there is no workspace and no second kernel.
//
// Streaming at HBM speed needs about 150-250 KB in flight per SM (the loaded
// DRAM latency is several microseconds), more than registers can hold, so B
// moves by TMA: warp 0 (one thread) loads 16 KB boxes of B into a ring of
// shared-memory stages, up to 12 of them, and 8 consumer warps compute from
// shared memory.  Boxes past the edges of B read as zero, so ragged N and K
// need no extra code.  Per CTA: one block of output columns, one contiguous K
// range.  The consumers first widen the range's slice of op(A) to FP32 in
// shared memory (zero beyond the M rows and past K) while the first boxes are
// in flight.  By the layout of B:
//   op(B) = B^T (B stored N x K, K contiguous; a linear layer's weight):
//     boxes of 256 K x 32 rows; each consumer warp owns 4 rows (output
//     columns), lane l takes elements 8l..8l+7 of each row, and a shuffle
//     butterfly sums the 32 lanes at the end;
//   op(B) = B (B stored K x N, N contiguous): boxes of 128 columns x 64 K
//     rows (or, from separate W1 and W2, 64 columns of each side by side);
//     16 threads cover the 128 columns (8 each) and 16 row lanes take every
//     16th row; the 2 row lanes of a warp are summed by a shuffle, the 8 warps
//     in shared memory.
//   e4m3 B is read N x K only, in boxes of 256 K x 64 rows (8 rows a warp).
// Every sum runs in a fixed order.  The output is D = alpha * sum + beta * C
// with C read only when beta != 0.  Each wait on a stage barrier is bounded:
// past the limit the CTA records ERR_TIMEOUT in the error word, the producer
// waits (bounded again) for its boxes in flight, and the kernel returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <type_traits>

#include "launch_impl.cuh"

namespace swg {
namespace {

constexpr int GV_CONSUMERS = 256;                   // 8 consumer warps
constexpr int GV_WARPS = GV_CONSUMERS / 32;
constexpr int GV_THREADS = GV_CONSUMERS + 32;       // + the producer warp
constexpr int GV_STAGE_BYTES = 16384;
constexpr int NK_KS = 256;                          // B stored N x K: K elements per box
constexpr int KN_CW = 128;                          // B stored K x N: columns per box
constexpr int KN_KS = 64;                           //   K rows per box
constexpr int KN_RPT = KN_KS / 16;                  //   rows per thread and box (4)

// Input kinds: IK 0 = binary16, 1 = bfloat16, 2 = e4m3 (8-bit).
template <int IK> using Elem = std::conditional_t<IK == 2, uint8_t, uint16_t>;
template <int IK> using Vec8 = std::conditional_t<IK == 2, uint2, uint4>;   // 8 elements
template <int IK> __host__ __device__ constexpr int esize() { return IK == 2 ? 1 : 2; }
// B stored N x K: rows (output columns) per 16 KB box of NK_KS elements each.
__host__ __device__ constexpr int nk_rows(int esz) { return GV_STAGE_BYTES / (NK_KS * esz); }

template <int IK>
__device__ __forceinline__ float widen1(uint32_t bits)
{
    if constexpr (IK == 1) return __uint_as_float(bits << 16);   // bfloat16 = top half of binary32
    if constexpr (IK == 0) return __half2float(__ushort_as_half((unsigned short)bits));
    return __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)bits, __NV_E4M3)));
}

// The eight values of one 8-element load, widened to FP32 (exact: e4m3 and
// binary16 both widen to binary16 without rounding, bfloat16 by a shift).
template <int IK>
__device__ __forceinline__ void widen8(const Vec8<IK> &v, float (&f)[8])
{
    if constexpr (IK == 2) {
        const uint32_t w[2] = {v.x, v.y};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)(w[h >> 1] >> (16 * (h & 1)));
            const __half2 t2 = __half2(__nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3));
            const float2 t = __half22float2(t2);
            f[2 * h] = t.x;
            f[2 * h + 1] = t.y;
        }
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            if constexpr (IK == 1) {
                f[2 * h] = __uint_as_float(w[h] << 16);
                f[2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
            } else {
                const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w[h]));
                f[2 * h] = t.x;
                f[2 * h + 1] = t.y;
            }
        }
    }
}

template <int IK>
__device__ __forceinline__ Vec8<IK> ld8(const Elem<IK> *p)
{
    return __ldg(reinterpret_cast<const Vec8<IK> *>(p));
}

// Up to eight elements at p (cnt of them, the rest zero) as one 8-element vector.
template <int IK>
__device__ __forceinline__ Vec8<IK> ld_partial(const Elem<IK> *p, int cnt)
{
    constexpr int B = 8 * esize<IK>();                 // bits per element
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (e < cnt) w[(e * B) >> 5] |= (uint32_t)__ldg(p + e) << ((e * B) & 31);
    if constexpr (IK == 2) return make_uint2(w[0], w[1]);
    else return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// op(A)[m][k0 + kk] for m < MR, kk < kr, widened to FP32 into As, zero where
// m >= M or kk >= klen.  M_MAJOR (the N x K consumer): row m at As + m * kr,
// each 8-element chunk c split in halves, elements 8c..8c+3 at 4c and
// 8c+4..8c+7 at kr/2 + 4c, so that lanes reading consecutive chunks touch
// consecutive 16-byte words (no bank conflicts); else As[kk * MR + m].
// A stored M x K (a_t = 0) is read 8 elements per load; A stored K x M
// (a_t = 1, 16-bit inputs only) one element at a time.  Runs on the 256
// consumer threads (ct = 0..255).
template <int MR, int IK, bool M_MAJOR>
__device__ __forceinline__ void stage_a(float *As, const GemvArgs &g, int k0, int klen, int ct)
{
    const Elem<IK> *A = static_cast<const Elem<IK> *>(g.A);
    const int kr = g.kr;
    if (!g.a_t) {
        const int per_row = kr >> 3;            // 8-element groups per row
        const int groups = MR * per_row;
        constexpr int U = 4;
        for (int g0 = ct; g0 < groups; g0 += U * GV_CONSUMERS) {
            Vec8<IK> v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = g0 + u * GV_CONSUMERS;
                const int m = q / per_row, kk = (q - m * per_row) * 8;
                const int cnt = klen - kk;
                v[u] = Vec8<IK>{};
                if (q < groups && m < g.M && cnt > 0) {
                    const Elem<IK> *p = A + (long long)m * g.lda + k0 + kk;
                    v[u] = cnt >= 8 ? ld8<IK>(p) : ld_partial<IK>(p, cnt);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = g0 + u * GV_CONSUMERS;
                if (q >= groups) break;
                const int m = q / per_row, kk = (q - m * per_row) * 8;
                float f[8];
                widen8<IK>(v[u], f);
                if (M_MAJOR) {
                    float *row = As + m * kr + (kk >> 1);
                    *reinterpret_cast<float4 *>(row) = make_float4(f[0], f[1], f[2], f[3]);
                    *reinterpret_cast<float4 *>(row + (kr >> 1)) =
                        make_float4(f[4], f[5], f[6], f[7]);
                } else if (MR == 1) {                  // one row: As[kk]
                    float4 *d = reinterpret_cast<float4 *>(As + kk);
                    d[0] = make_float4(f[0], f[1], f[2], f[3]);
                    d[1] = make_float4(f[4], f[5], f[6], f[7]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) As[(kk + e) * MR + m] = f[e];
                }
            }
        }
    } else {
        const int total = MR * kr;
        constexpr int U = 8;
        for (int i0 = ct; i0 < total; i0 += U * GV_CONSUMERS) {
            uint32_t v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u * GV_CONSUMERS;
                int m, kk;
                if (M_MAJOR) { m = i / kr; kk = i - m * kr; }
                else { kk = i / MR; m = i - kk * MR; }
                v[u] = 0u;
                if (i < total && m < g.M && kk < klen)
                    v[u] = __ldg(A + (long long)(k0 + kk) * g.lda + m);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u * GV_CONSUMERS;
                if (i >= total) continue;
                int dst = i;
                if (M_MAJOR) {
                    const int m = i / kr, kk = i - m * kr;
                    dst = m * kr + ((kk & 4) ? (kr >> 1) : 0) + ((kk >> 3) << 2) + (kk & 3);
                }
                As[dst] = widen1<IK>(v[u]);
            }
        }
    }
}

// Shared memory of one CTA, from a 128-byte aligned base: the ring of boxes,
// the op(A) slice (MR x kr FP32), this CTA's partial block (MR x CW FP32),
// the per-warp sums of the K x N layout (8 x MR x 128 FP32), the stage
// barriers full[ns] and empty[ns], and the abort flag.  cw: output columns
// per CTA (gemv_cols_per_block).
struct GvLayout {
    int as, part, red, bars, abort_off, total;
};

__host__ __device__ inline GvLayout gv_layout(int mr, bool b_kn, int cw, int kr, int ns)
{
    GvLayout L;
    L.as = ns * GV_STAGE_BYTES;
    L.part = L.as + 4 * mr * kr;
    L.red = L.part + 4 * mr * cw;
    L.bars = L.red + (b_kn ? 4 * GV_WARPS * mr * KN_CW : 0);
    L.abort_off = L.bars + 16 * ns;
    L.total = L.abort_off + 16 + 128;                  // + alignment slack
    return L;
}

// The 8 warps of a box agree on whether to go on: a wait that ran out, or
// the abort flag, stops all of them together.
__device__ __forceinline__ bool stage_ready(const uint64_t *full, int s, int ns,
                                            volatile int *abort_flag, int *err)
{
    const bool got = wait_bounded(smem_u32(&full[s % ns]), (uint32_t)((s / ns) & 1), abort_flag, err);
    return __all_sync(0xffffffffu, got);
}

// B stored N x K.  Box s of the range holds rows n0 .. n0 + ROWS - 1 (32 for
// 16-bit, 64 for 8-bit elements), K elements k0 + 256 s .. + 255, row-major.
// Consumer warp w owns rows w * RPW .. + RPW - 1; lane l takes elements
// 8l .. 8l + 7 of each.
template <int MR, int IK>
__device__ __forceinline__ void consume_nk(const GemvArgs &g, const uint8_t *ring,
                                           const uint64_t *full, uint64_t *empty,
                                           volatile int *abort_flag, float *As, float *part,
                                           int k0, int klen, int nst, int ct)
{
    constexpr int ROWS = nk_rows(esize<IK>());
    constexpr int RPW = ROWS / GV_WARPS;
    stage_a<MR, IK, true>(As, g, k0, klen, ct);
    named_bar_sync(1, GV_CONSUMERS);
    const int cw = ct >> 5, lane = ct & 31;
    // Two partial sums per output, over the even and the odd elements of each
    // 8-element chunk, advanced together by one packed FP32 FMA (16-bit B;
    // e4m3 B keeps one scalar sum).
    using Acc = std::conditional_t<IK != 2, float2, float>;
    Acc acc[MR][RPW];
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
        for (int r = 0; r < RPW; ++r) acc[m][r] = Acc{};

    for (int s = 0; s < nst; ++s) {
        if (!stage_ready(full, s, g.stages, abort_flag, g.err)) break;
        const int slot = s % g.stages;
        const Elem<IK> *st = reinterpret_cast<const Elem<IK> *>(ring + slot * GV_STAGE_BYTES) +
                             cw * RPW * NK_KS + 8 * lane;
        Vec8<IK> bv[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) bv[r] = *reinterpret_cast<const Vec8<IK> *>(st + r * NK_KS);
        float a[MR][8];
#pragma unroll
        for (int m = 0; m < MR; ++m) {
            const float *ap = As + m * g.kr + ((s * NK_KS + 8 * lane) >> 1);   // chunk halves
            const float4 a0 = *reinterpret_cast<const float4 *>(ap);
            const float4 a1 = *reinterpret_cast<const float4 *>(ap + (g.kr >> 1));
            a[m][0] = a0.x; a[m][1] = a0.y; a[m][2] = a0.z; a[m][3] = a0.w;
            a[m][4] = a1.x; a[m][5] = a1.y; a[m][6] = a1.z; a[m][7] = a1.w;
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            float b[8];
            widen8<IK>(bv[r], b);
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                if constexpr (IK != 2) {
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        acc[m][r] = __ffma2_rn(make_float2(a[m][e], a[m][e + 1]),
                                               make_float2(b[e], b[e + 1]), acc[m][r]);
                } else {   // 8 rows a warp: scalar FMAs keep the registers for 3 CTAs per SM
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[m][r] = fmaf(a[m][e], b[e], acc[m][r]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
    }
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            float v;
            if constexpr (IK != 2) v = acc[m][r].x + acc[m][r].y;
            else v = acc[m][r];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) part[m * ROWS + cw * RPW + r] = v;
        }
}

// B stored K x N.  Box s of the range holds K rows k0 + 64 s .. + 63,
// columns n0..n0+127 (row-major, 256 bytes a row).
template <int MR, int IK, bool DUAL>
__device__ __forceinline__ void consume_kn(const GemvArgs &g, const uint8_t *ring,
                                           const uint64_t *full, uint64_t *empty,
                                           volatile int *abort_flag, float *As, float *red,
                                           float *part, int k0, int klen, int nst, int ct)
{
    static_assert(IK != 2, "8-bit B is read N x K only");
    stage_a<MR, IK, false>(As, g, k0, klen, ct);
    named_bar_sync(1, GV_CONSUMERS);
    const int cx = ct & 15, rl = ct >> 4;              // 16 column threads x 16 row lanes
    const int cw = ct >> 5, lane = ct & 31;
    float acc[MR][8];
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[m][e] = 0.0f;

    for (int s = 0; s < nst; ++s) {
        if (!stage_ready(full, s, g.stages, abort_flag, g.err)) break;
        const int slot = s % g.stages;
        // One box of 128 columns, or (DUAL) two boxes of 64 columns, W1's
        // then W2's, each 64 rows of 128 bytes.
        constexpr int ROW = DUAL ? KN_CW / 2 : KN_CW;
        const uint16_t *st = reinterpret_cast<const uint16_t *>(ring + slot * GV_STAGE_BYTES) +
                             (DUAL ? (cx >> 3) * (KN_KS * ROW) + 8 * (cx & 7) : 8 * cx);
        uint4 bv[KN_RPT];
#pragma unroll
        for (int i = 0; i < KN_RPT; ++i)
            bv[i] = *reinterpret_cast<const uint4 *>(st + (rl + 16 * i) * ROW);
#pragma unroll
        for (int i = 0; i < KN_RPT; ++i) {
            const int kk = s * KN_KS + rl + 16 * i;
            float a[MR];
            if constexpr (MR == 2) {
                const float2 t = *reinterpret_cast<const float2 *>(As + kk * 2);
                a[0] = t.x; a[1] = t.y;
            } else {
                a[0] = As[kk];
            }
            float b[8];
            widen8<IK>(bv[i], b);
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                const float2 am = make_float2(a[m], a[m]);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {   // two adjacent columns per packed FMA
                    const float2 t = __ffma2_rn(am, make_float2(b[e], b[e + 1]),
                                                make_float2(acc[m][e], acc[m][e + 1]));
                    acc[m][e] = t.x;
                    acc[m][e + 1] = t.y;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
    }
    // The 2 row lanes of this warp (lanes cx and cx + 16).
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float v = acc[m][e];
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            if (lane < 16) red[(cw * MR + m) * KN_CW + 8 * lane + e] = v;
        }
    named_bar_sync(1, GV_CONSUMERS);
    for (int t = ct; t < MR * KN_CW; t += GV_CONSUMERS) {
        const int m = t / KN_CW, col = t - m * KN_CW;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < GV_WARPS; ++w) sum += red[(w * MR + m) * KN_CW + col];
        part[t] = sum;
    }
}

// Grid: clusters of g.ranges CTAs, one cluster per block of output columns;
// CTA rank r of a cluster covers K range [r kr, min(K, (r + 1) kr)).
template <int MR, bool B_KN, int IK, bool DUAL>
__global__ void __launch_bounds__(GV_THREADS, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                const GemvArgs g)
{
    static_assert(!DUAL || (B_KN && IK == 1), "two weights: bf16 B stored K x N");
    static_assert(MR == 1 || MR == 2, "the op(A) loads are written for one or two rows");
    constexpr int CW = B_KN ? KN_CW : nk_rows(esize<IK>());
    constexpr int KS = B_KN ? KN_KS : NK_KS;
    extern __shared__ uint8_t gv_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(gv_raw) + 127) & ~static_cast<uintptr_t>(127));
    const GvLayout L = gv_layout(MR, B_KN, CW, g.kr, g.stages);
    const uint8_t *ring = base;
    float *As = reinterpret_cast<float *>(base + L.as);
    float *part = reinterpret_cast<float *>(base + L.part);
    float *red = reinterpret_cast<float *>(base + L.red);
    uint64_t *full = reinterpret_cast<uint64_t *>(base + L.bars);
    uint64_t *empty = full + g.stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + L.abort_off);

    const int rank = (int)cluster_ctarank();
    const int block = blockIdx.x / g.ranges;
    const int k0 = rank * g.kr;
    const int klen = g.K - k0 < g.kr ? g.K - k0 : g.kr;
    const int nst = (klen + KS - 1) / KS;
    const int n0 = block * CW;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < g.stages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), GV_WARPS);
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmB);
        if (DUAL) tma_prefetch_desc(&tmB2);
    }
    __syncthreads();
    // B and op(A) may come from the kernel before this one on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        if (lane == 0) {
            const int ns = g.stages;
            int issued = 0;
            for (int s = 0; s < nst; ++s) {
                const int slot = s % ns;
                if (s >= ns && !wait_bounded(smem_u32(&empty[slot]), (uint32_t)(((s / ns) - 1) & 1),
                                             abort_flag, g.err))
                    break;
                const uint32_t fb = smem_u32(&full[slot]);
                mbar_arrive_expect_tx(fb, GV_STAGE_BYTES);
                const uint32_t dst = smem_u32(ring + slot * GV_STAGE_BYTES);
                if (DUAL) {               // 64 Gate columns, then the same 64 Up columns
                    tma_load_2d(dst, &tmB, fb, n0 / 2, k0 + s * KS);
                    tma_load_2d(dst + GV_STAGE_BYTES / 2, &tmB2, fb, n0 / 2, k0 + s * KS);
                } else if (B_KN) {
                    tma_load_2d(dst, &tmB, fb, n0, k0 + s * KS);
                } else {
                    tma_load_2d(dst, &tmB, fb, k0 + s * KS, n0);
                }
                issued = s + 1;
            }
            // Boxes still in flight (only after an abort) land before the CTA
            // leaves; after a normal run every one of these phases is complete.
            for (int s = issued > ns ? issued - ns : 0; s < issued; ++s)
                wait_bounded(smem_u32(&full[s % ns]), (uint32_t)((s / ns) & 1), abort_flag, g.err,
                             false, DRAIN_LIMIT_NS);
        }
    } else {
        const int ct = threadIdx.x - 32;
        if constexpr (B_KN)
            consume_kn<MR, IK, DUAL>(g, ring, full, empty, abort_flag, As, red, part, k0, klen, nst,
                                     ct);
        else
            consume_nk<MR, IK>(g, ring, full, empty, abort_flag, As, part, k0, klen, nst, ct);
    }

    cluster_sync_all();     // every partial block of the cluster is written
    if (DUAL && rank == 0 && warp > 0) {
        // Column j of the block is Gate j (from W1), column 64 + j Up j (W2).
        const uint32_t part_s = smem_u32(part);
        for (int t = threadIdx.x - 32; t < MR * (CW / 2); t += GV_CONSUMERS) {
            const int m = t / (CW / 2), j = t - m * (CW / 2), n = n0 / 2 + j;
            if (m < g.M && n < g.N) {
                const uint32_t at = part_s + 4u * (uint32_t)(m * CW + j);
                float gs = 0.0f, us = 0.0f;
                for (int r = 0; r < g.ranges; ++r) {
                    gs += ld_shared_cluster_f32(mapa_shared(at, (uint32_t)r));
                    us += ld_shared_cluster_f32(mapa_shared(at + 4u * (CW / 2), (uint32_t)r));
                }
                const float y = silu_f32(g.alpha * gs) * (g.alpha * us);
                store_out(g.D, (long long)m * g.ldd + n, y, g.out_kind);
            }
        }
    } else if (rank == 0 && warp > 0 && g.swiglu) {
        // Column pairs (Gate, Up) of the interleaved weight -> one output
        // column each, the SwiGLU page's pair-multiply epilogue.
        const uint32_t part_s = smem_u32(part);
        for (int t = threadIdx.x - 32; t < MR * (CW / 2); t += GV_CONSUMERS) {
            const int m = t / (CW / 2), c = 2 * (t - m * (CW / 2)), n = n0 + c;
            if (m < g.M && n < g.N) {
                const uint32_t at = part_s + 4u * (uint32_t)(m * CW + c);
                float gs = 0.0f, us = 0.0f;
                for (int r = 0; r < g.ranges; ++r) {
                    gs += ld_shared_cluster_f32(mapa_shared(at, (uint32_t)r));
                    us += ld_shared_cluster_f32(mapa_shared(at + 4u, (uint32_t)r));
                }
                const float y = silu_f32(g.alpha * gs) * (g.alpha * us);
                store_out(g.D, (long long)m * g.ldd + (n >> 1), y, g.out_kind);
            }
        }
    } else if (rank == 0 && warp > 0) {
        const uint32_t part_s = smem_u32(part);
        for (int t = threadIdx.x - 32; t < MR * CW; t += GV_CONSUMERS) {
            const int m = t / CW, n = n0 + (t - m * CW);
            if (m < g.M && n < g.N) {
                float sum = 0.0f;
                for (int r = 0; r < g.ranges; ++r)
                    sum += ld_shared_cluster_f32(mapa_shared(part_s + 4u * (uint32_t)t, (uint32_t)r));
                float v = g.alpha * sum;
                const long long off = (long long)m * g.ldd + n;
                if (g.beta != 0.0f) v += g.beta * load_out(g.D, off, g.out_kind);
                store_out(g.D, off, v, g.out_kind);
            }
        }
    }
    cluster_sync_all();     // no CTA leaves while CTA 0 still reads its partials
}

template <int MR, bool B_KN, int IK, bool DUAL = false>
cudaError_t launch_gemv_impl(const CUtensorMap &tmB, const CUtensorMap &tmB2, const GemvArgs &g,
                             int col_blocks, cudaStream_t s)
{
    static DeviceOnce configured;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto kernel = gemv_kernel<MR, B_KN, IK, DUAL>;
    if (configured.needed(dev)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 GV_MAX_SMEM);
        if (e != cudaSuccess) return e;
        configured.mark(dev);
    }
    constexpr int CW = B_KN ? KN_CW : nk_rows(esize<IK>());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(col_blocks * g.ranges));
    cfg.blockDim = dim3(GV_THREADS);
    cfg.dynamicSmemBytes = (size_t)gv_layout(MR, B_KN, CW, g.kr, g.stages).total;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)g.ranges;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, tmB, tmB2, g);
}

template <int MR>
cudaError_t launch_gemv_mr(const CUtensorMap &tmB, const CUtensorMap *tmB2, const GemvArgs &g,
                           bool b_kn, int in_kind, int col_blocks, cudaStream_t s)
{
    if (tmB2)
        return b_kn && in_kind == 1 ? launch_gemv_impl<MR, true, 1, true>(tmB, *tmB2, g, col_blocks, s)
                                    : cudaErrorInvalidValue;
    if (in_kind == 2)
        return b_kn ? cudaErrorInvalidValue
                    : launch_gemv_impl<MR, false, 2>(tmB, tmB, g, col_blocks, s);
    if (b_kn)
        return in_kind == 1 ? launch_gemv_impl<MR, true, 1>(tmB, tmB, g, col_blocks, s)
                            : launch_gemv_impl<MR, true, 0>(tmB, tmB, g, col_blocks, s);
    return in_kind == 1 ? launch_gemv_impl<MR, false, 1>(tmB, tmB, g, col_blocks, s)
                        : launch_gemv_impl<MR, false, 0>(tmB, tmB, g, col_blocks, s);
}

}  // namespace

int gemv_cols_per_block(bool b_kn, int in_kind)
{
    return b_kn ? KN_CW : nk_rows(in_kind == 2 ? 1 : 2);
}
int gemv_k_per_stage(bool b_kn) { return b_kn ? KN_KS : NK_KS; }
int gemv_box_inner(bool b_kn) { return b_kn ? KN_CW : NK_KS; }
int gemv_box_outer(bool b_kn, int in_kind) { return b_kn ? KN_KS : nk_rows(in_kind == 2 ? 1 : 2); }

int gemv_smem_bytes(int mr, bool b_kn, int in_kind, int kr, int stages)
{
    return gv_layout(mr, b_kn, gemv_cols_per_block(b_kn, in_kind), kr, stages).total;
}

cudaError_t launch_gemv(const CUtensorMap &tmB, const CUtensorMap *tmB2, const GemvArgs &g, int mr,
                        bool b_kn, int in_kind, int col_blocks, cudaStream_t s)
{
    switch (mr) {
    case 1: return launch_gemv_mr<1>(tmB, tmB2, g, b_kn, in_kind, col_blocks, s);
    case 2: return launch_gemv_mr<2>(tmB, tmB2, g, b_kn, in_kind, col_blocks, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace swg
