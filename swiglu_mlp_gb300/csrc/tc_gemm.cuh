// tc_gemm.cuh — persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// One CTA per SM walks a static list of output tiles (BM x BN, BM = 128).
// Roles inside a CTA (320 threads):
//   warp 0, lane 0 : TMA producer.  For every 64-wide K block it waits for a
//                    free shared-memory stage, arms the stage's "full" barrier
//                    with the byte count and issues the tile loads of op(A)
//                    and op(B) (128-byte swizzle; the tensor map's box and the
//                    operand's major-ness realise op = N / T without copies;
//                    an MN-major operand whose extent is a multiple of 64
//                    arrives as one 3-D box holding all its 64-wide atoms).
//   warp 1         : allocates tensor memory (TMEM); lane 0 issues
//                    tcgen05.mma (M=128, N=BN, K=16, FP32 accumulate) into one
//                    of two TMEM accumulators and commits each stage back to
//                    its "empty" barrier, each finished tile to "acc_full".
//   warps 2..9     : epilogue.  Each thread owns one accumulator row (TMEM
//                    lane) and half of the tile's columns (two warps per lane
//                    quarter), reads them 32 columns at a time with
//                    tcgen05.ld and applies the fused epilogue:
//                      EPI_STORE  D = alpha*acc + beta*C, cast, 16-byte stores;
//                      EPI_SWIGLU Y = SiLU(acc[2j]) * acc[2j+1] per column pair;
//                      EPI_SPLITK FP32 partial of one K range to the
//                                 workspace; splitk_reduce_kernel (launched
//                                 right behind, programmatic dependent launch)
//                                 sums the partials in split order and stores
//                                 alpha*sum + beta*C.
// The double TMEM accumulator lets the epilogue of tile t overlap the main
// loop of tile t+1.  A CTA's last tile, when every pipeline stage has been
// consumed, is written into the stage area in the 128-byte swizzle layout and
// stored with TMA bulk stores (whole lines, clipped at the matrix edges).
//
// CTA pairs (PAIR): clusters of two CTAs share one cta_group::2 MMA of
// 256 x BN; each CTA loads its 128 rows of A and half of B, and receives its
// own 128 accumulator rows.  Each epilogue warp hands a drained accumulator
// back on the leader's barrier with a release at CTA scope only: the hand-off
// orders tensor-memory reads, not the warp's global stores.  EPI_SPLITK_T and
// EPI_SWIGLU_DUAL are described at the EpiKind enumeration.
//
// Programmatic dependent launch: the kernel lets the next kernel on the stream
// be scheduled as soon as it starts, and touches global memory only after
// griddepcontrol.wait, so consecutive calls overlap set-up and tail safely.
//
// Every barrier wait is bounded (about two seconds): on expiry the thread
// records SWG_ERR_DEVICE_TIMEOUT in the error word, raises a CTA-wide abort
// flag that makes every other role leave its loop, the producer waits (again
// bounded) for its own loads in flight, the MMA thread for its own MMAs, and
// the CTA frees its TMEM and exits.
//
// Method sources: the GEMM statement of "GEMM o Coração Matemático" §1; the
// tiling, multi-buffering, split-K and epilogue fusion of
// "为什么 GEMM 是 CUDA 的必修课" (多级分块, 关键技术 items 3, 5, 6); the
// interleaved-weight SwiGLU epilogue of "Sobreposição de Ativação em Nível de
// Tile para Inferência Eficiente de LLM", Metodologia, Kernel-2.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace swg {

// EPI_SPLITK_T: split-K with swapped operands.  The kernel computes the
// transposed product (its rows are the output's columns), so each thread owns
// one output column and its registers hold output rows; the partial is written
// transposed back to ws[split][row][column].
// EPI_SWIGLU_DUAL: SwiGLU from separate W1 and W2.  The B tile's first BN/2
// columns come from W1 (Gate) and the last BN/2 from W2 (Up) -- in a CTA pair
// the even CTA loads its half of B from W1 and the odd CTA from W2 -- so the
// accumulator row holds Gate in columns [0, BN/2) and Up in [BN/2, BN).
// EPI_SPLITK_CL: swapped-operand split-K reduced inside a thread-block
// cluster.  The p.splits CTAs of a cluster (at most 8) compute the K ranges of
// one tile, one range per rank; each parks its FP32 partial in its own shared
// memory, and after a cluster barrier rank r reads its share of the tile's
// output rows from every rank's shared memory in rank order 0, 1, .., S-1,
// applies alpha and beta * C and stores D.  One launch, no workspace.  Each
// CTA runs exactly one unit, so the grid is tiles x S CTAs.
// EPI_SWIGLU_CL: the same cluster reduction for the fused SwiGLU in the
// output's own frame (rows = rows of A, columns = the 2N-space of W_fused):
// rank r sums its share of the tile's column pairs over the S ranks and
// stores SiLU(alpha * gate) * (alpha * up).
// EPI_STORE_CL: the same for a plain GEMM tile (128 x BN, output frame):
// rank r stores alpha * sum + beta * C for its share of the tile's columns.
enum EpiKind {
    EPI_STORE = 0,
    EPI_SWIGLU = 1,
    EPI_SPLITK = 2,
    EPI_SPLITK_T = 3,
    EPI_SWIGLU_DUAL = 4,
    EPI_SPLITK_CL = 5,
    EPI_SWIGLU_CL = 6,
    EPI_STORE_CL = 7
};

// The epilogues whose K ranges are reduced inside a cluster (one unit per CTA).
template <int EPI>
struct ClusterK {
    static constexpr bool value =
        EPI == EPI_SPLITK_CL || EPI == EPI_SWIGLU_CL || EPI == EPI_STORE_CL;
    // EPI_STORE_CL receives the partials in its consumed pipeline stages, so
    // its ranks first wait for every rank's main loop (one more barrier).
    static constexpr int barriers = EPI == EPI_STORE_CL ? 2 : 1;
};
enum OutKind { OUT_BF16 = 0, OUT_F16 = 1, OUT_F32 = 2 };

constexpr int BM = 128;
constexpr int BK = 64;               // 64 x 16-bit = one 128-byte swizzle row
constexpr int UMMA_K = 16;           // K of one kind::f16 MMA
constexpr int NUM_EPI_WARPS = 8;      // two per TMEM lane quarter
constexpr int NUM_EPI_THREADS = NUM_EPI_WARPS * 32;
constexpr int NUM_THREADS = 64 + NUM_EPI_THREADS;
constexpr int EPI_WARP0 = 2;
constexpr int ERR_TIMEOUT = 6;       // == SWG_ERR_DEVICE_TIMEOUT
constexpr int MAX_SPLITS = 16;       // split-K ranges per tile (host enforces)
constexpr int MAX_CLUSTER_SPLITS = 4; // K ranges of one tile reduced in a cluster
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // pipeline waits
constexpr uint64_t DRAIN_LIMIT_NS = 1000000ull;      // teardown drains

struct TileParams {
    int M, N, K;                 // N is the 2N-space width for SwiGLU
    int m_blocks, n_blocks, k_blocks;
    int tiles;                   // m_blocks * n_blocks
    int splits;                  // K ranges per tile (1 = no split)
    int kb_per_split;            // K blocks per range (last may be shorter)
    int units;                   // tiles * splits
    int group_m;                 // raster: m-blocks per group
    uint32_t idesc;              // tcgen05 instruction descriptor
    int bk;                      // elements per 128-byte K block: 64 (16-bit) or 128 (fp8)
    // 1: each CTA writes its last tile through shared memory with TMA stores
    // via the output map passed in the kernel's third tensor-map slot (D, Y,
    // or the 3-D split-K workspace); only with beta = 0 and whole 128-byte
    // output boxes.
    int tma_store;
    int a_mn_major;              // op(A) stored M-contiguous (transA = T)
    int b_mn_major;              // op(B) stored N-contiguous (transB = N)
    // MN-major operand mapped in 3-D (64 MN x K rows x atoms): one box per
    // stage fills all its 64-wide atoms (see make_tmap_mn3); 0: 2-D boxes.
    int a_mn3, b_mn3;
    float alpha, beta;
    void *D;                     // output (also C when beta != 0)
    long long ldd;
    int out_kind;                // OutKind
    float *ws;                   // split-K partials [splits][M][ld_ws]
    long long ld_ws;
    int *err;                    // device error word
};

// Tile configuration.  BN is the MMA's N (the tile width).  With PAIR, two
// CTAs of a cluster share one 256-row MMA: each holds its 128 rows of A and
// BN/2 columns of B per stage and receives its 128 accumulator rows.
template <int BN, bool PAIR, int EPI = EPI_STORE>
struct Cfg {
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;
    static constexpr int B_COLS = PAIR ? BN / 2 : BN;     // B columns held per CTA
    // 128-byte K atoms per pipeline stage.  The few-rows cluster kernel moves
    // two per stage (one barrier round and one TMA issue per 32 KB of the
    // weight instead of per 16 KB): its per-SM rate was bound by the
    // producer's per-stage latency, not by bytes.
    static constexpr int KPS = EPI == EPI_SPLITK_CL ? 2 : 1;
    static constexpr int A_BYTES = BM * BK * 2 * KPS;
    static constexpr int B_BYTES = B_COLS * BK * 2 * KPS;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // Cluster-reduced K ranges: a receive buffer for the partials sent by
    // every rank, beside the stages, so no rank has to wait for another's
    // main loop to end before sending (see the cluster epilogues).
    static constexpr int RECV_BYTES = EPI == EPI_SPLITK_CL   ? BN * BM * 4
                                      : EPI == EPI_SWIGLU_CL ? BM * (BN + 4 * MAX_CLUSTER_SPLITS) * 4
                                                             : 0;
    // 192 KB of stages (measured: a seventh 32 KB pair stage did not help
    // and shrank L1), at most 12, within the 227 KB a CTA can have.
    static constexpr int STAGE_BUDGET_RAW = 232448 - 2048 - RECV_BYTES;
    static constexpr int STAGE_BUDGET =
        STAGE_BUDGET_RAW < 192 * 1024 ? STAGE_BUDGET_RAW : 192 * 1024;
    static constexpr int STAGES_RAW = STAGE_BUDGET / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
    static constexpr int NUM_BARS = 2 * STAGES + 6;
    static constexpr int TMEM_COLS = (2 * BN) <= 32 ? 32 : (2 * BN) <= 64 ? 64
                                   : (2 * BN) <= 128 ? 128 : (2 * BN) <= 256 ? 256 : 512;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + RECV_BYTES + NUM_BARS * 8 + 64;
    static_assert(STAGES >= 3, "pipeline too shallow");
    static_assert(SMEM_BYTES <= 232448, "beyond the per-CTA shared memory");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "BN must be a multiple of 16, <= 256");
    static_assert(!PAIR || BN % 128 == 0, "pair tiles split B in 64-column boxes per CTA");
    static_assert(STAGES * STAGE_BYTES >= BM * BN * 4 || BN < 64,
                  "the stage area holds a staged FP32 output tile");
};

__device__ __forceinline__ void tile_coords(const TileParams &p, int tile, int &mb, int &nb);

// Tile coordinates of work unit u (grouped raster: walk GROUP m-blocks down a
// column of tiles before moving right, so concurrently running CTAs share A
// and B panels in L2).
__device__ __forceinline__ void unit_coords(const TileParams &p, int u, int &mb, int &nb,
                                            int &split, int &tile)
{
    // Integer division by a runtime value is a chain of tens of dependent
    // instructions on one thread; the first unit's coordinates sit on the
    // path to the first load (measured ~0.4 us), so the common shapes skip it.
    if (p.splits == 1) {
        split = 0;
        tile = u;
    } else {
        split = u / p.tiles;
        tile = u - split * p.tiles;
    }
    tile_coords(p, tile, mb, nb);
}

// Block coordinates of tile `tile` in the grouped raster (see unit_coords).
__device__ __forceinline__ void tile_coords(const TileParams &p, int tile, int &mb, int &nb)
{
    if (p.n_blocks == 1) {             // one column of tiles: the raster is the identity
        mb = tile;
        nb = 0;
        return;
    }
    if (p.m_blocks == 1) {             // one row of tiles
        mb = 0;
        nb = tile;
        return;
    }
    const int per_group = p.group_m * p.n_blocks;
    const int group = tile / per_group;
    const int first_m = group * p.group_m;
    int gm = p.m_blocks - first_m;
    gm = gm < p.group_m ? gm : p.group_m;
    const int local = tile - group * per_group;
    mb = first_m + local % gm;
    nb = local / gm;
}

// Waits for the phase of `bar` with the given parity.  Gives up (returning
// false) when another role has raised the abort flag, or after `limit_ns`;
// a time-out raises the abort flag and records ERR_TIMEOUT.  The drain waits
// at teardown pass honour_abort = false and a short limit.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             int *err, bool honour_abort = true,
                                             uint64_t limit_ns = WAIT_LIMIT_NS)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31) == 0) {
            if (honour_abort && *abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicCAS(err, 0, ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), version 1 at bit 46, 128-byte swizzle
// (layout type 2) at bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// SiLU(x) = x * sigmoid(x) = x / (1 + e^-x) in FP32 without a division
// slow path: __expf and __fdividef are the CUDA fast intrinsics.  Limits:
// x -> -inf gives 1 + e^-x = inf and x * (1/inf) = -0; x -> +inf gives x.
__device__ __forceinline__ float silu_f32(float x)
{
    return __fdividef(x, 1.0f + __expf(-x));
}

__device__ __forceinline__ uint32_t pack2(float a, float b, int out_kind)
{
    if (out_kind == OUT_F16) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float load_out(const void *base, long long idx, int out_kind)
{
    if (out_kind == OUT_F32) return reinterpret_cast<const float *>(base)[idx];
    if (out_kind == OUT_F16) return __half2float(reinterpret_cast<const __half *>(base)[idx]);
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
}

__device__ __forceinline__ void store_out(void *base, long long idx, float v, int out_kind)
{
    if (out_kind == OUT_F32)
        reinterpret_cast<float *>(base)[idx] = v;
    else if (out_kind == OUT_F16)
        reinterpret_cast<__half *>(base)[idx] = __float2half_rn(v);
    else
        reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(v);
}

// alpha*acc + beta*C for `cnt` (<= 32) consecutive outputs of one row,
// starting at element offset `off` of D.  `full` = all 32 in range and the
// row chunk is 16-byte aligned (guaranteed by the host's alignment rules).
__device__ __forceinline__ void store_row_chunk(const TileParams &p, long long off, const float *acc,
                                                int cnt)
{
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = p.alpha * acc[j];
    const bool full = cnt == 32;
    if (p.beta != 0.0f) {
        if (full && p.out_kind != OUT_F32) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const uint16_t *>(p.D) + off);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 w = src[q];
                uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    float lo, hi;
                    if (p.out_kind == OUT_F16) {
                        __half2 c2 = *reinterpret_cast<__half2 *>(&ww[h]);
                        lo = __low2float(c2);
                        hi = __high2float(c2);
                    } else {
                        __nv_bfloat162 c2 = *reinterpret_cast<__nv_bfloat162 *>(&ww[h]);
                        lo = __low2float(c2);
                        hi = __high2float(c2);
                    }
                    v[q * 8 + h * 2] += p.beta * lo;
                    v[q * 8 + h * 2 + 1] += p.beta * hi;
                }
            }
        } else if (full) {
            const float4 *src = reinterpret_cast<const float4 *>(
                reinterpret_cast<const float *>(p.D) + off);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float4 c4 = src[q];
                v[q * 4 + 0] += p.beta * c4.x;
                v[q * 4 + 1] += p.beta * c4.y;
                v[q * 4 + 2] += p.beta * c4.z;
                v[q * 4 + 3] += p.beta * c4.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < cnt) v[j] += p.beta * load_out(p.D, off + j, p.out_kind);
        }
    }
    if (full && p.out_kind != OUT_F32) {
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.D) + off);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack2(v[q * 8 + 0], v[q * 8 + 1], p.out_kind);
            w.y = pack2(v[q * 8 + 2], v[q * 8 + 3], p.out_kind);
            w.z = pack2(v[q * 8 + 4], v[q * 8 + 5], p.out_kind);
            w.w = pack2(v[q * 8 + 6], v[q * 8 + 7], p.out_kind);
            dst[q] = w;
        }
    } else if (full) {
        float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.D) + off);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(v[q * 4], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < cnt) store_out(p.D, off + j, v[j], p.out_kind);
    }
}

// One 32-column chunk of one accumulator row (row m of the output, first
// column n of the tile's column space) through the epilogue EPI.
template <int EPI>
__device__ __forceinline__ void epi_chunk(const TileParams &p, const uint32_t (&r)[32], int m, int n,
                                          int split)
{
    if (n >= p.N) return;
    const int cnt = (p.N - n) < 32 ? (p.N - n) : 32;
    if (EPI == EPI_STORE) {
        float a[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) a[j] = __uint_as_float(r[j]);
        store_row_chunk(p, (long long)m * p.ldd + n, a, cnt);
    } else if (EPI == EPI_SWIGLU) {
        // Column pair (2j, 2j+1) of the 2N-space is (Gate_j, Up_j); output
        // column n/2 + j.
        const long long off = (long long)m * p.ldd + n / 2;
        // alpha = product of per-tensor dequantisation scales (1 for bf16),
        // applied to Gate and Up before the SiLU.
        float y[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            y[j] = silu_f32(p.alpha * __uint_as_float(r[2 * j])) *
                   (p.alpha * __uint_as_float(r[2 * j + 1]));
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.D) + off;
        if (cnt == 32) {
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = pack2(y[2 * j], y[2 * j + 1], OUT_BF16);
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
            d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (2 * j < cnt) dst[j] = __float2bfloat16_rn(y[j]);
        }
    } else {
        // Split-K: raw FP32 partial of this K range; reduced by a second kernel.
        float *dst = p.ws + ((long long)split * p.M + m) * p.ld_ws + n;
        if (cnt == 32) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                reinterpret_cast<float4 *>(dst)[j] =
                    make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < cnt) dst[j] = __uint_as_float(r[j]);
        }
    }
}

// ------------------------------------------------ staged last-tile stores
// A CTA's last tile is written to shared memory (the pipeline stages, all
// consumed by then) as boxes of 128 rows x 128 bytes -- 64 16-bit or 32 FP32
// output columns -- and stored with TMA: whole cache lines instead of one
// 16-byte piece of 32 different rows per warp store.  Within a box, row r's
// eight 16-byte chunks sit at chunk (j XOR r mod 8): the tensor map's 128-byte
// swizzle, which also spreads a warp's writes of one chunk over all banks.
__device__ __forceinline__ void stage16(uint32_t base, int row, int byte_col, uint4 v)
{
    const int box = byte_col >> 7;
    const int j = (byte_col >> 4) & 7;
    st_shared_v4(base + (uint32_t)(box * 16384 + row * 128 + ((j ^ (row & 7)) << 4)), v);
}

__device__ __forceinline__ uint4 f32x4(float a, float b, float c, float d)
{
    return make_uint4(__float_as_uint(a), __float_as_uint(b), __float_as_uint(c),
                      __float_as_uint(d));
}

// Output values of one 32-column accumulator chunk (tile columns
// [c0, c0 + 32)) of tile row `row`, staged: the same arithmetic as epi_chunk
// with beta = 0.
template <int EPI>
__device__ __forceinline__ void stage_epi_chunk(const TileParams &p, const uint32_t (&r)[32],
                                                uint32_t base, int row, int c0)
{
    if (EPI == EPI_STORE) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = p.alpha * __uint_as_float(r[j]);
        if (p.out_kind == OUT_F32) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                stage16(base, row, (c0 + 4 * q) * 4,
                        f32x4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                stage16(base, row, (c0 + 8 * q) * 2,
                        make_uint4(pack2(v[8 * q], v[8 * q + 1], p.out_kind),
                                   pack2(v[8 * q + 2], v[8 * q + 3], p.out_kind),
                                   pack2(v[8 * q + 4], v[8 * q + 5], p.out_kind),
                                   pack2(v[8 * q + 6], v[8 * q + 7], p.out_kind)));
        }
    } else if (EPI == EPI_SWIGLU) {
        float y[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            y[j] = silu_f32(p.alpha * __uint_as_float(r[2 * j])) *
                   (p.alpha * __uint_as_float(r[2 * j + 1]));
#pragma unroll
        for (int q = 0; q < 2; ++q)
            stage16(base, row, (c0 / 2 + 8 * q) * 2,
                    make_uint4(pack2(y[8 * q], y[8 * q + 1], OUT_BF16),
                               pack2(y[8 * q + 2], y[8 * q + 3], OUT_BF16),
                               pack2(y[8 * q + 4], y[8 * q + 5], OUT_BF16),
                               pack2(y[8 * q + 6], y[8 * q + 7], OUT_BF16)));
    } else {   // EPI_SPLITK: the raw FP32 partial
#pragma unroll
        for (int q = 0; q < 8; ++q)
            stage16(base, row, (c0 + 4 * q) * 4,
                    f32x4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                          __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])));
    }
}

// TMA stores of the staged boxes of tile (mb, nb) for this CTA's rows [m0,
// m0 + 128): boxes wholly right of the output's last column are skipped,
// the rest are clipped by the tensor map.
template <int EPI, int BN>
__device__ __forceinline__ void store_staged(const TileParams &p, const CUtensorMap *tm,
                                             uint32_t base, int m0, int nb, int split)
{
    const int esize = (EPI == EPI_SPLITK || (EPI == EPI_STORE && p.out_kind == OUT_F32)) ? 4 : 2;
    const int out_cols = EPI == EPI_SWIGLU ? BN / 2 : BN;
    const int n_out = EPI == EPI_SWIGLU ? p.N / 2 : p.N;
    const int box_cols = 128 / esize;
    const int x0 = nb * out_cols;
    for (int b = 0; b < out_cols / box_cols; ++b) {
        const int x = x0 + b * box_cols;
        if (x >= n_out) break;
        if (EPI == EPI_SPLITK)
            tma_store_3d(tm, base + b * 16384, x, m0, split);
        else
            tma_store_2d(tm, base + b * 16384, x, m0);
    }
    bulk_commit_group();
    // The staged tile is the CTA's last: only its shared-memory source has to
    // outlive the copy.
    bulk_wait_read_all();
}

// ------------------------------------------------ cluster split-K epilogues
// The K ranges of one tile run on the S = p.splits CTAs of a cluster, one
// range per rank.  Rank r owns a share of the tile's outputs.  As soon as its
// accumulator is complete, each CTA pushes every piece of its FP32 partial
// to the owner's receive buffer recv[source rank][...] (a region of that
// CTA's shared memory beside its pipeline stages; stores to distributed
// shared memory are posted, loads from it would wait a round trip each).
// One cluster barrier (release/acquire at cluster scope; the producer and
// MMA warps take part too) makes them visible, and the owner sums recv[0],
// recv[1], .., recv[S-1] from its own shared memory, in that order starting
// from 0, before the epilogue arithmetic.  After that barrier no CTA touches
// another's shared memory.

// EPI_SPLITK_CL (swapped-operand frame: TMEM lane = output column n of the
// tile, TMEM column j = output row m).  Rank r owns output rows
// [r * BN / S, (r + 1) * BN / S) of the tile.  recv[s] holds, per column n,
// G = BN / S / 4 groups of four rows; group g of column n sits at 16-byte
// slot n * G + (g XOR ((n * G / 8) mod G)), so each thread pushes four
// consecutive rows of its column with one 16-byte store and eight
// consecutive columns of one group fall in eight different bank groups.
// Before the accumulator is ready each thread loads the C values of the
// outputs it will produce (beta != 0), so that read overlaps the main loop.
__device__ __forceinline__ int recv_slot(int n, int g, int G)
{
    return n * G + (g ^ ((n * G / 8) % G));
}

template <int BN>
__device__ __forceinline__ void splitk_cluster_epilogue(const TileParams &p, uint32_t tmem_base,
                                                        uint8_t *recv_buf, uint64_t *acc_full,
                                                        volatile int *abort_flag, int unit,
                                                        int krank)
{
    // items (4 rows x 1 column) per thread: (BN / S / 4) * 128 / 256; the
    // host runs BN = 64 with S >= 2 only
    constexpr int ITEMS = BN / 8 > 4 ? 4 : BN / 8;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int et = threadIdx.x - EPI_WARP0 * 32;     // 0 .. 255
    const int S = p.splits;
    int mb, nb, split, tile;
    unit_coords(p, unit, mb, nb, split, tile);
    const int rows = BN / S;                   // output rows this rank reduces (4 .. 32)
    const int G = rows / 4;                    // four-row groups per column
    const int n_items = G * BM;
    const int Mo = p.N, No = p.M;              // output rows / columns
    // item idx: column n = idx % BM of the tile, rows 4 * (idx / BM) .. + 3 of this rank's share
    float c[ITEMS][4];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        c[it][0] = c[it][1] = c[it][2] = c[it][3] = 0.0f;
        const int idx = et + it * NUM_EPI_THREADS;
        if (p.beta == 0.0f || idx >= n_items) continue;
        const int n = mb * BM + idx % BM;
        const int m0 = nb * BN + krank * rows + 4 * (idx / BM);
        if (n >= No) continue;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (m0 + i < Mo) c[it][i] = load_out(p.D, (long long)(m0 + i) * p.ldd + n, p.out_kind);
    }

    // push: rows jj .. jj + 3 of this thread's column go to rank jj / rows
    const uint32_t recv = smem_u32(recv_buf);
    const uint32_t slice = (uint32_t)(rows * BM * 4);        // bytes of one source's slice
    constexpr int W = BN >= 32 ? 32 : 16;
    const int q = warp & 3;
    const int h = (warp - EPI_WARP0) / 4;
    const bool active = (BN == 64) || h == 0;
    const int j0 = BN == 64 ? h * 32 : 0;
    const int n_local = q * 32 + lane;
    bool ok = wait_bounded(smem_u32(&acc_full[0]), 0, abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
        tc_fence_after();
        if (active) {
            uint32_t r[W];
            tmem_ld_cols(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + j0, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int g = 0; g < W / 4; ++g) {
                const int jj = j0 + 4 * g;
                if (nb * BN + jj >= Mo) break;     // rows past the output are not sent
                const int owner = jj / rows;
                const uint32_t a = recv + (uint32_t)krank * slice +
                                   (uint32_t)(recv_slot(n_local, (jj - owner * rows) / 4, G) * 16);
                if (owner == krank)                // own share: a local store
                    st_shared_v4(a, make_uint4(r[4 * g], r[4 * g + 1], r[4 * g + 2], r[4 * g + 3]));
                else
                    st_dsmem_v4(mapa_shared(a, (uint32_t)owner), r[4 * g], r[4 * g + 1],
                                r[4 * g + 2], r[4 * g + 3]);
            }
        }
    }
    tc_fence_before();
    cluster_sync_all();
    // reduce this rank's rows from the local receive buffer, sources in order
    const float *rb = reinterpret_cast<const float *>(recv_buf);
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int idx = et + it * NUM_EPI_THREADS;
        if (idx >= n_items) continue;
        const int nl = idx % BM;
        const int g = idx / BM;
        const int n = mb * BM + nl;
        const int m0 = nb * BN + krank * rows + 4 * g;
        if (n >= No) continue;
        const int slot = recv_slot(nl, g, G);
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int r = 0; r < MAX_CLUSTER_SPLITS; ++r) {
            if (r < S) {
                const float4 v = *reinterpret_cast<const float4 *>(
                    rb + (size_t)r * (slice / 4) + slot * 4);
                acc[0] += v.x;
                acc[1] += v.y;
                acc[2] += v.z;
                acc[3] += v.w;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (m0 + i < Mo) {
                const float out = p.beta != 0.0f ? __fmaf_rn(p.beta, c[it][i], p.alpha * acc[i])
                                                 : p.alpha * acc[i];
                store_out(p.D, (long long)(m0 + i) * p.ldd + n, out, p.out_kind);
            }
        }
    }
}

// EPI_SWIGLU_CL (output frame: TMEM lane = row of the tile, TMEM column =
// 2N-space column, Gate at even and Up at odd columns).  Rank r owns the
// tile's 2N-space columns [r * BN / S, (r + 1) * BN / S);
// recv[s][row][column - r * BN / S], rows padded by 4 floats (16-byte stores
// and loads without bank conflicts).  For each row and group of 16 columns
// (8 outputs) the owner forms y = SiLU(alpha * gate) * (alpha * up) per
// pair, rounds once to bf16 and stores 16 bytes of Y.
template <int BN>
__device__ __forceinline__ void swiglu_cluster_epilogue(const TileParams &p, uint32_t tmem_base,
                                                        uint8_t *recv_buf, uint64_t *acc_full,
                                                        volatile int *abort_flag, int unit,
                                                        int krank)
{
    constexpr int NC = BN / 32;                // 32-column chunks per tile row
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int et = threadIdx.x - EPI_WARP0 * 32;
    const int S = p.splits;
    const int cols = BN / S;                   // 2N-space columns per rank (>= 32)
    const int ld = cols + 4;                   // row stride of a receive slice, floats
    const uint32_t slice = (uint32_t)(BM * ld * 4);
    int mb, nb, split, tile;
    unit_coords(p, unit, mb, nb, split, tile);
    const uint32_t recv = smem_u32(recv_buf);
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int c_begin = ((warp - EPI_WARP0) / 4) * (NC / 2);
    bool ok = wait_bounded(smem_u32(&acc_full[0]), 0, abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    if (ok && __any_sync(0xffffffffu, mb * BM + row < p.M)) {
        tc_fence_after();
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        const bool send = mb * BM + row < p.M;  // rows past the output are not sent
#pragma unroll 1
        for (int c = c_begin; c < c_begin + NC / 2; ++c) {
            uint32_t r[32];
            tmem_ld_32cols(t_row + c * 32, r);   // whole warp (.sync.aligned)
            tmem_ld_wait(r);
            if (!send) continue;
            const int owner = (c * 32) / cols;
            const uint32_t al =
                recv + (uint32_t)krank * slice + (uint32_t)((row * ld + c * 32 - owner * cols) * 4);
            if (owner == krank) {                 // own share: local stores
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(al + 16 * j,
                                 make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]));
            } else {
                const uint32_t a = mapa_shared(al, (uint32_t)owner);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_dsmem_v4(a + 16 * j, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            }
        }
    }
    tc_fence_before();
    cluster_sync_all();
    const float *rb = reinterpret_cast<const float *>(recv_buf);
    const int n_items = BM * (cols / 16);
    const int n_out = p.N / 2;                 // output columns (p.N is the 2N-space width)
#pragma unroll 1
    for (int idx = et; idx < n_items; idx += NUM_EPI_THREADS) {
        // consecutive threads take consecutive groups of a row (wider stores)
        const int rr = idx / (cols / 16);
        const int cl = (idx % (cols / 16)) * 16;   // column within this rank's share
        const int m = mb * BM + rr;
        const int n = (nb * BN + krank * cols + cl) / 2;   // first output column
        if (m >= p.M || n >= n_out) continue;
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
#pragma unroll
        for (int r = 0; r < MAX_CLUSTER_SPLITS; ++r) {
            if (r < S) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    rb + (size_t)r * (slice / 4) + rr * ld + cl);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float4 v = src[w];
                    acc[4 * w] += v.x;
                    acc[4 * w + 1] += v.y;
                    acc[4 * w + 2] += v.z;
                    acc[4 * w + 3] += v.w;
                }
            }
        }
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            y[j] = silu_f32(p.alpha * acc[2 * j]) * (p.alpha * acc[2 * j + 1]);
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.D) + (long long)m * p.ldd + n;
        if (n_out - n >= 8) {
            *reinterpret_cast<uint4 *>(dst) =
                make_uint4(pack2(y[0], y[1], OUT_BF16), pack2(y[2], y[3], OUT_BF16),
                           pack2(y[4], y[5], OUT_BF16), pack2(y[6], y[7], OUT_BF16));
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < n_out - n) dst[j] = __float2bfloat16_rn(y[j]);
        }
    }
}

// EPI_STORE_CL (output frame, 128 x BN tile, TMEM lane = row).  Rank r owns
// the tile's columns [r * BN / S, (r + 1) * BN / S); recv[s][row][column -
// r * BN / S] with rows padded by 4 floats sits in the consumed stages, so the
// ranks first pass a cluster barrier once every main loop has finished.  C
// for this rank's outputs is loaded (beta != 0) before the accumulator is
// ready.  For each row and group of 32 columns the owner stores
// alpha * (recv[0] + .. + recv[S-1]) + beta * C, summed in rank order from 0.
template <int BN>
__device__ __forceinline__ void store_cluster_epilogue(const TileParams &p, uint32_t tmem_base,
                                                       uint8_t *recv_buf, uint64_t *acc_full,
                                                       volatile int *abort_flag, int krank, int cid)
{
    constexpr int NC = BN / 32;
    // Output columns per item: a thread loads C, reads each slice and stores
    // D in 64-byte runs.  Measured on the small MLP's down projection (one
    // call, isolated): 53.7-54.0 us with 32 columns, 54.1-54.4 with 16,
    // 55.9-56.3 with 8 and 58.3-58.7 with 4 (conflict-free 16-byte reads):
    // the number of global load and store instructions decides, not the
    // shared-memory bank conflicts of the wider items.
    constexpr int GW = 32;
    // items per thread with S >= 2 (instantiated for BN = 256 only; the
    // floor of one keeps other instantiations of the kernel compilable)
    constexpr int ITEMS_RAW = BM * (BN / 2) / GW / NUM_EPI_THREADS;
    constexpr int ITEMS = ITEMS_RAW > 0 ? ITEMS_RAW : 1;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int et = threadIdx.x - EPI_WARP0 * 32;
    const int S = p.splits;
    const int cols = BN / S;                   // this rank's columns (>= 64)
    const int ld = cols + 4;
    const uint32_t slice = (uint32_t)(BM * ld * 4);
    int mb, nb;
    tile_coords(p, cid, mb, nb);
    const int n_items = BM * (cols / GW);
    // 1. C of this rank's outputs
    float c[ITEMS][GW];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
#pragma unroll
        for (int j = 0; j < GW; ++j) c[it][j] = 0.0f;
        const int idx = et + it * NUM_EPI_THREADS;
        if (p.beta == 0.0f || idx >= n_items) continue;
        // consecutive threads take consecutive groups of a row: whole lines
        const int m = mb * BM + idx / (cols / GW);
        const int n = nb * BN + krank * cols + (idx % (cols / GW)) * GW;
        if (m >= p.M || n >= p.N) continue;
        const long long off = (long long)m * p.ldd + n;
        if (p.N - n >= GW && p.out_kind != OUT_F32) {
            uint32_t ww[GW / 2];
#pragma unroll
            for (int v = 0; v < GW / 8; ++v) {
                const uint4 w = *reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const uint16_t *>(p.D) + off + 8 * v);
                ww[4 * v] = w.x; ww[4 * v + 1] = w.y; ww[4 * v + 2] = w.z; ww[4 * v + 3] = w.w;
            }
#pragma unroll
            for (int h = 0; h < GW / 2; ++h) {
                if (p.out_kind == OUT_F16) {
                    const __half2 c2 = *reinterpret_cast<const __half2 *>(&ww[h]);
                    c[it][2 * h] = __low2float(c2);
                    c[it][2 * h + 1] = __high2float(c2);
                } else {
                    const __nv_bfloat162 c2 = *reinterpret_cast<const __nv_bfloat162 *>(&ww[h]);
                    c[it][2 * h] = __low2float(c2);
                    c[it][2 * h + 1] = __high2float(c2);
                }
            }
        } else if (p.N - n >= GW) {
            const float4 *src = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.D) + off);
#pragma unroll
            for (int h = 0; h < GW / 4; ++h) {
                const float4 a = src[h];
                c[it][4 * h] = a.x; c[it][4 * h + 1] = a.y; c[it][4 * h + 2] = a.z; c[it][4 * h + 3] = a.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < GW; ++j)
                if (j < p.N - n) c[it][j] = load_out(p.D, off + j, p.out_kind);
        }
    }
    // 2. every rank's main loop is over: its stages may receive partials
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int c_begin = ((warp - EPI_WARP0) / 4) * (NC / 2);
    bool ok = wait_bounded(smem_u32(&acc_full[0]), 0, abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    cluster_sync_all();
    const uint32_t recv = smem_u32(recv_buf);
    if (ok && __any_sync(0xffffffffu, mb * BM + row < p.M)) {
        tc_fence_after();
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        const bool send = mb * BM + row < p.M;  // rows past the output are not sent
#pragma unroll 1
        for (int cc = c_begin; cc < c_begin + NC / 2; ++cc) {
            uint32_t r[32];
            tmem_ld_32cols(t_row + cc * 32, r);  // whole warp (.sync.aligned)
            tmem_ld_wait(r);
            if (!send) continue;
            const int owner = (cc * 32) / cols;
            const uint32_t al =
                recv + (uint32_t)krank * slice + (uint32_t)((row * ld + cc * 32 - owner * cols) * 4);
            if (owner == krank) {                 // own share: local stores
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(al + 16 * j,
                                 make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]));
            } else {
                const uint32_t a = mapa_shared(al, (uint32_t)owner);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_dsmem_v4(a + 16 * j, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            }
        }
    }
    tc_fence_before();
    cluster_sync_all();
    // 3. reduce this rank's columns from the local receive buffer
    const float *rb = reinterpret_cast<const float *>(recv_buf);
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int idx = et + it * NUM_EPI_THREADS;
        if (idx >= n_items) continue;
        const int rr = idx / (cols / GW);
        const int cl = (idx % (cols / GW)) * GW;
        const int m = mb * BM + rr;
        const int n = nb * BN + krank * cols + cl;
        if (m >= p.M || n >= p.N) continue;
        float acc[GW];
#pragma unroll
        for (int j = 0; j < GW; ++j) acc[j] = 0.0f;
#pragma unroll
        for (int r = 0; r < MAX_CLUSTER_SPLITS; ++r) {
            if (r < S) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    rb + (size_t)r * (slice / 4) + rr * ld + cl);
#pragma unroll
                for (int h = 0; h < GW / 4; ++h) {
                    const float4 a = src[h];
                    acc[4 * h] += a.x; acc[4 * h + 1] += a.y; acc[4 * h + 2] += a.z; acc[4 * h + 3] += a.w;
                }
            }
        }
        float out[GW];
#pragma unroll
        for (int j = 0; j < GW; ++j)
            out[j] = p.beta != 0.0f ? __fmaf_rn(p.beta, c[it][j], p.alpha * acc[j])
                                    : p.alpha * acc[j];
        const long long off = (long long)m * p.ldd + n;
        if (p.N - n >= GW && p.out_kind != OUT_F32) {
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.D) + off);
#pragma unroll
            for (int v = 0; v < GW / 8; ++v)
                dst[v] = make_uint4(pack2(out[8 * v], out[8 * v + 1], p.out_kind),
                                    pack2(out[8 * v + 2], out[8 * v + 3], p.out_kind),
                                    pack2(out[8 * v + 4], out[8 * v + 5], p.out_kind),
                                    pack2(out[8 * v + 6], out[8 * v + 7], p.out_kind));
        } else if (p.N - n >= GW) {
            float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.D) + off);
#pragma unroll
            for (int h = 0; h < GW / 4; ++h)
                dst[h] = make_float4(out[4 * h], out[4 * h + 1], out[4 * h + 2], out[4 * h + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < GW; ++j)
                if (j < p.N - n) store_out(p.D, off + j, out[j], p.out_kind);
        }
    }
}

// FP8: operands are 8-bit (e4m3/e5m2) and the MMA is kind::f8f6f4.  In bytes
// nothing else changes: a 128-byte swizzled stage row holds 128 elements and
// each MMA (K = 32) consumes 32 bytes of it, as a kind::f16 MMA (K = 16) does.
template <int BN, int EPI, bool PAIR, bool FP8 = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmX, const TileParams p)
{
    using C = Cfg<BN, PAIR, EPI>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzled stages need 1024-byte alignment.
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + S * C::A_BYTES;
    uint8_t *recv = sB + S * C::B_BYTES;     // cluster-reduced K: partials received
    uint64_t *bars = reinterpret_cast<uint64_t *>(recv + C::RECV_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = bars + S;
    uint64_t *acc_full = bars + 2 * S;
    uint64_t *acc_empty = bars + 2 * S + 2;
    uint64_t *mma_done = bars + 2 * S + 4;
    uint64_t *staged = bars + 2 * S + 5;     // last tile written to shared memory
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + C::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Pair mode: rank 0 of the cluster issues the MMAs; work is indexed by
    // cluster, and this CTA owns rows [128*rank, 128*rank + 128) of the tile.
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    // Cluster-reduced K: cluster c is tile c, rank r its K range r (unit r * tiles + c).
    constexpr bool CLK = ClusterK<EPI>::value;
    const int krank = CLK ? (int)cluster_ctarank() : 0;
    const int cid = CLK ? (int)(blockIdx.x >> (p.splits >> 1)) : 0;   // cluster sizes 1, 2, 4
    const int first_unit = PAIR ? (int)(blockIdx.x >> 1) : CLK ? krank * p.tiles + cid
                                                               : (int)blockIdx.x;
    const int unit_step = PAIR ? (int)(gridDim.x >> 1) : CLK ? p.units : (int)gridDim.x;

    // Programmatic dependent launch: the kernel queued behind this one on the
    // stream (the split-K reduction, or the next GEMM of a chain) may be
    // scheduled from now on.  It runs its set-up as SMs free up and then waits
    // (griddepcontrol.wait) until this grid has completed and its writes are
    // visible.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // The kernel parameters sit in constant memory, which a CTA's first
    // access fetches from L2 or DRAM (about half a microsecond measured at
    // the producer's first unit): touch the scheduling fields now, so that
    // miss overlaps the set-up instead of delaying the first loads.
    asm volatile("" ::"r"(p.units), "r"(p.tiles), "r"(p.kb_per_split), "r"(p.k_blocks),
                 "r"(p.group_m), "r"(p.n_blocks), "r"(p.m_blocks), "r"(p.bk));

    if (threadIdx.x == 0) {
        // Tensor maps are fetched from memory on first use: start that now.
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            // one arrival per epilogue warp, from both CTAs in pair mode
            mbar_init(smem_u32(&acc_empty[b]), NUM_EPI_WARPS * (PAIR ? 2 : 1));
        }
        mbar_init(smem_u32(mma_done), 1);
        mbar_init(smem_u32(staged), NUM_EPI_WARPS);
        *abort_flag = 0;
        fence_barrier_init();
        if (EPI == EPI_SWIGLU_DUAL || p.tma_store) tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    // Pair mode: the peer's loads signal the leader's barriers, so both CTAs'
    // barriers must be initialised before either starts.  Single CTA: the
    // producer initialised the barriers itself and needs no tensor memory, so
    // it starts loading at once and only releases the other warps, which
    // wait for the barrier set-up and the TMEM address.
    if (PAIR) {
        cluster_sync_all();
    } else if (warp == 0) {
        __syncwarp();
        named_bar_arrive(2, NUM_THREADS);
    } else {
        named_bar_sync(2, NUM_THREADS);
    }
    tc_fence_after();
    const uint32_t tmem_base = (PAIR || warp != 0) ? *tmem_holder : 0u;
    // Everything above touches only this CTA's own resources and the kernel
    // parameters.  Global memory is read and written only after the grid this
    // one was launched behind (if any) has completed: a no-op without one.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            bool ok = true;
            for (int u = first_unit; u < p.units && ok; u += unit_step) {
                int mb, nb, split, tile;
                if (CLK) {                     // the one unit: K range krank of tile cid
                    split = krank;
                    tile = cid;
                    tile_coords(p, tile, mb, nb);
                } else {
                    unit_coords(p, u, mb, nb, split, tile);
                }
                const int kb0 = split * p.kb_per_split;
                int kb1 = kb0 + p.kb_per_split;
                kb1 = kb1 < p.k_blocks ? kb1 : p.k_blocks;
                const int m0 = mb * C::TILE_M + (int)rank * BM;
                const int n0 = nb * BN + (int)rank * C::B_COLS;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(smem_u32(&empty[stage]), phase ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&full[stage]);
                    uint32_t fb = fb_local;
                    if (PAIR) {
                        // both CTAs' bytes complete on the leader's barrier
                        fb = mapa_shared(fb_local, 0);
                        if (leader) mbar_arrive_expect_tx(fb_local, 2 * C::STAGE_BYTES);
                    } else {
                        mbar_arrive_expect_tx(fb_local, C::STAGE_BYTES);
                    }
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    const uint32_t a_dst = smem_u32(sA + stage * C::A_BYTES);
                    const uint32_t b_dst = smem_u32(sB + stage * C::B_BYTES);
                    const int k0 = kb * p.bk * C::KPS;       // first K element of the stage
                    auto load = [&](uint32_t dst, const CUtensorMap *tm, int x, int y) {
                        if (PAIR)
                            tma_load_2d_pair(dst, tm, fb, x, y);
                        else
                            tma_load_2d(dst, tm, fb, x, y);
                    };
                    auto load3 = [&](uint32_t dst, const CUtensorMap *tm, int y, int z) {
                        if (PAIR)
                            tma_load_3d_pair(dst, tm, fb, 0, y, z);
                        else
                            tma_load_3d(dst, tm, fb, 0, y, z);
                    };
                    // (MN-major boxes span all C::KPS atoms of K rows: {64, 64 KPS, ..})
                    if (!p.a_mn_major) {
#pragma unroll
                        for (int j = 0; j < C::KPS; ++j)                  // box {64 K, 128 M}
                            load(a_dst + j * (BM * 128), &tmA, k0 + j * p.bk, m0);
                    } else if (p.a_mn3) {
                        load3(a_dst, &tmA, k0, m0 / 64);                    // box {64 M, 64 K, 2}
                    } else {
                        load(a_dst, &tmA, m0, k0);                          // box {64 M, 64 K}
                        load(a_dst + 8192 * C::KPS, &tmA, m0 + 64, k0);
                    }
                    if (EPI == EPI_SWIGLU_DUAL) {
                        // W1 / W2 are K x N (N-major), boxes {64 N, 64 K}.  Pair:
                        // this CTA's B_COLS columns come from W1 (rank 0) or
                        // W2 (rank 1); single CTA: BN/2 from each.
                        const int nd = nb * (BN / 2);
                        if (p.b_mn3 && PAIR) {
                            // box {64 N, 64 K, B_COLS / 64} of this CTA's weight
                            load3(b_dst, rank != 0 ? &tmX : &tmB, k0, nd / 64);
                        } else if (p.b_mn3) {
                            // boxes {64 N, 64 K, BN / 128}: Gate atoms, then Up atoms
                            load3(b_dst, &tmB, k0, nd / 64);
                            load3(b_dst + (BN / 128) * 8192, &tmX, k0, nd / 64);
                        } else {
#pragma unroll
                            for (int c = 0; c < C::B_COLS / 64; ++c) {
                                const bool up = PAIR ? (rank != 0) : (c >= BN / 128);
                                const int cc = PAIR ? c : (c % (BN / 128));
                                load(b_dst + c * 8192, up ? &tmX : &tmB, nd + cc * 64, k0);
                            }
                        }
                    } else if (!p.b_mn_major) {
#pragma unroll
                        for (int j = 0; j < C::KPS; ++j)                  // box {64 K, B_COLS N}
                            load(b_dst + j * (C::B_COLS * 128), &tmB, k0 + j * p.bk, n0);
                    } else if (p.b_mn3) {
                        load3(b_dst, &tmB, k0, n0 / 64);                    // box {64 N, 64 K, B_COLS / 64}
                    } else {
#pragma unroll
                        for (int c = 0; c < C::B_COLS / 64; ++c)            // box {64 N, 64 K}
                            load(b_dst + c * 8192 * C::KPS, &tmB, n0 + c * 64, k0);
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // Never leave with loads in flight into this CTA's shared memory.
            if (!PAIR || leader) {
                for (int s = 0; s < S; ++s)
                    if (armed & (1u << s))
                        wait_bounded(smem_u32(&full[s]), (armed_parity >> s) & 1, abort_flag,
                                     p.err, false, DRAIN_LIMIT_NS);
            } else if (!ok) {
                // The peer's loads complete on the leader's barriers, which
                // it cannot poll; after an abort give them time to land.
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 200000ull) {
                }
            }
        }
        __syncwarp();
        if (CLK) {                     // (see the cluster epilogues)
            for (int b = 0; b < ClusterK<EPI>::barriers; ++b) cluster_sync_all();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && leader) {
            // K-major operand: next K=16 slice is 32 bytes further in the
            // swizzled row; MN-major: two 8-row K groups (2 x 1024 bytes) further.
            // With C::KPS > 1 a K-major operand's atoms follow each other
            // (rows x 128 bytes apart); an MN-major atom holds 64 KPS K rows.
            const uint32_t a_kstep = p.a_mn_major ? 2048u : 32u;
            const uint32_t b_kstep = p.b_mn_major ? 2048u : 32u;
            const uint32_t a_lbo = p.a_mn_major ? 8192u * C::KPS : 16u;
            const uint32_t b_lbo = p.b_mn_major ? 8192u * C::KPS : 16u;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int t = 0;
            for (int u = first_unit; u < p.units && ok; u += unit_step, ++t) {
                int mb, nb, split, tile;
                unit_coords(p, u, mb, nb, split, tile);
                const int kb0 = split * p.kb_per_split;
                int kb1 = kb0 + p.kb_per_split;
                kb1 = kb1 < p.k_blocks ? kb1 : p.k_blocks;
                const int acc = t & 1;
                const uint32_t acc_phase = (t >> 1) & 1;
                if (!wait_bounded(smem_u32(&acc_empty[acc]), acc_phase ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(smem_u32(&full[stage]), phase, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + stage * C::A_BYTES);
                    const uint32_t b_base = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < C::KPS * (BK / UMMA_K); ++kk) {
                        const int j = kk / (BK / UMMA_K), kq = kk % (BK / UMMA_K);
                        const uint32_t a_off = p.a_mn_major ? kk * a_kstep
                                                            : j * (BM * 128) + kq * a_kstep;
                        const uint32_t b_off = p.b_mn_major ? kk * b_kstep
                                                            : j * (C::B_COLS * 128) + kq * b_kstep;
                        const uint64_t ad = smem_desc(a_base + a_off, a_lbo, 1024);
                        const uint64_t bd = smem_desc(b_base + b_off, b_lbo, 1024);
                        const uint32_t accum = (kb > kb0 || kk > 0) ? 1u : 0u;
                        if (PAIR && FP8)
                            tc_mma_f8_pair(d_tmem, ad, bd, p.idesc, accum);
                        else if (PAIR)
                            tc_mma_f16_pair(d_tmem, ad, bd, p.idesc, accum);
                        else if (FP8)
                            tc_mma_f8(d_tmem, ad, bd, p.idesc, accum);
                        else
                            tc_mma_f16(d_tmem, ad, bd, p.idesc, accum);
                    }
                    if (PAIR)
                        tc_commit_pair(smem_u32(&empty[stage]));
                    else
                        tc_commit(smem_u32(&empty[stage]));
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if (PAIR)
                    tc_commit_pair(smem_u32(&acc_full[acc]));
                else
                    tc_commit(smem_u32(&acc_full[acc]));
            }
            // Never free TMEM under a running MMA.
            if (PAIR)
                tc_commit_pair_local(smem_u32(mma_done));
            else
                tc_commit(smem_u32(mma_done));
            wait_bounded(smem_u32(mma_done), 0, abort_flag, p.err, false, DRAIN_LIMIT_NS);
        }
        __syncwarp();
        if (CLK) {                     // (see the cluster epilogues)
            for (int b = 0; b < ClusterK<EPI>::barriers; ++b) cluster_sync_all();
        }
    } else if (EPI == EPI_SPLITK_CL) {
        splitk_cluster_epilogue<BN>(p, tmem_base, recv, acc_full, abort_flag, first_unit, krank);
    } else if (EPI == EPI_SWIGLU_CL) {
        swiglu_cluster_epilogue<BN>(p, tmem_base, recv, acc_full, abort_flag, first_unit, krank);
    } else if (EPI == EPI_STORE_CL) {
        // the partials go to the consumed stages (at most 139 KB of 192 KB)
        store_cluster_epilogue<BN>(p, tmem_base, smem, acc_full, abort_flag, krank, cid);
    } else if (EPI == EPI_SWIGLU_DUAL) {
        // ------------------------------------------ epilogue (separate W1, W2)
        // Output column j of the tile = SiLU(acc[j]) * acc[BN/2 + j]; warps
        // 2..5 take output columns [0, BN/4), warps 6..9 [BN/4, BN/2).
        constexpr int HALF = BN / 2;
        constexpr int PER_WARP = HALF / 2;     // instantiated for BN = 128, 256 only
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int h = (warp - EPI_WARP0) / 4;
        int t = 0;
        for (int u = first_unit; u < p.units; u += unit_step, ++t) {
            int mb, nb, split, tile;
            unit_coords(p, u, mb, nb, split, tile);
            const int acc = t & 1;
            const uint32_t acc_phase = (t >> 1) & 1;
            bool ok = wait_bounded(smem_u32(&acc_full[acc]), acc_phase, abort_flag, p.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            const int m = mb * C::TILE_M + (int)rank * BM + row;
#pragma unroll 1
            for (int c = 0; c < PER_WARP / 32; ++c) {
                const int j0 = h * PER_WARP + c * 32;
                uint32_t g[32], v[32];
                tmem_ld_32cols(t_row + j0, g);
                tmem_ld_32cols(t_row + HALF + j0, v);
                tmem_ld_wait(g);
                tmem_ld_wait(v);
                const int n = nb * HALF + j0;                   // output column
                if (m < p.M && n < p.N) {
                    const int cnt = (p.N - n) < 32 ? (p.N - n) : 32;
                    float y[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        y[j] = silu_f32(__uint_as_float(g[j])) * __uint_as_float(v[j]);
                    __nv_bfloat16 *dst =
                        reinterpret_cast<__nv_bfloat16 *>(p.D) + (long long)m * p.ldd + n;
                    if (cnt == 32) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                        for (int w = 0; w < 4; ++w)
                            d4[w] = make_uint4(pack2(y[8 * w], y[8 * w + 1], OUT_BF16),
                                               pack2(y[8 * w + 2], y[8 * w + 3], OUT_BF16),
                                               pack2(y[8 * w + 4], y[8 * w + 5], OUT_BF16),
                                               pack2(y[8 * w + 6], y[8 * w + 7], OUT_BF16));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < cnt) dst[j] = __float2bfloat16_rn(y[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR)
                    mbar_arrive_remote_tmem(mapa_shared(smem_u32(&acc_empty[acc]), 0));
                else
                    mbar_arrive(smem_u32(&acc_empty[acc]));
            }
        }
    } else if (EPI == EPI_SPLITK_T) {
        // ------------------------------------------------- epilogue (swapped)
        // TMEM lane = output column n (kernel row), TMEM column j = output row
        // m (kernel column).  BN <= 32: warps 2..5 read all BN columns; BN = 64:
        // warps 2..5 take columns 0..31 and warps 6..9 columns 32..63.
        constexpr int W = BN >= 32 ? 32 : 16;
        const int q = warp & 3;
        const int h = (warp - EPI_WARP0) / 4;
        const bool active = (BN == 64) || h == 0;
        const int j0 = BN == 64 ? h * 32 : 0;
        int t = 0;
        for (int u = first_unit; u < p.units; u += unit_step, ++t) {
            int mb, nb, split, tile;
            unit_coords(p, u, mb, nb, split, tile);
            const int acc = t & 1;
            const uint32_t acc_phase = (t >> 1) & 1;
            bool ok = wait_bounded(smem_u32(&acc_full[acc]), acc_phase, abort_flag, p.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            if (active) {
                uint32_t r[W];
                tmem_ld_cols(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + j0, r);
                tmem_ld_wait(r);
                const int n = mb * BM + q * 32 + lane;          // output column
                if (n < p.M) {
#pragma unroll
                    for (int j = 0; j < W; ++j) {
                        const int m = nb * BN + j0 + j;         // output row
                        if (m < p.N)
                            p.ws[((long long)split * p.N + m) * p.ld_ws + n] = __uint_as_float(r[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[acc]));
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp w may only read TMEM lanes 32*(w%4) .. 32*(w%4)+31; warps 2..5
        // take the first half of the tile's 32-column chunks, warps 6..9 the
        // second half.
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int row = q * 32 + lane;
        constexpr int NC = BN / 32;             // 32-column chunks per tile (>= 2)
        const int c_begin = ((warp - EPI_WARP0) / 4) * (NC / 2);
        const int c_end = c_begin + NC / 2;
        int t = 0;
        for (int u = first_unit; u < p.units; u += unit_step, ++t) {
            int mb, nb, split, tile;
            unit_coords(p, u, mb, nb, split, tile);
            const int acc = t & 1;
            const uint32_t acc_phase = (t >> 1) & 1;
            bool ok = wait_bounded(smem_u32(&acc_full[acc]), acc_phase, abort_flag, p.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            const int m = mb * C::TILE_M + (int)rank * BM + row;
            const bool row_ok = m < p.M;
            // The CTA's last tile goes through shared memory (see
            // stage_epi_chunk); earlier tiles overlap the next main loop and
            // are stored directly.
            const bool stage_out = p.tma_store && u + unit_step >= p.units;
            const uint32_t sbase = smem_u32(smem);
            auto emit = [&](const uint32_t(&r)[32], int c) {
                if (stage_out)
                    stage_epi_chunk<EPI>(p, r, sbase, row, c * 32);
                else if (row_ok)
                    epi_chunk<EPI>(p, r, m, nb * BN + c * 32, split);
            };
            // Two register buffers: the load of chunk c+1 is in flight while
            // chunk c is converted and stored (tcgen05.wait::ld waits for all
            // earlier loads, so each wait retires exactly the older chunk).
            uint32_t ra[32], rb[32];
            tmem_ld_32cols(t_row + c_begin * 32, ra);
#pragma unroll 1
            for (int c = c_begin; c < c_end; c += 2) {
                tmem_ld_wait(ra);
                if (c + 1 < c_end) tmem_ld_32cols(t_row + (c + 1) * 32, rb);
                emit(ra, c);
                if (c + 1 < c_end) {
                    tmem_ld_wait(rb);
                    if (c + 2 < c_end) tmem_ld_32cols(t_row + (c + 2) * 32, ra);
                    emit(rb, c + 1);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (stage_out) {
                // This warp's rows are staged: publish them to the TMA (async
                // proxy) and count the warp in.  Warp 2's lane 0 waits, with
                // a bound, for all eight warps and issues the stores.
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(staged));
                if (warp == EPI_WARP0 && lane == 0 &&
                    wait_bounded(smem_u32(staged), 0, abort_flag, p.err))
                    store_staged<EPI, BN>(p, &tmX, sbase, mb * C::TILE_M + (int)rank * BM, nb,
                                          split);
                __syncwarp();
            }
            // Accumulator drained: hand it back to the MMA warp (the leader's
            // barrier in pair mode), one arrival per warp.
            if (lane == 0) {
                if (PAIR)
                    mbar_arrive_remote_tmem(mapa_shared(smem_u32(&acc_empty[acc]), 0));
                else
                    mbar_arrive(smem_u32(&acc_empty[acc]));
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    // Pair mode: neither CTA may free its tensor memory or exit while the
    // leader's MMAs or the peer's arrivals can still reach it.  (Cluster-
    // reduced K: after the cluster barrier of the epilogue nothing reaches
    // another CTA's shared memory any more.)
    if (PAIR)
        cluster_sync_all();
    else
        __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        if (PAIR)
            tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace swg
