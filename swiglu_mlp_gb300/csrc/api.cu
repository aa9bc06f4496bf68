// api.cu — the C ABI declared in include/swiglu_mlp.h: argument validation,
// tile/split selection, tensor-map encoding, library-owned workspace, and the
// two small auxiliary kernels (K == 0 scaling, weight interleave).
//
// Validation happens before any CUDA call, so a rejected call has no side
// effects and the checks run on machines without a GPU.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <vector>

#include "swiglu_mlp.h"
#include "launch.h"

namespace {

using swg::TileParams;

// Why this thread's most recent call failed with SWG_ERR_CUDA: the CUDA
// runtime error, or 10000 + the driver result of a failed tensor-map encoding.
thread_local int t_last_cuda_error = 0;

// Records the runtime's pending error of this thread (if any) and returns
// SWG_ERR_CUDA.
int cuda_fail()
{
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) t_last_cuda_error = (int)e;
    return SWG_ERR_CUDA;
}

// The calling thread's current device, with that device's primary context
// made current to the thread (once per thread and device): the tensor-map
// encoder is a driver call and fails without a current context, which a
// thread that has made no runtime call yet does not have.
int current_device(int &dev)
{
    thread_local int t_bound = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();
    if (t_bound != dev) {
        if (cudaSetDevice(dev) != cudaSuccess) return cuda_fail();
        t_bound = dev;
    }
    return SWG_OK;
}

// SWG_OK if the launches just made left no error, else SWG_ERR_CUDA (recorded).
int launch_status()
{
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return SWG_OK;
    t_last_cuda_error = (int)e;
    return SWG_ERR_CUDA;
}

std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;

}  // namespace

namespace swg {
std::atomic<unsigned> g_setup_epoch{0};
}

void noalloc_forget();

namespace {

// Device error word: written by kernels whose bounded waits ran out.
__device__ int g_err_word;

constexpr int64_t kMaxDim = 0x7fffffff;

// ----------------------------------------------------------------- dtypes

struct TypeInfo {
    bool in_bf16;    // A, B bfloat16 (else binary16)
    int out_kind;    // swg::OutKind
    int out_bytes;
};

bool type_info(int dtype, TypeInfo &t)
{
    switch (dtype) {
    case SWG_F16_F32OUT: t = {false, swg::OUT_F32, 4}; return true;
    case SWG_BF16: t = {true, swg::OUT_BF16, 2}; return true;
    case SWG_F16: t = {false, swg::OUT_F16, 2}; return true;
    case SWG_BF16_F32OUT: t = {true, swg::OUT_F32, 4}; return true;
    default: return false;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ----------------------------------------------------------------- per device

struct Workspace {
    void *base = nullptr;   // split-K FP32 partials
    size_t bytes = 0;
    void *raw = nullptr;    // the allocation: base, or base - kGuardBytes with guards
    // Smaller workspaces this one replaced (their raw allocations).  Work
    // already queued, or a CUDA graph captured earlier, may still address
    // them, so they are freed only by swg_shutdown.
    std::vector<void *> retired;
};

// Test switch SWG_TEST_WS_GUARD=1: every split-K workspace (and the fixed
// array of gemm_splitk_noalloc) gets kGuardBytes of kGuardByte before and
// after it, which swg_debug_workspace_guards checks.  A kernel that wrote
// past either end of its partials would change them.
constexpr size_t kGuardBytes = 64 * 1024;
constexpr unsigned char kGuardByte = 0xA5;

bool ws_guards_enabled()
{
    const char *v = std::getenv("SWG_TEST_WS_GUARD");
    return v && v[0] == '1';
}

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int *err = nullptr;                          // address of g_err_word
    std::map<cudaStream_t, Workspace> ws;
    std::map<int, int> max_pairs;                // (kind, bn) -> resident CTA pairs
};

std::map<int, DeviceState> g_dev;

int device_state(DeviceState *&out)
{
    int dev = 0;
    if (int rc = current_device(dev)) return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cuda_fail();
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return cuda_fail();
        d.err = static_cast<int *>(p);
        d.ready = true;
    }
    out = &d;
    return SWG_OK;
}

// Grow-only split-K workspace for (device, stream).  Only the stream that
// owns it uses it, so stream order keeps calls from overlapping.
int workspace(DeviceState *d, cudaStream_t s, size_t bytes, Workspace *&out)
{
    if (std::getenv("SWG_TEST_FAIL_ALLOC")) return SWG_ERR_NO_MEMORY;
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = d->ws[s];
    if (w.base == nullptr || w.bytes < bytes) {
        // No allocation while the stream is being captured into a graph:
        // the caller runs the call once before capturing.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return cuda_fail();
        if (cs != cudaStreamCaptureStatusNone) return SWG_ERR_UNSUPPORTED;
        const bool guards = ws_guards_enabled();
        const size_t extra = guards ? 2 * kGuardBytes : 0;
        void *p = nullptr;
        if (cudaMalloc(&p, bytes + extra) != cudaSuccess) {
            cudaGetLastError();
            return SWG_ERR_NO_MEMORY;
        }
        if (guards) {
            uint8_t *b = static_cast<uint8_t *>(p);
            if (cudaMemsetAsync(b, kGuardByte, kGuardBytes, s) != cudaSuccess ||
                cudaMemsetAsync(b + kGuardBytes + bytes, kGuardByte, kGuardBytes, s) !=
                    cudaSuccess) {
                cudaFree(p);
                return cuda_fail();
            }
        }
        if (w.raw) w.retired.push_back(w.raw);
        w.raw = p;
        w.base = static_cast<uint8_t *>(p) + (guards ? kGuardBytes : 0);
        w.bytes = bytes;
    }
    out = &w;
    return SWG_OK;
}

// Where a split-K call's FP32 partials go: the (device, stream) workspace
// above, or -- for gemm_splitk_noalloc -- a fixed array of `bytes` bytes at
// `base` that belongs to the library's device image.
struct FixedScratch {
    float *base;
    size_t bytes;
};

int split_workspace(DeviceState *d, cudaStream_t s, size_t bytes, const FixedScratch *fx,
                    float *&out)
{
    if (fx) {
        if (bytes > fx->bytes) return SWG_ERR_UNSUPPORTED;   // partials would not fit
        out = fx->base;
        return SWG_OK;
    }
    Workspace *w = nullptr;
    if (int rc = workspace(d, s, bytes, w)) return rc;
    out = static_cast<float *>(w->base);
    return SWG_OK;
}

// The fixed array of gemm_splitk_noalloc on the current device (defined at
// the end of this file); called after argument validation.
int noalloc_scratch(cudaStream_t s, FixedScratch &out);

// Tuning and testing: SWG_MN_3D=0 keeps two 2-D boxes per MN-major operand
// and stage instead of one 3-D box.
bool mn_3d_disabled()
{
    const char *v = std::getenv("SWG_MN_3D");
    return v && v[0] == '0';
}

// ----------------------------------------------------------------- tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major matrix of `outer` rows x `inner` contiguous 16-bit elements with
// row stride `ld`, read in boxes of 64 x box_outer with the 128-byte swizzle.
// Rows/columns past the matrix read as zero.
bool make_tmap(CUtensorMap *m, const void *ptr, bool bf16, int64_t inner, int64_t outer,
               int64_t ld, int box_outer)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        t_last_cuda_error = 10000 + (int)CUDA_ERROR_NOT_FOUND;
        return false;
    }
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_outer};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) t_last_cuda_error = 10000 + (int)r;
    return r == CUDA_SUCCESS;
}

// MN-major operand whose MN extent `mn` is a multiple of 64, viewed in 3-D
// as (64 contiguous MN elements, K rows at the row stride, mn / 64 atoms 128
// bytes apart): one box of {64, kbox, atoms} fills `atoms` consecutive
// (kbox x 128-byte) swizzle atoms of a stage, the layout separate 2-D
// {64, kbox} boxes give, with one TMA instruction.  Rows past K read as zero; with mn a multiple of 64 no box
// reaches past a row's last element.  Returns false (and the caller keeps the
// 2-D map) if the driver declines the encoding.
bool make_tmap_mn3(CUtensorMap *m, const void *ptr, bool bf16, int64_t mn, int64_t k, int64_t ld,
                   int atoms, int kbox = 64)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || mn % 64 != 0 || mn_3d_disabled()) return false;
    cuuint64_t dims[3] = {64u, (cuuint64_t)k, (cuuint64_t)(mn / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128u};
    cuuint32_t box[3] = {64u, (cuuint32_t)kbox, (cuuint32_t)atoms};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major matrix of 8-bit elements (e4m3), boxes of 128 x box_outer: one
// 128-byte swizzle row per box row, as for the 16-bit maps.
bool make_tmap_u8(CUtensorMap *m, const void *ptr, int64_t inner, int64_t outer, int64_t ld,
                  int box_outer)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        t_last_cuda_error = 10000 + (int)CUDA_ERROR_NOT_FOUND;
        return false;
    }
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_outer};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) t_last_cuda_error = 10000 + (int)r;
    return r == CUDA_SUCCESS;
}

// Output map of the staged last-tile stores: `cols` x `rows` elements of
// `esize` (2 or 4) bytes with a row stride of `ld` elements -- and with
// `depth` > 0, a third dimension of that many slices `dstride` elements
// apart (the split-K workspace).  Box: 128 bytes x 128 rows, 128-byte swizzle.
// Stores are clipped at the map's bounds, but along a row only at 16-byte
// granules: callers use the map only where cols * esize is a multiple of 16
// or the row's padding up to the next granule is scratch.
bool make_tmap_store(CUtensorMap *m, void *ptr, int esize, int64_t cols, int64_t rows, int64_t ld,
                     int64_t depth = 0, int64_t dstride = 0)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        t_last_cuda_error = 10000 + (int)CUDA_ERROR_NOT_FOUND;
        return false;
    }
    const cuuint32_t rank = depth > 0 ? 3u : 2u;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)(depth > 0 ? depth : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * esize), (cuuint64_t)(dstride * esize)};
    cuuint32_t box[3] = {(cuuint32_t)(128 / esize), 128u, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(m, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                    rank, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) t_last_cuda_error = 10000 + (int)r;
    return r == CUDA_SUCCESS;
}

// tcgen05 instruction descriptor, kind::f16: D=F32 (bits 4-5 = 1), A/B type
// (bits 7-9, 10-12: 0 = f16, 1 = bf16), A/B major (bits 15, 16: 1 = MN-major),
// N >> 3 (bits 17-22), M >> 4 (bits 24-28).  With bf16 = false the same
// bits describe kind::f8f6f4 with e4m3 A and B (format code 0).
uint32_t make_idesc(bool bf16, bool a_mn, bool b_mn, int m, int n)
{
    const uint32_t t = bf16 ? 1u : 0u;
    return (1u << 4) | (t << 7) | (t << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tile width with the best last-wave fill; ties and near-ties keep the wider
// tile (more operand reuse per byte loaded).
int pick_bn(int64_t M, int64_t N, int sms, const int *cands, int ncand)
{
    int best = cands[0];
    double best_score = -1.0;
    for (int i = 0; i < ncand; ++i) {
        const int bn = cands[i];
        const int64_t tiles = cdiv(M, swg::BM) * cdiv(N, bn);
        const int64_t waves = cdiv(tiles, sms);
        double eff = double(tiles) / double(waves * sms);
        // Narrow tiles re-read A more often; only take one for a clear gain.
        const double penalty = bn == 256 ? 1.0 : bn == 128 ? 0.90 : 0.80;
        const double score = eff * penalty;
        if (score > best_score + 1e-9) {
            best_score = score;
            best = bn;
        }
    }
    return best;
}

// Resident CTA pairs of a pair kernel (kind 0 = GEMM store, 1 = SwiGLU,
// 2 = split-K partials, 3 = SwiGLU from separate weights, 4 = FP8 GEMM,
// 5 = FP8 SwiGLU).
int max_pairs(DeviceState *d, int kind, int bn)
{
    const int key = kind * 1024 + bn;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = d->max_pairs.find(key);
        if (it != d->max_pairs.end()) return it->second;
    }
    const int n = kind == 0   ? swg::max_active_pairs_store(bn, d->sms)
                  : kind == 1 ? swg::max_active_pairs_swiglu(bn, d->sms)
                  : kind == 2 ? swg::max_active_pairs_splitk(bn, d->sms)
                  : kind == 3 ? swg::max_active_pairs_dual(bn, d->sms)
                  : kind == 4 ? swg::max_active_pairs_fp8(0, bn, d->sms)
                              : swg::max_active_pairs_fp8(1, bn, d->sms);
    std::lock_guard<std::mutex> lk(g_mu);
    d->max_pairs[key] = n;
    return n;
}

// Resident clusters of `csize` CTAs of a cluster-reduced split kernel
// (kind 0 = few-rows GEMM, 1 = the same with e4m3, 2 = SwiGLU, 3 = GEMM
// tiles of 128 x 256), cached per device like max_pairs.
int max_clusters(DeviceState *d, int kind, int bn, int csize)
{
    const int key = (16 + kind) * 65536 + bn * 16 + csize;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = d->max_pairs.find(key);
        if (it != d->max_pairs.end()) return it->second;
    }
    const int n = kind == 0   ? swg::max_active_clusters_splitk_cl(bn, csize, d->sms)
                  : kind == 1 ? swg::max_active_clusters_splitk_cl_fp8(bn, csize, d->sms)
                  : kind == 2 ? swg::max_active_clusters_swiglu_cl(bn, csize, d->sms)
                              : swg::max_active_clusters_store_cl(csize, d->sms);
    std::lock_guard<std::mutex> lk(g_mu);
    d->max_pairs[key] = n;
    return n;
}

// Tile mode override for tests and tuning: SWG_TILE_MODE=1cta forces
// single-CTA 128-row tiles, =2cta forces CTA-pair 256-row tiles, =2cta128
// and =2cta256 also fix the pair tile's width.
int forced_tile_mode(int *pair_bn)
{
    const char *v = std::getenv("SWG_TILE_MODE");
    *pair_bn = 0;
    if (!v) return 0;
    if (v[0] == '1') return 1;
    if (v[0] == '2') {
        *pair_bn = std::atoi(v + 4);   // "2cta" -> 0, "2cta128" -> 128
        return 2;
    }
    return 0;
}

struct TileChoice {
    bool pair = false;
    int bn = 256;
    int units = 0;      // CTAs (single) or CTA pairs (pair) to launch
};

// Chooses single-CTA or CTA-pair tiles and the tile width for an output of
// M x N (N in the tile-column space), by last-wave fill; pairs halve the B
// operand each SM loads, so they win ties and are used whenever M > 128.
TileChoice choose_tiles(DeviceState *d, int kind, int64_t M, int64_t N, const int *single_bns,
                        int n_single)
{
    TileChoice c;
    int only_bn = 0;
    const int mode = forced_tile_mode(&only_bn);
    bool try_pair = (M > swg::BM && mode != 1) || mode == 2;
    if (try_pair) {
        // 128-wide pair tiles measured well below 256-wide ones (they load
        // 24 KB per 256 MMA cycles), so only a forced mode selects them.
        static const int pair_bns_auto[] = {256};
        static const int pair_bns_forced[] = {256, 128};
        const int *pair_bns = only_bn ? pair_bns_forced : pair_bns_auto;
        const int n_pair_bns = only_bn ? 2 : 1;
        double best = -1.0;
        for (int i = 0; i < n_pair_bns; ++i) {
            const int bn = pair_bns[i];
            if (only_bn && bn != only_bn) continue;
            const int slots = max_pairs(d, kind, bn);
            if (slots <= 0) continue;
            const int64_t tiles = cdiv(M, 2 * swg::BM) * cdiv(N, bn);
            const int64_t waves = cdiv(tiles, slots);
            const double eff = double(tiles) / double(waves * slots);
            const double score = eff * (bn == 256 ? 1.0 : 0.9);
            if (score > best + 1e-9) {
                best = score;
                c.pair = true;
                c.bn = bn;
                c.units = (int)std::min<int64_t>(tiles, slots);
            }
        }
        if (c.pair) return c;
    }
    c.bn = pick_bn(M, N, d->sms, single_bns, n_single);
    c.units = (int)std::min<int64_t>(cdiv(M, swg::BM) * cdiv(N, c.bn), d->sms);
    return c;
}

// SWG_CLUSTER_SPLITK=0 keeps automatic few-rows splits on the workspace path
// (tests compare the two reductions).
bool cluster_splitk_disabled()
{
    const char *v = std::getenv("SWG_CLUSTER_SPLITK");
    return v && v[0] == '0';
}

// Split-K GEMM with swapped operands for M <= 64: the kernel computes
// D^T = op(B)^T op(A)^T with op(B)^T (N x K) as its 128-row operand and
// op(A)^T as its BN-column operand.  With an automatic split the K ranges of
// a tile run as one thread-block cluster that reduces them itself (one
// launch, EPI_SPLITK_CL); otherwise the kernel writes transposed FP32
// partials ws[split][m][n] and the usual in-order reduction forms D.
// With fp8 (e4m3 A and B; op(A) = A and op(B) = B^T, both K-major) the
// K blocks are 128 elements, the same 128-byte rows, and the MMA is
// kind::f8f6f4; everything else is shared.
int splitk_swapped(DeviceState *d, const TypeInfo &ti, int transA, int transB, int64_t M,
                   int64_t N, int64_t K, float alpha, const void *A, int64_t lda, const void *B,
                   int64_t ldb, float beta, void *C, int64_t ldc, int split_k, cudaStream_t s,
                   bool fp8, const FixedScratch *fx)
{
    const int bk = fp8 ? 128 : swg::BK;
    const int64_t kb = cdiv(K, bk);
    // op(A)^T is the kernel's B operand: K-major when A is stored M x K
    // (op N), MN-major (one 64-wide atom) when stored K x M (op T).
    const bool bT_mn = transA == SWG_OP_T;
    const int bn = bT_mn ? 64 : (M <= 16 ? 16 : M <= 32 ? 32 : 64);
    const int64_t tiles = cdiv(N, swg::BM) * cdiv(M, bn);
    int splits;
    if (split_k == 0)
        splits = (int)std::min<int64_t>(std::max<int64_t>(d->sms / tiles, 1), std::max<int64_t>(kb / 4, 1));
    else
        splits = (int)std::min<int64_t>(split_k, kb);
    splits = std::max(1, std::min(splits, swg::MAX_SPLITS));
    const int kbps = (int)cdiv(kb, splits);
    splits = (int)cdiv(kb, kbps);

    // Automatic split: the K ranges of a tile run as one thread-block cluster
    // whose CTAs sum their partials through shared memory -- one launch, no
    // workspace.  Cluster size: the largest of 4, 2, 1 whose clusters are all
    // resident at once (one per tile) and whose ranges are at least 4 K
    // blocks.  Used when it gives as many ranges as the workspace path would,
    // or at least half the SMs; otherwise (small N) the workspace path
    // splits K further.
    int cl = 0;
    if (split_k == 0 && !cluster_splitk_disabled()) {
        int S = 1;
        while (S < swg::MAX_CLUSTER_SPLITS && tiles * 2 * S <= d->sms && kb >= 8 * S &&
               tiles <= max_clusters(d, fp8 ? 1 : 0, bn, 2 * S))
            S *= 2;
        // (64-row tiles keep at most 16 rows of the reduction per rank)
        if ((S == splits || tiles * S * 2 >= d->sms) && S * 32 >= bn) cl = S;
    }
    // K atoms (128 bytes of K) per pipeline stage: two on the cluster path
    // (MN-major boxes then span 128 K rows), one on the workspace path.
    const int kps = cl > 0 ? 2 : 1;

    // op(B)^T is the kernel's A operand: MN-major when B is stored K x N (op N).
    const bool aT_mn = transB == SWG_OP_N;
    CUtensorMap ta, tb;
    bool ok;
    if (fp8) {
        ok = make_tmap_u8(&ta, B, K, N, ldb, swg::BM) && make_tmap_u8(&tb, A, K, M, lda, bn);
    } else {
        ok = aT_mn ? make_tmap(&ta, B, ti.in_bf16, N, K, ldb, 64 * kps)
                   : make_tmap(&ta, B, ti.in_bf16, K, N, ldb, swg::BM);
        ok = ok && (bT_mn ? make_tmap(&tb, A, ti.in_bf16, M, K, lda, 64 * kps)
                          : make_tmap(&tb, A, ti.in_bf16, K, M, lda, bn));
    }
    if (!ok) return cuda_fail();
    // MN-major operands: one 3-D box per stage where the extent allows.
    CUtensorMap t3;
    const bool a3 =
        !fp8 && aT_mn && make_tmap_mn3(&t3, B, ti.in_bf16, N, K, ldb, swg::BM / 64, 64 * kps);
    if (a3) ta = t3;
    const bool b3 = !fp8 && bT_mn && make_tmap_mn3(&t3, A, ti.in_bf16, M, K, lda, bn / 64, 64 * kps);
    if (b3) tb = t3;

    TileParams p{};           // in the kernel's (transposed) frame
    p.a_mn3 = a3;
    p.b_mn3 = b3;
    p.M = (int)N;
    p.N = (int)M;
    p.K = (int)K;
    p.m_blocks = (int)cdiv(N, swg::BM);
    p.n_blocks = (int)cdiv(M, bn);
    p.k_blocks = (int)kb;
    p.bk = bk;
    p.tiles = p.m_blocks * p.n_blocks;
    p.group_m = 16;
    p.idesc = make_idesc(fp8 ? false : ti.in_bf16, aT_mn, bT_mn, swg::BM, bn);
    p.a_mn_major = aT_mn;
    p.b_mn_major = bT_mn;
    p.err = d->err;

    if (cl > 0) {
        // K is walked in stages of kps atoms: k_blocks counts stages
        const int64_t ks = cdiv(K, (int64_t)bk * kps);
        p.k_blocks = (int)ks;
        p.splits = cl;
        p.kb_per_split = (int)cdiv(ks, cl);
        p.units = p.tiles * cl;
        // every rank has at least one stage (ranges of >= 4 atoms guarantee it)
        if ((int64_t)(cl - 1) * p.kb_per_split >= ks) return SWG_ERR_UNSUPPORTED;
        p.alpha = alpha;
        p.beta = beta;
        p.D = C;
        p.ldd = ldc;
        p.out_kind = ti.out_kind;
        if ((fp8 ? swg::launch_tc_splitk_cl_fp8(bn, ta, tb, p, p.units, s)
                 : swg::launch_tc_splitk_cl(bn, ta, tb, p, p.units, s)) != cudaSuccess)
            return cuda_fail();
        g_launches++;
        return SWG_OK;
    }

    const int64_t ld_ws = cdiv(N, 4) * 4;
    float *ws = nullptr;
    if (int rc = split_workspace(d, s, sizeof(float) * (size_t)splits * (size_t)M * (size_t)ld_ws,
                                 fx, ws))
        return rc;

    p.splits = splits;
    p.kb_per_split = kbps;
    p.units = p.tiles * splits;
    p.ws = ws;
    p.ld_ws = ld_ws;
    const int grid = (int)std::min<int64_t>(p.units, d->sms);
    if ((fp8 ? swg::launch_tc_splitk_t_fp8(bn, ta, tb, p, grid, s)
             : swg::launch_tc_splitk_t(bn, ta, tb, p, grid, s)) != cudaSuccess)
        return cuda_fail();
    g_launches++;

    TileParams r{};           // the reduction works in the output's frame
    r.M = (int)M;
    r.N = (int)N;
    r.splits = splits;
    r.alpha = alpha;
    r.beta = beta;
    r.D = C;
    r.ldd = ldc;
    r.out_kind = ti.out_kind;
    r.ws = p.ws;
    r.ld_ws = ld_ws;
    if (swg::launch_splitk_reduce(r, d->sms, s) != cudaSuccess) return cuda_fail();
    g_launches++;
    return SWG_OK;
}

// GEMM over 128 x 256 tiles with the K range of each tile split over a
// cluster of S CTAs (EPI_STORE_CL): the ranks exchange their FP32 partials
// through shared memory and each stores alpha * sum + beta * C for its share
// of the tile's columns, summed in rank order.
int gemm_store_cluster(DeviceState *d, const TypeInfo &ti, int transA, int transB, int64_t M,
                       int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                       const void *B, int64_t ldb, float beta, void *C, int64_t ldc, int S,
                       cudaStream_t s)
{
    const bool a_mn = transA == SWG_OP_T;
    const bool b_mn = transB == SWG_OP_N;
    CUtensorMap ta, tb, t3;
    bool ok = a_mn ? make_tmap(&ta, A, ti.in_bf16, M, K, lda, 64)
                   : make_tmap(&ta, A, ti.in_bf16, K, M, lda, swg::BM);
    ok = ok && (b_mn ? make_tmap(&tb, B, ti.in_bf16, N, K, ldb, 64)
                     : make_tmap(&tb, B, ti.in_bf16, K, N, ldb, 256));
    if (!ok) return cuda_fail();
    TileParams p{};
    p.a_mn3 = a_mn && make_tmap_mn3(&t3, A, ti.in_bf16, M, K, lda, swg::BM / 64);
    if (p.a_mn3) ta = t3;
    p.b_mn3 = b_mn && make_tmap_mn3(&t3, B, ti.in_bf16, N, K, ldb, 256 / 64);
    if (p.b_mn3) tb = t3;
    const int64_t kb = cdiv(K, swg::BK);
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.m_blocks = (int)cdiv(M, swg::BM);
    p.n_blocks = (int)cdiv(N, 256);
    p.k_blocks = (int)kb;
    p.bk = swg::BK;
    p.tiles = p.m_blocks * p.n_blocks;
    p.splits = S;
    p.kb_per_split = (int)cdiv(kb, S);
    p.units = p.tiles * S;
    p.group_m = 16;
    p.idesc = make_idesc(ti.in_bf16, a_mn, b_mn, swg::BM, 256);
    p.a_mn_major = a_mn;
    p.b_mn_major = b_mn;
    p.alpha = alpha;
    p.beta = beta;
    p.D = C;
    p.ldd = ldc;
    p.out_kind = ti.out_kind;
    p.err = d->err;
    if (swg::launch_tc_store_cl(ta, tb, p, p.units, s) != cudaSuccess) return cuda_fail();
    g_launches++;
    return SWG_OK;
}

// One or two rows (16-bit or e4m3 inputs): one launch of the cluster kernel
// of k_gemv.cu on the FP32 pipes (the product streams op(B) once; tensor-core
// tiles would be almost all padding).  Measured on GB300 at 4096 x 4096: one
// row 8.3 us back to back against 9.5-10.0 us for the split-K tensor-core
// path; three or four rows were slower there (10.9-13.6 us) than on the
// tensor cores.  Blocks of 32 (B stored N x K; 64 for e4m3) or 128 (B stored
// K x N) output columns.  K is cut into up to 8 ranges: as many as bring the
// grid to about one CTA per SM, at least as many as keep the FP32 op(A) slice
// a CTA stages within kGemvSlice / rows elements, each range a whole number
// of boxes (256 or 64 K elements) except the last.  The ring of 16 KB boxes
// is as deep as 227 KB of shared memory allows (12 at most), or as a half or
// a third of it allows when the grid is larger than the GPU (two or three
// CTAs per SM).  SWG_ERR_UNSUPPORTED, with nothing launched, when K needs
// more ranges, N is beyond 2^30 or the tensor map cannot be encoded.
constexpr int64_t kGemvMaxRows = 2;
constexpr int64_t kGemvSlice = 8192;

bool gemv_disabled()
{
    const char *v = std::getenv("SWG_GEMV");
    return v && v[0] == '0';
}

// Row-major matrix of `outer` rows x `inner` contiguous elements (in_kind 0
// binary16, 1 bfloat16, 2 e4m3 as bytes), read without swizzle in boxes of
// box_inner x box_outer; past the edges reads zero.
bool make_tmap_plain(CUtensorMap *m, const void *ptr, int in_kind, int64_t inner, int64_t outer,
                     int64_t ld, int box_inner, int box_outer)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int esz = in_kind == 2 ? 1 : 2;
    const CUtensorMapDataType dt = in_kind == 2   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : in_kind == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * esz)};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// in_kind: 0 binary16, 1 bfloat16, 2 e4m3 (A stored M x K, B stored N x K).
// swiglu: B is the interleaved weight W_fused (K x N with N = 2 x the output
// columns) and C is Y; the kernel's last step forms SiLU(Gate) * Up.  B2
// non-null: SwiGLU from separate bf16 W1 = B and W2 = B2, both K x N with
// row stride ldb, N the output width (64 output columns per block).
int gemv_path(DeviceState *d, int in_kind, int out_kind, int transA, int transB, int64_t M,
              int64_t N, int64_t K, float alpha, const void *A, int64_t lda, const void *B,
              int64_t ldb, float beta, void *C, int64_t ldc, cudaStream_t s, bool swiglu = false,
              const void *B2 = nullptr)
{
    const int mr = M <= 1 ? 1 : 2;
    const bool b_kn = transB == SWG_OP_N;
    const bool dual = B2 != nullptr;
    if (dual && (!b_kn || in_kind != 1)) return SWG_ERR_UNSUPPORTED;
    const int64_t ks = swg::gemv_k_per_stage(b_kn);
    const int64_t blocks = cdiv(N, swg::gemv_cols_per_block(b_kn, in_kind) / (dual ? 2 : 1));
    const int64_t kr_max = kGemvSlice / mr;          // a multiple of both box lengths
    const int64_t s_min = cdiv(K, kr_max);
    if (s_min > 8 || N > (int64_t(1) << 30)) return SWG_ERR_UNSUPPORTED;
    int64_t ranges = std::min<int64_t>(8, std::max<int64_t>(1, d->sms / blocks));
    ranges = std::min<int64_t>(ranges, cdiv(K, ks));
    ranges = std::max<int64_t>(ranges, s_min);
    const int64_t kr = cdiv(cdiv(K, ranges), ks) * ks;
    ranges = cdiv(K, kr);
    // Up to three CTAs per SM when the grid is larger than the GPU (228 KB of
    // shared memory per SM, 1 KB of it reserved per CTA; every instantiation
    // of the kernel uses at most 72 registers, so three 288-thread CTAs fit).
    const int64_t per_sm = std::min<int64_t>(3, cdiv(blocks * ranges, d->sms));
    const int64_t budget = per_sm == 1 ? swg::GV_MAX_SMEM : 233472 / per_sm - 1024;
    const int64_t fixed = swg::gemv_smem_bytes(mr, b_kn, in_kind, (int)kr, 0);
    const int64_t per_stage = swg::gemv_smem_bytes(mr, b_kn, in_kind, (int)kr, 1) - fixed;
    const int64_t stages = std::min<int64_t>({12, cdiv(kr, ks), (budget - fixed) / per_stage});
    if (stages < 1) return SWG_ERR_UNSUPPORTED;

    CUtensorMap tm, tm2;
    bool ok;
    if (dual) {
        const int bi = swg::gemv_box_inner(true) / 2, bo = swg::gemv_box_outer(true, in_kind);
        ok = make_tmap_plain(&tm, B, in_kind, N, K, ldb, bi, bo) &&
             make_tmap_plain(&tm2, B2, in_kind, N, K, ldb, bi, bo);
    } else {
        ok = b_kn ? make_tmap_plain(&tm, B, in_kind, N, K, ldb, swg::gemv_box_inner(true),
                                    swg::gemv_box_outer(true, in_kind))
                  : make_tmap_plain(&tm, B, in_kind, K, N, ldb, swg::gemv_box_inner(false),
                                    swg::gemv_box_outer(false, in_kind));
    }
    if (!ok) return SWG_ERR_UNSUPPORTED;

    swg::GemvArgs g{};
    g.A = A;
    g.lda = lda;
    g.a_t = transA == SWG_OP_T;
    g.D = C;
    g.ldd = ldc;
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    g.kr = (int)kr;
    g.ranges = (int)ranges;
    g.stages = (int)stages;
    g.alpha = alpha;
    g.beta = beta;
    g.out_kind = out_kind;
    g.err = d->err;
    g.swiglu = swiglu || dual ? 1 : 0;
    if (swg::launch_gemv(tm, dual ? &tm2 : nullptr, g, mr, b_kn, in_kind, (int)blocks, s) !=
        cudaSuccess)
        return cuda_fail();
    g_launches++;
    return SWG_OK;
}

// ----------------------------------------------------------------- small kernels

__global__ void scale_kernel(void *D, long long ldd, int M, int N, float beta, int out_kind)
{
    const long long total = (long long)M * N;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / N, c = i - r * N;
        const long long o = r * ldd + c;
        if (out_kind == swg::OUT_F32) {
            float *d = static_cast<float *>(D);
            d[o] = beta == 0.0f ? 0.0f : beta * d[o];
        } else if (out_kind == swg::OUT_F16) {
            __half *d = static_cast<__half *>(D);
            d[o] = __float2half_rn(beta == 0.0f ? 0.0f : beta * __half2float(d[o]));
        } else {
            __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(D);
            d[o] = __float2bfloat16_rn(beta == 0.0f ? 0.0f : beta * __bfloat162float(d[o]));
        }
    }
}

// Four output column pairs per thread: 8-byte loads from W1 and W2, one
// 16-byte store of (g0,u0,g1,u1,g2,u2,g3,u3).
__global__ void interleave_kernel(const uint16_t *W1, const uint16_t *W2, uint16_t *Wf, long long K,
                                  long long N)
{
    const long long quads = N / 4;
    const long long total = K * quads;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long k = i / quads, n = (i - k * quads) * 4;
        const uint2 g = *reinterpret_cast<const uint2 *>(W1 + k * N + n);
        const uint2 u = *reinterpret_cast<const uint2 *>(W2 + k * N + n);
        uint4 o;
        o.x = (g.x & 0xffffu) | (u.x << 16);
        o.y = (g.x >> 16) | (u.x & 0xffff0000u);
        o.z = (g.y & 0xffffu) | (u.y << 16);
        o.w = (g.y >> 16) | (u.y & 0xffff0000u);
        *reinterpret_cast<uint4 *>(Wf + k * 2 * N + 2 * n) = o;
    }
}

// One warp waits, through the pipeline kernels' own bounded wait, on an
// mbarrier that nothing ever arrives on; after limit_ns it records
// SWG_ERR_DEVICE_TIMEOUT in the error word and returns, like a pipeline
// kernel whose partner never shows up.
__global__ void selftest_wait_kernel(int *err, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        swg::mbar_init(swg::smem_u32(&bar), 1);
        abort_flag = 0;
        swg::fence_barrier_init();
    }
    __syncthreads();
    bool ok = true;
    if (threadIdx.x == 0)
        ok = swg::wait_bounded(swg::smem_u32(&bar), 0, &abort_flag, err, true, limit_ns);
    __syncthreads();
    (void)ok;
}

int grid_for(long long work, int sms)
{
    long long g = cdiv(work, 256);
    const long long cap = (long long)sms * 8;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

}  // namespace

// =================================================================== C ABI

extern "C" {

const char *swg_status_string(int status)
{
    switch (status) {
    case SWG_OK: return "SWG_OK";
    case SWG_ERR_INVALID_ARG: return "SWG_ERR_INVALID_ARG";
    case SWG_ERR_MISALIGNED: return "SWG_ERR_MISALIGNED";
    case SWG_ERR_UNSUPPORTED: return "SWG_ERR_UNSUPPORTED";
    case SWG_ERR_CUDA: return "SWG_ERR_CUDA";
    case SWG_ERR_NO_MEMORY: return "SWG_ERR_NO_MEMORY";
    case SWG_ERR_DEVICE_TIMEOUT: return "SWG_ERR_DEVICE_TIMEOUT";
    default: return "SWG_ERR_UNKNOWN";
    }
}

uint64_t swg_launch_count(void) { return g_launches.load(); }

int swg_selftest_wait_timeout(int64_t limit_ns, void *stream)
{
    if (limit_ns <= 0 || limit_ns > 1000000000) return SWG_ERR_INVALID_ARG;
    DeviceState *d = nullptr;
    if (int rc = device_state(d)) return rc;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        d->err, (unsigned long long)limit_ns);
    g_launches++;
    return launch_status();
}

// GEMM with e4m3 A and B (kind::f8f6f4): A stored M x K and B stored N x K,
// both K-major; per-tensor dequantisation scales are folded into alpha.
static int gemm_fp8(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                    const void *A, int64_t lda, const void *B, int64_t ldb, float beta, void *C,
                    int64_t ldc, int out_kind, int out_bytes, int split_k, void *stream,
                    bool noalloc)
{
    if ((transA != SWG_OP_N && transA != SWG_OP_T) || (transB != SWG_OP_N && transB != SWG_OP_T))
        return SWG_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || split_k < 0) return SWG_ERR_INVALID_ARG;
    if (transA != SWG_OP_N || transB != SWG_OP_T) return SWG_ERR_UNSUPPORTED;
    if (split_k > 1 && M > 64) return SWG_ERR_UNSUPPORTED;   // FP8 split-K: few rows only
    if (M == 0 || N == 0) return SWG_OK;
    if (C == nullptr || ldc < N) return SWG_ERR_INVALID_ARG;
    if (K > 0 && (A == nullptr || B == nullptr || lda < K || ldb < K)) return SWG_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim || ldc > kMaxDim || lda > kMaxDim ||
        ldb > kMaxDim)
        return SWG_ERR_UNSUPPORTED;
    if (!aligned16(C) || (ldc * out_bytes) % 16 != 0) return SWG_ERR_MISALIGNED;
    if (K > 0 && (!aligned16(A) || !aligned16(B) || lda % 16 != 0 || ldb % 16 != 0))
        return SWG_ERR_MISALIGNED;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FixedScratch fxs{};
    const FixedScratch *fx = nullptr;
    if (noalloc) {
        if (int rc = noalloc_scratch(s, fxs)) return rc;
        fx = &fxs;
    }
    DeviceState *d = nullptr;
    if (int rc = device_state(d)) return rc;
    if (K == 0) {
        scale_kernel<<<grid_for(M * N, d->sms), 256, 0, s>>>(C, ldc, (int)M, (int)N, beta, out_kind);
        g_launches++;
        return launch_status();
    }
    // One or two rows with an automatic split: the FP32-pipe kernel, as for
    // 16-bit inputs (8-bit weights halve the bytes it streams).
    if (split_k == 0 && M <= kGemvMaxRows && !gemv_disabled()) {
        const int rc = gemv_path(d, 2, out_kind, transA, transB, M, N, K, alpha, A, lda, B, ldb,
                                 beta, C, ldc, s);
        if (rc != SWG_ERR_UNSUPPORTED) return rc;
    }
    // Few rows (decode): the transposed product with the K loop split, as
    // for 16-bit inputs, unless the caller asked for no split.
    if (M <= 64 && split_k != 1) {
        const int64_t kb = cdiv(K, 128);
        const int64_t swapped_tiles = cdiv(N, swg::BM);
        if (split_k > 1 || (kb >= 8 && swapped_tiles * 2 <= d->sms)) {
            TypeInfo ti{false, out_kind, out_bytes};
            return splitk_swapped(d, ti, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta,
                                  C, ldc, split_k, s, true, fx);
        }
    }
    static const int cands[] = {256, 128};
    const TileChoice tc = choose_tiles(d, 4, M, N, cands, 2);
    const int bn = tc.bn;
    const bool pair = tc.pair;
    CUtensorMap ta, tb;
    if (!make_tmap_u8(&ta, A, K, M, lda, swg::BM) ||
        !make_tmap_u8(&tb, B, K, N, ldb, pair ? bn / 2 : bn))
        return cuda_fail();
    TileParams p{};
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.m_blocks = (int)cdiv(M, pair ? 2 * swg::BM : swg::BM);
    p.n_blocks = (int)cdiv(N, bn);
    p.k_blocks = (int)cdiv(K, 128);
    p.bk = 128;
    p.tiles = p.m_blocks * p.n_blocks;
    p.splits = 1;
    p.kb_per_split = p.k_blocks;
    p.units = p.tiles;
    p.group_m = pair ? 8 : 16;
    p.idesc = make_idesc(false, false, false, pair ? 2 * swg::BM : swg::BM, bn);
    p.alpha = alpha;
    p.beta = beta;
    p.D = C;
    p.ldd = ldc;
    p.out_kind = out_kind;
    p.err = d->err;
    CUtensorMap td;
    if (beta == 0.0f && (N * (out_kind == swg::OUT_F32 ? 4 : 2)) % 16 == 0) {
        if (!make_tmap_store(&td, C, out_kind == swg::OUT_F32 ? 4 : 2, N, M, ldc))
            return cuda_fail();
        p.tma_store = 1;
    }
    if (swg::launch_tc_store_fp8(bn, pair, ta, tb, p, tc.units, s, p.tma_store ? &td : nullptr) !=
        cudaSuccess)
        return cuda_fail();
    g_launches++;
    return SWG_OK;
}

// gemm_ex and gemm_splitk_noalloc: one plan (kernels, tiles, split) for
// both; they differ only in where split-K partials go (fx).
static int gemm_impl(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                     const void *A, int64_t lda, const void *B, int64_t ldb, float beta, void *C,
                     int64_t ldc, int dtype, int split_k, void *stream, bool noalloc)
{
    if (dtype == SWG_E4M3_BF16OUT || dtype == SWG_E4M3_F32OUT)
        return gemm_fp8(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                        dtype == SWG_E4M3_BF16OUT ? swg::OUT_BF16 : swg::OUT_F32,
                        dtype == SWG_E4M3_BF16OUT ? 2 : 4, split_k, stream, noalloc);
    TypeInfo ti;
    if (!type_info(dtype, ti)) return SWG_ERR_UNSUPPORTED;
    if ((transA != SWG_OP_N && transA != SWG_OP_T) || (transB != SWG_OP_N && transB != SWG_OP_T))
        return SWG_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || split_k < 0) return SWG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SWG_OK;
    const int64_t a_cols = transA ? M : K, b_cols = transB ? K : N;
    if (C == nullptr || ldc < N) return SWG_ERR_INVALID_ARG;
    if (K > 0 && (A == nullptr || B == nullptr || lda < a_cols || ldb < b_cols))
        return SWG_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim || ldc > kMaxDim || lda > kMaxDim ||
        ldb > kMaxDim)
        return SWG_ERR_UNSUPPORTED;
    if (!aligned16(C) || (ldc * ti.out_bytes) % 16 != 0) return SWG_ERR_MISALIGNED;
    if (K > 0 && (!aligned16(A) || !aligned16(B) || (lda * 2) % 16 != 0 || (ldb * 2) % 16 != 0))
        return SWG_ERR_MISALIGNED;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FixedScratch fxs{};
    const FixedScratch *fx = nullptr;
    if (noalloc) {
        if (int rc = noalloc_scratch(s, fxs)) return rc;
        fx = &fxs;
    }
    DeviceState *d = nullptr;
    if (int rc = device_state(d)) return rc;

    if (K == 0) {
        scale_kernel<<<grid_for(M * N, d->sms), 256, 0, s>>>(C, ldc, (int)M, (int)N, beta,
                                                              ti.out_kind);
        g_launches++;
        return launch_status();
    }

    if (split_k == 0 && M <= kGemvMaxRows && !gemv_disabled()) {
        const int rc = gemv_path(d, ti.in_bf16 ? 1 : 0, ti.out_kind, transA, transB, M, N, K,
                                 alpha, A, lda, B, ldb, beta, C, ldc, s);
        if (rc != SWG_ERR_UNSUPPORTED) return rc;
    }

    const int64_t kb = cdiv(K, swg::BK);
    const int64_t mblk = cdiv(M, swg::BM);
    // Tile shape first (single-CTA or CTA pair, and width), then the split:
    // K is split when the tiles would fill at most half of the slots that
    // shape can keep resident ("为什么 GEMM 是 CUDA 的必修课", 关键技术 item 5).
    static const int cands[] = {256, 128};
    TileChoice tc = choose_tiles(d, 0, M, N, cands, 2);
    // A small output with a short K (no split below): when its tiles would
    // occupy at most a quarter of the SMs, 128 x 64 single-CTA tiles spread
    // the main loop and the epilogue's C reads and D writes over more SMs
    // (a 256^3 GEMM: 8 CTAs instead of one CTA pair).
    int forced_bn = 0;
    if (kb < 8 && forced_tile_mode(&forced_bn) == 0) {
        const int64_t sms_used = tc.pair ? 2 * (int64_t)tc.units : (int64_t)tc.units;
        const int64_t narrow = mblk * cdiv(N, 64);
        if (sms_used * 4 <= d->sms && narrow > sms_used) {
            tc.pair = false;
            tc.bn = 64;
            tc.units = (int)std::min<int64_t>(narrow, d->sms);
        }
    }
    const bool pair = tc.pair;
    const int bn = tc.bn;
    const int64_t tiles = (pair ? cdiv(M, 2 * swg::BM) : mblk) * cdiv(N, bn);
    const int slots = pair ? max_pairs(d, 2, bn) : d->sms;
    int splits = 1;
    if (split_k == 0) {
        if (slots > 0 && tiles * 2 <= slots && kb >= 8) {
            splits = (int)std::min<int64_t>(slots / tiles, kb / 4);
            if (splits < 2) splits = 1;
        }
    } else if (split_k > 1) {
        splits = (int)std::min<int64_t>(split_k, kb);
    }
    splits = std::min(splits, swg::MAX_SPLITS);
    // More rows and an automatic split: 128 x 256 tiles whose K ranges run as
    // one cluster of S CTAs that sum their partials through shared memory
    // (one launch, no workspace), when S clusters per tile are resident at
    // once and fill at least half of the SMs.
    if (split_k == 0 && splits > 1 && M > 64 && !cluster_splitk_disabled() &&
        forced_tile_mode(&forced_bn) == 0) {
        const int64_t t1 = cdiv(M, swg::BM) * cdiv(N, 256);
        int S = 0;
        for (int s_c = 2; s_c <= swg::MAX_CLUSTER_SPLITS; s_c *= 2)
            if (t1 * s_c <= d->sms && kb >= 4 * s_c && t1 <= max_clusters(d, 3, 256, s_c))
                S = s_c;
        if (S > 0 && t1 * S * 2 >= d->sms && (int64_t)(S - 1) * cdiv(kb, S) < kb)
            return gemm_store_cluster(d, ti, transA, transB, M, N, K, alpha, A, lda, B, ldb,
                                      beta, C, ldc, S, static_cast<cudaStream_t>(stream));
    }
    // Few rows and a split K: compute the transposed product instead, so the
    // large operand fills the MMA's 128 rows and the <= 64 rows of op(A)
    // become its N (smaller stages, deeper pipeline, fewer partials).
    if (splits > 1 && M <= 64)
        return splitk_swapped(d, ti, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C,
                              ldc, split_k, static_cast<cudaStream_t>(stream), false, fx);
    int kbps = (int)kb;
    if (splits > 1) {
        kbps = (int)cdiv(kb, splits);
        splits = (int)cdiv(kb, kbps);
    }

    const bool a_mn = transA == SWG_OP_T;
    const bool b_mn = transB == SWG_OP_N;
    CUtensorMap ta, tb;
    bool ok = a_mn ? make_tmap(&ta, A, ti.in_bf16, M, K, lda, 64)
                   : make_tmap(&ta, A, ti.in_bf16, K, M, lda, swg::BM);
    ok = ok && (b_mn ? make_tmap(&tb, B, ti.in_bf16, N, K, ldb, 64)
                     : make_tmap(&tb, B, ti.in_bf16, K, N, ldb, pair ? bn / 2 : bn));
    if (!ok) return cuda_fail();
    // MN-major operands: one 3-D box per stage where the extent allows.
    CUtensorMap t3;
    const bool a3 = a_mn && make_tmap_mn3(&t3, A, ti.in_bf16, M, K, lda, swg::BM / 64);
    if (a3) ta = t3;
    const bool b3 = b_mn && make_tmap_mn3(&t3, B, ti.in_bf16, N, K, ldb, (pair ? bn / 2 : bn) / 64);
    if (b3) tb = t3;

    TileParams p{};
    p.a_mn3 = a3;
    p.b_mn3 = b3;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.m_blocks = (int)(pair ? cdiv(M, 2 * swg::BM) : mblk);
    p.n_blocks = (int)cdiv(N, bn);
    p.k_blocks = (int)kb;
    p.bk = swg::BK;
    p.tiles = p.m_blocks * p.n_blocks;
    p.splits = splits;
    p.kb_per_split = kbps;
    p.units = p.tiles * splits;
    // Raster groups: about as many A panels as B panels per wave of tiles
    // (256-row pair tiles: 8 m-blocks; 128-row tiles: 16).
    p.group_m = pair ? 8 : 16;
    p.idesc = make_idesc(ti.in_bf16, a_mn, b_mn, pair ? 2 * swg::BM : swg::BM, bn);
    p.a_mn_major = a_mn;
    p.b_mn_major = b_mn;
    p.alpha = alpha;
    p.beta = beta;
    p.D = C;
    p.ldd = ldc;
    p.out_kind = ti.out_kind;
    p.err = d->err;

    cudaError_t e;
    if (splits > 1) {
        const int units = (int)std::min<int64_t>(p.units, slots);
        const int64_t ld_ws = cdiv(N, 4) * 4;
        float *ws = nullptr;
        if (int rc = split_workspace(d, s,
                                     sizeof(float) * (size_t)splits * (size_t)M * (size_t)ld_ws,
                                     fx, ws))
            return rc;
        p.ws = ws;
        p.ld_ws = ld_ws;
        // Each CTA's last partial tile leaves through shared memory and TMA
        // stores into ws viewed as [splits][M][ld_ws].
        CUtensorMap tw;
        if (!make_tmap_store(&tw, p.ws, 4, N, M, ld_ws, splits, M * ld_ws)) return cuda_fail();
        p.tma_store = 1;
        e = swg::launch_tc_splitk(bn, pair, ta, tb, p, units, s, &tw);
        if (e == cudaSuccess) {
            g_launches++;
            e = swg::launch_splitk_reduce(p, d->sms, s);
        }
    } else {
        // beta = 0: each CTA's last tile leaves through shared memory and TMA
        // stores (beta != 0 reads C and keeps the direct stores).  TMA clips
        // a row only at 16-byte granules, so N must end on one.
        CUtensorMap td;
        if (beta == 0.0f && (N * ti.out_bytes) % 16 == 0) {
            if (!make_tmap_store(&td, C, ti.out_bytes, N, M, ldc)) return cuda_fail();
            p.tma_store = 1;
        }
        e = swg::launch_tc_store(bn, pair, ta, tb, p, tc.units, s, p.tma_store ? &td : nullptr);
    }
    if (e != cudaSuccess) return cuda_fail();
    g_launches++;
    return SWG_OK;
}

int gemm_ex(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha, const void *A,
            int64_t lda, const void *B, int64_t ldb, float beta, void *C, int64_t ldc, int dtype,
            int split_k, void *stream)
{
    return gemm_impl(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, split_k,
                     stream, false);
}

int gemm(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha, const void *A,
         int64_t lda, const void *B, int64_t ldb, float beta, void *C, int64_t ldc, int dtype,
         void *stream)
{
    return gemm_ex(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, 0,
                   stream);
}

int swiglu_mlp(const void *A, const void *W_fused, void *Y, int64_t M, int64_t N, int64_t K,
               void *stream)
{
    if (M < 0 || N < 0 || K < 0) return SWG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SWG_OK;
    if (Y == nullptr || (K > 0 && (A == nullptr || W_fused == nullptr)))
        return SWG_ERR_INVALID_ARG;
    if (M > kMaxDim || 2 * N > kMaxDim || K > kMaxDim) return SWG_ERR_UNSUPPORTED;
    if (!aligned16(Y) || N % 8 != 0) return SWG_ERR_MISALIGNED;
    if (K > 0 && (!aligned16(A) || !aligned16(W_fused) || K % 8 != 0)) return SWG_ERR_MISALIGNED;

    DeviceState *d = nullptr;
    if (int rc = device_state(d)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (K == 0) {   // Gate = Up = 0, so Y = SiLU(0) * 0 = 0.
        scale_kernel<<<grid_for(M * N, d->sms), 256, 0, s>>>(Y, N, (int)M, (int)N, 0.0f,
                                                              swg::OUT_BF16);
        g_launches++;
        return launch_status();
    }

    const int64_t N2 = 2 * N;
    // One or two rows (decode): one launch of the FP32-pipe kernel, which
    // streams W_fused once and forms SiLU(Gate) * Up in its final reduction.
    if (M <= kGemvMaxRows && !gemv_disabled()) {
        const int rc = gemv_path(d, 1, swg::OUT_BF16, SWG_OP_N, SWG_OP_N, M, N2, K, 1.0f, A, K,
                                 W_fused, N2, 0.0f, Y, N, s, true);
        if (rc != SWG_ERR_UNSUPPORTED) return rc;
    }
    // At most 64 rows (decode of a few sequences): one 128 x 128 tile per
    // block of the 2N-space, only its first M rows used and exchanged, with
    // its K range cut into S pieces that run as one
    // thread-block cluster and are summed through shared memory before the
    // pair-multiply (one launch, no workspace).  Otherwise (many tiles, or
    // no cluster configuration that is resident at once) the persistent
    // kernel below.
    if (M <= 64 && !cluster_splitk_disabled()) {
        const int64_t kb = cdiv(K, swg::BK);
        // The cluster size using the most CTAs with every cluster resident at
        // once.  Tiles are 128 x 128: the receive buffer of a 256-column tile
        // would leave room for a single pipeline stage.
        const int bn = 128;
        const int64_t tiles = cdiv(N2, bn);
        int S = 0;
        for (int s_c = 2; s_c <= swg::MAX_CLUSTER_SPLITS; s_c *= 2) {
            if (tiles * s_c > d->sms || (s_c - 1) * cdiv(kb, s_c) >= kb) continue;
            if (tiles > max_clusters(d, 2, bn, s_c)) continue;
            S = s_c;
        }
        // worth it when the tiles alone would leave half of the SMs idle
        if (S > 0 && tiles * 2 <= d->sms) {
            CUtensorMap ta, tb, t3;
            if (!make_tmap(&ta, A, true, K, M, K, swg::BM) ||
                !make_tmap(&tb, W_fused, true, N2, K, N2, 64))
                return cuda_fail();
            TileParams p{};
            p.b_mn3 = make_tmap_mn3(&t3, W_fused, true, N2, K, N2, bn / 64);
            if (p.b_mn3) tb = t3;
            p.M = (int)M;
            p.N = (int)N2;
            p.K = (int)K;
            p.m_blocks = 1;
            p.n_blocks = (int)tiles;
            p.k_blocks = (int)kb;
            p.bk = swg::BK;
            p.tiles = (int)tiles;
            p.splits = S;
            p.kb_per_split = (int)cdiv(kb, S);
            p.units = p.tiles * S;
            p.group_m = 16;
            p.idesc = make_idesc(true, false, true, swg::BM, bn);
            p.b_mn_major = 1;
            p.alpha = 1.0f;
            p.D = Y;
            p.ldd = N;
            p.out_kind = swg::OUT_BF16;
            p.err = d->err;
            if (swg::launch_tc_swiglu_cl(bn, ta, tb, p, p.units, s) != cudaSuccess)
                return cuda_fail();
            g_launches++;
            return SWG_OK;
        }
    }
    static const int cands[] = {256, 128, 64};
    const TileChoice tc = choose_tiles(d, 1, M, N2, cands, 3);
    const int bn = tc.bn;
    const bool pair = tc.pair;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, A, true, K, M, K, swg::BM) || !make_tmap(&tb, W_fused, true, N2, K, N2, 64))
        return cuda_fail();
    // W_fused is MN-major: one 3-D box per stage where 2N allows.
    CUtensorMap t3;
    const bool b3 = make_tmap_mn3(&t3, W_fused, true, N2, K, N2, (pair ? bn / 2 : bn) / 64);
    if (b3) tb = t3;

    TileParams p{};
    p.b_mn3 = b3;
    p.M = (int)M;
    p.N = (int)N2;
    p.K = (int)K;
    p.m_blocks = (int)cdiv(M, pair ? 2 * swg::BM : swg::BM);
    p.n_blocks = (int)cdiv(N2, bn);
    p.k_blocks = (int)cdiv(K, swg::BK);
    p.bk = swg::BK;
    p.tiles = p.m_blocks * p.n_blocks;
    p.splits = 1;
    p.kb_per_split = p.k_blocks;
    p.units = p.tiles;
    p.group_m = pair ? 8 : 16;
    p.idesc = make_idesc(true, false, true, pair ? 2 * swg::BM : swg::BM, bn);
    p.a_mn_major = 0;
    p.b_mn_major = 1;
    p.alpha = 1.0f;
    p.beta = 0.0f;
    p.D = Y;
    p.ldd = N;
    p.out_kind = swg::OUT_BF16;
    p.err = d->err;
    // Each CTA's last tile leaves through shared memory and TMA stores (whole
    // 128-byte boxes: 64 output columns per tile, so bn >= 128).
    CUtensorMap ty;
    if (bn >= 128) {
        if (!make_tmap_store(&ty, Y, 2, N, M, N)) return cuda_fail();
        p.tma_store = 1;
    }
    if (swg::launch_tc_swiglu(bn, pair, ta, tb, p, tc.units, s, p.tma_store ? &ty : nullptr) !=
        cudaSuccess)
        return cuda_fail();
    g_launches++;
    return SWG_OK;
}

int swiglu_mlp_fp8(const void *A, const void *W_fused_t, void *Y, int64_t M, int64_t N,
                   int64_t K, float scale, void *stream)
{
    if (M < 0 || N < 0 || K < 0) return SWG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SWG_OK;
    if (Y == nullptr || (K > 0 && (A == nullptr || W_fused_t == nullptr)))
        return SWG_ERR_INVALID_ARG;
    if (M > kMaxDim || 2 * N > kMaxDim || K > kMaxDim) return SWG_ERR_UNSUPPORTED;
    if (!aligned16(Y) || N % 8 != 0) return SWG_ERR_MISALIGNED;
    if (K > 0 && (!aligned16(A) || !aligned16(W_fused_t) || K % 16 != 0))
        return SWG_ERR_MISALIGNED;

    DeviceState *d = nullptr;
    if (int rc = device_state(d)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        scale_kernel<<<grid_for(M * N, d->sms), 256, 0, s>>>(Y, N, (int)M, (int)N, 0.0f,
                                                              swg::OUT_BF16);
        g_launches++;
        return launch_status();
    }
    const int64_t N2 = 2 * N;
    // One or two rows (decode): the FP32-pipe kernel over the transposed
    // interleaved weight (its N x K layout), SiLU(Gate) * Up in its final
    // reduction, the scale applied to Gate and Up first.
    if (M <= kGemvMaxRows && !gemv_disabled()) {
        const int rc = gemv_path(d, 2, swg::OUT_BF16, SWG_OP_N, SWG_OP_T, M, N2, K, scale, A, K,
                                 W_fused_t, K, 0.0f, Y, N, s, true);
        if (rc != SWG_ERR_UNSUPPORTED) return rc;
    }
    static const int cands[] = {256, 128, 64};
    const TileChoice tc = choose_tiles(d, 5, M, N2, cands, 3);
    const int bn = tc.bn;
    const bool pair = tc.pair;
    CUtensorMap ta, tb;
    if (!make_tmap_u8(&ta, A, K, M, K, swg::BM) ||
        !make_tmap_u8(&tb, W_fused_t, K, N2, K, pair ? bn / 2 : bn))
        return cuda_fail();
    TileParams p{};
    p.M = (int)M;
    p.N = (int)N2;
    p.K = (int)K;
    p.m_blocks = (int)cdiv(M, pair ? 2 * swg::BM : swg::BM);
    p.n_blocks = (int)cdiv(N2, bn);
    p.k_blocks = (int)cdiv(K, 128);
    p.bk = 128;
    p.tiles = p.m_blocks * p.n_blocks;
    p.splits = 1;
    p.kb_per_split = p.k_blocks;
    p.units = p.tiles;
    p.group_m = pair ? 8 : 16;
    p.idesc = make_idesc(false, false, false, pair ? 2 * swg::BM : swg::BM, bn);
    p.alpha = scale;
    p.beta = 0.0f;
    p.D = Y;
    p.ldd = N;
    p.out_kind = swg::OUT_BF16;
    p.err = d->err;
    CUtensorMap ty;
    if (bn >= 128) {
        if (!make_tmap_store(&ty, Y, 2, N, M, N)) return cuda_fail();
        p.tma_store = 1;
    }
    if (swg::launch_tc_swiglu_fp8(bn, pair, ta, tb, p, tc.units, s, p.tma_store ? &ty : nullptr) !=
        cudaSuccess)
        return cuda_fail();
    g_launches++;
    return SWG_OK;
}

int swiglu_mlp_dual(const void *A, const void *W1, const void *W2, void *Y, int64_t M, int64_t N,
                    int64_t K, void *stream)
{
    if (M < 0 || N < 0 || K < 0) return SWG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SWG_OK;
    if (Y == nullptr || (K > 0 && (A == nullptr || W1 == nullptr || W2 == nullptr)))
        return SWG_ERR_INVALID_ARG;
    if (M > kMaxDim || 2 * N > kMaxDim || K > kMaxDim) return SWG_ERR_UNSUPPORTED;
    if (!aligned16(Y) || N % 8 != 0) return SWG_ERR_MISALIGNED;
    if (K > 0 && (!aligned16(A) || !aligned16(W1) || !aligned16(W2) || K % 8 != 0))
        return SWG_ERR_MISALIGNED;

    DeviceState *d = nullptr;
    if (int rc = device_state(d)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {   // Gate = Up = 0, so Y = 0.
        scale_kernel<<<grid_for(M * N, d->sms), 256, 0, s>>>(Y, N, (int)M, (int)N, 0.0f,
                                                              swg::OUT_BF16);
        g_launches++;
        return launch_status();
    }

    // One or two rows (decode): the FP32-pipe kernel reading W1 and W2 in
    // 64-column boxes side by side, SiLU(Gate) * Up in its final reduction.
    if (M <= kGemvMaxRows && !gemv_disabled()) {
        const int rc = gemv_path(d, 1, swg::OUT_BF16, SWG_OP_N, SWG_OP_N, M, N, K, 1.0f, A, K, W1,
                                 N, 0.0f, Y, N, s, true, W2);
        if (rc != SWG_ERR_UNSUPPORTED) return rc;
    }
    // Tiles are chosen in the 2N-wide Gate|Up column space, as for swiglu_mlp.
    static const int cands[] = {256, 128};
    const TileChoice tc = choose_tiles(d, 3, M, 2 * N, cands, 2);
    const int bn = tc.bn;
    const bool pair = tc.pair;
    CUtensorMap ta, tw1, tw2;
    if (!make_tmap(&ta, A, true, K, M, K, swg::BM) || !make_tmap(&tw1, W1, true, N, K, N, 64) ||
        !make_tmap(&tw2, W2, true, N, K, N, 64))
        return cuda_fail();
    // W1 and W2 are MN-major: 3-D boxes of a pair CTA's whole half (or a
    // single CTA's Gate or Up atoms) where N allows; both maps or neither.
    CUtensorMap t31, t32;
    const int w_atoms = bn / 128;
    const bool w3 = make_tmap_mn3(&t31, W1, true, N, K, N, w_atoms) &&
                    make_tmap_mn3(&t32, W2, true, N, K, N, w_atoms);
    if (w3) {
        tw1 = t31;
        tw2 = t32;
    }

    TileParams p{};
    p.b_mn3 = w3;
    p.M = (int)M;
    p.N = (int)N;              // output columns; a tile covers bn/2 of them
    p.K = (int)K;
    p.m_blocks = (int)cdiv(M, pair ? 2 * swg::BM : swg::BM);
    p.n_blocks = (int)cdiv(N, bn / 2);
    p.k_blocks = (int)cdiv(K, swg::BK);
    p.bk = swg::BK;
    p.tiles = p.m_blocks * p.n_blocks;
    p.splits = 1;
    p.kb_per_split = p.k_blocks;
    p.units = p.tiles;
    p.group_m = pair ? 8 : 16;
    p.idesc = make_idesc(true, false, true, pair ? 2 * swg::BM : swg::BM, bn);
    p.a_mn_major = 0;
    p.b_mn_major = 1;
    p.alpha = 1.0f;
    p.beta = 0.0f;
    p.D = Y;
    p.ldd = N;
    p.out_kind = swg::OUT_BF16;
    p.err = d->err;
    if (swg::launch_tc_swiglu_dual(bn, pair, ta, tw1, tw2, p, tc.units, s) != cudaSuccess)
        return cuda_fail();
    g_launches++;
    return SWG_OK;
}

int swiglu_mlp_forward(const void *A, const void *W_fused, const void *W_down, void *Y, void *Out,
                       int64_t M, int64_t N, int64_t K, float beta, void *stream)
{
    // Everything both launches need is checked first, so a rejected call
    // writes nothing.
    if (M < 0 || N < 0 || K < 0) return SWG_ERR_INVALID_ARG;
    if (M == 0 || K == 0) return SWG_OK;          // Out is M x K
    if (Out == nullptr || A == nullptr || W_fused == nullptr) return SWG_ERR_INVALID_ARG;
    if (N > 0 && (Y == nullptr || W_down == nullptr)) return SWG_ERR_INVALID_ARG;
    if (M > kMaxDim || 2 * N > kMaxDim || K > kMaxDim) return SWG_ERR_UNSUPPORTED;
    if (!aligned16(Out) || !aligned16(A) || !aligned16(W_fused) || K % 8 != 0)
        return SWG_ERR_MISALIGNED;
    if (N > 0 && (!aligned16(Y) || !aligned16(W_down) || N % 8 != 0)) return SWG_ERR_MISALIGNED;
    // Y = SiLU(A W1) (.) (A W2) through the fused kernel, then the down
    // projection Out = Y W_down + beta * Out through gemm.
    if (int rc = swiglu_mlp(A, W_fused, Y, M, N, K, stream)) return rc;
    return gemm(SWG_OP_N, SWG_OP_N, M, K, N, 1.0f, Y, N, W_down, K, beta, Out, K, SWG_BF16,
                stream);
}

int swiglu_interleave(const void *W1, const void *W2, void *W_fused, int64_t K, int64_t N,
                      void *stream)
{
    if (K < 0 || N < 0) return SWG_ERR_INVALID_ARG;
    if (K == 0 || N == 0) return SWG_OK;
    if (!W1 || !W2 || !W_fused) return SWG_ERR_INVALID_ARG;
    if (K > kMaxDim || 2 * N > kMaxDim) return SWG_ERR_UNSUPPORTED;
    if (!aligned16(W1) || !aligned16(W2) || !aligned16(W_fused) || N % 4 != 0)
        return SWG_ERR_MISALIGNED;
    DeviceState *d = nullptr;
    if (int rc = device_state(d)) return rc;
    interleave_kernel<<<grid_for(K * N / 4, d->sms), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(W1), static_cast<const uint16_t *>(W2),
        static_cast<uint16_t *>(W_fused), K, N);
    g_launches++;
    return launch_status();
}

int swg_get_device_error(void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return cuda_fail();
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_word, sizeof(int)) != cudaSuccess) return cuda_fail();
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_err_word, &zero, sizeof(int)) != cudaSuccess) return cuda_fail();
        return v;
    }
    return SWG_OK;
}

int swg_last_cuda_error(void) { return t_last_cuda_error; }

const char *swg_cuda_error_name(int code)
{
    if (code == 0) return "none";
    if (code >= 10000) return "tensor-map encoding failed (driver result = code - 10000)";
    return cudaGetErrorName(static_cast<cudaError_t>(code));
}

void swg_shutdown(void)
{
    {
        std::lock_guard<std::mutex> lk(g_mu);
        int cur = 0;
        const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
        for (auto &dv : g_dev) {
            bool any = false;
            for (auto &kv : dv.second.ws) any = any || kv.second.raw != nullptr;
            if (any && cudaSetDevice(dv.first) == cudaSuccess) {
                for (auto &kv : dv.second.ws) {
                    if (kv.second.raw) cudaFree(kv.second.raw);
                    for (void *r : kv.second.retired) cudaFree(r);
                }
            }
            dv.second.ws.clear();
            // Device addresses, occupancy figures and kernel attributes are
            // looked up again by the next call: after a cudaDeviceReset the
            // cached ones would be stale.
            dv.second.ready = false;
            dv.second.max_pairs.clear();
        }
        if (have_cur) cudaSetDevice(cur);
        swg::g_setup_epoch.fetch_add(1);
    }
    noalloc_forget();
}

}  // extern "C"

// =================================================================== no-allocation GEMM
//
// gemm_splitk_noalloc runs exactly what gemm_ex plans for the same arguments
// (the same kernels, tile shapes, split count and fixed-order reduction), but
// a split-K call keeps its FP32 partial sums in a fixed array that is part of
// the library's device image instead of a workspace from cudaMalloc.  It is
// for callers that must not allocate device memory once they are running:
// for example a host framework that has already reserved nearly all device
// memory in its own pool (a cudaMalloc would fail, or fragment that pool), or
// a serving loop that forbids cudaMalloc/cudaFree because they can
// synchronise the whole device.

namespace {

constexpr size_t kNoallocGuardFloats = kGuardBytes / sizeof(float);
constexpr size_t kNoallocScratchFloats = SWG_NOALLOC_SCRATCH_BYTES / sizeof(float);

// The partials, between two guard bands of kGuardBytes that no kernel writes
// (filled and checked only under SWG_TEST_WS_GUARD=1).  Every GPU on which
// the library's kernels are loaded holds these bytes until the process exits.
// All calls share them; a call writes every partial it later reads, so
// nothing here has to start at zero.
static __device__ __align__(256) float
    g_noalloc_scratch[kNoallocGuardFloats + kNoallocScratchFloats + kNoallocGuardFloats];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
bool g_noalloc_ready[kNoallocMaxDevices];
bool g_noalloc_guarded[kNoallocMaxDevices];
float *g_noalloc_ptr[kNoallocMaxDevices];   // device address of g_noalloc_scratch

// Once per device, with that device current: the array's device address.
// In host code the symbol g_noalloc_scratch is a host-side stand-in, not a
// device address, so kernels are given this address instead.  swg_shutdown
// forgets it (a cudaDeviceReset invalidates it).
int noalloc_setup(int &dev, cudaStream_t s)
{
    if (int rc = current_device(dev)) return rc;
    if (dev < 0 || dev >= kNoallocMaxDevices) return SWG_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ready[dev]) return SWG_OK;
    void *scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess) return cuda_fail();
    g_noalloc_ptr[dev] = static_cast<float *>(scratch);
    g_noalloc_guarded[dev] = false;
    if (ws_guards_enabled()) {
        uint8_t *b = static_cast<uint8_t *>(scratch);
        if (cudaMemsetAsync(b, kGuardByte, kGuardBytes, s) != cudaSuccess ||
            cudaMemsetAsync(b + kGuardBytes + SWG_NOALLOC_SCRATCH_BYTES, kGuardByte, kGuardBytes,
                            s) != cudaSuccess)
            return cuda_fail();
        g_noalloc_guarded[dev] = true;
    }
    g_noalloc_ready[dev] = true;
    return SWG_OK;
}

// Number of bytes in [p, p + n) on the device that differ from kGuardByte
// (-1 if they cannot be read).
int64_t guard_damage(const void *p, size_t n)
{
    std::vector<unsigned char> h(n);
    if (cudaMemcpy(h.data(), p, n, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
    int64_t bad = 0;
    for (unsigned char c : h) bad += c != kGuardByte;
    return bad;
}

int noalloc_scratch(cudaStream_t s, FixedScratch &out)
{
    int dev = 0;
    if (int rc = noalloc_setup(dev, s)) return rc;
    out.base = g_noalloc_ptr[dev] + kNoallocGuardFloats;
    out.bytes = SWG_NOALLOC_SCRATCH_BYTES;
    return SWG_OK;
}

}  // namespace

extern "C" {

int gemm_splitk_noalloc(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                        const void *A, int64_t lda, const void *B, int64_t ldb, float beta,
                        void *C, int64_t ldc, int dtype, int split_k, void *stream)
{
    // Arguments are validated (before any CUDA call) and planned exactly as
    // by gemm_ex; the array's set-up follows validation.
    return gemm_impl(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, split_k,
                     stream, true);
}

int swg_debug_workspace_guards(void *stream, int64_t *bad_bytes)
{
    if (bad_bytes == nullptr) return SWG_ERR_INVALID_ARG;
    *bad_bytes = 0;
    int dev = 0;
    if (int rc = current_device(dev)) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return cuda_fail();
    int64_t bad = 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_dev.find(dev);
        if (it != g_dev.end()) {
            for (auto &kv : it->second.ws) {
                const Workspace &w = kv.second;
                if (!w.raw || w.raw == w.base) continue;          // allocated without guards
                const uint8_t *lo = static_cast<const uint8_t *>(w.raw);
                const int64_t a = guard_damage(lo, kGuardBytes);
                const int64_t b = guard_damage(lo + kGuardBytes + w.bytes, kGuardBytes);
                if (a < 0 || b < 0) return cuda_fail();
                bad += a + b;
            }
        }
    }
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (dev < kNoallocMaxDevices && g_noalloc_ready[dev] && g_noalloc_guarded[dev]) {
            const uint8_t *lo = reinterpret_cast<const uint8_t *>(g_noalloc_ptr[dev]);
            const int64_t a = guard_damage(lo, kGuardBytes);
            const int64_t b = guard_damage(lo + kGuardBytes + SWG_NOALLOC_SCRATCH_BYTES,
                                           kGuardBytes);
            if (a < 0 || b < 0) return cuda_fail();
            bad += a + b;
        }
    }
    *bad_bytes = bad;
    return SWG_OK;
}

}  // extern "C"

// Forgets the device addresses cached by gemm_splitk_noalloc (swg_shutdown).
void noalloc_forget()
{
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    for (int i = 0; i < kNoallocMaxDevices; ++i) g_noalloc_ready[i] = false;
}
