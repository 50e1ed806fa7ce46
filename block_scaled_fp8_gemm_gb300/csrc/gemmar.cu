// gemmar.cu -- the C ABI of libgemmar (declared in include/gemmar.h): context
// and workspace, argument and shape validation, TMA tensor maps, launches,
// the device status word and the closed-form self-test.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "gemmar.h"
#include "kernels.h"

#define GEMMAR_API extern "C" __attribute__((visibility("default")))

using namespace gemmar;

struct gemmar_ctx {
    int device = -1;
    int num_sms = 0;
    int64_t max_M = 0, N = 0, K = 0;
    int max_P = 0;
    uint32_t flags = 0;
    uint64_t timeout_ns = 0;
    float *W = nullptr;               // fp32 partials, max_P * (max_M + 128 * max_P) * N (tile-blocked)
    int64_t W_floats = 0;
    uint32_t *band_done = nullptr;    // kMaxBands retire counters, then as many claim counters
    ptx::DevStatus *status = nullptr;
    uint8_t *sfa = nullptr;           // mx repack images of A scales
    int64_t sfa_bytes = 0;
    uint8_t *sfb = nullptr;           // mx repack images of B scales
    int64_t sfb_bytes = 0;
    uint8_t *wire_q = nullptr;        // fp8-wire codes, max_M * N
    float *wire_s = nullptr;          // fp8-wire row scales, max_M
    int disabled = 0;
    int64_t total_bytes = 0;
    // the last fused band-path call, for gemmar_overlap_stats
    int ov_bands = 0;                 // bands whose claim counters it used (0: no in-kernel reduce)
    int64_t ov_bpb = 0;               // 32 x 32 blocks per band
    int64_t ov_total = 0;             // blocks of the call
    // phase timing: one set of GEMMAR_NUM_PHASES + 1 events per recorded call
    int timing = 0;
    std::vector<cudaEvent_t> events;
    int recorded = 0;
};

namespace gemmar {

cudaError_t ensure_dynamic_smem(const void *kernel, int bytes)
{
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({kernel, dev}))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        done.insert({kernel, dev});
    return e;
}

}  // namespace gemmar

namespace {

constexpr int kMaxTimedCalls = 65536;
constexpr int kEventsPerCall = GEMMAR_NUM_PHASES + 1;

// Event marking the start of phase `ph` (ph == GEMMAR_NUM_PHASES: the end) of
// the current recorded call, or nullptr when timing is off or the record is full.
cudaEvent_t phase_event(gemmar_ctx *ctx, int ph)
{
    if (!ctx->timing || ctx->recorded >= kMaxTimedCalls)
        return nullptr;
    const size_t idx = (size_t)ctx->recorded * kEventsPerCall + ph;
    while (ctx->events.size() <= idx) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess)
            return nullptr;
        ctx->events.push_back(e);
    }
    return ctx->events[idx];
}

void mark(gemmar_ctx *ctx, int ph, cudaStream_t st)
{
    cudaEvent_t e = phase_event(ctx, ph);
    if (e)
        cudaEventRecord(e, st);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// 2-D uint8 tensor [rows, cols] (cols contiguous), box {128 bytes, box_rows},
// 128-byte swizzle; rows past the end read as zero.
bool make_tmap_u8(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int box_rows)
{
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

int check_ctx(gemmar_ctx *ctx)
{
    if (ctx == nullptr)
        return GEMMAR_ERR_ARG;
    if (ctx->disabled)
        return GEMMAR_ERR_DISABLED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    if (dev != ctx->device)
        return GEMMAR_ERR_DEVICE;
    return GEMMAR_OK;
}

int shape_rules(int P, int64_t M, int64_t N, int64_t K, int bands, int scale_kind)
{
    if (P < 1 || P > kMaxP || M < 1 || N < 1 || K < 1 || bands < 1)
        return GEMMAR_ERR_ARG;
    if (bands > kMaxBands || bands > M || M % bands != 0)
        return GEMMAR_ERR_SHAPE;
    // N is tiled by 256/128 (blockscale: also the B-scale block; ptpc) or 224/128 (mx)
    const bool n_ok = scale_kind == GEMMAR_SCALE_MX32 ? (N % 128 == 0 || N % 224 == 0) : (N % 128 == 0);
    if (!n_ok || K % 128 != 0)
        return GEMMAR_ERR_SHAPE;
    if (N > 65536 || K > 65536 || M > (int64_t(1) << 24))
        return GEMMAR_ERR_SHAPE;
    return GEMMAR_OK;
}

int mx_tile_n(int64_t N) { return (N % 224 == 0) ? 224 : 128; }
int ptpc_tile_n(int64_t N) { return (N % 256 == 0) ? 256 : 128; }

bool known_scale_kind(int k)
{
    return k == GEMMAR_SCALE_BLOCK128 || k == GEMMAR_SCALE_MX32 || k == GEMMAR_SCALE_PTPC;
}

TileGrid make_grid(int P, int64_t M, int64_t N, int64_t K, int bands, int bn, int slice_loop = 0)
{
    TileGrid g;
    if (slice_loop)
        bands = 1;
    g.P = P;
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    g.bands = bands;
    g.rows_per_band = (int)(M / bands);
    g.mt_per_band = (g.rows_per_band + 127) / 128;
    g.ntiles_n = (int)(N / bn);
    g.slice_loop = slice_loop;
    g.num_tiles = (slice_loop ? 1 : P) * bands * g.mt_per_band * g.ntiles_n;
    return g;
}

// The blockscale kernel splits 65536 registers between its warp roles with
// setmaxnreg; that split needs the kernel to have been built for 128 per thread
// (512 threads).
bool register_split_ok(int bn)
{
    return gemm_blockscale_split_ok(bn);
}

int64_t mx_sfa_bytes(int P, int64_t M, int64_t K, int bands)
{
    const int64_t rpb = M / bands, mtpb = (rpb + 127) / 128;
    return (int64_t)P * bands * mtpb * (K / 128) * 512;
}

int64_t mx_sfb_bytes(int P, int64_t N, int64_t K, int bn) { return (int64_t)P * (N / bn) * (K / 128) * 1024; }

#define CUDA_OK(x)                          \
    do {                                    \
        if ((x) != cudaSuccess)             \
            return GEMMAR_ERR_CUDA;         \
    } while (0)

// One GEMM launch over P slices.  scale_kind selects the kernel; o says where
// the result goes.
int run_gemm(gemmar_ctx *ctx, int P, const uint8_t *const *A, const void *const *sa, const uint8_t *const *B,
             const void *const *sb, int scale_kind, int64_t M, int64_t N, int64_t K, int bands, const GemmOut &o,
             cudaStream_t st, int slice_loop = 0)
{
    if (!load_encode())
        return GEMMAR_ERR_CUDA;
    if (scale_kind == GEMMAR_SCALE_BLOCK128) {
        // slice_loop 2 (partials summed on chip) exists on the CTA-pair kernel only
        const BsPlan pl = plan_blockscale(P, M, N, K, bands, slice_loop, ctx->num_sms,
                                          (slice_loop == 2 || (ctx->flags & GEMMAR_CTA_PAIR)) ? 1 : 0);
        if (slice_loop == 2 && !pl.pair)
            return GEMMAR_ERR_DEVICE;
        if (!pl.pair && !register_split_ok(pl.bn))
            return GEMMAR_ERR_DEVICE;
        BsParams prm;
        std::memset(&prm, 0, sizeof(prm));
        for (int p = 0; p < P; ++p) {
            if (!make_tmap_u8(&prm.tmA[p], A[p], M, K, 128) || !make_tmap_u8(&prm.tmB[p], B[p], N, K, pl.box_b_rows))
                return GEMMAR_ERR_CUDA;
            prm.sa[p] = static_cast<const float *>(sa[p]);
            prm.sb[p] = static_cast<const float *>(sb[p]);
        }
        prm.g = pl.g;
        prm.o = o;
        prm.status = ctx->status;
        prm.timeout_ns = ctx->timeout_ns;
        CUDA_OK(launch_blockscale(prm, pl, st));
    } else if (scale_kind == GEMMAR_SCALE_PTPC) {
        // one fp32 scale per row of A and of B: whole-K accumulation, scaled in the epilogue
        const int bn = ptpc_tile_n(N);
        if (slice_loop)
            bands = 1;
        if (!gemm_mx_split_ok(gemm_ptpc_num_regs(bn)))
            return GEMMAR_ERR_DEVICE;
        MxParams prm;
        std::memset(&prm, 0, sizeof(prm));
        for (int p = 0; p < P; ++p) {
            if (!make_tmap_u8(&prm.tmA[p], A[p], M, K, 128) || !make_tmap_u8(&prm.tmB[p], B[p], N, K, bn))
                return GEMMAR_ERR_CUDA;
            prm.pa[p] = static_cast<const float *>(sa[p]);
            prm.pb[p] = static_cast<const float *>(sb[p]);
        }
        prm.g = make_grid(P, M, N, K, bands, bn, slice_loop);
        prm.o = o;
        prm.status = ctx->status;
        prm.timeout_ns = ctx->timeout_ns;
        const int grid = std::min(prm.g.num_tiles, ctx->num_sms);
        CUDA_OK(launch_gemm_ptpc(prm, bn, grid, st));
    } else {
        const int bn = mx_tile_n(N);
        if (slice_loop)
            bands = 1;
        if (!gemm_mx_split_ok(gemm_mx_num_regs(bn)))
            return GEMMAR_ERR_DEVICE;
        if (mx_sfa_bytes(P, M, K, bands) > ctx->sfa_bytes || mx_sfb_bytes(P, N, K, bn) > ctx->sfb_bytes)
            return GEMMAR_ERR_WORKSPACE;
        CUDA_OK(launch_mx_repack(reinterpret_cast<const uint8_t *const *>(sa),
                                 reinterpret_cast<const uint8_t *const *>(sb), P, (int)M, (int)N, (int)K, bands, bn,
                                 ctx->sfa, ctx->sfb, st));
        MxParams prm;
        std::memset(&prm, 0, sizeof(prm));
        for (int p = 0; p < P; ++p)
            if (!make_tmap_u8(&prm.tmA[p], A[p], M, K, 128) || !make_tmap_u8(&prm.tmB[p], B[p], N, K, bn))
                return GEMMAR_ERR_CUDA;
        prm.sfa = ctx->sfa;
        prm.sfb = ctx->sfb;
        prm.g = make_grid(P, M, N, K, bands, bn, slice_loop);
        prm.o = o;
        prm.status = ctx->status;
        prm.timeout_ns = ctx->timeout_ns;
        const int grid = std::min(prm.g.num_tiles, ctx->num_sms);
        CUDA_OK(launch_gemm_mx(prm, bn, grid, st));
    }
    return GEMMAR_OK;
}

int gemm_single(gemmar_ctx *ctx, const uint8_t *A, const void *sa, const uint8_t *B, const void *sb, void *C,
                int c_dtype, int64_t M, int64_t N, int64_t K, int scale_kind, void *stream)
{
    int rc = check_ctx(ctx);
    if (rc)
        return rc;
    if (!A || !sa || !B || !sb || !C || (c_dtype != GEMMAR_DTYPE_F32 && c_dtype != GEMMAR_DTYPE_BF16))
        return GEMMAR_ERR_ARG;
    if ((rc = shape_rules(1, M, N, K, 1, scale_kind)))
        return rc;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(sa) || !aligned16(sb))
        return GEMMAR_ERR_ALIGN;
    GemmOut o{C, nullptr, c_dtype == GEMMAR_DTYPE_BF16 ? OUT_BF16 : OUT_F32, -1};
    return run_gemm(ctx, 1, &A, &sa, &B, &sb, scale_kind, M, N, K, 1, o, as_stream(stream));
}

}  // namespace

// ============================================================================ ABI

GEMMAR_API int gemmar_supports(int P, int64_t M, int64_t N, int64_t K, int bands, int scale_kind)
{
    if (!known_scale_kind(scale_kind))
        return GEMMAR_ERR_ARG;
    return shape_rules(P, M, N, K, bands, scale_kind);
}

GEMMAR_API int64_t gemmar_workspace_bytes(const gemmar_ctx *ctx) { return ctx ? ctx->total_bytes : 0; }

GEMMAR_API int gemmar_status(gemmar_ctx *ctx, int *detail)
{
    if (ctx == nullptr)
        return GEMMAR_ERR_ARG;
    ptx::DevStatus st{0, 0};
    if (cudaMemcpy(&st, ctx->status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    if (detail)
        *detail = st.detail;
    if (st.code != 0)
        ctx->disabled = 1;
    return st.code;
}

GEMMAR_API int gemmar_overlap_stats(gemmar_ctx *ctx, int64_t *overlapped, int64_t *total)
{
    if (ctx == nullptr || overlapped == nullptr || total == nullptr)
        return GEMMAR_ERR_ARG;
    *overlapped = 0;
    *total = ctx->ov_total;
    if (ctx->ov_bands == 0)
        return GEMMAR_OK;
    std::vector<uint32_t> claimed((size_t)ctx->ov_bands);
    if (cudaMemcpy(claimed.data(), ctx->band_done + ctx->ov_bands, sizeof(uint32_t) * claimed.size(),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    for (uint32_t c : claimed)   // a counter can pass the band's block count by the claims that found it empty
        *overlapped += std::min<int64_t>(c, ctx->ov_bpb);
    return GEMMAR_OK;
}

GEMMAR_API int gemmar_destroy(gemmar_ctx *ctx)
{
    if (ctx == nullptr)
        return GEMMAR_ERR_ARG;
    int prev = -1;
    cudaGetDevice(&prev);
    if (ctx->device >= 0)
        cudaSetDevice(ctx->device);
    cudaDeviceSynchronize();
    cudaFree(ctx->W);
    cudaFree(ctx->band_done);
    cudaFree(ctx->status);
    cudaFree(ctx->sfa);
    cudaFree(ctx->sfb);
    cudaFree(ctx->wire_q);
    cudaFree(ctx->wire_s);
    for (cudaEvent_t e : ctx->events)
        cudaEventDestroy(e);
    if (prev >= 0)
        cudaSetDevice(prev);
    delete ctx;
    return GEMMAR_OK;
}

GEMMAR_API int gemm_blockscale_fp8(gemmar_ctx *ctx, const uint8_t *A, const float *sa, const uint8_t *B,
                                   const float *sb, void *C, int c_dtype, int64_t M, int64_t N, int64_t K,
                                   void *stream)
{
    return gemm_single(ctx, A, sa, B, sb, C, c_dtype, M, N, K, GEMMAR_SCALE_BLOCK128, stream);
}

GEMMAR_API int gemm_ptpc_fp8(gemmar_ctx *ctx, const uint8_t *A, const float *sa, const uint8_t *B, const float *sb,
                             void *C, int c_dtype, int64_t M, int64_t N, int64_t K, void *stream)
{
    return gemm_single(ctx, A, sa, B, sb, C, c_dtype, M, N, K, GEMMAR_SCALE_PTPC, stream);
}

GEMMAR_API int gemm_mxfp8(gemmar_ctx *ctx, const uint8_t *A, const uint8_t *ea, const uint8_t *B, const uint8_t *eb,
                          void *C, int c_dtype, int64_t M, int64_t N, int64_t K, void *stream)
{
    return gemm_single(ctx, A, ea, B, eb, C, c_dtype, M, N, K, GEMMAR_SCALE_MX32, stream);
}

GEMMAR_API int band_reduce(gemmar_ctx *ctx, const float *W, int P, int64_t M, int64_t N, int bands, uint16_t *out,
                           void *stream)
{
    int rc = check_ctx(ctx);
    if (rc)
        return rc;
    if (!W || !out)
        return GEMMAR_ERR_ARG;
    if (P < 1 || P > kMaxP || M < 1 || N < 1 || bands < 1)
        return GEMMAR_ERR_ARG;
    if (M % bands != 0 || N % 8 != 0 || bands > kMaxBands)
        return GEMMAR_ERR_SHAPE;
    if (!aligned16(W) || !aligned16(out))
        return GEMMAR_ERR_ALIGN;
    CUDA_OK(launch_band_reduce(W, out, P, M, N, bands, nullptr, 0, ctx->status, ctx->timeout_ns, ctx->num_sms,
                               as_stream(stream)));
    return GEMMAR_OK;
}

GEMMAR_API int rowquant_e4m3(gemmar_ctx *ctx, const void *x, int x_dtype, int64_t M, int64_t N, uint8_t *q,
                             float *row_scale, void *stream)
{
    int rc = check_ctx(ctx);
    if (rc)
        return rc;
    if (!x || !q || !row_scale || (x_dtype != GEMMAR_DTYPE_F32 && x_dtype != GEMMAR_DTYPE_BF16) || M < 1 || N < 1)
        return GEMMAR_ERR_ARG;
    if (N % 16 != 0)
        return GEMMAR_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(row_scale))
        return GEMMAR_ERR_ALIGN;
    CUDA_OK(launch_rowquant(x, x_dtype == GEMMAR_DTYPE_BF16, M, N, q, row_scale, ctx->num_sms, as_stream(stream)));
    return GEMMAR_OK;
}

GEMMAR_API int rowdequant_e4m3(gemmar_ctx *ctx, const uint8_t *q, const float *row_scale, int64_t M, int64_t N,
                               uint16_t *y, void *stream)
{
    int rc = check_ctx(ctx);
    if (rc)
        return rc;
    if (!q || !row_scale || !y || M < 1 || N < 1)
        return GEMMAR_ERR_ARG;
    if (N % 16 != 0)
        return GEMMAR_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(row_scale) || !aligned16(y))
        return GEMMAR_ERR_ALIGN;
    CUDA_OK(launch_rowdequant(q, row_scale, M, N, y, ctx->num_sms, as_stream(stream)));
    return GEMMAR_OK;
}

GEMMAR_API int quant_blockscale_e4m3(gemmar_ctx *ctx, const void *x, int x_dtype, int64_t R, int64_t C,
                                     int group_rows, uint8_t *q, float *scales, void *stream)
{
    int rc = check_ctx(ctx);
    if (rc)
        return rc;
    if (!x || !q || !scales || R < 1 || C < 1 || (group_rows != 1 && group_rows != 128) ||
        (x_dtype != GEMMAR_DTYPE_F32 && x_dtype != GEMMAR_DTYPE_BF16))
        return GEMMAR_ERR_ARG;
    if (C % 128 != 0)
        return GEMMAR_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scales))
        return GEMMAR_ERR_ALIGN;
    CUDA_OK(launch_quant_blockscale(x, x_dtype == GEMMAR_DTYPE_BF16, R, C, group_rows, q, scales, ctx->num_sms,
                                    as_stream(stream)));
    return GEMMAR_OK;
}

GEMMAR_API int quant_mx_e4m3(gemmar_ctx *ctx, const void *x, int x_dtype, int64_t R, int64_t C, uint8_t *q,
                             uint8_t *e8m0, void *stream)
{
    int rc = check_ctx(ctx);
    if (rc)
        return rc;
    if (!x || !q || !e8m0 || R < 1 || C < 1 || (x_dtype != GEMMAR_DTYPE_F32 && x_dtype != GEMMAR_DTYPE_BF16))
        return GEMMAR_ERR_ARG;
    if (C % 32 != 0)
        return GEMMAR_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(e8m0))
        return GEMMAR_ERR_ALIGN;
    CUDA_OK(launch_quant_mx(x, x_dtype == GEMMAR_DTYPE_BF16, R, C, q, e8m0, ctx->num_sms, as_stream(stream)));
    return GEMMAR_OK;
}

GEMMAR_API int fused_gemm_reduce(gemmar_ctx *ctx, int P, const uint8_t *const *A, const void *const *sa,
                                 const uint8_t *const *B, const void *const *sb, int scale_kind, int64_t M,
                                 int64_t N, int64_t K, int bands, uint32_t flags, uint16_t *out, void *stream)
{
    int rc = check_ctx(ctx);
    if (rc)
        return rc;
    if (!A || !sa || !B || !sb || !out || !known_scale_kind(scale_kind))
        return GEMMAR_ERR_ARG;
    if (bands == 0)
        bands = P;
    if ((rc = shape_rules(P, M, N, K, bands, scale_kind)))
        return rc;
    for (int p = 0; p < P; ++p) {
        if (!A[p] || !sa[p] || !B[p] || !sb[p])
            return GEMMAR_ERR_ARG;
        if (!aligned16(A[p]) || !aligned16(sa[p]) || !aligned16(B[p]) || !aligned16(sb[p]))
            return GEMMAR_ERR_ALIGN;
    }
    if (!aligned16(out))
        return GEMMAR_ERR_ALIGN;
    // on-chip partial sums: mx on the mx kernel, blockscale on the CTA-pair kernel
    // (N % 256 == 0); other blockscale shapes take the band path, whose bits they reproduce
    // ptpc applies its scales after the whole K of a slice, so its only in-tile
    // reduction is the on-chip one (GEMMAR_FUSE_SLICES takes it too)
    const bool onchip = ((flags & GEMMAR_FUSE_ONCHIP) ||
                         (scale_kind == GEMMAR_SCALE_PTPC && (flags & GEMMAR_FUSE_SLICES))) &&
                        (scale_kind != GEMMAR_SCALE_BLOCK128 || plan_blockscale(P, M, N, K, bands, 2, ctx->num_sms, 1).pair);
    const bool slices = onchip || ((flags & GEMMAR_FUSE_SLICES) != 0 && !(flags & GEMMAR_FUSE_ONCHIP));
    if (!slices && blocked_partial_floats(P, M, bands, N) > ctx->W_floats)
        return GEMMAR_ERR_WORKSPACE;
    if ((flags & GEMMAR_FP8_WIRE) && M * N > ctx->max_M * ctx->N)
        return GEMMAR_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    ctx->ov_bands = 0;
    ctx->ov_total = 0;
    // fp8 wire on the band path: the band reduce can quantise the rows itself
    const bool fuse_q = !slices && (flags & GEMMAR_FP8_WIRE) && (flags & GEMMAR_FUSE_QUANTIZE) &&
                        N <= kBandQuantMaxN;
    if (slices) {
        // every tile accumulates all P slices itself: no partials, no band reduce
        if (flags & GEMMAR_DEBUG_CANARY)
            CUDA_OK(cudaMemsetAsync(out, 0xFF, sizeof(uint16_t) * (size_t)(M * N), st));
        mark(ctx, GEMMAR_PHASE_GEMM, st);
        GemmOut os{out, nullptr, OUT_BF16, -1};
        if ((rc = run_gemm(ctx, P, A, sa, B, sb, scale_kind, M, N, K, 1, os, st, onchip ? 2 : 1)))
            return rc;
        mark(ctx, GEMMAR_PHASE_REDUCE, st);
    } else {
        int bn;
        uint32_t expected;   // every epilogue warp signals once per retired tile
        bool inkernel = false;   // the GEMM's reducer warps take the bands that retire while it runs
        if (scale_kind == GEMMAR_SCALE_BLOCK128) {
            const BsPlan pl = plan_blockscale(P, M, N, K, bands, 0, ctx->num_sms,
                                              (ctx->flags & GEMMAR_CTA_PAIR) ? 1 : 0);
            bn = pl.bn;
            expected = pl.band_signals;
            inkernel = !pl.pair && !(flags & GEMMAR_SERIAL_REDUCE);
        } else {
            bn = scale_kind == GEMMAR_SCALE_PTPC ? ptpc_tile_n(N) : mx_tile_n(N);
            const TileGrid g = make_grid(P, M, N, K, bands, bn);
            expected = (uint32_t)(g.mt_per_band * g.ntiles_n * P * 8);
            inkernel = !(flags & GEMMAR_SERIAL_REDUCE);
        }
        // band retire counters, then the reducer warps' per-band claim counters
        uint32_t *claim = ctx->band_done + bands;
        CUDA_OK(cudaMemsetAsync(ctx->band_done, 0, sizeof(uint32_t) * 2 * bands, st));
        if (flags & GEMMAR_DEBUG_CANARY) {
            CUDA_OK(cudaMemsetAsync(ctx->W, 0xFF, sizeof(float) * (size_t)blocked_partial_floats(P, M, bands, N), st));
            CUDA_OK(cudaMemsetAsync(out, 0xFF, sizeof(uint16_t) * (size_t)(M * N), st));
        }
        GemmOut o{ctx->W, ctx->band_done, OUT_PARTIAL_F32, (flags & GEMMAR_FAULT_SKIP_BAND) ? 0 : -1,
                  inkernel ? claim : nullptr, out, expected};
        {
            const int64_t mtpb = (M / bands + 127) / 128;
            ctx->ov_bpb = mtpb * (N / bn) * 4 * (bn / 32);
            ctx->ov_bands = inkernel ? bands : 0;
            ctx->ov_total = inkernel ? ctx->ov_bpb * bands : 0;
        }
        mark(ctx, GEMMAR_PHASE_GEMM, st);
        if ((rc = run_gemm(ctx, P, A, sa, B, sb, scale_kind, M, N, K, bands, o, st)))
            return rc;
        mark(ctx, GEMMAR_PHASE_REDUCE, st);
        if (fuse_q) {
            // the remaining blocks' sums go straight to the row quantiser
            CUDA_OK(launch_band_reduce_quant(ctx->W, out, P, M, N, bands, bn, ctx->band_done, expected,
                                             inkernel ? claim : nullptr, ctx->wire_q, ctx->wire_s, ctx->status,
                                             ctx->timeout_ns, st));
        } else {
            CUDA_OK(launch_band_reduce_blocked(ctx->W, out, P, M, N, bands, bn, ctx->band_done, expected,
                                               inkernel ? claim : nullptr, ctx->status, ctx->timeout_ns,
                                               ctx->num_sms, st));
        }
    }
    mark(ctx, GEMMAR_PHASE_QUANTIZE, st);
    if ((flags & GEMMAR_FP8_WIRE) && !fuse_q)
        CUDA_OK(launch_rowquant(out, 1, M, N, ctx->wire_q, ctx->wire_s, ctx->num_sms, st));
    mark(ctx, GEMMAR_PHASE_DEQUANTIZE, st);
    if (flags & GEMMAR_FP8_WIRE)
        CUDA_OK(launch_rowdequant(ctx->wire_q, ctx->wire_s, M, N, out, ctx->num_sms, st));
    mark(ctx, GEMMAR_NUM_PHASES, st);
    if (ctx->timing && ctx->recorded < kMaxTimedCalls)
        ++ctx->recorded;
    return GEMMAR_OK;
}

GEMMAR_API int gemmar_set_phase_timing(gemmar_ctx *ctx, int enable)
{
    if (ctx == nullptr)
        return GEMMAR_ERR_ARG;
    ctx->timing = enable ? 1 : 0;
    return GEMMAR_OK;
}

GEMMAR_API int gemmar_phase_times(gemmar_ctx *ctx, float *ms, int *calls)
{
    if (ctx == nullptr || ms == nullptr)
        return GEMMAR_ERR_ARG;
    for (int ph = 0; ph < GEMMAR_NUM_PHASES; ++ph)
        ms[ph] = 0.0f;
    for (int c = 0; c < ctx->recorded; ++c) {
        cudaEvent_t *ev = &ctx->events[(size_t)c * kEventsPerCall];
        if (cudaEventSynchronize(ev[GEMMAR_NUM_PHASES]) != cudaSuccess)
            return GEMMAR_ERR_CUDA;
        for (int ph = 0; ph < GEMMAR_NUM_PHASES; ++ph) {
            float t = 0.0f;
            if (cudaEventElapsedTime(&t, ev[ph], ev[ph + 1]) != cudaSuccess)
                return GEMMAR_ERR_CUDA;
            ms[ph] += t;
        }
    }
    if (calls)
        *calls = ctx->recorded;
    ctx->recorded = 0;
    return GEMMAR_OK;
}

// ---------------------------------------------------------------- create + self-test

namespace {

// Closed-form self-test: every code 0x38 (= 1.0), every scale 1 (fp32 1.0 or
// ue8m0 byte 127) -> every output equals P * K exactly.
int self_test(gemmar_ctx *ctx)
{
    const int P = std::min(2, ctx->max_P);
    const int64_t M = 128 * P, N = 256, K = 128;
    if ((int64_t)P * M * N > ctx->W_floats || ctx->N < N || ctx->K < K || ctx->max_M < M)
        return GEMMAR_OK;   // workspace too small for the test shape: nothing to run
    uint8_t *ops = nullptr;
    const size_t a_bytes = M * K, b_bytes = N * K;
    const size_t sa_bytes = M * (K / 32) * 4 + 64, sb_bytes = N * (K / 32) * 4 + 64;
    const size_t out_bytes = M * N * 2;
    const size_t total = a_bytes + b_bytes + sa_bytes + sb_bytes + out_bytes + 5 * 256;
    if (cudaMalloc(&ops, total) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    uint8_t *dA = ops, *dB = dA + al(a_bytes);
    uint8_t *dsa = dB + al(b_bytes), *dsb = dsa + al(sa_bytes);
    uint16_t *dout = reinterpret_cast<uint16_t *>(dsb + al(sb_bytes));
    int rc = GEMMAR_OK;
    cudaStream_t st;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
        cudaFree(ops);
        return GEMMAR_ERR_CUDA;
    }
    std::vector<float> ones(std::max(sa_bytes, sb_bytes) / 4, 1.0f);
    std::vector<uint16_t> host(M * N);
    // every scale kind, on the band path and with the partials summed on chip
    for (int run = 0; run < 6 && rc == GEMMAR_OK; ++run) {
        const int kind = run % 3;
        const uint32_t flags = run < 3 ? 0u : GEMMAR_FUSE_ONCHIP;
        const uint16_t expect = (P * K == 256) ? 0x4380 : 0x4300;   // bf16 of 256 (P=2) or 128 (P=1)
        bool ok = cudaMemsetAsync(dA, 0x38, a_bytes, st) == cudaSuccess &&
                  cudaMemsetAsync(dB, 0x38, b_bytes, st) == cudaSuccess;
        if (kind == GEMMAR_SCALE_BLOCK128)
            ok = ok && cudaMemcpyAsync(dsa, ones.data(), M * (K / 128) * 4, cudaMemcpyHostToDevice, st) == cudaSuccess &&
                 cudaMemcpyAsync(dsb, ones.data(), (N / 128) * (K / 128) * 4, cudaMemcpyHostToDevice, st) == cudaSuccess;
        else if (kind == GEMMAR_SCALE_MX32)
            ok = ok && cudaMemsetAsync(dsa, 127, M * (K / 32), st) == cudaSuccess &&
                 cudaMemsetAsync(dsb, 127, N * (K / 32), st) == cudaSuccess;
        else
            ok = ok && cudaMemcpyAsync(dsa, ones.data(), M * 4, cudaMemcpyHostToDevice, st) == cudaSuccess &&
                 cudaMemcpyAsync(dsb, ones.data(), N * 4, cudaMemcpyHostToDevice, st) == cudaSuccess;
        ok = ok && cudaMemsetAsync(dout, 0, out_bytes, st) == cudaSuccess;
        if (!ok) {
            rc = GEMMAR_ERR_CUDA;
            break;
        }
        const uint8_t *As[2] = {dA, dA}, *Bs[2] = {dB, dB};
        const void *SA[2] = {dsa, dsa}, *SB[2] = {dsb, dsb};
        rc = fused_gemm_reduce(ctx, P, As, SA, Bs, SB, kind, M, N, K, P, flags, dout, st);
        if (rc == GEMMAR_OK && cudaStreamSynchronize(st) != cudaSuccess)
            rc = GEMMAR_ERR_CUDA;
        if (rc == GEMMAR_OK)
            rc = gemmar_status(ctx, nullptr);
        if (rc == GEMMAR_OK) {
            if (cudaMemcpy(host.data(), dout, out_bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
                rc = GEMMAR_ERR_CUDA;
            else
                for (size_t i = 0; i < host.size(); ++i)
                    if (host[i] != expect) {
                        rc = GEMMAR_ERR_DEVICE;
                        break;
                    }
        }
    }
    cudaStreamDestroy(st);
    cudaFree(ops);
    return rc;
}

}  // namespace

GEMMAR_API int gemmar_create(gemmar_ctx **out, int device, int64_t max_M, int64_t N, int64_t K, int max_P,
                             uint32_t flags, int64_t wait_timeout_ns)
{
    if (out == nullptr)
        return GEMMAR_ERR_ARG;
    *out = nullptr;
    if (max_P < 1 || max_P > kMaxP || max_M < 1 || N < 1 || K < 1 || wait_timeout_ns < 0)
        return GEMMAR_ERR_ARG;
    if ((N % 128 != 0 && N % 224 != 0) || K % 128 != 0 || N > 65536 || K > 65536 || max_M > (int64_t(1) << 24))
        return GEMMAR_ERR_SHAPE;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    if (cur != device)
        return GEMMAR_ERR_DEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    if (!(prop.major == 10 && prop.minor == 3))
        return GEMMAR_ERR_DEVICE;   // built for sm_103a only
    if (!load_encode())
        return GEMMAR_ERR_CUDA;

    gemmar_ctx *ctx = new gemmar_ctx();
    ctx->device = device;
    ctx->num_sms = prop.multiProcessorCount;
    ctx->max_M = max_M;
    ctx->N = N;
    ctx->K = K;
    ctx->max_P = max_P;
    ctx->flags = flags;
    ctx->timeout_ns = wait_timeout_ns > 0 ? (uint64_t)wait_timeout_ns : 2000000000ull;
    // fp32 partials in the tile-blocked layout: every band padded to whole
    // 128-row tiles, for up to max_P bands
    ctx->W_floats = (int64_t)max_P * (max_M + 128 * max_P) * N;
    // mx repack images, sized for the largest tile count any band split can give
    ctx->sfa_bytes = (int64_t)max_P * ((max_M + 127) / 128 + kMaxBands) * (K / 128) * 512;
    ctx->sfb_bytes = (int64_t)max_P * (N / 128) * (K / 128) * 1024;
    int rc = GEMMAR_OK;
    auto alloc = [&](void **p, size_t bytes) {
        if (rc == GEMMAR_OK && cudaMalloc(p, bytes) != cudaSuccess)
            rc = GEMMAR_ERR_CUDA;
        if (rc == GEMMAR_OK)
            ctx->total_bytes += (int64_t)bytes;
    };
    alloc(reinterpret_cast<void **>(&ctx->W), sizeof(float) * (size_t)ctx->W_floats);
    alloc(reinterpret_cast<void **>(&ctx->band_done), sizeof(uint32_t) * 2 * kMaxBands);   // + claim counters
    alloc(reinterpret_cast<void **>(&ctx->status), sizeof(ptx::DevStatus));
    alloc(reinterpret_cast<void **>(&ctx->sfa), (size_t)ctx->sfa_bytes);
    alloc(reinterpret_cast<void **>(&ctx->sfb), (size_t)ctx->sfb_bytes);
    alloc(reinterpret_cast<void **>(&ctx->wire_q), (size_t)(max_M * N));
    alloc(reinterpret_cast<void **>(&ctx->wire_s), sizeof(float) * (size_t)max_M);
    if (rc == GEMMAR_OK && cudaMemset(ctx->status, 0, sizeof(ptx::DevStatus)) != cudaSuccess)
        rc = GEMMAR_ERR_CUDA;
    if (rc == GEMMAR_OK && !register_split_ok(256))
        rc = GEMMAR_ERR_DEVICE;
    if (rc == GEMMAR_OK && !(flags & GEMMAR_NO_SELF_TEST))
        rc = self_test(ctx);
    if (rc != GEMMAR_OK) {
        gemmar_destroy(ctx);
        return rc;
    }
    *out = ctx;
    return GEMMAR_OK;
}
