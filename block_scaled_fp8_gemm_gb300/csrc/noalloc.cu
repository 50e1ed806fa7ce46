// noalloc.cu -- fused_gemm_reduce_noalloc: the blockscale fused GEMM + band
// reduce for callers that cannot allocate device memory.
//
// Who needs it: engines that reserve all of the GPU's memory for their own
// pool at start-up and forbid any later cudaMalloc (a late allocation would
// fail or split their arena), and host frameworks that load this library as
// a plugin and require every device byte to come from the host's allocator.
// Such callers cannot create a gemmar_ctx, because gemmar_create allocates the
// workspace.  This entry point instead keeps its scratch -- the fp32 partials,
// the band counters and the device status word -- in file-scope __device__
// arrays of a fixed size that the CUDA driver reserves when it loads this
// library's device code on a GPU, and keeps until the process exits.
//
// The kernels are the ones fused_gemm_reduce launches (same tiles, same
// fixed-order reduce), so the result equals that call's bit for bit.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "gemmar.h"
#include "kernels.h"

using namespace gemmar;

// Scratch shared by every call on a device.  The name of each array is, in
// host code, only a stand-in for the symbol: the device address comes from
// cudaGetSymbolAddress (see scratch_for_device).
static __device__ __align__(256) float g_noalloc_partials[GEMMAR_NOALLOC_MAX_PARTIALS];
static __device__ __align__(256) uint32_t g_noalloc_band_done[2 * 1024];   // retire, then claim counters
static __device__ __align__(256) ptx::DevStatus g_noalloc_status;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct Scratch {
    bool ready = false;
    float *partials = nullptr;
    uint32_t *band_done = nullptr;
    ptx::DevStatus *status = nullptr;
    int num_sms = 0;
};

Scratch g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode_na = nullptr;

// Device addresses of the scratch arrays on `device` (which must be current),
// looked up once per device.
int scratch_for_device(int device, Scratch **out)
{
    if (device < 0 || device >= kMaxDevices)
        return GEMMAR_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    Scratch &s = g_scratch[device];
    if (!s.ready) {
        if (g_encode_na == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess)
                return GEMMAR_ERR_CUDA;
            g_encode_na = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, device) != cudaSuccess)
            return GEMMAR_ERR_CUDA;
        if (!(prop.major == 10 && prop.minor == 3))
            return GEMMAR_ERR_DEVICE;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&s.partials), g_noalloc_partials) != cudaSuccess ||
            cudaGetSymbolAddress(reinterpret_cast<void **>(&s.band_done), g_noalloc_band_done) != cudaSuccess ||
            cudaGetSymbolAddress(reinterpret_cast<void **>(&s.status), g_noalloc_status) != cudaSuccess)
            return GEMMAR_ERR_CUDA;
        s.num_sms = prop.multiProcessorCount;
        s.ready = true;
    }
    *out = &s;
    return GEMMAR_OK;
}

bool tmap_u8(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int box_rows)
{
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    return g_encode_na(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" __attribute__((visibility("default"))) int fused_gemm_reduce_noalloc(
    int P, const uint8_t *const *A, const float *const *sa, const uint8_t *const *B, const float *const *sb,
    int64_t M, int64_t N, int64_t K, int bands, uint16_t *out, void *stream)
{
    if (!A || !sa || !B || !sb || !out)
        return GEMMAR_ERR_ARG;
    if (bands == 0)
        bands = P;
    if (P < 1 || P > kMaxP || M < 1 || N < 1 || K < 1 || bands < 1)
        return GEMMAR_ERR_ARG;
    if (bands > 1024 || bands > M || M % bands != 0 || N % 128 != 0 || K % 128 != 0 || N > 65536 || K > 65536 ||
        M > (int64_t(1) << 24))
        return GEMMAR_ERR_SHAPE;
    if (blocked_partial_floats(P, M, bands, N) > GEMMAR_NOALLOC_MAX_PARTIALS)
        return GEMMAR_ERR_WORKSPACE;   // beyond the fixed scratch: use fused_gemm_reduce
    for (int p = 0; p < P; ++p) {
        if (!A[p] || !sa[p] || !B[p] || !sb[p])
            return GEMMAR_ERR_ARG;
        if (!al16(A[p]) || !al16(sa[p]) || !al16(B[p]) || !al16(sb[p]))
            return GEMMAR_ERR_ALIGN;
    }
    if (!al16(out))
        return GEMMAR_ERR_ALIGN;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    Scratch *s = nullptr;
    int rc = scratch_for_device(device, &s);
    if (rc != GEMMAR_OK)
        return rc;
    const BsPlan pl = plan_blockscale(P, M, N, K, bands, 0, s->num_sms);
    if (!pl.pair) {
        if (!gemm_blockscale_split_ok(pl.bn))
            return GEMMAR_ERR_DEVICE;
    }
    const int bn = pl.bn;

    BsParams prm;
    std::memset(&prm, 0, sizeof(prm));
    for (int p = 0; p < P; ++p) {
        if (!tmap_u8(&prm.tmA[p], A[p], M, K, 128) || !tmap_u8(&prm.tmB[p], B[p], N, K, pl.box_b_rows))
            return GEMMAR_ERR_CUDA;
        prm.sa[p] = sa[p];
        prm.sb[p] = sb[p];
    }
    prm.g = pl.g;
    // one-CTA plans run the GEMM kernel's reducer warps: claim counters after the retire counters
    uint32_t *claim = pl.pair ? nullptr : s->band_done + bands;
    prm.o = GemmOut{s->partials, s->band_done, OUT_PARTIAL_F32, -1, claim, out, pl.band_signals};
    prm.status = s->status;
    prm.timeout_ns = kTimeoutNs;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the counters and the status word keep the previous call's values: clear them
    if (cudaMemsetAsync(s->band_done, 0, sizeof(uint32_t) * 2 * bands, st) != cudaSuccess ||
        cudaMemsetAsync(s->status, 0, sizeof(ptx::DevStatus), st) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    if (launch_blockscale(prm, pl, st) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    const uint32_t expected = pl.band_signals;
    if (launch_band_reduce_blocked(s->partials, out, P, M, N, bands, bn, s->band_done, expected, claim, s->status,
                                   kTimeoutNs, s->num_sms, st) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    return GEMMAR_OK;
}

extern "C" __attribute__((visibility("default"))) int fused_gemm_reduce_noalloc_status(int *detail)
{
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    if (device < 0 || device >= kMaxDevices)
        return GEMMAR_ERR_DEVICE;
    ptx::DevStatus *dst = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        if (!g_scratch[device].ready)
            return GEMMAR_ERR_DEVICE;   // no call on this device yet
        dst = g_scratch[device].status;
    }
    ptx::DevStatus st{};
    if (cudaMemcpy(&st, dst, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMMAR_ERR_CUDA;
    if (detail)
        *detail = st.detail;
    return st.code == 0 ? GEMMAR_OK : st.code;
}
