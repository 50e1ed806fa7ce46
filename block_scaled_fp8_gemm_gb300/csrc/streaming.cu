// streaming.cu -- the HBM-bound kernels of the path: the fixed-order band
// reduce, the per-row e4m3 codec (fp8 wire), the device quantisers and the
// mxfp8 scale repack.  All are coalesced, 16-byte vectorised, grid-stride
// kernels sized in multiples of the SM count.
#include <cuda_bf16.h>

#include <atomic>

#include "kernels.h"

namespace gemmar {
using namespace ptx;

namespace {

__host__ __device__ inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ float4 ldcg4(const float *p) { return __ldcg(reinterpret_cast<const float4 *>(p)); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// --------------------------------------------------------------------------
// band_reduce: out[m,n] = bf16_rn(((W[b][0] + W[b][1]) + ...) + W[b][P-1]), fp32,
// p ascending.  One thread reduces 8 consecutive columns of one row across all
// P slices with 2P independent 16-byte loads in flight.  When band_done is
// given, the CTA first waits (bounded) until that band's tiles have all
// retired; the counter is read with acquire semantics and W with L2-coherent
// (.cg) loads.
// --------------------------------------------------------------------------
template <int P>
__global__ void __launch_bounds__(256) band_reduce_kernel(const float *__restrict__ W, uint16_t *__restrict__ out,
                                                          int64_t rows_per_band, int64_t N, int bands,
                                                          const uint32_t *band_done, uint32_t expected,
                                                          DevStatus *status, uint64_t timeout_ns)
{
    __shared__ int band_ok;
    const int64_t band_elems = rows_per_band * N;
    const int64_t npk = band_elems / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int b = 0; b < bands; ++b) {
        if (band_done != nullptr) {
            if (threadIdx.x == 0) {
                int ok = 1;
                if (ld_acquire(band_done + b) < expected) {
                    const uint64_t t0 = globaltimer();
                    while (ld_acquire(band_done + b) < expected) {
                        if (*(volatile int *)&status->code != 0) { ok = 0; break; }
                        if (globaltimer() - t0 > timeout_ns) {
                            report(status, kErrTimeout, SITE_REDUCE_BAND);
                            ok = 0;
                            break;
                        }
                        __nanosleep(256);
                    }
                }
                band_ok = ok;
            }
            __syncthreads();
            if (!band_ok)
                return;
        }
        const float *Wb = W + (int64_t)b * P * band_elems;
        uint16_t *ob = out + (int64_t)b * band_elems;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < npk; i += stride) {
            const float *src = Wb + i * 8;
            float4 lo[P], hi[P];
#pragma unroll
            for (int p = 0; p < P; ++p) {
                lo[p] = ldcg4(src + p * band_elems);
                hi[p] = ldcg4(src + p * band_elems + 4);
            }
            float4 a = lo[0], c = hi[0];
#pragma unroll
            for (int p = 1; p < P; ++p) {
                a.x = a.x + lo[p].x; a.y = a.y + lo[p].y; a.z = a.z + lo[p].z; a.w = a.w + lo[p].w;
                c.x = c.x + hi[p].x; c.y = c.y + hi[p].y; c.z = c.z + hi[p].z; c.w = c.w + hi[p].w;
            }
            uint4 o;
            o.x = bf16x2_from_f32(a.x, a.y);
            o.y = bf16x2_from_f32(a.z, a.w);
            o.z = bf16x2_from_f32(c.x, c.y);
            o.w = bf16x2_from_f32(c.z, c.w);
            *reinterpret_cast<uint4 *>(ob + i * 8) = o;
        }
    }
}

// --------------------------------------------------------------------------
// band_reduce over the fused path's blocked partials (layout: epilogue.cuh).
// One warp reduces one 32-row x 32-column block of a tile: for each of its
// 8 column units it loads the unit from every slice (512 contiguous bytes per
// slice and warp), sums in fp32 with p ascending, rounds to bf16 and parks
// the row's 64 bytes in registers; a warp-private shared transpose then
// writes 8 rows x 64 bytes per store instruction.  Rows past the band end
// (ragged bands) are not written.  Same arithmetic as band_reduce_kernel.
// Blocks are numbered within a band (column chunk fastest, then lane quarter,
// then tile); with `claimed` the kernel starts band b at block claimed[b], the
// ones before it having been reduced by the GEMM kernel's reducer warps.
// --------------------------------------------------------------------------
template <int P>
__global__ void __launch_bounds__(256, 2) band_reduce_blocked_kernel(const float4 *__restrict__ W,
                                                                  uint16_t *__restrict__ out, int M, int N,
                                                                  int bands, int rows_per_band, int mt_per_band,
                                                                  int ntiles_n, int bn, const uint32_t *band_done,
                                                                  uint32_t expected, const uint32_t *claimed,
                                                                  DevStatus *status, uint64_t timeout_ns)
{
    __shared__ __align__(16) uint32_t stage[8][32 * 16];   // per warp: 32 rows x 64 bytes
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nchunk = bn / 32;
    const int64_t tiles_per_band = (int64_t)mt_per_band * ntiles_n;
    const int64_t blocks_per_band = tiles_per_band * 4 * nchunk;   // (tile, q, c) blocks
    const int64_t tile_f4 = 128 * bn / 4;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    uint32_t *st = stage[warp];
    for (int b = 0; b < bands; ++b) {
        if (band_done != nullptr) {
            // each warp checks the band itself: no CTA-wide barrier per band, so a
            // warp with fewer blocks in the last band moves on to the next one
            int ok = 1;
            if (lane == 0 && ld_acquire(band_done + b) < expected) {
                const uint64_t t0 = globaltimer();
                while (ld_acquire(band_done + b) < expected) {
                    if (*(volatile int *)&status->code != 0) { ok = 0; break; }
                    if (globaltimer() - t0 > timeout_ns) {
                        report(status, kErrTimeout, SITE_REDUCE_BAND);
                        ok = 0;
                        break;
                    }
                    __nanosleep(256);
                }
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            __syncwarp();
            if (!ok)
                return;
        }
        const int64_t blk0 = claimed != nullptr ? min64((int64_t)claimed[b], blocks_per_band) : 0;
        if (blk0 >= blocks_per_band)
            continue;
        for (int64_t blk = blk0 + (int64_t)blockIdx.x * (blockDim.x >> 5) + warp; blk < blocks_per_band;
             blk += warps_total) {
            const int c = (int)(blk % nchunk);
            const int q = (int)((blk / nchunk) % 4);
            const int64_t i = blk / (4 * nchunk);
            const int mt = (int)(i / ntiles_n), nt = (int)(i % ntiles_n);
            // float4 index of (band b, slice 0, tile i, q, c, unit 0, lane)
            const float4 *src = W + ((int64_t)b * P * tiles_per_band + i) * tile_f4 + ((q * nchunk + c) * 8) * 32 + lane;
            uint32_t o[16];
            // the next item's P loads are issued before this item is summed: two items
            // (2P 16-byte loads per lane) in flight keep HBM busy at two CTAs per SM
            float4 nx[P];
#pragma unroll
            for (int p = 0; p < P; ++p)
                nx[p] = __ldcs(src + (int64_t)p * tiles_per_band * tile_f4);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                float4 v[P];
#pragma unroll
                for (int p = 0; p < P; ++p)
                    v[p] = nx[p];
                if (u + 1 < 8) {
#pragma unroll
                    for (int p = 0; p < P; ++p)
                        nx[p] = __ldcs(src + (int64_t)p * tiles_per_band * tile_f4 + (u + 1) * 32);
                }
                float4 a = v[0];
#pragma unroll
                for (int p = 1; p < P; ++p) {
                    a.x = a.x + v[p].x; a.y = a.y + v[p].y; a.z = a.z + v[p].z; a.w = a.w + v[p].w;
                }
                o[2 * u] = bf16x2_from_f32(a.x, a.y);
                o[2 * u + 1] = bf16x2_from_f32(a.z, a.w);
            }
            // transpose: row `lane` holds 64 bytes (16 words), XOR-swizzled by 16-byte unit
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4 *>(st + lane * 16 + ((j ^ ((lane >> 1) & 3)) * 4)) =
                    make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            __syncwarp();
            const int row0 = mt * 128 + q * 32;                      // tile row within the band
            const int64_t col = (int64_t)nt * bn + c * 32;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int r = k * 8 + (lane >> 2), j = lane & 3;
                const uint4 val = *reinterpret_cast<const uint4 *>(st + r * 16 + ((j ^ ((r >> 1) & 3)) * 4));
                if (row0 + r < rows_per_band) {
                    const int64_t m = (int64_t)b * rows_per_band + row0 + r;
                    *reinterpret_cast<uint4 *>(out + m * N + col + j * 8) = val;
                }
            }
            __syncwarp();
        }
    }
}

// --------------------------------------------------------------------------
// rowquant: one warp per row.  Pass 1 streams the row for its amax (warp
// shuffle max); pass 2 re-reads it (L1/L2 hit) and writes the codes.
// s = fp32(amax / 448) and codes = e4m3_rn_sat(fp32(x / s)), IEEE divisions.
// --------------------------------------------------------------------------
template <bool BF16>
__device__ __forceinline__ void load8(const void *x, int64_t idx, float (&v)[8])
{
    if constexpr (BF16) {
        uint4 w = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(x) + idx);
        v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
        v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
    } else {
        const float *f = reinterpret_cast<const float *>(x) + idx;
        float4 a = *reinterpret_cast<const float4 *>(f);
        float4 b = *reinterpret_cast<const float4 *>(f + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

__device__ __forceinline__ uint32_t enc4(float a, float b, float c, float d, float s)
{
    if (s == 0.0f)
        return 0u;
    uint32_t lo = e4m3x2_from_f32(__fdiv_rn(a, s), __fdiv_rn(b, s));
    uint32_t hi = e4m3x2_from_f32(__fdiv_rn(c, s), __fdiv_rn(d, s));
    return lo | (hi << 16);
}

// e4m3 codes of RN(a/s) and RN(b/s) without dividing, given yl = RN(y(1 - 2^-21))
// and yh = RN(y(1 + 2^-21)) for y = RN(1/s) (s > 0, y a normal number).  The
// products l = RN(a yl) and h = RN(a yh) are a/s times (1 -+ 2^-21) and three
// rounding factors, each within 2^-24 of 1; (1 + 2^-24)^3 < 1 + 2^-21, so |l| <
// |a/s| < |h| (below the normal range, all three round to a zero code anyway).
// Rounding to e4m3 (nearest-even, saturating) is monotone, so when l and h give
// the same code every value between them does, RN(a/s) included.  Otherwise a/s
// lies within ~2^-21 of a code midpoint: divide exactly.  With bf16 inputs this
// happens to ~0.5% of the values (x 448 / amax is then exactly a midpoint), so
// the division stays per pair: a fallback for a whole lane's values would be
// taken by most warps.
__device__ __forceinline__ uint32_t enc2_guarded(float a, float b, float s, float yl, float yh)
{
    // the products two per packed instruction
    const float2 l = mul2(a, b, yl, yl);
    const float2 h = mul2(a, b, yh, yh);
    const uint32_t lo = e4m3x2_from_f32(l.x, l.y);
    const uint32_t hi = e4m3x2_from_f32(h.x, h.y);
    if (lo == hi)
        return lo;
    return e4m3x2_from_f32(__fdiv_rn(a, s), __fdiv_rn(b, s));
}

// Row/group encoder: the guarded products when 1/s is a normal number below
// 2^125, exact division otherwise (s == 0 gives +0 codes).  s = amax / 448 is at
// most FLT_MAX / 448, so y is never subnormal; s = inf gives y = 0 and products
// equal to the exact quotients' codes (+-0, and NaN for an infinite input).
struct Enc {
    float s, yl, yh;
    bool fast;
    __device__ __forceinline__ explicit Enc(float sc) : s(sc)
    {
        const float y = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
        yl = __fmul_rn(y, 1.0f - 0x1p-21f);
        yh = __fmul_rn(y, 1.0f + 0x1p-21f);
        fast = sc >= 0x1p-125f;   // 1/s <= 2^125: finite, and y (1 + 2^-21) cannot overflow
    }
    // from the fields of an encoder built earlier (kept in shared memory)
    __device__ __forceinline__ Enc(float sc, float yl_, float yh_, bool fast_) : s(sc), yl(yl_), yh(yh_), fast(fast_) {}
    __device__ __forceinline__ uint32_t operator()(float a, float b, float c, float d) const
    {
        if (!fast)
            return enc4(a, b, c, d, s);
        return enc2_guarded(a, b, s, yl, yh) | (enc2_guarded(c, d, s, yl, yh) << 16);
    }
};

template <bool BF16>
__global__ void __launch_bounds__(256) rowquant_kernel(const void *__restrict__ x, int64_t M, int64_t N,
                                                       uint8_t *__restrict__ q, float *__restrict__ s)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < M; row += warps_total) {
        const int64_t base = row * N;
        float amax = 0.0f;
#pragma unroll 4
        for (int64_t c = (int64_t)lane * 8; c < N; c += 256) {
            float v[8];
            load8<BF16>(x, base + c, v);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                amax = fmaxf(amax, fabsf(v[j]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float sc = __fdiv_rn(amax, 448.0f);
        if (lane == 0)
            s[row] = sc;
        const Enc enc(sc);
#pragma unroll 4
        for (int64_t c = (int64_t)lane * 8; c < N; c += 256) {
            float v[8];
            load8<BF16>(x, base + c, v);
            uint2 w;
            w.x = enc(v[0], v[1], v[2], v[3]);
            w.y = enc(v[4], v[5], v[6], v[7]);
            *reinterpret_cast<uint2 *>(q + base + c) = w;
        }
    }
}

// Single-pass variant for bf16 rows with N % 1024 == 0 and N <= 8192: one
// CTA of N/32 threads per row; thread t holds the row's 16-byte chunks t,
// t+T, t+2T, t+3T (T = N/32, so every load and store is warp-contiguous) in
// registers, the CTA reduces the amax through shared memory, and the row is
// read from HBM exactly once.  Many small CTAs per SM keep the loads of
// several rows in flight while other rows divide: the 32-register bound lets
// nine rows (126 KB) be resident per SM.  The kernel is close to issue-bound,
// so the amax is taken on packed pairs (64 us instead of 68 us for
// 16384 x 7168 on GB300; a persistent variant that prefetched the next row
// into shared memory ran 80 us).
__global__ void __launch_bounds__(256, 8) rowquant_bf16_cta_kernel(const uint16_t *__restrict__ x, int64_t N,
                                                                 uint8_t *__restrict__ q, float *__restrict__ s)
{
    __shared__ float red[32];
    const int T = blockDim.x;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t row = blockIdx.x;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + row * N);
    uint4 w[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        w[c] = __ldcs(xr + t + c * T);
    // amax on packed pairs: max.xorsign.abs.bf16x2 keeps the larger magnitude
    // of each half exactly (its sign is a xor of the inputs', dropped below)
    uint32_t m2 = 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t u[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(u[j]));
    }
    float amax = fmaxf(fabsf(bf16_lo(m2)), fabsf(bf16_hi(m2)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0)
        red[warp] = amax;
    __syncthreads();
    amax = red[0];
    for (int i = 1; i < (T >> 5); ++i)
        amax = fmaxf(amax, red[i]);
    const float sc = __fdiv_rn(amax, 448.0f);
    if (t == 0)
        s[row] = sc;
    const Enc enc(sc);
    uint2 *qr = reinterpret_cast<uint2 *>(q + row * N);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint2 o;
        o.x = enc(bf16_lo(w[c].x), bf16_hi(w[c].x), bf16_lo(w[c].y), bf16_hi(w[c].y));
        o.y = enc(bf16_lo(w[c].z), bf16_hi(w[c].z), bf16_lo(w[c].w), bf16_hi(w[c].w));
        __stcs(qr + t + c * T, o);
    }
}

// --------------------------------------------------------------------------
// Band reduce with the row quantiser folded in (the fp8 wire without the bf16
// round trip): one CTA per 8 consecutive rows of a 32-row lane group of a band's
// tile row.  Phase 1 forms each element of those rows exactly as the band
// reduce does -- ((W_0 + W_1) + ...) in fp32, rounded to bf16 -- or, for the
// 32 x 32 blocks the GEMM kernel's reducer warps already summed (block index
// below claimed[b]), reads their bf16 result from `out`; it parks the 8 bf16
// rows in shared memory and takes each row's amax on the way.  Phase 2 codes
// the parked rows exactly as rowquant_bf16_cta_kernel does: s = amax / 448
// (IEEE), codes = e4m3_rn_sat(x / s).  Loads: a warp covers 8 rows x 4 column
// units of one chunk, four 128-byte pieces per slice.  The thread's row
// (t & 7) is fixed, so its amax is one register.
// --------------------------------------------------------------------------
constexpr int kRqRows = 8;
constexpr int kRqThreads = 512;

template <int P>
__global__ void __launch_bounds__(kRqThreads, 2) band_reduce_quant_kernel(
    const float4 *__restrict__ W, const uint16_t *out, int N, int bands, int rows_per_band, int mt_per_band,
    int ntiles_n, int bn, const uint32_t *band_done, uint32_t expected, const uint32_t *claimed,
    uint8_t *__restrict__ q, float *__restrict__ s, DevStatus *status, uint64_t timeout_ns)
{
    extern __shared__ __align__(16) uint8_t rq_smem[];
    uint16_t *park = reinterpret_cast<uint16_t *>(rq_smem);   // [kRqRows][N] bf16
    __shared__ float red[kRqThreads / 32][kRqRows];
    __shared__ float enc_s[kRqRows], enc_yl[kRqRows], enc_yh[kRqRows];
    __shared__ int enc_fast[kRqRows];
    __shared__ int band_ok;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    // CTA -> (band, tile row, lane quarter, 8-row group)
    int rest = blockIdx.x;
    const int g8 = rest & 3;
    rest >>= 2;
    const int qq = rest & 3;
    rest >>= 2;
    const int mt = rest % mt_per_band;
    const int b = rest / mt_per_band;
    const int row0 = mt * 128 + qq * 32 + g8 * kRqRows;   // first row within the band
    if (row0 >= rows_per_band)
        return;
    if (band_done != nullptr) {
        if (t == 0) {
            int ok = 1;
            if (ld_acquire(band_done + b) < expected) {
                const uint64_t t0 = globaltimer();
                while (ld_acquire(band_done + b) < expected) {
                    if (*(volatile int *)&status->code != 0) { ok = 0; break; }
                    if (globaltimer() - t0 > timeout_ns) {
                        report(status, kErrTimeout, SITE_REDUCE_BAND);
                        ok = 0;
                        break;
                    }
                    __nanosleep(256);
                }
            }
            band_ok = ok;
        }
        __syncthreads();
        if (!band_ok)
            return;
    }
    const int nchunk = bn / 32;
    const int64_t tiles_per_band = (int64_t)mt_per_band * ntiles_n;
    const int64_t tile_f4 = 128 * (int64_t)bn / 4;
    const int64_t slice_f4 = tiles_per_band * tile_f4;
    const int64_t done = claimed != nullptr ? (int64_t)claimed[b] : 0;
    const int r = t & (kRqRows - 1);
    const bool row_ok = row0 + r < rows_per_band;
    const int64_t m = (int64_t)b * rows_per_band + row0 + r;
    const float4 *Wt = W + (int64_t)b * P * slice_f4 + qq * (nchunk * 8 * 32) + g8 * kRqRows + r;
    float amax = 0.0f;
    // phase 1: column quad cq of row r; a thread keeps r, steps cq by 32
    for (int cq = t >> 3; cq < N / 4; cq += kRqThreads / kRqRows) {
        const int col = cq * 4;
        const int nt = col / bn, cin = col - nt * bn;
        const int c = cin >> 5, u = (cin & 31) >> 2;
        uint2 v = make_uint2(0u, 0u);
        if (row_ok) {
            const int64_t tile = (int64_t)mt * ntiles_n + nt;
            const int64_t blk = (tile * 4 + qq) * nchunk + c;
            if (blk < done) {
                v = *reinterpret_cast<const uint2 *>(out + m * N + col);
            } else {
                const float4 *src = Wt + tile * tile_f4 + (c * 8 + u) * 32;
                float4 w[P];
#pragma unroll
                for (int p = 0; p < P; ++p)
                    w[p] = __ldcs(src + p * slice_f4);
                float4 a = w[0];
#pragma unroll
                for (int p = 1; p < P; ++p) {
                    a.x = a.x + w[p].x; a.y = a.y + w[p].y; a.z = a.z + w[p].z; a.w = a.w + w[p].w;
                }
                v = make_uint2(bf16x2_from_f32(a.x, a.y), bf16x2_from_f32(a.z, a.w));
            }
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                                     fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))));
        }
        *reinterpret_cast<uint2 *>(park + r * N + col) = v;
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 8));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 16));
    if (lane < kRqRows)
        red[warp][lane] = amax;
    __syncthreads();
    if (t < kRqRows) {
        float a = red[0][t];
        for (int w = 1; w < kRqThreads / 32; ++w)
            a = fmaxf(a, red[w][t]);
        const float sc = __fdiv_rn(a, 448.0f);
        const Enc e(sc);
        enc_s[t] = e.s;
        enc_yl[t] = e.yl;
        enc_yh[t] = e.yh;
        enc_fast[t] = e.fast ? 1 : 0;
        if (row0 + t < rows_per_band)
            s[(int64_t)b * rows_per_band + row0 + t] = sc;
    }
    __syncthreads();
    // phase 2: 8 elements per item, row-major over the parked rows
    const int per_row = N / 8;
    for (int i = t; i < kRqRows * per_row; i += kRqThreads) {
        const int rr = i / per_row, g = i - rr * per_row;
        if (row0 + rr >= rows_per_band)
            break;   // rows past the band end come last
        const Enc e(enc_s[rr], enc_yl[rr], enc_yh[rr], enc_fast[rr] != 0);
        const uint4 w = *reinterpret_cast<const uint4 *>(park + rr * N + g * 8);
        uint2 o;
        o.x = e(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
        o.y = e(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
        __stcs(reinterpret_cast<uint2 *>(q + ((int64_t)b * rows_per_band + row0 + rr) * N) + g, o);
    }
}

// --------------------------------------------------------------------------
// rowdequant: y = bf16_rn(fp32(decode(q) * s[row])), 16 codes per thread.
// --------------------------------------------------------------------------
__device__ __forceinline__ void dequant16(const uint4 c, float sc, uint16_t *y)
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float2 a = f32x2_from_e4m3x2((uint16_t)(w[j] & 0xFFFFu));
        float2 b = f32x2_from_e4m3x2((uint16_t)(w[j] >> 16));
        o[2 * j] = bf16x2_from_f32(__fmul_rn(a.x, sc), __fmul_rn(a.y, sc));
        o[2 * j + 1] = bf16x2_from_f32(__fmul_rn(b.x, sc), __fmul_rn(b.y, sc));
    }
    uint4 *dst = reinterpret_cast<uint4 *>(y);
    __stcs(dst, make_uint4(o[0], o[1], o[2], o[3]));
    __stcs(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
}

// 16 codes per pack, one pack per thread per loop trip; the launch gives 16
// blocks per SM, so the latency is covered by resident warps rather than by
// deep per-thread unrolling (which throttled the load/store unit).
__global__ void __launch_bounds__(256) rowdequant_kernel(const uint8_t *__restrict__ q, const float *__restrict__ s,
                                                         int64_t M, int64_t N, uint16_t *__restrict__ y)
{
    const int64_t n16 = M * N / 16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
        dequant16(__ldcs(reinterpret_cast<const uint4 *>(q + i * 16)), __ldg(s + i * 16 / N), y + i * 16);
}

// --------------------------------------------------------------------------
// Blockscale quantisers, on fp32 or bf16 input (the call site quantises the
// layer's bf16 activations itself).  Every lane loads 16 bytes: V = 4 fp32 or
// 8 bf16 values (bf16 -> fp32 is exact, so both inputs meet the same fp32
// arithmetic).  s = fp32(amax/448), codes = e4m3_rn_sat(fp32(x/s)); a zero
// group gives s = 0 and +0 codes.
// --------------------------------------------------------------------------
template <bool BF16>
struct Lane16 {
    static constexpr int V = BF16 ? 8 : 4;   // values per 16-byte lane load
    float v[V];
    __device__ __forceinline__ void load(const void *x, int64_t e)
    {
        if constexpr (BF16) {
            const uint4 w = __ldcs(reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(x) + e));
            v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
            v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
        } else {
            const float4 a = __ldcs(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + e));
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        }
    }
    // max |v| with NaN skipped (fmaxf returns the other operand), from 0: a lane of
    // NaN alone gives 0, as a group of NaN alone must (scale 0, +0 codes)
    __device__ __forceinline__ float amax() const
    {
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i)
            m = fmaxf(m, fabsf(v[i]));
        return m;
    }
    // the V codes of this lane, stored with one 4- or 8-byte write
    __device__ __forceinline__ void store_codes(uint8_t *q, int64_t e, const Enc &enc) const
    {
        const uint32_t lo = enc(v[0], v[1], v[2], v[3]);
        if constexpr (BF16)
            *reinterpret_cast<uint2 *>(q + e) = make_uint2(lo, enc(v[4], v[5], v[6], v[7]));
        else
            *reinterpret_cast<uint32_t *>(q + e) = lo;
    }
};

// max over the L lanes of an aligned L-lane segment of the warp; only the
// lanes of that segment need to take part
template <int L>
__device__ __forceinline__ float segment_max(float m)
{
    uint32_t mask = 0xFFFFFFFFu;
    if constexpr (L < 32)
        mask = ((1u << L) - 1u) << ((threadIdx.x & 31) & ~(L - 1));
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(mask, m, o));
    return m;
}

// 1x128: eight lanes per (row, 128-group), 16 values per lane (two 16-byte
// loads of bf16 or four of fp32), so a warp step covers four groups and the
// per-group scale arithmetic (an IEEE division and reciprocal, executed by
// every lane of the group) is spread over 16 values per lane.  (Four lanes of
// 32 values halve that share but need 93 registers, two CTAs per SM, and ran
// slower; one division per two warp steps, lane j of a group dividing for step
// j % 2, ran slower too.)  With C % 128 == 0 group gi = row * (C/128) + g
// starts at element 128 * gi, so the groups are walked as one flat sequence.
constexpr int kQSteps = 2;    // warp steps with loads in flight together
constexpr int kQLanes = 8;    // lanes per group
constexpr int kQVals = 128 / kQLanes;

// A lane's 16 values as loaded: bf16 as 8 packed pairs, unpacked where they are
// used (holding them unpacked cost registers and 12% of the kernel's time), or
// 16 fp32 bit patterns.
template <bool BF16>
struct Lane16x {
    static constexpr int NW = BF16 ? kQVals / 2 : kQVals;
    uint32_t w[NW];
    __device__ __forceinline__ void load(const void *x, int64_t e)
    {
        const uint4 *src = BF16 ? reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(x) + e)
                                : reinterpret_cast<const uint4 *>(reinterpret_cast<const float *>(x) + e);
#pragma unroll
        for (int i = 0; i < NW / 4; ++i) {
            const uint4 v = __ldcs(src + i);
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
    }
    // the k-th of the four-value quads, as fp32
    __device__ __forceinline__ float4 quad(int k) const
    {
        if constexpr (BF16)
            return make_float4(bf16_lo(w[2 * k]), bf16_hi(w[2 * k]), bf16_lo(w[2 * k + 1]), bf16_hi(w[2 * k + 1]));
        else
            return make_float4(__uint_as_float(w[4 * k]), __uint_as_float(w[4 * k + 1]), __uint_as_float(w[4 * k + 2]),
                               __uint_as_float(w[4 * k + 3]));
    }
    // max |v| with NaN skipped, from 0 (a group of NaN alone gives 0)
    __device__ __forceinline__ float amax() const
    {
        float m = 0.0f;
#pragma unroll
        for (int k = 0; k < kQVals / 4; ++k) {
            const float4 v = quad(k);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        return m;
    }
    __device__ __forceinline__ void store_codes(uint8_t *q, int64_t e, const Enc &enc) const
    {
        uint32_t c[kQVals / 4];
        if (enc.fast) {
#pragma unroll
            for (int k = 0; k < kQVals / 4; ++k) {
                const float4 v = quad(k);
                c[k] = enc2_guarded(v.x, v.y, enc.s, enc.yl, enc.yh) | (enc2_guarded(v.z, v.w, enc.s, enc.yl, enc.yh) << 16);
            }
        } else {
#pragma unroll
            for (int k = 0; k < kQVals / 4; ++k) {
                const float4 v = quad(k);
                c[k] = enc4(v.x, v.y, v.z, v.w, enc.s);
            }
        }
        *reinterpret_cast<uint4 *>(q + e) = make_uint4(c[0], c[1], c[2], c[3]);
    }
};

template <bool BF16>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const void *__restrict__ x, int64_t ngroups,
                                                          uint8_t *__restrict__ q, float *__restrict__ scales)
{
    constexpr int L = kQLanes;    // lanes per group
    constexpr int GPW = 32 / L;   // groups per warp step
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (int64_t step = w0 * kQSteps; step * GPW < ngroups; step += warps_total * kQSteps) {
        int64_t gi[kQSteps];
        Lane16x<BF16> d[kQSteps];
#pragma unroll
        for (int u = 0; u < kQSteps; ++u) {
            gi[u] = (step + u) * GPW + lane / L;
            if (gi[u] < ngroups)
                d[u].load(x, gi[u] * 128 + (lane % L) * kQVals);
        }
#pragma unroll
        for (int u = 0; u < kQSteps; ++u) {
            const float m = segment_max<L>(gi[u] < ngroups ? d[u].amax() : 0.0f);
            if (gi[u] < ngroups) {
                const float sc = __fdiv_rn(m, 448.0f);
                if (lane % L == 0)
                    scales[gi[u]] = sc;
                d[u].store_codes(q, gi[u] * 128 + (lane % L) * kQVals, Enc(sc));
            }
        }
    }
}

// 128x128: one 256-thread CTA per block; each warp row-step covers 32V/128 rows.
template <bool BF16>
__global__ void __launch_bounds__(256) quant_128x128_kernel(const void *__restrict__ x, int64_t R, int64_t C,
                                                            uint8_t *__restrict__ q, float *__restrict__ scales)
{
    using L16 = Lane16<BF16>;
    constexpr int L = 128 / L16::V;   // lanes per row of the block
    constexpr int RPW = 32 / L;       // rows per warp step
    __shared__ float red[8];
    const int64_t G = C / 128;
    const int64_t nblk = ((R + 127) / 128) * G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane / L, col = (lane % L) * L16::V;
    for (int64_t bi = blockIdx.x; bi < nblk; bi += gridDim.x) {
        const int64_t br = bi / G, bc = bi % G;
        const int64_t r0 = br * 128;
        const int rows = (int)min64(128, R - r0);
        float amax = 0.0f;
        for (int rr = warp * RPW + sub; rr < rows; rr += 8 * RPW) {
            L16 d;
            d.load(x, (r0 + rr) * C + bc * 128 + col);
            amax = fmaxf(amax, d.amax());
        }
        amax = segment_max<32>(amax);
        if (lane == 0)
            red[warp] = amax;
        __syncthreads();
        float m = red[0];
#pragma unroll
        for (int w = 1; w < 8; ++w)
            m = fmaxf(m, red[w]);
        const float sc = __fdiv_rn(m, 448.0f);
        if (tid == 0)
            scales[bi] = sc;
        const Enc enc(sc);
        for (int rr = warp * RPW + sub; rr < rows; rr += 8 * RPW) {
            const int64_t e = (r0 + rr) * C + bc * 128 + col;
            L16 d;
            d.load(x, e);
            d.store_codes(q, e, enc);
        }
        __syncthreads();
    }
}

// ue8m0 byte of r = fp32(amax/448): ceil(log2 r) + 127 from the IEEE fields,
// exact at powers of two; 0 for r == 0; clamped to [0, 254].
__device__ __forceinline__ uint32_t ue8m0_of(float r)
{
    const uint32_t bits = __float_as_uint(r);
    if (r == 0.0f)
        return 0u;
    const uint32_t ef = (bits >> 23) & 0xFFu, man = bits & 0x7FFFFFu;
    int e;
    if (ef == 0) {   // subnormal: man * 2^-149
        const int fl = (31 - __clz(man)) - 149;
        e = fl + ((__popc(man) == 1) ? 0 : 1);
    } else {
        e = (int)ef - 127 + (man != 0 ? 1 : 0);
    }
    int b = e + 127;
    b = b < 0 ? 0 : (b > 254 ? 254 : b);
    return (uint32_t)b;
}

// 2^(127 - byte) as fp32 (byte 254 -> 2^-127, a subnormal).
__device__ __forceinline__ float inv_scale_of(uint32_t byte)
{
    return byte == 254u ? __uint_as_float(0x00400000u) : __uint_as_float((254u - byte) << 23);
}

// mx quantiser: an aligned segment of 32/V lanes per 32-wide group (V values
// per lane: 4 fp32 or 8 bf16).
template <bool BF16>
__global__ void __launch_bounds__(256) quant_mx_kernel(const void *__restrict__ x, int64_t R, int64_t C,
                                                       uint8_t *__restrict__ q, uint8_t *__restrict__ e8)
{
    using L16 = Lane16<BF16>;
    constexpr int L = 32 / L16::V;   // lanes per group
    const int64_t nvec = R * C / L16::V;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // the grid stride is a multiple of 32 threads, so the lanes of one group stay together
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const int64_t e = i * L16::V;
        L16 d;
        d.load(x, e);
        const float amax = segment_max<L>(d.amax());
        const uint32_t b = ue8m0_of(__fdiv_rn(amax, 448.0f));
        if ((threadIdx.x & (L - 1)) == 0)
            e8[e / 32] = (uint8_t)b;
        uint32_t w[2] = {0u, 0u};
        if (amax != 0.0f) {
            const float inv = inv_scale_of(b);
#pragma unroll
            for (int h = 0; h < L16::V / 4; ++h)
                w[h] = e4m3x2_from_f32(__fmul_rn(d.v[4 * h], inv), __fmul_rn(d.v[4 * h + 1], inv)) |
                       (e4m3x2_from_f32(__fmul_rn(d.v[4 * h + 2], inv), __fmul_rn(d.v[4 * h + 3], inv)) << 16);
        }
        if constexpr (BF16)
            *reinterpret_cast<uint2 *>(q + e) = make_uint2(w[0], w[1]);
        else
            *reinterpret_cast<uint32_t *>(q + e) = w[0];
    }
}

// --------------------------------------------------------------------------
// mx scale repack.  The block-scaled MMA reads the scale of row r (of A, or
// of B along N) for 32-wide K group j of a 128-K stage from TMEM column
// base + r/32, lane r%32, byte j.  tcgen05.cp 32x128b copies shared-memory
// row l (16 bytes = 4 words) into lane l, columns +0..+3, so the image of
// one stage is word[l*4 + c] = scale word of row c*32 + l (rows past the
// tile: 0).  A: one 512-byte image per (slice, band, 128-row tile of the
// band, stage), following the GEMM's tile decomposition; B: two per (slice,
// BN-column tile, stage) -> rows 0..127 and 128..255 of the tile.
// --------------------------------------------------------------------------
struct SlicePtrs {
    const uint8_t *p[kMaxP];
};

__global__ void mx_repack_a_kernel(SlicePtrs ea, int P, int M, int K, int bands, int rows_per_band,
                                   int mt_per_band, uint32_t *__restrict__ out)
{
    const int KB = K / 128, G = K / 32;
    const int64_t total = (int64_t)P * bands * mt_per_band * KB * 128;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int w = (int)(i % 128);
        int64_t r = i / 128;
        const int kb = (int)(r % KB); r /= KB;
        const int mt = (int)(r % mt_per_band); r /= mt_per_band;
        const int b = (int)(r % bands);
        const int p = (int)(r / bands);
        const int lane = w >> 2, c = w & 3;
        const int band_end = min((b + 1) * rows_per_band, M);
        const int row = b * rows_per_band + mt * 128 + c * 32 + lane;
        uint32_t v = 0;
        if (row < band_end)
            v = *reinterpret_cast<const uint32_t *>(ea.p[p] + (int64_t)row * G + kb * 4);
        out[i] = v;
    }
}

__global__ void mx_repack_b_kernel(SlicePtrs eb, int P, int N, int K, int BN, uint32_t *__restrict__ out)
{
    const int KB = K / 128, NT = N / BN, G = K / 32;
    const int64_t total = (int64_t)P * NT * KB * 256;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int w = (int)(i % 256);
        int64_t r = i / 256;
        const int kb = (int)(r % KB); r /= KB;
        const int nt = (int)(r % NT);
        const int p = (int)(r / NT);
        const int half = w >> 7, lane = (w & 127) >> 2, c = w & 3;
        const int rt = half * 128 + c * 32 + lane;   // row within the BN tile
        uint32_t v = 0;
        if (rt < BN)
            v = *reinterpret_cast<const uint32_t *>(eb.p[p] + (int64_t)(nt * BN + rt) * G + kb * 4);
        out[i] = v;
    }
}

}  // namespace

// ------------------------------------------------------------------ launchers

// CTAs of `kernel` (256 threads, no dynamic shared memory) resident per SM on the
// current device, asked once per device and kept in `cache` (0: not asked yet).
template <typename Kernel>
int resident_per_sm(Kernel kernel, std::atomic<int> (&cache)[64])
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 1;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess || n < 1)
            n = 1;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

std::atomic<int> g_plain_per_sm[kMaxP + 1][64];
std::atomic<int> g_blocked_per_sm[kMaxP + 1][64];

cudaError_t launch_band_reduce(const float *W, uint16_t *out, int P, int64_t M, int64_t N, int bands,
                               const uint32_t *band_done, uint32_t expected, DevStatus *status,
                               uint64_t timeout_ns, int num_sms, cudaStream_t s)
{
    const int64_t rpb = M / bands;
    // two whole waves of resident CTAs (measured at the headline size: 576 us
    // against 581 for one wave and 591 for 8 CTAs per SM, 2.67 waves)
    const dim3 block(256);
#define GEMMAR_REDUCE_CASE(PP)                                                                            \
    case PP: {                                                                                            \
        const dim3 grid((unsigned)(2 * num_sms * resident_per_sm(band_reduce_kernel<PP>, g_plain_per_sm[PP]))); \
        band_reduce_kernel<PP><<<grid, block, 0, s>>>(W, out, rpb, N, bands, band_done, expected, status, \
                                                      timeout_ns);                                        \
        break;                                                                                            \
    }
    switch (P) {
        GEMMAR_REDUCE_CASE(1) GEMMAR_REDUCE_CASE(2) GEMMAR_REDUCE_CASE(3) GEMMAR_REDUCE_CASE(4)
        GEMMAR_REDUCE_CASE(5) GEMMAR_REDUCE_CASE(6) GEMMAR_REDUCE_CASE(7) GEMMAR_REDUCE_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef GEMMAR_REDUCE_CASE
    return cudaGetLastError();
}

template <int P>
int blocked_per_sm()
{
    return resident_per_sm(band_reduce_blocked_kernel<P>, g_blocked_per_sm[P]);
}

cudaError_t launch_band_reduce_blocked(const float *W, uint16_t *out, int P, int64_t M, int64_t N, int bands,
                                       int bn, const uint32_t *band_done, uint32_t expected,
                                       const uint32_t *claimed, DevStatus *status, uint64_t timeout_ns,
                                       int num_sms, cudaStream_t s)
{
    const int rpb = (int)(M / bands), mtpb = (rpb + 127) / 128, ntn = (int)(N / bn);
    const float4 *w4 = reinterpret_cast<const float4 *>(W);
    // one wave: every CTA resident from the start, none left for a partial second
    // wave (its warps stride over the blocks, so the count only sets the schedule)
    const dim3 block(256);
#define GEMMAR_REDUCE_BLK_CASE(PP)                                                                                \
    case PP: {                                                                                                    \
        const dim3 grid((unsigned)(num_sms * blocked_per_sm<PP>()));                                              \
        band_reduce_blocked_kernel<PP><<<grid, block, 0, s>>>(w4, out, (int)M, (int)N, bands, rpb, mtpb, ntn, bn, \
                                                              band_done, expected, claimed, status, timeout_ns);   \
        break;                                                                                                    \
    }
    switch (P) {
        GEMMAR_REDUCE_BLK_CASE(1) GEMMAR_REDUCE_BLK_CASE(2) GEMMAR_REDUCE_BLK_CASE(3) GEMMAR_REDUCE_BLK_CASE(4)
        GEMMAR_REDUCE_BLK_CASE(5) GEMMAR_REDUCE_BLK_CASE(6) GEMMAR_REDUCE_BLK_CASE(7) GEMMAR_REDUCE_BLK_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef GEMMAR_REDUCE_BLK_CASE
    return cudaGetLastError();
}

cudaError_t launch_rowquant(const void *x, int x_is_bf16, int64_t M, int64_t N, uint8_t *q, float *s, int num_sms,
                            cudaStream_t st)
{
    const int64_t blocks_needed = (M + 7) / 8;
    const int grid = (int)min64(blocks_needed, (int64_t)num_sms * 8);
    if (x_is_bf16 && N % 1024 == 0 && N <= 8192 && M <= 0x7FFFFFFF)
        rowquant_bf16_cta_kernel<<<(unsigned)M, (unsigned)(N / 32), 0, st>>>(static_cast<const uint16_t *>(x), N, q, s);
    else if (x_is_bf16)
        rowquant_kernel<true><<<grid, 256, 0, st>>>(x, M, N, q, s);
    else
        rowquant_kernel<false><<<grid, 256, 0, st>>>(x, M, N, q, s);
    return cudaGetLastError();
}

cudaError_t launch_band_reduce_quant(const float *W, const uint16_t *out, int P, int64_t M, int64_t N, int bands,
                                     int bn, const uint32_t *band_done, uint32_t expected, const uint32_t *claimed,
                                     uint8_t *q, float *s, DevStatus *status, uint64_t timeout_ns, cudaStream_t st)
{
    if (N > kBandQuantMaxN || N % bn != 0 || bn % 32 != 0)
        return cudaErrorInvalidValue;
    const int rpb = (int)(M / bands), mtpb = (rpb + 127) / 128, ntn = (int)(N / bn);
    const float4 *w4 = reinterpret_cast<const float4 *>(W);
    const size_t smem = (size_t)kRqRows * N * 2;
    const unsigned grid = (unsigned)bands * mtpb * 16;
#define GEMMAR_RQ_CASE(PP)                                                                                     \
    case PP: {                                                                                                 \
        const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(band_reduce_quant_kernel<PP>), \
                                                  (int)(kRqRows * kBandQuantMaxN * 2));                         \
        if (e != cudaSuccess)                                                                                  \
            return e;                                                                                          \
        band_reduce_quant_kernel<PP><<<grid, kRqThreads, smem, st>>>(w4, out, (int)N, bands, rpb, mtpb, ntn, bn, \
                                                                     band_done, expected, claimed, q, s, status, \
                                                                     timeout_ns);                              \
        break;                                                                                                 \
    }
    switch (P) {
        GEMMAR_RQ_CASE(1) GEMMAR_RQ_CASE(2) GEMMAR_RQ_CASE(3) GEMMAR_RQ_CASE(4)
        GEMMAR_RQ_CASE(5) GEMMAR_RQ_CASE(6) GEMMAR_RQ_CASE(7) GEMMAR_RQ_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef GEMMAR_RQ_CASE
    return cudaGetLastError();
}

cudaError_t launch_rowdequant(const uint8_t *q, const float *s, int64_t M, int64_t N, uint16_t *y, int num_sms,
                              cudaStream_t st)
{
    const int64_t need = (M * N / 16 + 255) / 256;
    const int grid = (int)max64(1, min64(need, (int64_t)num_sms * 16));
    rowdequant_kernel<<<grid, 256, 0, st>>>(q, s, M, N, y);
    return cudaGetLastError();
}

cudaError_t launch_quant_blockscale(const void *x, int x_is_bf16, int64_t R, int64_t C, int group_rows, uint8_t *q,
                                    float *scales, int num_sms, cudaStream_t st)
{
    if (group_rows == 1) {
        const int64_t ngroups = R * (C / 128);
        const int64_t per_cta = 8 * (32 / kQLanes) * kQSteps;   // 8 warps, 32 / kQLanes groups per warp step
        const int64_t need = (ngroups + per_cta - 1) / per_cta;
        const int grid = (int)max64(1, min64(need, (int64_t)num_sms * 8));
        if (x_is_bf16)
            quant_1x128_kernel<true><<<grid, 256, 0, st>>>(x, ngroups, q, scales);
        else
            quant_1x128_kernel<false><<<grid, 256, 0, st>>>(x, ngroups, q, scales);
    } else {
        const int64_t nblk = ((R + 127) / 128) * (C / 128);
        const int grid = (int)max64(1, min64(nblk, (int64_t)num_sms * 8));
        if (x_is_bf16)
            quant_128x128_kernel<true><<<grid, 256, 0, st>>>(x, R, C, q, scales);
        else
            quant_128x128_kernel<false><<<grid, 256, 0, st>>>(x, R, C, q, scales);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_mx(const void *x, int x_is_bf16, int64_t R, int64_t C, uint8_t *q, uint8_t *e8, int num_sms,
                            cudaStream_t st)
{
    const int64_t need = (R * C / (x_is_bf16 ? 8 : 4) + 255) / 256;
    const int grid = (int)max64(1, min64(need, (int64_t)num_sms * 8));
    if (x_is_bf16)
        quant_mx_kernel<true><<<grid, 256, 0, st>>>(x, R, C, q, e8);
    else
        quant_mx_kernel<false><<<grid, 256, 0, st>>>(x, R, C, q, e8);
    return cudaGetLastError();
}

cudaError_t launch_mx_repack(const uint8_t *const *ea, const uint8_t *const *eb, int P, int M, int N, int K,
                             int bands, int bn, uint8_t *sfa_out, uint8_t *sfb_out, cudaStream_t s)
{
    SlicePtrs pa{}, pb{};
    for (int p = 0; p < P; ++p) {
        pa.p[p] = ea[p];
        pb.p[p] = eb[p];
    }
    const int rpb = M / bands, mtpb = (rpb + 127) / 128;
    const int64_t ta = (int64_t)P * bands * mtpb * (K / 128) * 128;
    const int64_t tb = (int64_t)P * (N / bn) * (K / 128) * 256;
    const int ga = (int)max64(1, min64((ta + 255) / 256, 4096));
    const int gb = (int)max64(1, min64((tb + 255) / 256, 4096));
    mx_repack_a_kernel<<<ga, 256, 0, s>>>(pa, P, M, K, bands, rpb, mtpb, reinterpret_cast<uint32_t *>(sfa_out));
    mx_repack_b_kernel<<<gb, 256, 0, s>>>(pb, P, N, K, bn, reinterpret_cast<uint32_t *>(sfb_out));
    return cudaGetLastError();
}

}  // namespace gemmar
