// epilogue.cuh -- tile bookkeeping and the coalesced row-chunk store shared by
// the two GEMM kernels.
#pragma once

#include "kernels.h"

namespace gemmar {

struct TileCoord {
    int b, p, m0, n0, valid_rows;
};

template <int BN>
__device__ __forceinline__ TileCoord decode_tile(int t, const TileGrid &g)
{
    TileCoord c;
    if (g.slice_loop) {
        // A tile reads all P slices' operands.  Tiles go in groups of 16 row
        // tiles, column-major inside a group, so that the CTAs running at one
        // time share A rows and B columns (about 16 x 9 tiles on 152 SMs) and
        // each K-step's operands come from L2 more often than from HBM.
        constexpr int kGroupM = 16;
        const int mt_total = (g.M + 127) / 128;
        const int per_group = kGroupM * g.ntiles_n;
        const int m_first = (t / per_group) * kGroupM;
        const int idx = t % per_group;
        const int gm = min(kGroupM, mt_total - m_first);
        c.p = 0;
        c.b = 0;
        c.m0 = (m_first + idx % gm) * 128;
        c.n0 = (idx / gm) * BN;
        c.valid_rows = min(128, g.M - c.m0);
        return c;
    }
    const int nt = t % g.ntiles_n;
    int r = t / g.ntiles_n;
    const int mt = r % g.mt_per_band;
    r /= g.mt_per_band;
    c.p = r % g.P;
    c.b = r / g.P;
    c.m0 = c.b * g.rows_per_band + mt * 128;
    c.n0 = nt * BN;
    int band_end = (c.b + 1) * g.rows_per_band;
    if (band_end > g.M) band_end = g.M;
    c.valid_rows = min(128, band_end - c.m0);
    return c;
}

// Global address of tile row 0 (the caller adds rows) for a tile's output.
// OUT_PARTIAL_F32 writes W[b][p][row - b*rows_per_band][n].
__device__ __forceinline__ char *tile_out_base(const GemmOut &o, const TileGrid &g, const TileCoord &c,
                                               int elem_bytes)
{
    int64_t row;
    if (o.out_mode == OUT_PARTIAL_F32)
        row = ((int64_t)c.b * g.P + c.p) * g.rows_per_band + (c.m0 - (int64_t)c.b * g.rows_per_band);
    else
        row = c.m0;
    return reinterpret_cast<char *>(o.out) + (row * g.N + c.n0) * elem_bytes;
}

// Store one 32-row chunk of a warp's output through a warp-private 32 x
// (UNITS*16)-byte shared staging buffer: each thread writes its own row
// (16-byte units, XOR-swizzled so the 8 threads of a shared-memory phase hit
// distinct banks), then the warp reads it back row-contiguously and issues
// coalesced 16-byte global stores (UNITS lanes per row).  rows_valid masks
// rows past the band or matrix end.  Whole warp must call.
template <int UNITS>
__device__ __forceinline__ void store_chunk(uint32_t stage, const uint4 (&v)[UNITS], char *gdst,
                                            int64_t row_stride_bytes, int rows_valid)
{
    static_assert(UNITS == 8 || UNITS == 4 || UNITS == 2, "chunk is 128, 64 or 32 bytes per row");
    constexpr int ROWB = UNITS * 16;
    const int lane = threadIdx.x & 31;
    const int sw = (UNITS == 8) ? (lane & 7) : (UNITS == 4) ? ((lane >> 1) & 3) : ((lane >> 2) & 1);
#pragma unroll
    for (int u = 0; u < UNITS; ++u)
        ptx::st_shared_v4(stage + lane * ROWB + ((u ^ sw) * 16), v[u]);
    __syncwarp();
    constexpr int RPI = 32 / UNITS;   // rows per store instruction
#pragma unroll
    for (int i = 0; i < UNITS; ++i) {
        const int r = i * RPI + lane / UNITS;
        const int u = lane % UNITS;
        const int rsw = (UNITS == 8) ? (r & 7) : (UNITS == 4) ? ((r >> 1) & 3) : ((r >> 2) & 1);
        const uint4 val = ptx::ld_shared_v4(stage + r * ROWB + ((u ^ rsw) * 16));
        if (r < rows_valid)
            *reinterpret_cast<uint4 *>(gdst + r * row_stride_bytes + u * 16) = val;
    }
    __syncwarp();
}

// Blocked layout of the fused path's fp32 partials (the context's own
// workspace).  Tile i of band b, slice p (i = mt * ntiles_n + nt) owns 128*BN
// floats at ((b * P + p) * tiles_per_band + i) * 128 * BN; inside it, the
// 16-byte unit u (columns c*32 + 4u .. +3) of tile row q*32 + l sits at
// float4 index ((q * BN/32 + c) * 8 + u) * 32 + l.  A warp's 32 rows of one
// unit are therefore 512 contiguous bytes: the epilogue stores its registers
// straight to HBM, fully coalesced and without shared-memory staging (shared
// memory is busy feeding the tensor cores), and the band reducer transposes.
__device__ __forceinline__ float4 *partial_tile_base(const GemmOut &o, const TileGrid &g, const TileCoord &c,
                                                     int bn)
{
    const int mt = (c.m0 - c.b * g.rows_per_band) / 128;
    const int64_t tiles_per_band = (int64_t)g.mt_per_band * g.ntiles_n;
    const int64_t i = (int64_t)mt * g.ntiles_n + c.n0 / bn;
    const int64_t tile = ((int64_t)c.b * g.P + c.p) * tiles_per_band + i;
    return reinterpret_cast<float4 *>(o.out) + tile * (128 * bn / 4);
}

// Store 32 fp32 columns (chunk c) of this thread's tile row into the blocked
// partial layout: 8 fully coalesced 512-byte warp stores.
template <int BN>
__device__ __forceinline__ void store_partial_chunk(float4 *tile_base, int q, int c, const float *v)
{
    const int lane = threadIdx.x & 31;
    float4 *dst = tile_base + ((q * (BN / 32) + c) * 8) * 32 + lane;
#pragma unroll
    for (int u = 0; u < 8; ++u)
        __stcg(dst + u * 32, make_float4(v[u * 4 + 0], v[u * 4 + 1], v[u * 4 + 2], v[u * 4 + 3]));
}

// Publish n retired tiles (per warp) of one band to the band reducer: the
// warp barrier orders every lane's stores before lane 0, whose gpu-scope fence
// and release add then make them visible to the reducer's acquire.
__device__ __forceinline__ void signal_band(const GemmOut &o, int band, uint32_t n = 1u)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0 && band != o.skip_band) {
        __threadfence();
        ptx::red_release_add(o.band_done + band, n);
    }
}

// A warp's band signals, batched per run of same-band tiles: the fence in
// signal_band waits until every partial store the warp has in flight is
// performed (about a microsecond after a tile's 128 KB), so a warp counts the
// tiles it retires and publishes a band's count once, when its next tile
// belongs to another band, or at the end.  The counts the reducer waits for
// are unchanged.  Whole warp must call.
struct BandSignals {
    int band = -1;
    uint32_t n = 0;
    __device__ __forceinline__ void add(const GemmOut &o, int b)
    {
        if (b != band)
            flush(o);
        band = b;
        ++n;
    }
    __device__ __forceinline__ void flush(const GemmOut &o)
    {
        if (n != 0)
            signal_band(o, band, n);
        n = 0;
    }
};

template <int N>
__device__ __forceinline__ void setmaxnreg_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void setmaxnreg_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Round a dynamic shared-memory pointer up to a 1024-byte boundary of the
// shared address space (the 128-byte swizzle pattern repeats every 1024 bytes).
__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    const uint32_t a = ptx::smem_u32(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}

}  // namespace gemmar
