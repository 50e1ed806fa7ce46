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
    __device__ __forceinline__ void add(const GemmOut &o, int b, uint32_t count = 1)
    {
        if (b != band)
            flush(o);
        band = b;
        n += count;
    }
    __device__ __forceinline__ void flush(const GemmOut &o)
    {
        if (n != 0)
            signal_band(o, band, n);
        n = 0;
    }
};

// ---------------------------------------------------------------------------
// In-kernel band reduce: two warps of a GEMM CTA sum retired bands while the
// CTA's other warps keep computing tiles.  It works on 32-row x 32-column
// blocks of the blocked partials (numbered within a band as in
// band_reduce_blocked_kernel: column chunk fastest, then lane quarter, then
// tile) and claims them with an atomic add on the band's own counter, and only
// in bands whose retire count is complete, so it never waits on a block that
// other CTAs have still to write: while the next band is incomplete it polls,
// and it leaves as soon as its own CTA's epilogue warps are done (the band
// reduce kernel launched after the GEMM takes, in every band, the blocks from
// the final counter value on).  A block is read in eight items (one 16-byte
// column unit of each lane's row, all P slices) through a four-stage cp.async
// ring in shared memory per warp; each lane loads and sums only its own row, so
// the ring needs no warp barrier.  The arithmetic is that of the band reduce:
// ((W_0 + W_1) + W_2) + ..., fp32, then bf16 RN.
// ---------------------------------------------------------------------------
constexpr int kReduceRingStages = 4;   // default ring depth (items in flight per reducer warp)
// shared-memory ring of one reducer warp with RS stages, and of the two reducer warps of a CTA
template <int RS = kReduceRingStages>
__host__ __device__ constexpr int reduce_warp_ring_bytes() { return RS * kMaxP * 512; }
template <int RS = kReduceRingStages>
__host__ __device__ constexpr int reduce_ring_bytes() { return 2 * reduce_warp_ring_bytes<RS>(); }

struct BandClaim {
    int band = 0;                // lowest band that may still have unclaimed blocks
    int ready_upto = -1;         // bands <= ready_upto have been seen complete
    uint32_t ahead = 0xFFFFFFFFu; // index taken in `band` by a claim issued one block early
};

// Lane 0 claims the next block of a complete band (band * bpb + index); -1
// when this CTA's epilogue has finished, every band is claimed, or the poll ran
// out of time.  After a successful claim the next one is issued at once (the
// atomic's round trip then overlaps the block's copies); its index, if inside
// the band, is a claimed block and is always returned by the next call.
__device__ __forceinline__ int claim_retired_block(const GemmOut &o, const TileGrid &g, uint32_t bpb, BandClaim &cl,
                                                   const volatile int *epi_done, int epi_warps, uint64_t timeout_ns)
{
    int blk = -1;
    if ((threadIdx.x & 31) == 0) {
        if (cl.ahead != 0xFFFFFFFFu) {
            const uint32_t r = cl.ahead;
            cl.ahead = 0xFFFFFFFFu;
            if (r < bpb)
                blk = (int)((uint32_t)cl.band * bpb + r);
            else
                ++cl.band;   // this band is all claimed
        }
        const uint64_t t0 = ptx::globaltimer();
        while (blk < 0 && cl.band < g.bands) {
            // once this CTA's tiles are all stored, the rest is the reduce kernel's: it
            // starts when every CTA has left, and runs on all of each SM's warps
            if (*epi_done >= epi_warps)
                break;
            if (cl.band > cl.ready_upto) {
                if (ptx::ld_acquire(o.band_done + cl.band) < o.band_expected) {
                    if (ptx::globaltimer() - t0 > timeout_ns)
                        break;
                    __nanosleep(1024);
                    continue;
                }
                cl.ready_upto = cl.band;
            }
            const uint32_t r = atomicAdd(o.reduce_next + cl.band, 1u);
            if (r < bpb)
                blk = (int)((uint32_t)cl.band * bpb + r);
            else
                ++cl.band;
        }
        if (blk >= 0 && *epi_done < epi_warps)
            cl.ahead = atomicAdd(o.reduce_next + cl.band, 1u);   // cl.band is complete
    }
    return __shfl_sync(0xffffffffu, blk, 0);
}

// ring: shared address of reduce_warp_ring_bytes<RS>() (16-byte aligned) that nothing
// else uses while this reducer warp runs.  A block is read as eight items, one
// 16-byte column unit (4 columns) of each lane's row from every slice (P x 512 B
// per item, one ring stage).  Whole warp calls.
template <int RS = kReduceRingStages>
__device__ __forceinline__ void band_reducer_warp(const GemmOut &o, const TileGrid &g, int bn, uint32_t ring,
                                                  const volatile int *epi_done, int epi_warps, uint64_t timeout_ns)
{
    constexpr int IPB = 8;                     // items per block
    constexpr int STAGE = kMaxP * 512;         // bytes per ring stage
    // the block of an item in flight is kept in one of two slots (even and odd
    // groups of IPB items): the ring may run at most one group ahead
    static_assert(RS >= 1 && RS <= IPB, "ring deeper than one block of items");
    const int lane = threadIdx.x & 31;
    const int P = g.P;
    const int nchunk = bn / 32;
    const int64_t tiles_per_band = (int64_t)g.mt_per_band * g.ntiles_n;
    const uint32_t bpb = (uint32_t)(tiles_per_band * 4 * nchunk);
    const int64_t tile_f4 = 128 * (int64_t)bn / 4;
    const int64_t slice_f4 = tiles_per_band * tile_f4;
    const float4 *W = reinterpret_cast<const float4 *>(o.out);
    // block of items 8j..8j+7 (slot j & 1), decomposed once per claim: the lane's
    // first source float4 of slice 0 and its row's first output column (null past
    // the band end)
    const float4 *src0 = nullptr, *src1 = nullptr;
    uint16_t *out0 = nullptr, *out1 = nullptr;
    auto decompose = [&](int blk, const float4 *&src, uint16_t *&out) {
        const uint32_t b = (uint32_t)blk / bpb, r = (uint32_t)blk % bpb;
        const int c = (int)(r % nchunk), q = (int)((r / nchunk) & 3);
        const int64_t i = r / (4 * nchunk);
        src = W + ((int64_t)b * P * tiles_per_band + i) * tile_f4 + ((q * nchunk + c) * 8) * 32 + lane;
        const int mt = (int)(i / g.ntiles_n), nt = (int)(i % g.ntiles_n);
        const int row = mt * 128 + q * 32 + lane;
        out = row < g.rows_per_band ? o.red_out + ((int64_t)b * g.rows_per_band + row) * g.N + (int64_t)nt * bn + c * 32
                                    : nullptr;
    };
    // bf16 sums of the last four items: 16 columns of the lane's row
    uint32_t o0 = 0, o1 = 0, o2 = 0, o3 = 0, o4 = 0, o5 = 0, o6 = 0, o7 = 0;
    const bool out32 = (reinterpret_cast<uintptr_t>(o.red_out) & 31) == 0;
    bool more = true;
    int issued = 0;
    BandClaim cl;
    // item k = column unit k % 8 of its block, in ring stage k % RS
    auto issue = [&](int k) {
        const int j = (k / IPB) & 1;
        if (more && k % IPB == 0) {
            const int claimed = claim_retired_block(o, g, bpb, cl, epi_done, epi_warps, timeout_ns);
            more = claimed >= 0;
            if (more) {
                if (j)
                    decompose(claimed, src1, out1);
                else
                    decompose(claimed, src0, out0);
            }
        }
        if (more) {
            const float4 *src = (j ? src1 : src0) + (k % IPB) * 32;
            const uint32_t dst = ring + (k % RS) * STAGE + lane * 16;
            for (int p = 0; p < P; ++p)
                ptx::cp_async_cg16(dst + p * 512, src + p * slice_f4);
            ++issued;
        }
        ptx::cp_async_commit();   // one group per item slot, empty past the last item
    };
#pragma unroll 1
    for (int k = 0; k < RS; ++k)
        issue(k);
#pragma unroll 1
    for (int k = 0; k < issued; ++k) {
        ptx::cp_async_wait<RS - 1>();   // this lane's copies of item k have landed
        const uint32_t st = ring + (k % RS) * STAGE + lane * 16;
        const uint4 w = ptx::ld_shared_v4(st);
        float a[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z), __uint_as_float(w.w)};
        for (int p = 1; p < P; ++p) {
            const uint4 v = ptx::ld_shared_v4(st + p * 512);
            a[0] = a[0] + __uint_as_float(v.x); a[1] = a[1] + __uint_as_float(v.y);
            a[2] = a[2] + __uint_as_float(v.z); a[3] = a[3] + __uint_as_float(v.w);
        }
        uint16_t *const out = ((k / IPB) & 1) ? out1 : out0;
        // four consecutive items are 16 consecutive columns of the lane's row: 32
        // bytes, stored as one full sector once the fourth is summed
        {
            const uint32_t lo = ptx::bf16x2_from_f32(a[0], a[1]), hi = ptx::bf16x2_from_f32(a[2], a[3]);
            const int slot = k & 3;   // registers, not an indexed array: selected moves
            o0 = slot == 0 ? lo : o0; o1 = slot == 0 ? hi : o1;
            o2 = slot == 1 ? lo : o2; o3 = slot == 1 ? hi : o3;
            o4 = slot == 2 ? lo : o4; o5 = slot == 2 ? hi : o5;
            o6 = slot == 3 ? lo : o6; o7 = slot == 3 ? hi : o7;
        }
        if ((k & 3) == 3 && out != nullptr) {
            uint16_t *dst = out + ((k % IPB) & 4) * 4;
            if (out32)   // rows are 32-byte multiples; the output base decides
                asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(o0),
                             "r"(o1), "r"(o2), "r"(o3), "r"(o4), "r"(o5), "r"(o6), "r"(o7)
                             : "memory");
            else {
                reinterpret_cast<uint4 *>(dst)[0] = make_uint4(o0, o1, o2, o3);
                reinterpret_cast<uint4 *>(dst)[1] = make_uint4(o4, o5, o6, o7);
            }
        }
        issue(k + RS);   // reuses this item's stage: this lane has read it
    }
    ptx::cp_async_wait<0>();
}

// Band-reduce work for warps with time and registers to spare between tiles
// (the whole-K kernel's epilogue warps, whose next tile computes in the other
// TMEM buffer): a warp holds one claimed 32 x 32 block at a time and sums one
// item of it per step -- one 16-byte column unit of each lane's row over all P
// slices, in the band reducer's order ((W_0 + W_1) + ...) in fp32 then bf16 --
// with plain loads into registers.  Claims never wait: a band that is not
// complete yet is tried again at the next call.  A block once claimed is
// finished (finish()) before the warp counts itself out, as band_reduce then
// skips it.
struct SpareReducer {
    const float4 *src = nullptr;   // the lane's 16 bytes of item 0, slice 0, of the held block
    uint16_t *out = nullptr;       // the lane's row, first column of the block (null past the band end)
    int item = 8;                  // next item of the held block; 8: none held
    int band = 0;                  // lowest band that may still have unclaimed blocks (lane 0)
    int ready_upto = -1;           // bands <= ready_upto have been seen complete (lane 0)

    // take a block if none is held and one is free; false if none is held afterwards.
    // Whole warp calls.
    __device__ __forceinline__ bool hold(const GemmOut &o, const TileGrid &g, int bn)
    {
        if (item < 8)
            return true;
        const int nchunk = bn / 32;
        const int64_t tiles_per_band = (int64_t)g.mt_per_band * g.ntiles_n;
        const uint32_t bpb = (uint32_t)(tiles_per_band * 4 * nchunk);
        int blk = -1;
        if ((threadIdx.x & 31) == 0) {
            while (band < g.bands) {
                if (band > ready_upto) {
                    if (ptx::ld_acquire(o.band_done + band) < o.band_expected)
                        break;   // not complete yet: the next call tries again
                    ready_upto = band;
                }
                const uint32_t r = atomicAdd(o.reduce_next + band, 1u);
                if (r < bpb) {
                    blk = (int)((uint32_t)band * bpb + r);
                    break;
                }
                ++band;
            }
        }
        blk = __shfl_sync(0xffffffffu, blk, 0);
        if (blk < 0)
            return false;
        const int lane = threadIdx.x & 31;
        const uint32_t b = (uint32_t)blk / bpb, r = (uint32_t)blk % bpb;
        const int c = (int)(r % nchunk), q = (int)((r / nchunk) & 3);
        const int64_t i = r / (4 * nchunk);
        const int64_t tile_f4 = 128 * (int64_t)bn / 4;
        src = reinterpret_cast<const float4 *>(o.out) + ((int64_t)b * g.P * tiles_per_band + i) * tile_f4 +
              ((q * nchunk + c) * 8) * 32 + lane;
        const int mt = (int)(i / g.ntiles_n), nt = (int)(i % g.ntiles_n);
        const int row = mt * 128 + q * 32 + lane;
        out = row < g.rows_per_band ? o.red_out + ((int64_t)b * g.rows_per_band + row) * g.N + (int64_t)nt * bn + c * 32
                                    : nullptr;
        item = 0;
        return true;
    }

    // sum and store the next item of the held block.  Whole warp calls.
    __device__ __forceinline__ void step(const GemmOut &o, const TileGrid &g, int bn)
    {
        const int64_t slice_f4 = (int64_t)g.mt_per_band * g.ntiles_n * (128 * (int64_t)bn / 4);
        const float4 *s = src + item * 32;
        float4 v[kMaxP];
#pragma unroll
        for (int p = 0; p < kMaxP; ++p)
            if (p < g.P)
                v[p] = __ldcs(s + p * slice_f4);
        float a0 = v[0].x, a1 = v[0].y, a2 = v[0].z, a3 = v[0].w;
#pragma unroll
        for (int p = 1; p < kMaxP; ++p)
            if (p < g.P) {
                a0 = a0 + v[p].x; a1 = a1 + v[p].y; a2 = a2 + v[p].z; a3 = a3 + v[p].w;
            }
        if (out != nullptr)
            *reinterpret_cast<uint2 *>(out + item * 4) = make_uint2(ptx::bf16x2_from_f32(a0, a1), ptx::bf16x2_from_f32(a2, a3));
        ++item;
    }

    // sum what is left of the held block.  Whole warp calls.
    __device__ __forceinline__ void finish(const GemmOut &o, const TileGrid &g, int bn)
    {
        while (item < 8)
            step(o, g, bn);
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
