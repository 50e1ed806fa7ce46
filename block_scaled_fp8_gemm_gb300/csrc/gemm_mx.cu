// gemm_mx.cu -- mxfp8 GEMM (e4m3 with one ue8m0 scale per 32 of K for every
// row of A and of B; sglang pull request #43480, "What") on the native
// block-scaled tensor-core MMA: tcgen05.mma kind::mxf8f6f4.block_scale with
// scale_vec::1X, the scales read from TMEM, accumulation over the whole K in
// TMEM -- no promotion on the CUDA cores.
//
// Persistent and warp-specialised, one CTA of 12 warps per SM:
//   warp 0     TMA producer: A 128x128, B BNx128 tiles (128-byte swizzle) and
//              the stage's repacked scale images (512 + 1024 bytes, bulk copy).
//   warp 1     MMA issuer: per stage, tcgen05.cp of the scale images into
//              TMEM (32x128b, replicated to the four lane quarters), then
//              4 block-scaled MMAs (K = 32 each; scale-factor id k selects the
//              byte of the 32-bit scale word).  tcgen05.cp and tcgen05.mma
//              issued by one thread execute in order, so one TMEM scale slot
//              serves every stage.
//   warps 2-3  band path: band reducers (epilogue.cuh).
//   warps 4-11 epilogue: drain the tile's fp32 accumulator (double-buffered
//              across tiles) in 32-column chunks and store it.  On the band
//              path with the in-kernel reduce they also sum band-reduce items
//              between tiles, until the next tile's accumulator is complete.
// With the slice partials summed on chip (TileGrid::slice_loop == 2) every
// slice of a tile accumulates from zero in its own TMEM buffer -- exactly the
// band path's partial -- and the epilogue folds it into a register running sum
// in the band reducer's order while the MMA fills the other buffer.
// TMEM: accumulators at columns [0, 2*BN), A scales at 480..483, B scales at
// 488..495.
#include "epilogue.cuh"

namespace gemmar {
using namespace ptx;

namespace {

constexpr uint32_t kSfaCol = 480;
constexpr uint32_t kSfbCol = 488;

template <int BN, bool PT>
struct MxCfg {
    static constexpr int kStages = PT ? (BN == 256 ? 4 : 6) : (BN == 224 ? 4 : 5);
    static constexpr int kABytes = 128 * 128;
    static constexpr int kBBytes = BN * 128;
    static constexpr int kSfBytes = PT ? 0 : 512 + 1024;
    static constexpr int kStageBytes = kABytes + kBBytes + kSfBytes;
    static constexpr int kEpiWarps = 8;
    static constexpr int kRingStages = kReduceRingStages;   // the band reducers' ring depth
    // 4 KB per epilogue warp for staged C stores; on the band path the two band
    // reducer warps use the same bytes as their ring
    static constexpr int kStagingBytes = kEpiWarps * 4096 > reduce_ring_bytes<kRingStages>()
                                             ? kEpiWarps * 4096 : reduce_ring_bytes<kRingStages>();
    static constexpr int kTmemCols = 512;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kStages * kABytes;
    static constexpr int kOffSf = kOffB + kStages * kBBytes;
    static constexpr int kOffStaging = kOffSf + kStages * kSfBytes;
    static constexpr int kOffBar = kOffStaging + kStagingBytes;
    static constexpr int kNumBars = 2 * kStages + 5;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static_assert(kBBytes % 1024 == 0, "B tiles stay 1024-byte aligned");
    static_assert(kStagingBytes >= reduce_ring_bytes<kRingStages>(), "the band reducer's ring reuses the staging");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(PT ? 2 * BN <= 512 : 2 * BN <= (int)kSfaCol, "accumulators below the scale columns");
};

constexpr int kThreads = 384;
// Band path: pause between a warp's partial-store chunks (4 KB per warp), so a
// tile's partial leaves over the next tile's compute rather than in one burst.
constexpr unsigned kStorePaceNs = 600;
constexpr int kRegsLow = 64;    // warpgroup 0 (producer, MMA, band reducers) after setmaxnreg.dec
constexpr int kRegsHigh = 216;  // warpgroups 1-2 (epilogue) after setmaxnreg.inc

// Four channel scales.  The load is ordered after the preceding TMEM wait (asm
// volatile) so the compiler keeps it next to its use instead of hoisting every
// group's scales to the top of the slice, which spills the running sum.
__device__ __forceinline__ float4 ld_scales4(const float *p)
{
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// Scale one 16-column group of a ptpc tile row in place: w = (sa * sb[n]) * acc,
// both products rounded to fp32 (the blockscale promotion's order).  The warp
// holds its 128 per-channel scales one float4 per lane (loaded before the
// TMEM-full wait, so the load latency hides under it); the group's 16 scales
// are lanes src0 .. src0+3, broadcast by shuffles.
__device__ __forceinline__ void ptpc_scale16(uint32_t *r, float sa, const float4 &mine, int src0)
{
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
        const float bs[4] = {__shfl_sync(0xFFFFFFFFu, mine.x, src0 + j4), __shfl_sync(0xFFFFFFFFu, mine.y, src0 + j4),
                             __shfl_sync(0xFFFFFFFFu, mine.z, src0 + j4), __shfl_sync(0xFFFFFFFFu, mine.w, src0 + j4)};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            r[j4 * 4 + j] = __float_as_uint(__fmul_rn(__fmul_rn(sa, bs[j]), __uint_as_float(r[j4 * 4 + j])));
    }
}

template <int BN, bool PT>
__global__ void __launch_bounds__(kThreads, 1) gemm_mx_kernel(const __grid_constant__ MxParams prm)
{
    using C = MxCfg<BN, PT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *empty = full + C::kStages;
    uint64_t *tfull = empty + C::kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *final_bar = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    volatile int *epi_done = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 8);   // epilogue warps finished

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const TileGrid &g = prm.g;
    const int KB = g.K / 128;
    const int NKS = (g.slice_loop ? g.P : 1) * KB;   // K-blocks per tile
    const bool exact = g.slice_loop == 2;            // slice partials summed on chip

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull + b, 1);
            mbar_init(tempty + b, C::kEpiWarps);
        }
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        *epi_done = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int p = 0; p < g.P; ++p) {
            prefetch_tmap(&prm.tmA[p]);
            prefetch_tmap(&prm.tmB[p]);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < 4) {
        // producer and MMA warps give registers to the epilogue warpgroups
        setmaxnreg_dec<kRegsLow>();
      if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0, issued = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x) {
                const TileCoord tc = decode_tile<BN>(t, g);
                const int mt = (tc.m0 - tc.b * g.rows_per_band) / 128;
                for (int ks = 0; ks < NKS; ++ks) {
                    const int p = g.slice_loop ? ks / KB : tc.p;
                    const int kb = ks % KB;
                    const int64_t a_img = ((int64_t)(p * g.bands + tc.b) * g.mt_per_band + mt) * KB;
                    const int64_t b_img = ((int64_t)p * g.ntiles_n + tc.n0 / BN) * KB;
                    if (!mbar_wait(empty + stage, ph ^ 1, abort_flag, prm.status, prm.timeout_ns,
                                   SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full + stage, C::kStageBytes);
                    tma_load_2d(smem + C::kOffA + stage * C::kABytes, &prm.tmA[p], full + stage, kb * 128, tc.m0);
                    tma_load_2d(smem + C::kOffB + stage * C::kBBytes, &prm.tmB[p], full + stage, kb * 128, tc.n0);
                    if constexpr (!PT) {
                        uint8_t *sf = smem + C::kOffSf + stage * C::kSfBytes;
                        bulk_load(sf, prm.sfa + (a_img + kb) * 512, 512, full + stage);
                        bulk_load(sf + 512, prm.sfb + (b_img + kb) * 1024, 1024, full + stage);
                    }
                    ++issued;
                    if (++stage == C::kStages) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            if (*abort_flag) {
                const int first = issued > C::kStages ? issued - C::kStages : 0;
                for (int j = first; j < issued; ++j) {
                    uint64_t *bar = full + (j % C::kStages);
                    const uint32_t par = (uint32_t)((j / C::kStages) & 1);
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(bar, par) && globaltimer() - t0 < prm.timeout_ns) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t ph = 0, titer = 0;
            bool ok = true;
            const uint32_t sfa_t = tmem_base + kSfaCol, sfb_t = tmem_base + kSfbCol;
            // An accumulation unit is a tile (band path, one-chain slice loop) or,
            // with the partials summed on chip, one slice of a tile: each unit
            // accumulates its K-blocks from zero into one TMEM buffer.
            const int units = exact ? g.P : 1;
            const int ks_per_unit = exact ? KB : NKS;
            for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x) {
                for (int un = 0; un < units && ok; ++un) {
                    const uint32_t buf = titer & 1, tph = (titer >> 1) & 1;
                    if (!mbar_wait(tempty + buf, tph ^ 1, abort_flag, prm.status, prm.timeout_ns,
                                   SITE_MMA_TMEM_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t d = tmem_base + buf * BN;
                    for (int ks = 0; ks < ks_per_unit; ++ks) {
                        if (!mbar_wait(full + stage, ph, abort_flag, prm.status, prm.timeout_ns, SITE_MMA_FULL)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = desc_kmajor_sw128(smem_u32(smem + C::kOffA + stage * C::kABytes));
                        const uint64_t bd = desc_kmajor_sw128(smem_u32(smem + C::kOffB + stage * C::kBBytes));
                        if constexpr (PT) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_f8(d, ad + 2 * k, bd + 2 * k, idesc_f8_e4m3(128, BN), (ks > 0 || k > 0) ? 1u : 0u);
                        } else {
                            const uint32_t sf = smem_u32(smem + C::kOffSf + stage * C::kSfBytes);
                            tc_cp_32x128b_warpx4(sfa_t, smem_desc(sf, 0, 128, 0));
                            tc_cp_32x128b_warpx4(sfb_t, smem_desc(sf + 512, 0, 128, 0));
                            tc_cp_32x128b_warpx4(sfb_t + 4, smem_desc(sf + 1024, 0, 128, 0));
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_mxf8(d, ad + 2 * k, bd + 2 * k, idesc_mx_e4m3(128, BN, (uint32_t)k), sfa_t, sfb_t,
                                         (ks > 0 || k > 0) ? 1u : 0u);
                        }
                        tc_commit(empty + stage);
                        if (ks == ks_per_unit - 1)
                            tc_commit(tfull + buf);
                        if (++stage == C::kStages) {
                            stage = 0;
                            ph ^= 1;
                        }
                    }
                    ++titer;
                }
            }
            tc_commit(final_bar);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(final_bar, 0)) {
                if (globaltimer() - t0 > prm.timeout_ns) {
                    report(prm.status, kErrTimeout, SITE_TEARDOWN_MMA);
                    break;
                }
            }
        }
      } else if (prm.o.out_mode == OUT_PARTIAL_F32 && prm.o.reduce_next != nullptr) {
            // ------------------------------------------------ band reducers (warps 2-3; the
            // staging is unused when the epilogue writes blocked partials): half of it each
            band_reducer_warp<C::kRingStages>(prm.o, g, BN,
                                              smem_u32(smem + C::kOffStaging) + (warp - 2) * reduce_warp_ring_bytes<C::kRingStages>(),
                                 epi_done, C::kEpiWarps, prm.timeout_ns);
      }
    } else {
        setmaxnreg_inc<kRegsHigh>();
        // ---------------------------------------------------- epilogue
        constexpr int NCH = BN / 32;
        const int ew = warp - 4;
        const int q = warp & 3;
        const int h = ew >> 2;
        const uint32_t staging = smem_u32(smem + C::kOffStaging + ew * 4096);
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
        uint32_t titer = 0;
        BandSignals signals;
        if (exact && BN % 128 == 0) {
            // Each slice's fp32 partial arrives in a TMEM buffer of its own; the
            // warp owns a contiguous half of the tile row (BN/2 columns), reads it
            // with 64-column loads (the buffer goes back to the MMA after the last
            // one), scales it (ptpc) and folds it into a running sum in the band
            // reducer's order, run = W_0, then run = run + W_p; bf16(run) is stored
            // once per tile.
            constexpr int HALF = BN / 2;
            constexpr int NL = HALF / 64;   // 64-column TMEM loads per slice
            bool ok = true;
            for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x) {
                const TileCoord tc = decode_tile<BN>(t, g);
                const int64_t mrow = min(tc.m0 + q * 32 + lane, g.M - 1);
                // -0 is the identity of IEEE addition (-0 + x == x for every x, +0 and -0
                // included), so run = -0, then run += W_p for p = 0.. gives W_0 first
                float run[HALF];
#pragma unroll
                for (int j = 0; j < HALF; ++j)
                    run[j] = -0.0f;
                for (int sl = 0; sl < g.P; ++sl) {
                    const float sa_m = PT ? __ldg(prm.pa[sl] + mrow) : 0.0f;
                    // lane l: the scales of columns 4l .. 4l+3 of the warp's half
                    float4 sb_mine = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (PT && lane < HALF / 4)
                        sb_mine = ld_scales4(prm.pb[sl] + tc.n0 + h * HALF + lane * 4);
                    const uint32_t buf = titer & 1, tph = (titer >> 1) & 1;
                    if (!mbar_wait(tfull + buf, tph, abort_flag, prm.status, prm.timeout_ns, SITE_EPI_TMEM_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < NL; ++c) {
                        uint32_t r[64];
                        tmem_ld_x64(lane_base + buf * BN + h * HALF + c * 64, r);
                        tmem_wait_ld(r);
                        if (c == NL - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(tempty + buf);
                        }
                        if constexpr (PT) {
#pragma unroll
                            for (int g16 = 0; g16 < 4; ++g16)
                                ptpc_scale16(r + g16 * 16, sa_m, sb_mine, c * 16 + g16 * 4);
                        }
#pragma unroll
                        for (int j = 0; j < 64; ++j)
                            run[c * 64 + j] = __fadd_rn(run[c * 64 + j], __uint_as_float(r[j]));
                    }
                    ++titer;
                }
                if (!ok)
                    break;
                const int rows_valid = max(0, min(32, tc.valid_rows - q * 32));
                char *base = tile_out_base(prm.o, g, tc, 2) + ((int64_t)q * 32 * g.N + h * HALF) * 2;
#pragma unroll
                for (int c = 0; c < HALF / 32; ++c) {
                    uint4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float *a = &run[c * 32 + u * 8];
                        v[u] = make_uint4(bf16x2_from_f32(a[0], a[1]), bf16x2_from_f32(a[2], a[3]),
                                          bf16x2_from_f32(a[4], a[5]), bf16x2_from_f32(a[6], a[7]));
                    }
                    store_chunk<4>(staging, v, base + c * 64, (int64_t)g.N * 2, rows_valid);
                }
            }
        } else if (exact) {
            // Each slice's fp32 partial arrives in a TMEM buffer of its own; the
            // warp folds its 16-column groups h, h+2, ... into a running sum in the
            // band reducer's order (run = W_0, then run = run + W_p) and stores
            // bf16(run) once per tile.
            constexpr int NH = BN / 32;   // 16-column groups per warp
            bool ok = true;
            for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x) {
                const TileCoord tc = decode_tile<BN>(t, g);
                const int64_t mrow = min(tc.m0 + q * 32 + lane, g.M - 1);
                // -0 is the identity of IEEE addition (-0 + x == x for every x, +0 and -0
                // included), so run = -0, then run += W_p for p = 0.. gives W_0 first
                float run[NH * 16];
#pragma unroll
                for (int j = 0; j < NH * 16; ++j)
                    run[j] = -0.0f;
                for (int sl = 0; sl < g.P; ++sl) {
                    const float sa_m = PT ? __ldg(prm.pa[sl] + mrow) : 0.0f;
                    // lane l: the scales of columns 4(l&3) .. +3 of the warp's 16-column group l>>2
                    float4 sb_mine = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (PT && (lane >> 2) < NH)
                        sb_mine = ld_scales4(prm.pb[sl] + tc.n0 + (h + 2 * (lane >> 2)) * 16 + (lane & 3) * 4);
                    const uint32_t buf = titer & 1, tph = (titer >> 1) & 1;
                    if (!mbar_wait(tfull + buf, tph, abort_flag, prm.status, prm.timeout_ns, SITE_EPI_TMEM_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int i = 0; i < NH; ++i) {
                        uint32_t r[16];
                        tmem_ld_x16(lane_base + buf * BN + (h + 2 * i) * 16, r);
                        tmem_wait_ld(r);
                        if constexpr (PT)
                            ptpc_scale16(r, sa_m, sb_mine, i * 4);
                        if (i == NH - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(tempty + buf);
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            run[i * 16 + j] = __fadd_rn(run[i * 16 + j], __uint_as_float(r[j]));
                    }
                    ++titer;
                }
                if (!ok)
                    break;
                const int rows_valid = max(0, min(32, tc.valid_rows - q * 32));
                char *base = tile_out_base(prm.o, g, tc, 2) + (int64_t)q * 32 * g.N * 2;
#pragma unroll
                for (int i = 0; i < NH; ++i) {
                    uint4 v[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float *a = &run[i * 16 + u * 8];
                        v[u] = make_uint4(bf16x2_from_f32(a[0], a[1]), bf16x2_from_f32(a[2], a[3]),
                                          bf16x2_from_f32(a[4], a[5]), bf16x2_from_f32(a[6], a[7]));
                    }
                    store_chunk<2>(staging, v, base + (h + 2 * i) * 32, (int64_t)g.N * 2, rows_valid);
                }
            }
        }
        // band path with the in-kernel reduce: between tiles the epilogue warps sum
        // band-reduce items too (their next tile computes in the other TMEM buffer)
        const bool assist = !exact && prm.o.out_mode == OUT_PARTIAL_F32 && prm.o.reduce_next != nullptr;
        SpareReducer spare;
        for (int t = blockIdx.x; t < g.num_tiles && !exact; t += gridDim.x) {
            const TileCoord tc = decode_tile<BN>(t, g);
            const float sa_m = PT ? __ldg(prm.pa[tc.p] + min(tc.m0 + q * 32 + lane, g.M - 1)) : 0.0f;
            // lane l: the scales of columns 4(l&7) .. +3 of the warp's 32-column chunk l>>3
            float4 sb_mine = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (PT && (lane >> 3) < NCH / 2)
                sb_mine = ld_scales4(prm.pb[tc.p] + tc.n0 + (h + 2 * (lane >> 3)) * 32 + (lane & 7) * 4);
            const uint32_t buf = titer & 1, tph = (titer >> 1) & 1;
            if (!mbar_wait(tfull + buf, tph, abort_flag, prm.status, prm.timeout_ns, SITE_EPI_TMEM_FULL))
                break;
            tc_fence_after();
            const int rows_valid = max(0, min(32, tc.valid_rows - q * 32));
            const int esz = prm.o.out_mode == OUT_BF16 ? 2 : 4;
            char *base = tile_out_base(prm.o, g, tc, esz) + (int64_t)q * 32 * g.N * esz;
            if (prm.o.out_mode == OUT_PARTIAL_F32) {
                // Band path: read the warp's whole share of the tile (its 32-column chunks
                // h, h+2, ...) out of TMEM first and hand the buffer back, then store the fp32
                // partial one chunk at a time with a pause between chunks.  The next tile's
                // MMAs run meanwhile; spreading the 112-128 KB of partial stores over that
                // time instead of sending them in one burst keeps the SM's memory path free
                // for the operand loads the tensor cores wait on.
                constexpr int NW = (NCH + 1) / 2;   // chunks per warp
                uint32_t r[NW][32];
#pragma unroll
                for (int j = 0; j < NW; ++j)
                    if (h + 2 * j < NCH)
                        tmem_ld_x32(lane_base + buf * BN + (h + 2 * j) * 32, r[j]);
#pragma unroll
                for (int j = 0; j < NW; ++j)
                    tmem_wait_ld(r[j]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(tempty + buf);
                if constexpr (PT) {
                    // ptpc: the per-token x per-channel scale, chunk by chunk (the empty asm
                    // keeps the compiler from hoisting every chunk's scale broadcasts at once)
#pragma unroll
                    for (int j = 0; j < NW; ++j) {
                        if (h + 2 * j < NCH) {
                            ptpc_scale16(r[j], sa_m, sb_mine, j * 8);
                            ptpc_scale16(r[j] + 16, sa_m, sb_mine, j * 8 + 4);
                        }
                        asm volatile("" ::: "memory");
                    }
                }
                float4 *tb = partial_tile_base(prm.o, g, tc, BN);
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    if (h + 2 * j >= NCH)
                        continue;
                    if (j > 0)
                        __nanosleep(kStorePaceNs);
                    store_partial_chunk<BN>(tb, q, h + 2 * j, reinterpret_cast<const float *>(r[j]));
                }
                signals.add(prm.o, tc.b);
                ++titer;
                if (assist && t + (int)gridDim.x < g.num_tiles) {
                    // until the next tile's accumulator is complete (the MMA needs this
                    // buffer back only for the tile after next); not after the last tile,
                    // whose band signals the flush below still has to publish
                    while (!mbar_test_wait(tfull + (titer & 1), (titer >> 1) & 1) && spare.hold(prm.o, g, BN))
                        spare.step(prm.o, g, BN);
                }
                continue;
            }
            for (int c = h; c < NCH; c += 2) {
                uint32_t r[32];
                tmem_ld_x32(lane_base + buf * BN + c * 32, r);
                tmem_wait_ld(r);
                if constexpr (PT) {
                    ptpc_scale16(r, sa_m, sb_mine, ((c - h) >> 1) * 8);
                    ptpc_scale16(r + 16, sa_m, sb_mine, ((c - h) >> 1) * 8 + 4);
                }
                if (c + 2 >= NCH) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(tempty + buf);
                }
                if (prm.o.out_mode == OUT_BF16) {
                    uint4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        v[u] = make_uint4(bf16x2_from_f32(__uint_as_float(r[u * 8 + 0]), __uint_as_float(r[u * 8 + 1])),
                                          bf16x2_from_f32(__uint_as_float(r[u * 8 + 2]), __uint_as_float(r[u * 8 + 3])),
                                          bf16x2_from_f32(__uint_as_float(r[u * 8 + 4]), __uint_as_float(r[u * 8 + 5])),
                                          bf16x2_from_f32(__uint_as_float(r[u * 8 + 6]), __uint_as_float(r[u * 8 + 7])));
                    store_chunk<4>(staging, v, base + c * 64, (int64_t)g.N * 2, rows_valid);
                } else if (prm.o.out_mode == OUT_PARTIAL_F32) {
                    store_partial_chunk<BN>(partial_tile_base(prm.o, g, tc, BN), q, c,
                                            reinterpret_cast<const float *>(r));
                } else {
                    uint4 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        v[u] = make_uint4(r[u * 4 + 0], r[u * 4 + 1], r[u * 4 + 2], r[u * 4 + 3]);
                    store_chunk<8>(staging, v, base + c * 128, (int64_t)g.N * 4, rows_valid);
                }
            }
            if (prm.o.out_mode == OUT_PARTIAL_F32)
                signals.add(prm.o, tc.b);
            ++titer;
        }
        if (!exact)
            signals.flush(prm.o);
        if (assist)
            spare.finish(prm.o, g, BN);   // band_reduce skips a claimed block
        __syncwarp();
        if (lane == 0)
            atomicAdd(const_cast<int *>(epi_done), 1);
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc(tmem_base, C::kTmemCols);
}

template <int BN, bool PT>
cudaError_t launch_bn(const MxParams &p, int grid, cudaStream_t s)
{
    using C = MxCfg<BN, PT>;
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(gemm_mx_kernel<BN, PT>), C::kSmemBytes);
    if (e != cudaSuccess)
        return e;
    gemm_mx_kernel<BN, PT><<<grid, kThreads, C::kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

template <int BN, bool PT>
int regs_of()
{
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, gemm_mx_kernel<BN, PT>) != cudaSuccess)
        return -1;
    return a.numRegs;
}

}  // namespace

cudaError_t launch_gemm_mx(const MxParams &p, int bn, int grid, cudaStream_t s)
{
    if (bn == 224)
        return launch_bn<224, false>(p, grid, s);
    if (bn == 128)
        return launch_bn<128, false>(p, grid, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_ptpc(const MxParams &p, int bn, int grid, cudaStream_t s)
{
    if (bn == 256)
        return launch_bn<256, true>(p, grid, s);
    if (bn == 128)
        return launch_bn<128, true>(p, grid, s);
    return cudaErrorInvalidValue;
}

int gemm_mx_num_regs(int bn) { return bn == 224 ? regs_of<224, false>() : regs_of<128, false>(); }

bool gemm_mx_split_ok(int regs) { return regs >= 0 && (int64_t)regs * kThreads >= 128 * kRegsLow + 256 * kRegsHigh; }

int gemm_ptpc_num_regs(int bn) { return bn == 256 ? regs_of<256, true>() : regs_of<128, true>(); }

}  // namespace gemmar
