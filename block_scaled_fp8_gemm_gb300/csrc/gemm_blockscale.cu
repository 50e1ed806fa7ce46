// gemm_blockscale.cu -- block-scaled e4m3 GEMM on the 5th-generation tensor
// cores (tcgen05) with the fp32 1x128 (A) and 128x128 (B) scales applied at
// K-block granularity while draining TMEM ("MORI GEMM + All-Reduce
// Benchmark", "Running the benchmark": A 1x128, B 128x128, fp32 scales).
//
// One persistent CTA per SM, 16 warps, warp-specialised:
//   warp 0      TMA producer: A tile 128x128 and B tile BNx128 (e4m3, 128-byte
//               swizzle) per 128-K stage into a STAGES-deep shared ring.
//   warp 1      MMA issuer: per stage, 4 x tcgen05.mma kind::f8f6f4
//               (128 x BN x 32) into one of two TMEM accumulators, a fresh
//               accumulation per K-block (the scale changes every K-block).
//   warps 2-3   band path: band reducers (epilogue.cuh).
//   warps 4-11  epilogue / scale promotion: each thread owns one tile row and
//               BN/2 columns in registers and, per K-block, applies
//               acc += (sa[m,kb] * sb[n/128,kb]) * P_kb as it drains TMEM,
//               releasing the TMEM buffer back to the MMA warp as soon as it
//               is read.  At tile end: bf16/fp32 store through shared staging,
//               or, on the band path, the tile's sums written back into the
//               TMEM buffer of its last K-block (a "park").
//   warps 12-15 band path: store warps, one per TMEM lane quarter.  They copy a
//               parked tile to the band-ordered fp32 partials, release the
//               buffer and signal the band, while the epilogue warps promote
//               the next tile -- 128 KB of stores per tile leave the SM at its
//               store rate without holding the promotion.
// TMEM holds 2 x BN fp32 columns (double-buffered K-blocks), so the tensor
// cores run K-block kb+1 while the epilogue promotes kb.  On the band path the
// first kParkLead K-blocks of a tile share the one buffer that is not parked.
#include "epilogue.cuh"

namespace gemmar {
using namespace ptx;

namespace {

template <int BN>
struct BsCfg {
    static constexpr int kStages = (BN == 256) ? 4 : 6;
    static constexpr int kABytes = 128 * 128;
    static constexpr int kBBytes = BN * 128;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kEpiWarps = 8;
    static constexpr int kRingStages = kReduceRingStages;   // the band reducers' ring depth
    // 4 KB per epilogue warp for staged C stores; on the band path the two band
    // reducer warps use the same bytes as their ring
    static constexpr int kStagingBytes = kEpiWarps * 4096 > reduce_ring_bytes<kRingStages>()
                                             ? kEpiWarps * 4096 : reduce_ring_bytes<kRingStages>();
    static constexpr int kTmemCols = 2 * BN;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kStages * kABytes;
    static constexpr int kOffStaging = kOffB + kStages * kBBytes;
    static constexpr int kOffBar = kOffStaging + kStagingBytes;
    static constexpr int kNumBars = 2 * kStages + 6;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kTmemCols <= 512, "TMEM budget");
    static_assert(kStagingBytes >= reduce_ring_bytes<kRingStages>(), "the band reducer's ring reuses the staging");
};

constexpr int kThreads = 512;
constexpr int kRegsLow = 64;    // warpgroup 0 (producer, MMA, band reducers) after setmaxnreg.dec
constexpr int kRegsStore = 48;  // warpgroup 3 (store warps) after setmaxnreg.dec
constexpr int kRegsHigh = 200;  // warpgroups 1-2 (epilogue) after setmaxnreg.inc
constexpr int kRegsNeeded = 128 * kRegsLow + 128 * kRegsStore + 256 * kRegsHigh;
static_assert(kRegsNeeded <= 65536, "register split");
constexpr int kStoreWarps = 4;
// K-blocks at the start of a band-path tile that run in one TMEM buffer while
// the store warps drain the previous tile's partial from the other.  Each of
// them waits for its own promotion round trip (about 0.45 us more than a
// double-buffered K-block), while 128 KB takes about 2 us to leave an SM; two
// is the measured optimum at the wo_b shapes (serial band GEMM at P=8,
// M=16384: lead 1 1744-1808 us, 2 1693-1718, 3 1718-1761, 5 1822-1835).
constexpr int kParkLead = 2;

// TMEM K-block buffer of each K-step; the MMA, epilogue and store warps step
// through the same sequence.  Without a park the two buffers alternate.  With
// one, the buffer of a tile's last K-step holds the tile's partial until the
// store warps have read it: the next tile's first kParkLead K-steps (at most
// all but its last) use the other buffer, then the two alternate again,
// starting with the parked one.
struct BufSeq {
    uint32_t use0 = 0, use1 = 0;   // K-steps given to each buffer so far (registers, not an array)
    int last = 1;                  // buffer of the previous tile's last K-step
    // buffer of K-step ks (of nks) of the current tile; n = its use index
    __device__ __forceinline__ int next(int ks, int nks, bool park, uint32_t &n)
    {
        // the tile's last K-step always reuses the parked buffer (lead <= nks - 1), so a
        // tile cannot be parked before the store warps have taken the previous one
        const int lead = min(kParkLead, nks - 1);
        int b;
        if (!park)
            b = (int)((use0 + use1) & 1u);
        else
            b = ks < lead ? 1 - last : last ^ ((ks - lead) & 1);
        n = b ? use1 : use0;
        use0 += b ? 0u : 1u;
        use1 += b ? 1u : 0u;
        if (ks == nks - 1)
            last = b;
        return b;
    }
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) gemm_blockscale_kernel(const __grid_constant__ BsParams prm)
{
    using C = BsCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *empty = full + C::kStages;
    uint64_t *tfull = empty + C::kStages;   // [2]
    uint64_t *tempty = tfull + 2;           // [2]
    uint64_t *final_bar = tempty + 2;
    uint64_t *park_full = final_bar + 1;    // a tile's partial is in TMEM (8 epilogue warps arrive)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    volatile int *epi_done = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 8);   // epilogue warps finished

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const TileGrid &g = prm.g;
    const int KB = g.K / 128;
    const int NKS = (g.slice_loop ? g.P : 1) * KB;   // K-blocks per tile
    const bool park = prm.o.out_mode == OUT_PARTIAL_F32;

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
        mbar_init(park_full, C::kEpiWarps);
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
        setmaxnreg_dec<kRegsLow>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0, issued = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x) {
                const TileCoord tc = decode_tile<BN>(t, g);
                for (int ks = 0; ks < NKS; ++ks) {
                    const int p = g.slice_loop ? ks / KB : tc.p;
                    const int kb = ks % KB;
                    if (!mbar_wait(empty + stage, ph ^ 1, abort_flag, prm.status, prm.timeout_ns,
                                   SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full + stage, C::kStageBytes);
                    tma_load_2d(smem + C::kOffA + stage * C::kABytes, &prm.tmA[p], full + stage, kb * 128, tc.m0);
                    tma_load_2d(smem + C::kOffB + stage * C::kBBytes, &prm.tmB[p], full + stage, kb * 128, tc.n0);
                    ++issued;
                    if (++stage == C::kStages) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            if (*abort_flag) {
                // the CTA is giving up: let the loads already in flight land before it exits
                const int first = issued > C::kStages ? issued - C::kStages : 0;
                for (int j = first; j < issued; ++j) {
                    uint64_t *bar = full + (j % C::kStages);
                    const uint32_t par = (uint32_t)((j / C::kStages) & 1);
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(bar, par) && globaltimer() - t0 < prm.timeout_ns) {
                    }
                }
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_f8_e4m3(128, BN);
            int stage = 0;
            uint32_t ph = 0;
            BufSeq seq;
            bool ok = true;
            for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x) {
                for (int ks = 0; ks < NKS; ++ks) {
                    uint32_t n;
                    const int buf = seq.next(ks, NKS, park, n);
                    if (!mbar_wait(tempty + buf, (n & 1) ^ 1, abort_flag, prm.status, prm.timeout_ns,
                                   SITE_MMA_TMEM_EMPTY) ||
                        !mbar_wait(full + stage, ph, abort_flag, prm.status, prm.timeout_ns, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_kmajor_sw128(smem_u32(smem + C::kOffA + stage * C::kABytes));
                    const uint64_t bd = desc_kmajor_sw128(smem_u32(smem + C::kOffB + stage * C::kBBytes));
                    const uint32_t d = tmem_base + buf * BN;
#pragma unroll
                    for (int k = 0; k < 4; ++k)   // 4 x 32 of K = one 128-byte swizzle row
                        mma_f8(d, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
                    tc_commit(empty + stage);   // stage reusable once these MMAs have read it
                    tc_commit(tfull + buf);     // K-block partial ready for promotion
                    if (++stage == C::kStages) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            // all MMAs issued by this thread complete before TMEM is released
            tc_commit(final_bar);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(final_bar, 0)) {
                if (globaltimer() - t0 > prm.timeout_ns) {
                    report(prm.status, kErrTimeout, SITE_TEARDOWN_MMA);
                    break;
                }
            }
        } else if (warp >= 2 && prm.o.out_mode == OUT_PARTIAL_F32 && prm.o.reduce_next != nullptr) {
            // ------------------------------------------------ band reducers (the staging is
            // unused when the epilogue writes blocked partials): one half of it each
            band_reducer_warp<C::kRingStages>(prm.o, g, BN,
                                              smem_u32(smem + C::kOffStaging) + (warp - 2) * reduce_warp_ring_bytes<C::kRingStages>(),
                                 epi_done, C::kEpiWarps + kStoreWarps, prm.timeout_ns);
        }
    } else if (warp < 12) {
        setmaxnreg_inc<kRegsHigh>();
        // ---------------------------------------------------- epilogue
        constexpr int HALF = BN / 2;
        constexpr int NCH = HALF / 32;   // 32-column store chunks per thread
        static_assert(HALF % 64 == 0, "promotion works in 64-column TMEM loads");
        const int ew = warp - 4;        // 0..7
        const int q = warp & 3;         // TMEM lane quarter this warp may access
        const int h = ew >> 2;          // column half of the tile
        const int row = q * 32 + lane;  // tile row owned by this thread
        const uint32_t staging = smem_u32(smem + C::kOffStaging + ew * 4096);
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) + h * HALF;
        BufSeq seq;
        bool ok = true;
        const int nsl = g.slice_loop ? g.P : 1;
        for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x) {
            const TileCoord tc = decode_tile<BN>(t, g);
            const int64_t mrow = min(tc.m0 + row, g.M - 1);
            const int64_t nblk = (tc.n0 + h * HALF) >> 7;
            float acc[HALF];
#pragma unroll
            for (int j = 0; j < HALF; ++j)
                acc[j] = 0.0f;
            // scales of the tile's K-steps, slice by slice: sa[p][row, kb] * sb[p][n/128, kb].
            // The two factors are loaded a step ahead and multiplied where used, so
            // the load latency overlaps the wait and the TMEM reads of a step.
            const float *sa_row = prm.sa[tc.p] + mrow * KB;
            const float *sb_blk = prm.sb[tc.p] + nblk * KB;
            float a_next = __ldg(sa_row), b_next = __ldg(sb_blk);
            for (int ks = 0, sl = 0, kb = 0; ks < NKS; ++ks) {
                const float a_cur = a_next, b_cur = b_next;
                if (++kb == KB) {
                    kb = 0;
                    if (++sl < nsl) {
                        sa_row = prm.sa[sl] + mrow * KB;
                        sb_blk = prm.sb[sl] + nblk * KB;
                    }
                }
                if (ks + 1 < NKS) {
                    a_next = __ldg(sa_row + kb);
                    b_next = __ldg(sb_blk + kb);
                }
                uint32_t n;
                const int buf = seq.next(ks, NKS, park, n);
                if (!mbar_wait(tfull + buf, n & 1, abort_flag, prm.status, prm.timeout_ns, SITE_EPI_TMEM_FULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float s = a_cur * b_cur;
                const uint32_t taddr = lane_base + buf * BN;
                const bool parks = park && ks == NKS - 1;   // this buffer takes the tile's partial
                // 16-column TMEM loads, two in flight: the next one is issued before the
                // current one's promotions.  The buffer is free again once the last load
                // has landed, before the last 16 promotions.
                constexpr int NC = HALF / 16;
                uint32_t ra[16], rb[16];
                tmem_ld_x16(taddr, ra);
                tmem_wait_ld(ra);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    uint32_t(&cur)[16] = (c & 1) ? rb : ra;
                    uint32_t(&nxt)[16] = (c & 1) ? ra : rb;
                    if (c + 1 < NC)
                        tmem_ld_x16(taddr + (c + 1) * 16, nxt);
#pragma unroll
                    for (int j = 0; j < 16; j += 2)
                        fma2(acc[c * 16 + j], acc[c * 16 + j + 1], s, cur[j], cur[j + 1]);
                    if (c + 1 < NC) {
                        tmem_wait_ld(nxt);
                        if (c + 2 == NC && !parks) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(tempty + buf);
                        }
                    }
                }
                if (parks) {
                    // the tile's sums go back into the columns this warp has just read;
                    // the store warps copy them out and release the buffer
#pragma unroll
                    for (int c = 0; c < HALF / 32; ++c)
                        tmem_st_x32(taddr + c * 32, &acc[c * 32]);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(park_full);
                }
            }
            if (!ok)
                break;
            if (park)
                continue;   // the store warps write the partial and signal its band
            // -------- tile store
            const int rows_valid = max(0, min(32, tc.valid_rows - q * 32));
            if (prm.o.out_mode == OUT_BF16) {
                char *base = tile_out_base(prm.o, g, tc, 2) + ((int64_t)q * 32 * g.N + h * HALF) * 2;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    uint4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float *a = &acc[c * 32 + u * 8];
                        v[u] = make_uint4(bf16x2_from_f32(a[0], a[1]), bf16x2_from_f32(a[2], a[3]),
                                          bf16x2_from_f32(a[4], a[5]), bf16x2_from_f32(a[6], a[7]));
                    }
                    store_chunk<4>(staging, v, base + c * 64, (int64_t)g.N * 2, rows_valid);
                }
            } else {
                char *base = tile_out_base(prm.o, g, tc, 4) + ((int64_t)q * 32 * g.N + h * HALF) * 4;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    uint4 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float *a = &acc[c * 32 + u * 4];
                        v[u] = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                          __float_as_uint(a[3]));
                    }
                    store_chunk<8>(staging, v, base + c * 128, (int64_t)g.N * 4, rows_valid);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            atomicAdd(const_cast<int *>(epi_done), 1);
    } else {
        setmaxnreg_dec<kRegsStore>();
        if (park) {
            // ------------------------------------------------ store warps: warp 12 + q copies
            // lane quarter q (32 rows x BN columns) of each parked tile to its blocked
            // partial, hands the buffer back to the MMA warp and publishes the band
            // (batched per run of same-band tiles; 4 warps x 2 = the 8 signals a tile owes)
            const int q = warp & 3;
            const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
            BufSeq seq;
            BandSignals signals;
            uint32_t parked = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x) {
                const TileCoord tc = decode_tile<BN>(t, g);
                int buf = 0;
                uint32_t n;
                for (int ks = 0; ks < NKS; ++ks)
                    buf = seq.next(ks, NKS, true, n);
                if (!mbar_wait(park_full, parked & 1, abort_flag, prm.status, prm.timeout_ns, SITE_PARK_FULL)) {
                    ok = false;
                    break;
                }
                ++parked;
                tc_fence_after();
                float4 *tb = partial_tile_base(prm.o, g, tc, BN);
                const uint32_t taddr = lane_base + buf * BN;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32], (&lo)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[0]),
                                    (&hi)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[16]);
                    tmem_ld_x16(taddr + c * 32, lo);
                    tmem_ld_x16(taddr + c * 32 + 16, hi);
                    tmem_wait_ld(lo);
                    tmem_wait_ld(hi);
                    if (c == BN / 32 - 1) {
                        // the whole park is read: the MMA may refill the buffer
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(tempty + buf);
                            mbar_arrive(tempty + buf);
                        }
                    }
                    store_partial_chunk<BN>(tb, q, c, reinterpret_cast<const float *>(r));
                }
                signals.add(prm.o, tc.b, 2);
            }
            if (ok)
                signals.flush(prm.o);
        }
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

template <int BN>
cudaError_t launch_bn(const BsParams &p, int grid, cudaStream_t s)
{
    using C = BsCfg<BN>;
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(gemm_blockscale_kernel<BN>),
                                              C::kSmemBytes);
    if (e != cudaSuccess)
        return e;
    gemm_blockscale_kernel<BN><<<grid, kThreads, C::kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

template <int BN>
int regs_of()
{
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, gemm_blockscale_kernel<BN>) != cudaSuccess)
        return -1;
    return a.numRegs;
}

}  // namespace

cudaError_t launch_gemm_blockscale(const BsParams &p, int bn, int grid, cudaStream_t s)
{
    if (bn == 256)
        return launch_bn<256>(p, grid, s);
    if (bn == 128)
        return launch_bn<128>(p, grid, s);
    return cudaErrorInvalidValue;
}

int gemm_blockscale_num_regs(int bn) { return bn == 256 ? regs_of<256>() : regs_of<128>(); }

bool gemm_blockscale_split_ok(int bn)
{
    const int regs = gemm_blockscale_num_regs(bn);
    return regs >= 0 && (int64_t)regs * kThreads >= kRegsNeeded;
}

}  // namespace gemmar
