// gemm_blockscale_2sm.cu -- the blockscale GEMM on CTA pairs (tcgen05
// cta_group::2), same arithmetic as gemm_blockscale.cu ("MORI GEMM +
// All-Reduce Benchmark", "Running the benchmark": A 1x128, B 128x128 fp32
// scales, applied per 128-K block while draining TMEM).
//
// A cluster of two CTAs on the two SMs of a TPC computes a 256 x 256 pair
// tile: CTA r owns rows m0 + 128r .. +127 (all 256 columns) in its TMEM, and
// per 128-K stage loads those 128 rows of A and rows n0 + 128r .. +127 of B
// (32 KB); the leader (rank 0) issues tcgen05.mma.cta_group::2 (M=256, N=256,
// K=32) reading both CTAs' stages.  Per SM that is the MMA shape of the
// one-CTA 128 x 256 tile with half of its B traffic, which frees the shared
// memory for what limits the one-CTA kernel on the band path: the tile's fp32
// partial (128 KB per SM) is parked in shared memory at tile end and two
// store warps copy it to HBM with ordinary 16-byte stores while the next tile
// computes, instead of stalling the epilogue on 128 KB of global stores.  (The
// stores do not go through the TMA unit, which must keep issuing the next
// stages' operand loads meanwhile.)
//
// Per CTA:
//   warp 0       TMA producer: 3 stages of 16 KB A + 16 KB B
//   warp 1       TMEM allocation (both CTAs); MMA issue (leader only: the
//                whole warp runs the loop, lane 0 polls, one lane issues)
//   warps 2-3    band path: park drain -- warp 2 + h copies the parks of the
//                four epilogue warps of column half h to the blocked partials
//                and publishes the band (batched per run of same-band tiles)
//   warps 4-11   epilogue: thread = one row x 128 columns (2 TMEM loads of 64
//                per K-step), promotion acc += (sa * sb) * P_kb, tile store
// Barriers: stage-full counts both CTAs' TMA bytes on the leader; stage-empty
// and TMEM-full are multicast-committed to both CTAs; TMEM-empty lives on the
// leader and collects 8 local + 8 remote arrivals; park-full / park-empty (one
// pair per epilogue warp) hand each 16 KB park between its epilogue warp and
// its store warp.
#include <algorithm>

#include "epilogue.cuh"

namespace gemmar {
using namespace ptx;

namespace {

constexpr int kThreads = 384;
constexpr int kStages = 3;
constexpr int kABytes = 128 * 128;           // this CTA's 128 rows of A, one 128-K stage
constexpr int kBBytes = 128 * 128;           // this CTA's 128 rows of B
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kBufs = 2;                     // TMEM K-block buffers of 256 columns
constexpr int kEpiWarps = 8;
constexpr int kParkBytes = 16384;            // per epilogue warp: 32 rows x 128 fp32
constexpr int kOffA = 0;
constexpr int kOffB = kStages * kABytes;
constexpr int kOffPark = kOffB + kStages * kBBytes;
constexpr int kOffBar = kOffPark + kEpiWarps * kParkBytes;
constexpr int kNumBars = 2 * kStages + 2 * kBufs + 1 + 2 * kEpiWarps;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr int kRegsLow = 56;
constexpr int kRegsHigh = 224;
constexpr uint32_t kAbortGraceNs = 200000;   // let in-flight copies land before an aborting CTA exits
constexpr int kGroupM = 8;                   // pair-rows per tile group in the slice loops

struct PairTile {
    int b, p, m0, n0, band_end;
};

__device__ __forceinline__ PairTile decode_pair(int t, const TileGrid &g)
{
    PairTile c;
    if (g.slice_loop) {
        // A tile reads all P slices' operands.  Tiles go in groups of kGroupM
        // pair-rows, column-major inside a group, so that the clusters running at
        // one time share A rows and B columns (about 8 x 9 tiles on 76 clusters)
        // and each K-step's operands come from L2 more often than from HBM.
        const int mt2_total = (g.M + 255) / 256;
        const int per_group = kGroupM * g.ntiles_n;
        const int m_first = (t / per_group) * kGroupM;
        const int idx = t % per_group;
        const int gm = min(kGroupM, mt2_total - m_first);
        c.b = 0;
        c.p = 0;
        c.n0 = (idx / gm) * 256;
        c.m0 = (m_first + idx % gm) * 256;
        c.band_end = g.M;
        return c;
    }
    const int nt = t % g.ntiles_n;
    int r = t / g.ntiles_n;
    c.n0 = nt * 256;
    const int mt2_per_band = (g.rows_per_band + 255) / 256;
    const int mt2 = r % mt2_per_band;
    r /= mt2_per_band;
    c.p = r % g.P;
    c.b = r / g.P;
    c.m0 = c.b * g.rows_per_band + mt2 * 256;
    c.band_end = min((c.b + 1) * g.rows_per_band, g.M);
    return c;
}

__global__ void __launch_bounds__(kThreads, 1) gemm_blockscale_2sm_kernel(const __grid_constant__ BsParams prm)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;     // [kBufs]
    uint64_t *tempty = tfull + kBufs;      // [kBufs], used on the leader
    uint64_t *final_bar = tempty + kBufs;
    uint64_t *park_full = final_bar + 1;           // [kEpiWarps]
    uint64_t *park_empty = park_full + kEpiWarps;  // [kEpiWarps]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;
    const TileGrid &g = prm.g;
    const int KB = g.K / 128;
    const int NKS = (g.slice_loop ? g.P : 1) * KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < kBufs; ++b) {
            mbar_init(tfull + b, 1);
            mbar_init(tempty + b, 2 * kEpiWarps);
        }
        mbar_init(final_bar, 1);
        for (int w = 0; w < kEpiWarps; ++w) {
            mbar_init(park_full + w, 1);
            mbar_init(park_empty + w, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int p = 0; p < g.P; ++p) {
            prefetch_tmap(&prm.tmA[p]);
            prefetch_tmap(&prm.tmB[p]);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // barriers initialised and TMEM allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < 4) {
        setmaxnreg_dec<kRegsLow>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = cluster; t < g.num_tiles && ok; t += nclusters) {
                const PairTile tc = decode_pair(t, g);
                for (int ks = 0; ks < NKS; ++ks) {
                    const int p = g.slice_loop ? ks / KB : tc.p;
                    const int kb = ks % KB;
                    if (!mbar_wait(empty + stage, ph ^ 1, abort_flag, prm.status, prm.timeout_ns,
                                   SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0)
                        mbar_arrive_expect_tx(full + stage, 2 * kStageBytes);
                    const uint32_t fb = full_leader + 8u * stage;
                    tma_load_2d_pair(smem + kOffA + stage * kABytes, &prm.tmA[p], fb, kb * 128,
                                     tc.m0 + 128 * (int)rank);
                    tma_load_2d_pair(smem + kOffB + stage * kBBytes, &prm.tmB[p], fb, kb * 128,
                                     tc.n0 + 128 * (int)rank);
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
        } else if (warp == 1 && rank == 0) {
            // ------------------------------------------------ MMA issuer (leader)
            // The whole warp runs the loop so that descriptors and TMEM addresses
            // stay warp-uniform; lane 0 polls the barriers and broadcasts the
            // outcome, one elected lane issues.
            const uint32_t idesc = idesc_f8_e4m3(256, 256);
            int stage = 0;
            uint32_t ph = 0, kiter = 0;
            bool ok = true;
            for (int t = cluster; t < g.num_tiles && ok; t += nclusters) {
                for (int ks = 0; ks < NKS; ++ks) {
                    const uint32_t buf = kiter % kBufs, tph = (kiter / kBufs) & 1;
                    bool w = true;
                    if (lane == 0) {
                        w = mbar_wait_cluster(tempty + buf, tph ^ 1, abort_flag, prm.status, prm.timeout_ns,
                                              SITE_MMA_TMEM_EMPTY);
                        w = w && mbar_wait(full + stage, ph, abort_flag, prm.status, prm.timeout_ns, SITE_MMA_FULL);
                    }
                    if (!__shfl_sync(0xffffffffu, (int)w, 0)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (elect_one()) {
                        const uint64_t ad = desc_kmajor_sw128(smem_u32(smem + kOffA + stage * kABytes));
                        const uint64_t bd = desc_kmajor_sw128(smem_u32(smem + kOffB + stage * kBBytes));
                        const uint32_t d = tmem_base + buf * 256;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_f8_pair(d, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
                        tc_commit_pair(empty + stage, 3);
                        tc_commit_pair(tfull + buf, 3);
                    }
                    __syncwarp();
                    ++kiter;
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            if (elect_one())
                tc_commit_pair(final_bar, 3);
            __syncwarp();
        } else if (warp >= 2 && prm.o.out_mode == OUT_PARTIAL_F32 && g.slice_loop != 2) {
            // ------------------------------------------------ park drain (band path)
            const int h = warp - 2;   // column half whose four epilogue warps this warp serves
            BandSignals signals;
            uint32_t pk = 0;          // parks of each of those warps drained so far
            bool ok = true;
            for (int t = cluster; t < g.num_tiles && ok; t += nclusters) {
                const PairTile tc = decode_pair(t, g);
                const int m_cta = tc.m0 + 128 * (int)rank;
                if (m_cta < tc.band_end) {
                    const TileCoord ct{tc.b, tc.p, m_cta, tc.n0, 0};
                    float4 *tb = partial_tile_base(prm.o, g, ct, 256);
                    for (int q = 0; q < 4 && ok; ++q) {
                        const int ew = h * 4 + q;   // epilogue warp 4 + ew owns lane quarter q, half h
                        if (!mbar_wait(park_full + ew, pk & 1, abort_flag, prm.status, prm.timeout_ns,
                                       SITE_PARK_FULL)) {
                            ok = false;
                            break;
                        }
                        const uint32_t park = smem_u32(smem + kOffPark + ew * kParkBytes);
                        float4 *dst = tb + ((q * 8 + h * 4) * 8) * 32 + lane;
#pragma unroll 1
                        for (int i = 0; i < kParkBytes / 512; i += 4) {
                            uint4 v[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                v[u] = ld_shared_v4(park + (uint32_t)(((i + u) * 32 + lane) * 16));
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                __stcg(dst + (i + u) * 32, make_float4(__uint_as_float(v[u].x), __uint_as_float(v[u].y),
                                                                       __uint_as_float(v[u].z), __uint_as_float(v[u].w)));
                        }
                        __syncwarp();   // every lane has read the park
                        if (lane == 0)
                            mbar_arrive(park_empty + ew);
                    }
                    ++pk;
                }
                if (ok)
                    signals.add(prm.o, tc.b, 4);   // this tile's four parks of half h (or none past the band end)
            }
            if (ok)
                signals.flush(prm.o);
        }
    } else {
        setmaxnreg_inc<kRegsHigh>();
        // ---------------------------------------------------- epilogue (both CTAs)
        const int ew = warp - 4;
        const int q = warp & 3;         // TMEM lane quarter
        const int h = ew >> 2;          // 128-column half of the CTA's 256 columns
        const int row = q * 32 + lane;  // row within this CTA's 128 rows
        const uint32_t park = smem_u32(smem + kOffPark + ew * kParkBytes);
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) + h * 128;
        const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
        const bool partial = prm.o.out_mode == OUT_PARTIAL_F32;
        const bool exact = g.slice_loop == 2;
        uint32_t pk = 0;      // partials parked so far (park-full/empty phase)
        uint32_t kiter = 0;
        bool ok = true;
        const int nsl = g.slice_loop ? g.P : 1;
        for (int t = cluster; t < g.num_tiles && ok; t += nclusters) {
            const PairTile tc = decode_pair(t, g);
            const int m_cta = tc.m0 + 128 * (int)rank;
            const int rows_valid = max(0, min(32, tc.band_end - m_cta - q * 32));
            const int64_t mrow = min(m_cta + row, g.M - 1);
            const int64_t nblk = (tc.n0 + h * 128) >> 7;
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j)
                acc[j] = 0.0f;
            // raw scale factors of the next K-step, loaded a step ahead and
            // multiplied where used, so the load latency overlaps a step
            const float *sa_row = prm.sa[tc.p] + mrow * KB;
            const float *sb_blk = prm.sb[tc.p] + nblk * KB;
            float a_next = __ldg(sa_row), b_next = __ldg(sb_blk);
            for (int sl = 0; sl < nsl && ok; ++sl) {
                for (int kb = 0; kb < KB; ++kb) {
                    const float a_cur = a_next, b_cur = b_next;
                    if (kb + 1 < KB) {
                        a_next = __ldg(sa_row + kb + 1);
                        b_next = __ldg(sb_blk + kb + 1);
                    } else if (sl + 1 < nsl) {
                        sa_row = prm.sa[sl + 1] + mrow * KB;
                        sb_blk = prm.sb[sl + 1] + nblk * KB;
                        a_next = __ldg(sa_row);
                        b_next = __ldg(sb_blk);
                    }
                    const uint32_t buf = kiter % kBufs, tph = (kiter / kBufs) & 1;
                    if (!mbar_wait(tfull + buf, tph, abort_flag, prm.status, prm.timeout_ns, SITE_EPI_TMEM_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float s = a_cur * b_cur;
                    const uint32_t taddr = lane_base + buf * 256;
                    uint32_t r[64];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        tmem_ld_x64(taddr + c * 64, r);
                        tmem_wait_ld(r);
                        if (c == 1) {
                            // the K-block buffer is read: hand it back to the MMA warp
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                if (rank == 0)
                                    mbar_arrive(tempty + buf);
                                else
                                    mbar_arrive_cluster(tempty_leader + 8u * buf);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 64; j += 2)
                            fma2(acc[c * 64 + j], acc[c * 64 + j + 1], s, r[j], r[j + 1]);
                    }
                    ++kiter;
                }
                if (exact && ok && nsl > 1) {
                    // acc is slice sl's fp32 partial W_sl of this row.  Fold it into
                    // the running sum in the reducer's order, run = W_0 then
                    // run = run + W_p; the last sum stays in acc.
                    if (sl == 0) {
#pragma unroll
                        for (int u = 0; u < 32; ++u)
                            st_shared_v4(park + (uint32_t)((u * 32 + lane) * 16),
                                         make_uint4(__float_as_uint(acc[4 * u]), __float_as_uint(acc[4 * u + 1]),
                                                    __float_as_uint(acc[4 * u + 2]), __float_as_uint(acc[4 * u + 3])));
                    } else {
                        const bool last = sl + 1 == nsl;
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            const uint32_t addr = park + (uint32_t)((u * 32 + lane) * 16);
                            const uint4 v = ld_shared_v4(addr);
                            acc[4 * u] = __fadd_rn(__uint_as_float(v.x), acc[4 * u]);
                            acc[4 * u + 1] = __fadd_rn(__uint_as_float(v.y), acc[4 * u + 1]);
                            acc[4 * u + 2] = __fadd_rn(__uint_as_float(v.z), acc[4 * u + 2]);
                            acc[4 * u + 3] = __fadd_rn(__uint_as_float(v.w), acc[4 * u + 3]);
                            if (!last)
                                st_shared_v4(addr, make_uint4(__float_as_uint(acc[4 * u]), __float_as_uint(acc[4 * u + 1]),
                                                              __float_as_uint(acc[4 * u + 2]),
                                                              __float_as_uint(acc[4 * u + 3])));
                        }
                        if (last)
                            continue;
                    }
#pragma unroll
                    for (int j = 0; j < 128; ++j)
                        acc[j] = 0.0f;
                }
            }
            if (!ok)
                break;
            __syncwarp();   // every lane's last read of the running sum precedes the staging writes
            // -------- tile store
            if (partial) {
                if (m_cta < tc.band_end) {
                    // park this warp's 32 rows x 128 columns in the blocked order of the
                    // partial layout (chunks h*4 .. h*4+3 of lane quarter q are 16 KB
                    // contiguous in W) once its store warp has copied the previous one
                    if (!mbar_wait(park_empty + ew, (pk & 1) ^ 1, abort_flag, prm.status, prm.timeout_ns,
                                   SITE_PARK_EMPTY)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const float *a = &acc[c * 32 + u * 4];
                            st_shared_v4(park + (uint32_t)(((c * 8 + u) * 32 + lane) * 16),
                                         make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]),
                                                    __float_as_uint(a[2]), __float_as_uint(a[3])));
                        }
                    __syncwarp();   // every lane's park writes precede the arrive
                    if (lane == 0)
                        mbar_arrive(park_full + ew);
                    ++pk;
                }
                // a CTA tile past the band end (ragged bands) owns no partial block: its
                // store warp publishes the band without waiting for a park
            } else if (prm.o.out_mode == OUT_BF16) {
                const TileCoord ct{tc.b, tc.p, m_cta, tc.n0, 0};
                char *base = tile_out_base(prm.o, g, ct, 2) + ((int64_t)q * 32 * g.N + h * 128) * 2;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float *a = &acc[c * 32 + u * 8];
                        v[u] = make_uint4(bf16x2_from_f32(a[0], a[1]), bf16x2_from_f32(a[2], a[3]),
                                          bf16x2_from_f32(a[4], a[5]), bf16x2_from_f32(a[6], a[7]));
                    }
                    store_chunk<4>(park, v, base + c * 64, (int64_t)g.N * 2, rows_valid);
                }
            } else {
                const TileCoord ct{tc.b, tc.p, m_cta, tc.n0, 0};
                char *base = tile_out_base(prm.o, g, ct, 4) + ((int64_t)q * 32 * g.N + h * 128) * 4;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float *a = &acc[c * 32 + u * 4];
                        v[u] = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                          __float_as_uint(a[3]));
                    }
                    store_chunk<8>(park, v, base + c * 128, (int64_t)g.N * 4, rows_valid);
                }
            }
        }
    }

    __syncwarp();
    __syncthreads();   // every role of this CTA is done
    if (warp == 1 && lane == 0) {
        // every pair MMA has completed before either CTA's TMEM goes away
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(final_bar, 0)) {
            if (globaltimer() - t0 > prm.timeout_ns) {
                report(prm.status, kErrTimeout, SITE_TEARDOWN_MMA);
                break;
            }
        }
    }
    __syncwarp();
    if (*abort_flag) {
        // copies already issued by this CTA complete on the leader's barrier, which this
        // CTA cannot observe: give them time to land before the shared memory is released
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < kAbortGraceNs) {
        }
    }
    tc_fence_before();
    cluster_sync();   // no CTA leaves while its peer may still signal it
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc_pair(tmem_base, 512);
}

constexpr int kMaxDevices = 64;
int max_clusters_cached[kMaxDevices];   // per device: 0 unknown, else clusters + 1

}  // namespace

int gemm_blockscale_2sm_max_clusters()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 0;
    if (max_clusters_cached[dev] > 0)
        return max_clusters_cached[dev] - 1;
    if (ensure_dynamic_smem(reinterpret_cast<const void *>(gemm_blockscale_2sm_kernel), kSmemBytes) != cudaSuccess) {
        max_clusters_cached[dev] = 1;
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_blockscale_2sm_kernel, &cfg) != cudaSuccess)
        n = 0;
    max_clusters_cached[dev] = n + 1;
    return n;
}

int gemm_blockscale_2sm_num_regs()
{
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, gemm_blockscale_2sm_kernel) != cudaSuccess)
        return -1;
    return a.numRegs;
}

BsPlan plan_blockscale(int P, int64_t M, int64_t N, int64_t K, int bands, int slice_loop, int num_sms, int use_pair)
{
    BsPlan pl{};
    if (slice_loop)
        bands = 1;
    TileGrid &g = pl.g;
    g.P = P;
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    g.bands = bands;
    g.rows_per_band = (int)(M / bands);
    g.mt_per_band = (g.rows_per_band + 127) / 128;   // 128-row tiles of the blocked partial layout
    g.slice_loop = slice_loop;
    if (use_pair && N % 256 == 0) {
        const int regs2 = gemm_blockscale_2sm_num_regs();
        const int clusters = gemm_blockscale_2sm_max_clusters();
        if (clusters > 0 && regs2 >= 0 && (int64_t)regs2 * kThreads >= kRegsLow * 128 + kRegsHigh * 256) {
            pl.pair = 1;
            pl.bn = 256;
            pl.box_b_rows = 128;
            g.ntiles_n = (int)(N / 256);
            const int mt2 = (g.rows_per_band + 255) / 256;
            g.num_tiles = (slice_loop ? 1 : P) * bands * mt2 * g.ntiles_n;
            pl.grid = 2 * std::min(g.num_tiles, clusters);
            pl.band_signals = (uint32_t)(mt2 * g.ntiles_n * P * 16);   // 8 warps x 2 CTAs per pair tile
            return pl;
        }
    }
    pl.pair = 0;
    pl.bn = (N % 256 == 0) ? 256 : 128;
    pl.box_b_rows = pl.bn;
    g.ntiles_n = (int)(N / pl.bn);
    g.num_tiles = (slice_loop ? 1 : P) * bands * g.mt_per_band * g.ntiles_n;
    pl.grid = std::min(g.num_tiles, num_sms);
    pl.band_signals = (uint32_t)(g.mt_per_band * g.ntiles_n * P * 8);
    return pl;
}

cudaError_t launch_blockscale(const BsParams &p, const BsPlan &plan, cudaStream_t s)
{
    if (plan.pair)
        return launch_gemm_blockscale_2sm(p, plan.grid / 2, s);
    return launch_gemm_blockscale(p, plan.bn, plan.grid, s);
}

cudaError_t launch_gemm_blockscale_2sm(const BsParams &p, int clusters, cudaStream_t s)
{
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(gemm_blockscale_2sm_kernel), kSmemBytes);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_blockscale_2sm_kernel, p);
}

}  // namespace gemmar
