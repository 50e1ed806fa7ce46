// gemm_blockscale_2sm.cu -- the blockscale GEMM on CTA pairs (tcgen05
// cta_group::2), same arithmetic as gemm_blockscale.cu ("MORI GEMM +
// All-Reduce Benchmark", "Running the benchmark": A 1x128, B 128x128 fp32
// scales, applied per 128-K block while draining TMEM).
//
// A cluster of two CTAs on two SMs computes a 256 x 128 pair tile: CTA r owns
// rows m0 + 128r .. +127 in its TMEM, loads those 128 rows of A and rows
// n0 + 64r .. +63 of B into its shared memory (24 KB per 128-K stage, 8
// stages), and the leader (rank 0) issues tcgen05.mma.cta_group::2 (M=256,
// N=128, K=32) that reads both CTAs' stages.  Per SM that is the operand
// traffic of a 128 x 256 single-CTA tile for half the TMEM, so:
//   - TMEM holds 4 K-block buffers of 128 columns (4-deep MMA/epilogue slack);
//   - each epilogue thread owns one row x 64 columns: acc[64] in registers,
//     leaving room to park a finished tile's fp32 partial in registers and
//     stream it to HBM one 16-byte unit per K-step of the next tile, so the
//     partial write of the band path overlaps the tensor cores instead of
//     stalling them.
// Barriers: stage-full counts both CTAs' TMA bytes on the leader; stage-empty,
// TMEM-full and the final barrier are multicast-committed to both CTAs;
// TMEM-empty lives on the leader and collects 8 local + 8 remote arrivals.
#include <algorithm>

#include "epilogue.cuh"

namespace gemmar {
using namespace ptx;

namespace {

constexpr int kThreads = 384;
constexpr int kStages = 8;
constexpr int kABytes = 128 * 128;           // this CTA's 128 rows of A, one 128-K stage
constexpr int kBBytes = 64 * 128;            // this CTA's 64 rows of B
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kBufs = 4;                     // TMEM K-block buffers of 128 columns
constexpr int kEpiWarps = 8;
constexpr int kOffA = 0;
constexpr int kOffB = kStages * kABytes;
constexpr int kOffStaging = kOffB + kStages * kBBytes;
constexpr int kOffBar = kOffStaging + kEpiWarps * 4096;
constexpr int kNumBars = 2 * kStages + 2 * kBufs + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kBBytes % 1024 == 0, "B stages stay 1024-byte aligned");
constexpr int kRegsLow = 56;
constexpr int kRegsHigh = 224;
constexpr uint32_t kAbortGraceNs = 200000;   // let in-flight copies land before an aborting CTA exits

struct PairTile {
    int b, p, m0, n0, band_end;
};

__device__ __forceinline__ PairTile decode_pair(int t, const TileGrid &g)
{
    PairTile c;
    const int nt = t % g.ntiles_n;
    int r = t / g.ntiles_n;
    c.n0 = nt * 128;
    if (g.slice_loop) {
        c.b = 0;
        c.p = 0;
        c.m0 = r * 256;
        c.band_end = g.M;
        return c;
    }
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
            int stage = 0, issued = 0;
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
                    tma_load_2d_pair(smem + kOffA + stage * kABytes, &prm.tmA[p], fb, kb * 128, tc.m0 + 128 * (int)rank);
                    tma_load_2d_pair(smem + kOffB + stage * kBBytes, &prm.tmB[p], fb, kb * 128, tc.n0 + 64 * (int)rank);
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            (void)issued;
        } else if (warp == 1 && rank == 0) {
            // ------------------------------------------------ MMA issuer (leader)
            // The whole warp runs the loop so that descriptors and TMEM addresses
            // stay warp-uniform; lane 0 polls the barriers and broadcasts the
            // outcome, one elected lane issues.
            const uint32_t idesc = idesc_f8_e4m3(256, 128);
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
                        const uint32_t d = tmem_base + buf * 128;
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
        }
    } else {
        setmaxnreg_inc<kRegsHigh>();
        // ---------------------------------------------------- epilogue (both CTAs)
        const int ew = warp - 4;
        const int q = warp & 3;         // TMEM lane quarter
        const int h = ew >> 2;          // 64-column half of the pair tile
        const int row = q * 32 + lane;  // row within this CTA's 128 rows
        const uint32_t staging = smem_u32(smem + kOffStaging + ew * 4096);
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) + h * 64;
        const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
        const bool partial = prm.o.out_mode == OUT_PARTIAL_F32;
        // the previous tile's fp32 partial, stored one unit per K-step
        float park[64];
        float4 *park_base = nullptr;   // null: nothing parked
        int park_band = 0;
        uint32_t kiter = 0;
        bool ok = true;
        for (int t = cluster; t < g.num_tiles && ok; t += nclusters) {
            const PairTile tc = decode_pair(t, g);
            const int m_cta = tc.m0 + 128 * (int)rank;
            const int rows_valid = max(0, min(32, tc.band_end - m_cta - q * 32));
            const int64_t mrow = min(m_cta + row, g.M - 1);
            const int64_t nblk = tc.n0 >> 7;
            float acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j)
                acc[j] = 0.0f;
            const int nsl = g.slice_loop ? g.P : 1;
            const float *sa_row = prm.sa[tc.p] + mrow * KB;
            const float *sb_blk = prm.sb[tc.p] + nblk * KB;
            // raw scale factors of the next K-step, loaded a step ahead and
            // multiplied only where used, so the load latency overlaps a step
            float a_next = __ldg(sa_row), b_next = __ldg(sb_blk);
            int sl = 0, kb = 0;
            for (int ks0 = 0; ks0 < NKS && ok; ks0 += 16) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (ks0 == 0 && park_base != nullptr) {
                        // stream unit j of the parked partial (chunk h*2 + j/8, unit j%8)
                        __stcg(park_base + ((q * 4 + h * 2 + (j >> 3)) * 8 + (j & 7)) * 32 + lane,
                               make_float4(park[4 * j], park[4 * j + 1], park[4 * j + 2], park[4 * j + 3]));
                        if (j == 15) {
                            signal_band(prm.o, park_band);
                            park_base = nullptr;
                        }
                    }
                    if (ks0 + j < NKS && ok) {
                        const float a_cur = a_next, b_cur = b_next;
                        if (++kb == KB) {
                            kb = 0;
                            if (++sl < nsl) {
                                sa_row = prm.sa[sl] + mrow * KB;
                                sb_blk = prm.sb[sl] + nblk * KB;
                            }
                        }
                        if (ks0 + j + 1 < NKS) {
                            a_next = __ldg(sa_row + kb);
                            b_next = __ldg(sb_blk + kb);
                        }
                        const uint32_t buf = kiter % kBufs, tph = (kiter / kBufs) & 1;
                        if (!mbar_wait(tfull + buf, tph, abort_flag, prm.status, prm.timeout_ns, SITE_EPI_TMEM_FULL)) {
                            ok = false;
                        } else {
                            tc_fence_after();
                            uint32_t r[64];
                            tmem_ld_x64(lane_base + buf * 128, r);
                            tmem_wait_ld(r);
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                if (rank == 0)
                                    mbar_arrive(tempty + buf);
                                else
                                    mbar_arrive_cluster(tempty_leader + 8u * buf);
                            }
                            const float s = a_cur * b_cur;
#pragma unroll
                            for (int i = 0; i < 64; i += 2)
                                fma2(acc[i], acc[i + 1], s, r[i], r[i + 1]);
                            ++kiter;
                        }
                    }
                }
            }
            if (!ok)
                break;
            // -------- tile store
            if (partial) {
                // park this tile's partial; it goes out during the next tile's K-steps
                if (park_base != nullptr) {   // a previous park not fully streamed (cannot happen: 16 units per first block)
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        __stcg(park_base + ((q * 4 + h * 2 + (j >> 3)) * 8 + (j & 7)) * 32 + lane,
                               make_float4(park[4 * j], park[4 * j + 1], park[4 * j + 2], park[4 * j + 3]));
                    signal_band(prm.o, park_band);
                }
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    park[j] = acc[j];
                park_band = tc.b;
                const TileCoord ct{tc.b, tc.p, m_cta, tc.n0, 0};
                // a CTA tile past the band end (ragged bands) owns no partial block
                park_base = (m_cta < tc.band_end) ? partial_tile_base(prm.o, g, ct, 128) : nullptr;
                if (park_base == nullptr)
                    signal_band(prm.o, tc.b);
            } else if (prm.o.out_mode == OUT_BF16) {
                const TileCoord ct{tc.b, tc.p, m_cta, tc.n0, 0};
                char *base = tile_out_base(prm.o, g, ct, 2) + ((int64_t)q * 32 * g.N + h * 64) * 2;
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float *a = &acc[u * 8];
                    v[u] = make_uint4(bf16x2_from_f32(a[0], a[1]), bf16x2_from_f32(a[2], a[3]),
                                      bf16x2_from_f32(a[4], a[5]), bf16x2_from_f32(a[6], a[7]));
                }
                store_chunk<8>(staging, v, base, (int64_t)g.N * 2, rows_valid);
            } else {
                const TileCoord ct{tc.b, tc.p, m_cta, tc.n0, 0};
                char *base = tile_out_base(prm.o, g, ct, 4) + ((int64_t)q * 32 * g.N + h * 64) * 4;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
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
        // the last parked partial
        if (ok && park_base != nullptr) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                __stcg(park_base + ((q * 4 + h * 2 + (j >> 3)) * 8 + (j & 7)) * 32 + lane,
                       make_float4(park[4 * j], park[4 * j + 1], park[4 * j + 2], park[4 * j + 3]));
            signal_band(prm.o, park_band);
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

int max_clusters_cached = -1;

}  // namespace

int gemm_blockscale_2sm_max_clusters()
{
    if (max_clusters_cached >= 0)
        return max_clusters_cached;
    if (cudaFuncSetAttribute(gemm_blockscale_2sm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess) {
        max_clusters_cached = 0;
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
    max_clusters_cached = n;
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
    const int regs2 = gemm_blockscale_2sm_num_regs();
    const int clusters = gemm_blockscale_2sm_max_clusters();
    pl.pair = use_pair && clusters > 0 && regs2 >= 0 && (int64_t)regs2 * gemm_threads() >= 56 * 128 + 224 * 256;
    if (pl.pair) {
        pl.bn = 128;
        pl.box_b_rows = 64;
        g.ntiles_n = (int)(N / 128);
        const int mt2 = (g.rows_per_band + 255) / 256;
        g.num_tiles = (slice_loop ? 1 : P) * bands * mt2 * g.ntiles_n;
        pl.grid = 2 * std::min(g.num_tiles, clusters);
        pl.band_signals = (uint32_t)(mt2 * g.ntiles_n * P * 16);   // 8 warps x 2 CTAs per pair tile
    } else {
        pl.bn = (N % 256 == 0) ? 256 : 128;
        pl.box_b_rows = pl.bn;
        g.ntiles_n = (int)(N / pl.bn);
        g.num_tiles = (slice_loop ? 1 : P) * bands * g.mt_per_band * g.ntiles_n;
        pl.grid = std::min(g.num_tiles, num_sms);
        pl.band_signals = (uint32_t)(g.mt_per_band * g.ntiles_n * P * 8);
    }
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
