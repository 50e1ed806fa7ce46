// kernels.h -- host-side launch interface between the C ABI (gemmar.cu) and
// the kernel translation units.  Internal to libgemmar.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace gemmar {

constexpr int kMaxP = 8;      // == GEMMAR_MAX_P
constexpr int kMaxBands = 1024;

enum OutMode : int {
    OUT_PARTIAL_F32 = 0,   // fp32 partial into W[band][p][row-in-band][N], then signal the band counter
    OUT_F32 = 1,           // fp32 C[M,N]
    OUT_BF16 = 2,          // bf16 C[M,N]
};

// Work decomposition shared by both GEMM kernels: tile t covers rows
// [m0, m0 + min(128, band end - m0)) and columns [n0, n0 + BN) of slice p in
// band b, with t = ((b * P + p) * mt_per_band + mt) * ntiles_n + nt, i.e. in
// band order so that band 0's partials are complete first.  With slice_loop
// a tile instead runs over every slice (K-steps p*K/128 + kb) and its one
// accumulator holds the P-way sum.
struct TileGrid {
    int P, M, N, K;
    int bands, rows_per_band, mt_per_band, ntiles_n, num_tiles;
    int slice_loop;   // 1: a tile covers all P slices (bands == 1, t = mt * ntiles_n + nt) in one
                      //    fp32 chain; 2 (CTA-pair kernel): the same tiles, each slice's partial
                      //    summed in the band reducer's order
};

struct GemmOut {
    void *out;               // W (OUT_PARTIAL_F32) or C
    uint32_t *band_done;     // per-band tile-retire counters (OUT_PARTIAL_F32)
    int out_mode;
    int skip_band;           // fault injection: this band is never signalled (-1: none)
    // In-kernel band reduce (OUT_PARTIAL_F32 only; reduce_next == nullptr: off).  A
    // warp of each CTA claims 32 x 32 blocks of retired bands from reduce_next[band]
    // and writes their bf16 sums to red_out [M, N]; the blocks it leaves are reduced
    // by the band reduce kernel that follows, in each band from the final count on.
    uint32_t *reduce_next;   // [bands] claim counters, zero before the launch
    uint16_t *red_out;
    uint32_t band_expected;  // release signals that complete a band
};

struct BsParams {
    CUtensorMap tmA[kMaxP];  // A_p: dims {K, M} bytes, box {128, 128}, 128B swizzle
    CUtensorMap tmB[kMaxP];  // B_p: dims {K, N} bytes, box {128, BN}, 128B swizzle
    const float *sa[kMaxP];  // [M, K/128]
    const float *sb[kMaxP];  // [N/128, K/128]
    TileGrid g;
    GemmOut o;
    ptx::DevStatus *status;
    uint64_t timeout_ns;
};

// Parameters of the whole-K kernel family (gemm_mx.cu): mxfp8 (native
// block-scaled MMA, the scale images below) and ptpc (plain e4m3 MMA, one fp32
// scale per row of A and per row of B applied to the tile in the epilogue).
struct MxParams {
    CUtensorMap tmA[kMaxP];
    CUtensorMap tmB[kMaxP];
    const uint8_t *sfa;      // mx: repacked A scale words: [P][bands][mt_per_band][K/128][512 B]
    const uint8_t *sfb;      // mx: repacked B scale words: [P][N/BN][K/128][1024 B]
    const float *pa[kMaxP];  // ptpc: per-token scales of A_p, [M]
    const float *pb[kMaxP];  // ptpc: per-channel scales of B_p, [N]
    TileGrid g;
    GemmOut o;
    ptx::DevStatus *status;
    uint64_t timeout_ns;
};

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for the current device, done
// once per (kernel, device): the attribute belongs to the kernel's instance on
// each device, so a process that drives several GPUs sets it on each.
cudaError_t ensure_dynamic_smem(const void *kernel, int bytes);

// GEMM launchers (bn: 256 or 128 for blockscale; 224 or 128 for mx).
cudaError_t launch_gemm_blockscale(const BsParams &p, int bn, int grid, cudaStream_t s);
cudaError_t launch_gemm_mx(const MxParams &p, int bn, int grid, cudaStream_t s);
cudaError_t launch_gemm_ptpc(const MxParams &p, int bn, int grid, cudaStream_t s);
// Register count each GEMM kernel was built with (the warp-role register split needs it).
int gemm_blockscale_num_regs(int bn);
int gemm_mx_num_regs(int bn);
int gemm_ptpc_num_regs(int bn);
// A whole-K kernel (mx or ptpc) built with `regs` per thread has registers enough for its
// warp-role split.
bool gemm_mx_split_ok(int regs);
// The one-CTA blockscale kernel was built with registers enough for its warp-role split
// (setmaxnreg would wait forever otherwise).
bool gemm_blockscale_split_ok(int bn);

// Blockscale launch plan: CTA pairs (gemm_blockscale_2sm.cu, 256 x 128 pair
// tiles) when the device can co-schedule two-CTA clusters, else one CTA per
// tile (gemm_blockscale.cu, 128 x bn).  Every blockscale path of the library
// goes through the same plan, so all of them share one arithmetic.
struct BsPlan {
    int pair;              // 1: CTA-pair kernel
    int bn;                // tile width along N (also the blocked-partial tile width)
    int box_b_rows;        // rows of B each CTA loads per stage (TMA box)
    int grid;              // CTAs to launch
    uint32_t band_signals; // release signals per band in the fused band path
    TileGrid g;
};
BsPlan plan_blockscale(int P, int64_t M, int64_t N, int64_t K, int bands, int slice_loop, int num_sms,
                       int use_pair = 0);
cudaError_t launch_blockscale(const BsParams &p, const BsPlan &plan, cudaStream_t s);
int gemm_blockscale_2sm_max_clusters();
int gemm_blockscale_2sm_num_regs();
cudaError_t launch_gemm_blockscale_2sm(const BsParams &p, int clusters, cudaStream_t s);

// Scale repack for the mx GEMM (row-major ue8m0 bytes -> the tcgen05.cp image).
// ea/eb are host arrays of P device pointers.  Image layout: see streaming.cu.
cudaError_t launch_mx_repack(const uint8_t *const *ea, const uint8_t *const *eb, int P, int M, int N, int K,
                             int bands, int bn, uint8_t *sfa_out, uint8_t *sfb_out, cudaStream_t s);

// Streaming kernels.
cudaError_t launch_band_reduce(const float *W, uint16_t *out, int P, int64_t M, int64_t N, int bands,
                               const uint32_t *band_done, uint32_t expected, ptx::DevStatus *status,
                               uint64_t timeout_ns, int num_sms, cudaStream_t s);
// The same reduce over the fused path's tile-blocked partials (layout: epilogue.cuh).
// claimed (device, [bands], may be nullptr): in band b the blocks below claimed[b]
// were already reduced by the GEMM kernel's reducer warps (GemmOut::reduce_next).
// The band reduce with the row quantiser folded in (fp8 wire): codes q [M, N] and
// row scales s [M] from the blocked partials, taking the bf16 sums of the blocks
// below claimed[b] (may be nullptr) from `out`.  N <= kBandQuantMaxN.
constexpr int kBandQuantMaxN = 12288;   // 8 bf16 rows of N parked in shared memory
cudaError_t launch_band_reduce_quant(const float *W, const uint16_t *out, int P, int64_t M, int64_t N, int bands,
                                     int bn, const uint32_t *band_done, uint32_t expected, const uint32_t *claimed,
                                     uint8_t *q, float *s, ptx::DevStatus *status, uint64_t timeout_ns,
                                     cudaStream_t st);
cudaError_t launch_band_reduce_blocked(const float *W, uint16_t *out, int P, int64_t M, int64_t N, int bands,
                                       int bn, const uint32_t *band_done, uint32_t expected,
                                       const uint32_t *claimed, ptx::DevStatus *status,
                                       uint64_t timeout_ns, int num_sms, cudaStream_t s);   // one wave of CTAs
// Floats of blocked partials a fused call needs (ragged bands pad tiles to 128 rows).
inline int64_t blocked_partial_floats(int P, int64_t M, int bands, int64_t N)
{
    const int64_t rpb = M / bands, mtpb = (rpb + 127) / 128;
    return (int64_t)P * bands * mtpb * 128 * N;
}
cudaError_t launch_rowquant(const void *x, int x_is_bf16, int64_t M, int64_t N, uint8_t *q, float *s,
                            int num_sms, cudaStream_t st);
cudaError_t launch_rowdequant(const uint8_t *q, const float *s, int64_t M, int64_t N, uint16_t *y, int num_sms,
                              cudaStream_t st);
// Device quantisers; x is fp32 or (x_is_bf16) bf16.
cudaError_t launch_quant_blockscale(const void *x, int x_is_bf16, int64_t R, int64_t C, int group_rows, uint8_t *q,
                                    float *scales, int num_sms, cudaStream_t st);
cudaError_t launch_quant_mx(const void *x, int x_is_bf16, int64_t R, int64_t C, uint8_t *q, uint8_t *e8, int num_sms,
                            cudaStream_t st);

}  // namespace gemmar
