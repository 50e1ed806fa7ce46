/*
 * gemmar.h -- C ABI of libgemmar: the block-scaled fp8 GEMM and row-parallel
 * reduce of a DeepSeek-style attention block's output projection (wo_b),
 * run on one GB300 GPU (sm_103a).
 *
 * What the path computes (sources are web pages, cited by title and section):
 *   - wo_b is a row-parallel linear layer: a block-scale fp8 GEMM whose
 *     [M, hidden] result is all-reduced over the ranks that each hold one
 *     K-slice of the weight (sglang pull request #40757, "What").
 *   - Quantisation "blockscale": A (activations) with one fp32 scale per 1x128
 *     group along K, B (weight) with one fp32 scale per 128x128 block
 *     ("MORI GEMM + All-Reduce Benchmark", "Running the benchmark").
 *   - Quantisation "mxfp8": e4m3 with a ue8m0 power-of-two scale per 1x32 group,
 *     the exponent taken from the IEEE bits (sglang pull request #43480,
 *     "What" and review item 7 "Duplicated ue8m0 scale rule").
 *   - The reduce accumulates in fp32 and the output is bf16; the optional
 *     "fp8 wire" sends each output row as e4m3 with one fp32 scale
 *     ("MORI GEMM + All-Reduce Benchmark", "The fp8 wire").
 *   - The fused kernel writes each destination's row band as soon as that
 *     band's tiles are done (sglang pull request #40757, "What"; MORI page,
 *     "Where the time goes").
 *
 * On one GPU the P "ranks" are P K-slices resident in this GPU's memory; the
 * exchange is the band reduce reading their fp32 partials.  No collective runs.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major,
 *     contiguous, 16-byte aligned (else GEMMAR_ERR_ALIGN).  Sizes are element
 *     counts.  e4m3 tensors are uint8 codes (OCP E4M3FN); bf16 tensors are
 *     uint16 bit patterns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; 0 = legacy
 *     default stream) and returns a host status at once.  Any status other
 *     than GEMMAR_OK returned by a call means nothing was launched, except
 *     GEMMAR_ERR_CUDA, which reports that a launch or CUDA call failed.
 *   - Device-side failures (a bounded wait that expired) are recorded in the
 *     context's device status word; gemmar_status() reads it after the work is
 *     complete and makes the context sticky-disabled: every later call
 *     returns GEMMAR_ERR_DISABLED.  No kernel traps, hangs or faults on
 *     purpose; every device wait has a time limit.
 *   - The context owns only its workspace (fp32 partials, band counters,
 *     scale repack area, fp8-wire staging) and status word.  The workspace is
 *     overwritten by the next call that uses it; calls on one context must be
 *     stream-ordered (the same stream, or joined by events).
 *   - The current CUDA device must be the context's device.
 */
#ifndef GEMMAR_H
#define GEMMAR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemmar_ctx gemmar_ctx;

/* Status codes. */
enum {
    GEMMAR_OK = 0,
    GEMMAR_ERR_ARG = 1,        /* NULL pointer, bad enum value, negative or zero size */
    GEMMAR_ERR_SHAPE = 2,      /* shape the kernels cannot express (see gemmar_supports) */
    GEMMAR_ERR_ALIGN = 3,      /* a pointer is not 16-byte aligned */
    GEMMAR_ERR_WORKSPACE = 4,  /* call needs more workspace than gemmar_create sized */
    GEMMAR_ERR_CUDA = 5,       /* a CUDA runtime or driver call failed */
    GEMMAR_ERR_TIMEOUT = 6,    /* a device-side bounded wait expired (read by gemmar_status) */
    GEMMAR_ERR_DISABLED = 7,   /* context disabled by an earlier device-side failure */
    GEMMAR_ERR_DEVICE = 8      /* not an sm_103 device, wrong current device, or self-test mismatch */
};

/* Element types of an output or input matrix. */
enum { GEMMAR_DTYPE_F32 = 0, GEMMAR_DTYPE_BF16 = 1 };

/* Scale kinds. BLOCK128: fp32 A scales [M, K/128], fp32 B scales [N/128, K/128].
 * MX32: ue8m0 bytes (value 2^(byte-127)), A [M, K/32], B [N, K/32].
 * PTPC: fp32 per-token A scales [M] and per-channel B scales [N] (one scale
 * per row of A and of B over the whole K). */
enum { GEMMAR_SCALE_BLOCK128 = 0, GEMMAR_SCALE_MX32 = 1, GEMMAR_SCALE_PTPC = 2 };

/* Flags of gemmar_create and fused_gemm_reduce. */
#define GEMMAR_FP8_WIRE        (1u << 0)  /* fused: per-row e4m3 quantise + dequantise of the output */
#define GEMMAR_DEBUG_CANARY    (1u << 1)  /* fused: pre-fill partials and output with NaN */
#define GEMMAR_FAULT_SKIP_BAND (1u << 2)  /* fused, testing only: band 0 is never signalled, so the
                                             reducer's bounded wait expires (GEMMAR_ERR_TIMEOUT) */
#define GEMMAR_NO_SELF_TEST    (1u << 3)  /* create: skip the closed-form self-test */
#define GEMMAR_CTA_PAIR        (1u << 5)  /* create: run blockscale GEMMs with N % 256 == 0 on the CTA-pair
                                             kernel (256 x 256 tiles over two SMs; band partials parked in
                                             shared memory and copied out by two store warps) instead of
                                             the one-CTA kernel; the same bits (tests); on the wo_b band
                                             path its GEMM runs ~1810 us against ~1680 for the one-CTA
                                             kernel (both with the band reduce after the GEMM) */
#define GEMMAR_FUSE_SLICES     (1u << 4)  /* fused: each output tile accumulates all P slices itself (no
                                             partials, no band reduce); see fused_gemm_reduce */
#define GEMMAR_FUSE_ONCHIP     (1u << 6)  /* fused: the P slice partials of a tile stay on chip and are
                                             summed in the band reducer's order; bit-equal to the band
                                             path; see fused_gemm_reduce */
#define GEMMAR_SERIAL_REDUCE   (1u << 7)  /* fused band path: the GEMM kernel reduces no band while it
                                             runs; band_reduce sums every block after it (same bits) */
#define GEMMAR_FUSE_QUANTIZE   (1u << 8)  /* fused band path with GEMMAR_FP8_WIRE, N <= 12288: the band
                                             reduce quantises each row itself, without writing and
                                             re-reading the bf16 rows (same bits); ignored otherwise */

/* Largest number of K-slices ("ranks") one call takes. */
#define GEMMAR_MAX_P 8

/*
 * gemmar_supports -- can the kernels express this shape?  (The pages' op has
 * the same question answered by its supports(); sglang pull request #40757,
 * "Worth a reviewer's attention", last item.)  Rules:
 *   M >= 1; 1 <= P <= GEMMAR_MAX_P; 1 <= bands <= min(M, 1024) and M % bands == 0;
 *   BLOCK128: N % 128 == 0 (the B scale block); MX32: N % 128 == 0 or N % 224 == 0;
 *   PTPC: N % 128 == 0;
 *   K % 128 == 0 (every scale kind: one MMA stage is 128 of K);
 *   N <= 65536, K <= 65536, M <= 2^24.
 * Returns GEMMAR_OK or GEMMAR_ERR_SHAPE / GEMMAR_ERR_ARG.  Needs no GPU.
 */
int gemmar_supports(int P, int64_t M, int64_t N, int64_t K, int bands, int scale_kind);

/*
 * gemmar_create -- make a context on `device` (which must be current) whose
 * workspace serves fused_gemm_reduce calls with P <= max_P, M <= max_M and the
 * given N and K: fp32 partials of max_P*(max_M + 128*max_P)*N floats (a tile-
 * blocked layout; each band's rows are rounded up to whole 128-row tiles),
 * band counters, the
 * mxfp8 scale repack area and the fp8-wire staging.  Like the pages' window
 * it is sized once and never grows (sglang pull request #40757, "Worth a
 * reviewer's attention": the window is sized from the chunked-prefill
 * ceiling, not from the first request).  wait_timeout_ns bounds every
 * device-side wait (0 = 2 s).  Unless GEMMAR_NO_SELF_TEST is set, runs the
 * fused path on a closed-form case (unit codes and scales: every output
 * equals P*K) for every scale kind, on the band path and with the partials
 * summed on chip, under that deadline, and fails with GEMMAR_ERR_DEVICE on a
 * mismatch (the pages' self_test(), sglang pull request #40757).
 * On success *out owns device memory until gemmar_destroy.
 */
int gemmar_create(gemmar_ctx **out, int device, int64_t max_M, int64_t N, int64_t K, int max_P,
                  uint32_t flags, int64_t wait_timeout_ns);

/* gemmar_destroy -- synchronise the context's device and free its workspace. */
int gemmar_destroy(gemmar_ctx *ctx);

/*
 * gemmar_status -- read (blocking) the device status word; call after the
 * work is complete.  Returns GEMMAR_OK or the first device-side error
 * (GEMMAR_ERR_TIMEOUT); *detail (if not NULL) receives where it happened
 * (see the kernels' wait-site codes).  A device error disables the context.
 */
int gemmar_status(gemmar_ctx *ctx, int *detail);

/* gemmar_workspace_bytes -- device bytes the context holds. */
int64_t gemmar_workspace_bytes(const gemmar_ctx *ctx);

/*
 * Phase timing of fused_gemm_reduce, the per-layer breakdown of the MORI
 * page's "Where the time goes" table.  gemmar_set_phase_timing(ctx, 1) makes
 * every later fused call record CUDA events on its stream between its kernel
 * launches (nothing is skipped or reordered).  gemmar_phase_times waits for
 * those events, writes the summed milliseconds of each phase over the
 * recorded calls into ms[GEMMAR_NUM_PHASES] and the number of calls into
 * *calls, and clears the record.  Phases: GEMMAR_PHASE_GEMM (scale repack,
 * GEMM with band-ordered partial stores), GEMMAR_PHASE_REDUCE (band_reduce),
 * GEMMAR_PHASE_QUANTIZE and GEMMAR_PHASE_DEQUANTIZE (the fp8 wire; 0 when off;
 * with GEMMAR_FUSE_QUANTIZE the quantiser runs inside GEMMAR_PHASE_REDUCE).  On
 * the band path with the in-kernel reduce, GEMMAR_PHASE_GEMM includes the blocks
 * the GEMM kernel summed (gemmar_overlap_stats) and GEMMAR_PHASE_REDUCE the rest.
 * At most 65536 calls are recorded between reads (later ones are not timed).
 */
enum { GEMMAR_PHASE_GEMM = 0, GEMMAR_PHASE_REDUCE = 1, GEMMAR_PHASE_QUANTIZE = 2,
       GEMMAR_PHASE_DEQUANTIZE = 3, GEMMAR_NUM_PHASES = 4 };
int gemmar_set_phase_timing(gemmar_ctx *ctx, int enable);
int gemmar_phase_times(gemmar_ctx *ctx, float *ms, int *calls);

/*
 * gemmar_overlap_stats -- of the last fused_gemm_reduce band-path call on this
 * context, *total = its 32-row x 32-column output blocks and *overlapped = how
 * many of them the GEMM kernel's reducer warps summed while the GEMM was still
 * running (the rest were summed by band_reduce after it).  Both 0 when the last
 * fused call did not take the band path, or took it without the in-kernel
 * reduce (GEMMAR_SERIAL_REDUCE, or the CTA-pair kernel).  Reads device
 * memory with a synchronous copy: call after that call's work has completed.
 */
int gemmar_overlap_stats(gemmar_ctx *ctx, int64_t *overlapped, int64_t *total);

/*
 * gemm_blockscale_fp8 -- C[M,N] = A[M,K] * B[N,K]^T for one K-slice, with
 *   C[m,n] = sum_kb (sa[m,kb]*sb[n/128,kb]) * sum_{k in kb} a[m,k]*b[n,k]
 * accumulated in fp32 (tcgen05 MMA per 128-K block into TMEM, the scales
 * applied while draining TMEM).  Blockscale quantisation as on the MORI page
 * ("Running the benchmark": A 1x128, B 128x128, fp32 scales).
 *   A: e4m3 [M,K]; sa: fp32 [M, K/128]; B: e4m3 [N,K]; sb: fp32 [N/128, K/128];
 *   C: [M,N] of c_dtype (GEMMAR_DTYPE_F32 or GEMMAR_DTYPE_BF16, RNE).
 * Shape rules as gemmar_supports with P = bands = 1.
 */
int gemm_blockscale_fp8(gemmar_ctx *ctx, const uint8_t *A, const float *sa, const uint8_t *B,
                        const float *sb, void *C, int c_dtype, int64_t M, int64_t N, int64_t K,
                        void *stream);

/*
 * gemm_ptpc_fp8 -- C[M,N] = (sa[m]*sb[n]) * sum_k a[m,k]*b[n,k] for one K-slice:
 * the "ptpc" quantisation the MORI benchmark runs by default ("Negative
 * results", the paragraph on pinning `--quant`), read as per-token A scales and
 * per-output-channel B scales.  The MMA accumulates the whole K in TMEM (no
 * promotion); the epilogue multiplies by the fp32 product sa[m]*sb[n].
 *   A: e4m3 [M,K]; sa: fp32 [M]; B: e4m3 [N,K]; sb: fp32 [N];
 *   C: [M,N] of c_dtype.  Shape rules as gemmar_supports with P = bands = 1.
 */
int gemm_ptpc_fp8(gemmar_ctx *ctx, const uint8_t *A, const float *sa, const uint8_t *B,
                  const float *sb, void *C, int c_dtype, int64_t M, int64_t N, int64_t K,
                  void *stream);

/*
 * gemm_mxfp8 -- C[M,N] = sum_g 2^(ea[m,g]+eb[n,g]-254) * sum_{k in g} a[m,k]*b[n,k]
 * for one K-slice, on the native block-scaled MMA (tcgen05 kind::mxf8f6f4,
 * one ue8m0 scale per 32 of K); the mxfp8 wo_b of sglang pull request #43480.
 *   A: e4m3 [M,K]; ea: ue8m0 bytes [M, K/32]; B: e4m3 [N,K]; eb: [N, K/32];
 *   C: [M,N] of c_dtype.  Uses the context's repack area (needs M <= max_M,
 *   N and K <= those of gemmar_create, else GEMMAR_ERR_WORKSPACE).
 */
int gemm_mxfp8(gemmar_ctx *ctx, const uint8_t *A, const uint8_t *ea, const uint8_t *B,
               const uint8_t *eb, void *C, int c_dtype, int64_t M, int64_t N, int64_t K,
               void *stream);

/*
 * band_reduce -- the fixed-order reduce of the row-parallel layer: for band
 * b (rows b*M/bands .. (b+1)*M/bands-1),
 *   out[m,n] = bf16_rn( ((W[b][0][r][n] + W[b][1][r][n]) + ...) + W[b][P-1][r][n] )
 * in fp32, p ascending ("MORI GEMM + All-Reduce Benchmark", "The fp8 wire":
 * the reduce accumulates in fp32; "Negative results": the reduce streams
 * through all source slices at once).  Bit-exact and deterministic.
 *   W: fp32 [bands][P][M/bands][N] (caller-owned); out: bf16 [M,N].
 */
int band_reduce(gemmar_ctx *ctx, const float *W, int P, int64_t M, int64_t N, int bands,
                uint16_t *out, void *stream);

/*
 * rowquant_e4m3 -- the fp8 wire's narrowing: per row m of x [M,N],
 *   s[m] = fp32(amax_n |x[m,n]| / 448),  q[m,n] = e4m3_rn_sat(fp32(x[m,n] / s[m]))
 * (IEEE division; a zero row gives s = 0 and +0 codes).  One fp32 scale per
 * row ("MORI GEMM + All-Reduce Benchmark", "The fp8 wire"; sglang pull
 * request #40757, "The optional fp8 gather").  Non-finite inputs: the amax
 * skips NaN (a row of NaN alone is a zero row; a NaN value codes to NaN); an
 * infinite value makes s infinite, so finite values code to +-0 and
 * infinities to NaN.
 *   x: [M,N] of x_dtype (GEMMAR_DTYPE_BF16 or GEMMAR_DTYPE_F32); q: uint8 [M,N];
 *   row_scale: fp32 [M].  N % 16 == 0.  Bit-exact against the definition.
 */
int rowquant_e4m3(gemmar_ctx *ctx, const void *x, int x_dtype, int64_t M, int64_t N,
                  uint8_t *q, float *row_scale, void *stream);

/*
 * rowdequant_e4m3 -- the fp8 wire's widening: y[m,n] = bf16_rn(fp32(decode(q[m,n]) * s[m]))
 * ("MORI GEMM + All-Reduce Benchmark", "Who moves the gather": the second
 * kernel that widens the landed fp8).
 *   q: uint8 [M,N]; row_scale: fp32 [M]; y: bf16 [M,N].  N % 16 == 0.
 */
int rowdequant_e4m3(gemmar_ctx *ctx, const uint8_t *q, const float *row_scale, int64_t M,
                    int64_t N, uint16_t *y, void *stream);

/*
 * quant_blockscale_e4m3 -- device quantiser for blockscale operands: groups
 * of group_rows x 128 (group_rows 1 for activations, 128 for weights) of an
 * [R,C] matrix x of x_dtype (GEMMAR_DTYPE_BF16 or GEMMAR_DTYPE_F32; bf16 is
 * widened to fp32 exactly); s = fp32(amax/448), q = e4m3_rn_sat(fp32(x/s));
 * a zero group gives s = 0 and +0 codes; non-finite values as in
 * rowquant_e4m3, per group.  The real call site quantises wo_b's
 * bf16 input itself (sglang pull request #43480, "Numerics, measured where
 * the path engages"), so bf16 is the input the layer sees.
 * q: uint8 [R,C]; scales: fp32 [ceil(R/group_rows), C/128].
 * C % 128 == 0.  Bit-exact against the definition.
 */
int quant_blockscale_e4m3(gemmar_ctx *ctx, const void *x, int x_dtype, int64_t R, int64_t C, int group_rows,
                          uint8_t *q, float *scales, void *stream);

/*
 * quant_mx_e4m3 -- device mxfp8 quantiser: per 1x32 group of an [R,C] matrix x
 * of x_dtype (GEMMAR_DTYPE_BF16 or GEMMAR_DTYPE_F32), byte =
 * ceil(log2(fp32(amax/448))) + 127 from the IEEE bits (exact at powers of two;
 * sglang pull request #43480, review item 7), clamped to [0,254], 0 for a
 * zero group; q = e4m3_rn_sat(fp32(x * 2^(127-byte))).  The amax skips NaN; an
 * infinite value gives byte 254, finite values then code to +-0 and
 * infinities saturate to +-448.
 * q: uint8 [R,C]; e8m0: uint8 [R, C/32].  C % 32 == 0.  Bit-exact.
 */
int quant_mx_e4m3(gemmar_ctx *ctx, const void *x, int x_dtype, int64_t R, int64_t C, uint8_t *q,
                  uint8_t *e8m0, void *stream);

/*
 * fused_gemm_reduce -- the whole wo_b path for P K-slices resident on this
 * GPU: one persistent GEMM launch over every (band, slice, tile) in band
 * order that stores each tile's fp32 partial into the context's workspace
 * W[band][p] and signals that band's counter as soon as the tile retires
 * (sglang pull request #40757, "What": the fused kernel hands each row band
 * over as soon as that band's tiles are done).  Two reducer warps of
 * every GEMM CTA take 32 x 32 output blocks of the bands already complete and
 * sum them while the GEMM still runs (the hand-over overlapped with the
 * compute, as the pages overlap their scatter with it; not on the CTA-pair
 * kernel, whose shared memory holds no room for it); band_reduce then waits
 * (bounded) for each band's counter and sums the P partials of the remaining
 * blocks in the same fixed order to bf16 out [M,N].  With GEMMAR_FP8_WIRE the
 * reduced rows then go through rowquant_e4m3 + rowdequant_e4m3 ("The fp8
 * wire"); with GEMMAR_FUSE_QUANTIZE as well (N <= 12288), the band reduce
 * parks each group of 8 summed bf16 rows in shared memory, takes their amax
 * and writes their codes and scales itself (MORI page, "Negative results":
 * folding the narrowing into the reduce), so the rows it sums are neither
 * written as bf16 nor read back before rowdequant_e4m3; the output is
 * bit-equal to the unfolded wire.
 *   A[p], B[p], sa[p], sb[p]: HOST arrays of P device pointers; per slice as in
 *   gemm_blockscale_fp8 (scale_kind GEMMAR_SCALE_BLOCK128) or gemm_mxfp8
 *   (GEMMAR_SCALE_MX32).  bands: row bands (0 = P).  out: bf16 [M,N].
 * Deterministic: equal, bit for bit, to P x gemm_*(F32) into W followed by
 * band_reduce, and to itself on a rerun.
 *
 * With GEMMAR_FUSE_SLICES the slices are instead summed inside each output
 * tile: one fp32 accumulation chain per output element over (p, K-block) in
 * the fixed order p = 0..P-1, K ascending, rounded once to bf16.  Nothing is
 * stored between the slices, so the partial write and the band reduce
 * (2 x P*M*N*4 bytes) disappear; the result is deterministic and within the
 * same tolerance of the definition, but its fp32 rounding order differs from
 * the band path's, so the two are not bit-equal.  bands is then ignored
 * (it must still satisfy the shape rules).
 *
 * With GEMMAR_FUSE_ONCHIP each output tile computes the P slice partials one
 * after another, each exactly as the band path computes it (fp32, its own
 * K-blocks from zero), and sums them in the band reducer's order, ((W_0 +
 * W_1) + W_2) + ..., in fp32 before the single bf16 rounding, without the
 * 2 x P*M*N*4 bytes of partial traffic.  Blockscale (N % 256 == 0, a GPU that
 * runs CTA pairs) runs on the CTA-pair kernel, the running sum in shared
 * memory: bit-equal to the band path, of the default one-CTA kernel as of a
 * GEMMAR_CTA_PAIR context (the two kernels give the same bits).  mx and
 * ptpc run on the whole-K kernel, each slice accumulating in a TMEM buffer of
 * its own (ptpc: then scaled) and the running sum in registers: bit-equal to
 * their band path.  Other blockscale shapes take the band path.  Takes
 * precedence over GEMMAR_FUSE_SLICES, which for ptpc means the same as
 * GEMMAR_FUSE_ONCHIP (its scales apply after a slice's whole K, so no single
 * chain over the slices exists).
 */
int fused_gemm_reduce(gemmar_ctx *ctx, int P, const uint8_t *const *A, const void *const *sa,
                      const uint8_t *const *B, const void *const *sb, int scale_kind,
                      int64_t M, int64_t N, int64_t K, int bands, uint32_t flags,
                      uint16_t *out, void *stream);

/*
 * fused_gemm_reduce_noalloc -- the blockscale fused_gemm_reduce for callers
 * that cannot allocate device memory.  The pages have no counterpart; it is
 * an addition of this library.
 *
 * Who needs it: an inference engine that takes all of the GPU's memory for
 * its own pool at start-up and allows no cudaMalloc afterwards (a late
 * allocation would fail or split its arena), or a host application that
 * loads this library as a plugin and wants every device byte to come from its
 * own allocator.  Neither can call gemmar_create, which allocates.  This call
 * takes no context and allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine): its scratch -- fp32 partials for up to
 * GEMMAR_NOALLOC_MAX_PARTIALS elements (P*M*N, each band's rows rounded up to
 * whole 128-row tiles), 1024 band counters, 1024 claim counters for the
 * GEMM's in-kernel band reduce and a status word -- lives in fixed-size arrays
 * in the library's device code, which the CUDA driver reserves on every GPU
 * that loads the library (32 MiB plus a few KiB per GPU) and keeps until the
 * process exits.
 *
 * Arguments as fused_gemm_reduce with scale_kind GEMMAR_SCALE_BLOCK128 and no
 * flags: A, sa, B, sb are HOST arrays of P device pointers, out is bf16 [M,N]
 * on the current device, bands 0 means P.  Returns GEMMAR_ERR_WORKSPACE when
 * that padded P*M*N exceeds GEMMAR_NOALLOC_MAX_PARTIALS (use fused_gemm_reduce
 * then), and
 * the other codes as fused_gemm_reduce.  The result equals fused_gemm_reduce's
 * bit for bit (same kernels, same fixed-order reduce).
 *
 * The first call on a device looks up the scratch's device addresses (and the
 * driver loads the device code there); make that first call before any
 * stream capture.  Every call on a device shares the one scratch, which keeps
 * the last call's contents; the call clears its counters and status word
 * itself.  Calls whose work overlaps on the GPU (different streams without an
 * ordering between them, or several host threads) race on the scratch and
 * give wrong results: keep them stream-ordered.
 *
 * Device-side failures: every wait inside the kernels is bounded (2 s).  If
 * one expires -- for instance a GEMM CTA whose operand loads or tensor-core
 * work stall that long on a GPU shared with other work -- the kernels stop
 * early, the call has still returned GEMMAR_OK (it returns before the work
 * runs), and `out` is left incomplete.  The failure is recorded in the
 * scratch's status word: read it with fused_gemm_reduce_noalloc_status after
 * the call's work has completed, before the next call on that device clears
 * it.
 */
#define GEMMAR_NOALLOC_MAX_PARTIALS (8 * 1024 * 1024)
int fused_gemm_reduce_noalloc(int P, const uint8_t *const *A, const float *const *sa,
                              const uint8_t *const *B, const float *const *sb,
                              int64_t M, int64_t N, int64_t K, int bands, uint16_t *out, void *stream);

/*
 * fused_gemm_reduce_noalloc_status -- the device status of the last
 * fused_gemm_reduce_noalloc call on the current device: GEMMAR_OK, or
 * GEMMAR_ERR_TIMEOUT when a bounded wait of its kernels expired (then its
 * `out` is incomplete), with *detail (if not NULL) set to the wait site.
 * Reads the 8-byte status word with a synchronous device-to-host copy (no
 * allocation): call it after that call's work has completed (for example
 * after synchronising its stream).  GEMMAR_ERR_DEVICE if the current device
 * has made no such call yet.  The pages have no counterpart.
 */
int fused_gemm_reduce_noalloc_status(int *detail);

#ifdef __cplusplus
}
#endif

#endif /* GEMMAR_H */
