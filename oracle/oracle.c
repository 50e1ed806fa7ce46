/*
 * oracle.c -- plain, slow, obviously-correct CPU definition of what the
 * block-scaled fp8 wo_b path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this code:
 * only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark load it.  It shares no code, header, table or constant generator
 * with the CUDA library; the two meet only through the seeded input
 * generator (package `synthetic`), which holds none of the method's
 * arithmetic.
 *
 * Sources (web pages; cited by title and section):
 *   [PR40757]  sglang pull request #40757, "fuse wo_b's GEMM with its
 *              all-reduce" (DeepSeek-V4-Pro, block-scale fp8).
 *   [PR43480]  sglang pull request #43480 (DeepSeek-V4.1-Flash, mxfp8), its
 *              review thread, item 7 "Duplicated ue8m0 scale rule".
 *   [MORI]     "MORI GEMM + All-Reduce Benchmark", sections "Running the
 *              benchmark", "Where the time goes", "The fp8 wire",
 *              "What fp8 costs, numerically".
 *
 * Readings taken where the pages are silent:
 *   R1  "e4m3" is OCP E4M3FN: bias 7, no infinities, S.1111.111 is NaN,
 *       largest finite 448 -- the only e4m3 variant whose maximum is the 448
 *       of the pages' "amax/448" scale rule.
 *   R2  Encoding rounds to nearest, ties to the even code, and saturates any
 *       |v| >= 448 to +-448; NaN encodes to 0x7F.
 *   R3  A group whose amax is 0 gets scale 0 and all-zero (+0) codes; it
 *       decodes to exact zeros.  For ue8m0 the byte is 0.
 *   R4  Scales are fp32: s = fp32(amax / 448.0f) with IEEE division, and the
 *       codes are e4m3(fp32(x / s)), an IEEE division (not a reciprocal
 *       multiply).
 *   R5  The reduced result is rounded once, to bf16 with round-to-nearest-even.
 *
 * Floating point: the GEMM and the P-way sum are carried out in fp64.  Each
 * 128-wide (or 32-wide) group sum of e4m3 products is exact in fp64: a
 * product has at most 8 significant bits and lies in [2^-18, 2^18), and 128
 * of them need fewer than 53 bits.  Build with -ffp-contract=off and no fast
 * math, so every fp32 operation below is one IEEE-rounded operation.
 *
 * Parity status: every function here is pinned by the CPU test suite against
 * values the pages print, closed forms, library routines or exact rational
 * brute force; none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* e4m3 (OCP E4M3FN) code table -- reading R1.                               */
/* ------------------------------------------------------------------------ */

static double e4m3_value[256];      /* decoded value of every code          */

/* Decode one code from its bit fields: sign | 4-bit exponent | 3-bit mantissa. */
static double e4m3_from_fields(int code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 15;
    int mant = code & 7;
    double mag;
    if (expo == 15 && mant == 7)
        return NAN;                           /* S.1111.111 */
    if (expo == 0)
        mag = ldexp((double)mant, -9);        /* subnormal: mant/8 * 2^-6 */
    else
        mag = ldexp(8.0 + mant, expo - 10);   /* (1 + mant/8) * 2^(expo-7) */
    return sign ? -mag : mag;
}

__attribute__((constructor)) static void orc_build_tables(void)
{
    for (int c = 0; c < 256; ++c)
        e4m3_value[c] = e4m3_from_fields(c);
}

double orc_e4m3_decode(uint8_t code) { return e4m3_value[code]; }

void orc_e4m3_decode_table(double *out256)
{
    memcpy(out256, e4m3_value, sizeof(e4m3_value));
}

/*
 * Encode an fp32 value to e4m3 -- reading R2.  Table driven: the non-negative
 * finite codes 0x00..0x7E decode to strictly increasing values, so the nearest
 * code is found by bisection over the table; an exact midpoint goes to the
 * even code (the code whose mantissa LSB is 0).
 */
uint8_t orc_e4m3_encode(float v)
{
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return sign | 0x7E;                   /* saturate */
    int lo = 0, hi = 126;                     /* largest code with value <= a */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (e4m3_value[mid] <= a) lo = mid; else hi = mid - 1;
    }
    double below = e4m3_value[lo], above = e4m3_value[lo + 1];
    double d_lo = a - below, d_hi = above - a;    /* exact in fp64 */
    int code;
    if (d_lo < d_hi)       code = lo;
    else if (d_hi < d_lo)  code = lo + 1;
    else                   code = (lo % 2 == 0) ? lo : lo + 1;
    return sign | (uint8_t)code;
}

void orc_e4m3_encode_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------------ */
/* bf16 rounding (reading R5).                                               */
/* ------------------------------------------------------------------------ */

/*
 * Round a real number (given in fp64) once to bf16, nearest-even, and return
 * the bf16 bit pattern.  bf16 keeps 8 significant bits with fp32's exponent
 * range; below 2^-126 its spacing is 2^-133.  The value is scaled by a power
 * of two (exact), rounded to an integer by nearbyint in the default
 * round-to-nearest-even mode, and scaled back.
 */
uint16_t orc_bf16_rn(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);                      /* a in [2^(e2-1), 2^e2) */
    int q = e2 - 8;                     /* spacing of 8 significant bits */
    if (q < -133) q = -133;             /* subnormal spacing */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;           /* overflow to infinity */
    float f = (float)r;                 /* exact: r has <= 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return sign | (uint16_t)(bits >> 16);
}

void orc_bf16_rn_array(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_rn(x[i]);
}

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Quantisers -- [MORI] "Running the benchmark" (A 1x128, B 128x128, fp32   */
/* scales); [PR43480] item 7 for the ue8m0 exponent rule.                   */
/* ------------------------------------------------------------------------ */

/*
 * Block quantiser over groups of gr rows x gc columns of a row-major [R,C]
 * fp32 matrix.  Per group: amax = max |x|, s = fp32(amax / 448), code =
 * e4m3(fp32(x / s)); amax == 0 gives s = 0 and +0 codes (R3, R4).
 * scales is row-major [ceil(R/gr), ceil(C/gc)].
 */
void orc_quant_block(const float *x, int64_t R, int64_t C, int64_t gr, int64_t gc,
                     uint8_t *codes, float *scales)
{
    int64_t nbr = (R + gr - 1) / gr, nbc = (C + gc - 1) / gc;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bi = 0; bi < nbr; ++bi) {
        for (int64_t bj = 0; bj < nbc; ++bj) {
            int64_t r0 = bi * gr, r1 = r0 + gr < R ? r0 + gr : R;
            int64_t c0 = bj * gc, c1 = c0 + gc < C ? c0 + gc : C;
            float amax = 0.0f;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = c0; c < c1; ++c) {
                    float v = fabsf(x[r * C + c]);
                    if (v > amax) amax = v;
                }
            float s = amax / 448.0f;
            scales[bi * nbc + bj] = s;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = c0; c < c1; ++c)
                    codes[r * C + c] = (s == 0.0f) ? 0x00 : orc_e4m3_encode(x[r * C + c] / s);
        }
    }
}

/*
 * ue8m0 exponent for a group whose ratio is r = fp32(amax / 448):
 * e = ceil(log2 r), taken from r's binary representation -- floor(log2 r)
 * plus one unless r is an exact power of two -- so it is exact at powers of
 * two, where a floating log2 can land one too high ([PR43480] item 7).
 * frexp gives the representation exactly, subnormals included.  Returns the
 * stored byte e + 127, clamped to [0, 254]; r == 0 gives byte 0 (R3).  An
 * infinite r (a group holding an infinity) lies above every power of two and
 * takes the upper clamp; frexp does not define an exponent for it.
 */
uint8_t orc_ue8m0_byte(float r)
{
    if (!(r > 0.0f))
        return 0;
    if (isinf(r))
        return 254;
    int e2;
    double fr = frexp((double)r, &e2);   /* r = fr * 2^e2, fr in [0.5, 1) */
    int e = (fr == 0.5) ? e2 - 1 : e2;   /* exact power of two: log2 r = e2-1 */
    int b = e + 127;
    if (b < 0) b = 0;
    if (b > 254) b = 254;
    return (uint8_t)b;
}

/*
 * mxfp8 quantiser: 1x32 groups along each row of a row-major [R,C] matrix.
 * byte = ue8m0(fp32(amax/448)); code = e4m3(fp32(x * 2^-(byte-127))).
 * An amax of 0 gives byte 0 and +0 codes (R3).  sbytes is [R, ceil(C/32)].
 */
void orc_quant_mx(const float *x, int64_t R, int64_t C, uint8_t *codes, uint8_t *sbytes)
{
    int64_t ng = (C + 31) / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t g = 0; g < ng; ++g) {
            int64_t c0 = g * 32, c1 = c0 + 32 < C ? c0 + 32 : C;
            float amax = 0.0f;
            for (int64_t c = c0; c < c1; ++c) {
                float v = fabsf(x[r * C + c]);
                if (v > amax) amax = v;
            }
            uint8_t b = orc_ue8m0_byte(amax / 448.0f);
            sbytes[r * ng + g] = b;
            float inv = (float)ldexp(1.0, 127 - (int)b);   /* 2^-e, exact in fp32 */
            for (int64_t c = c0; c < c1; ++c)
                codes[r * C + c] = (amax == 0.0f) ? 0x00 : orc_e4m3_encode(x[r * C + c] * inv);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Scaled GEMM per K-slice and the P-way reduction, in fp64.                */
/* ------------------------------------------------------------------------ */

/*
 * Block-scaled GEMM of one K-slice ([MORI] "Running the benchmark":
 * A 1x128 and B 128x128 fp32 scales), for the listed output rows:
 *   G[m,n] = sum_kb (sa[m,kb] * sb[n/128,kb]) * sum_{k in kb} a[m,k] b[n,k]
 * with a, b the decoded e4m3 values.  A is [M,K], B is [N,K] (both K
 * contiguous), sa is [M,K/128], sb is [ceil(N/128),K/128].  rows==NULL means
 * every row.  The result is ADDED to acc[i*N + n] (fp64), so that calling it
 * for p = 0..P-1 forms the P-way sum.
 */
void orc_gemm_blockscale_acc(const uint8_t *A, const float *sa, const uint8_t *B, const float *sb,
                             int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                             double *acc)
{
    int64_t KB = K / 128;
    int64_t NB = (N + 127) / 128;
    if (rows == NULL) nrows = M;
    double *bdec = (double *)malloc(sizeof(double) * (size_t)(N * K));
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N * K; ++i)
        bdec[i] = e4m3_value[B[i]];
#pragma omp parallel
    {
        double *arow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t m = rows ? rows[i] : i;
            for (int64_t k = 0; k < K; ++k)
                arow[k] = e4m3_value[A[m * K + k]];
            for (int64_t n = 0; n < N; ++n) {
                const double *brow = bdec + n * K;
                double g = 0.0;
                for (int64_t kb = 0; kb < KB; ++kb) {
                    double dot = 0.0;
                    for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
                        dot += arow[k] * brow[k];
                    double scale = (double)sa[m * KB + kb] * (double)sb[(n / 128) * KB + kb];
                    g += scale * dot;
                }
                acc[i * N + n] += g;
            }
        }
        free(arow);
    }
    (void)NB;
    free(bdec);
}

/*
 * mxfp8 GEMM of one K-slice ([PR43480] "What": 32-wide ue8m0 scales):
 *   G[m,n] = sum_g 2^(ea[m,g] + eb[n,g] - 254) * sum_{k in g} a[m,k] b[n,k]
 * ea is [M,K/32], eb is [N,K/32] (stored bytes).  Added into acc as above.
 */
void orc_gemm_mx_acc(const uint8_t *A, const uint8_t *ea, const uint8_t *B, const uint8_t *eb,
                     int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                     double *acc)
{
    int64_t G = K / 32;
    if (rows == NULL) nrows = M;
    double *bdec = (double *)malloc(sizeof(double) * (size_t)(N * K));
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N * K; ++i)
        bdec[i] = e4m3_value[B[i]];
#pragma omp parallel
    {
        double *arow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t m = rows ? rows[i] : i;
            for (int64_t k = 0; k < K; ++k)
                arow[k] = e4m3_value[A[m * K + k]];
            for (int64_t n = 0; n < N; ++n) {
                const double *brow = bdec + n * K;
                double g = 0.0;
                for (int64_t gi = 0; gi < G; ++gi) {
                    double dot = 0.0;
                    for (int64_t k = gi * 32; k < gi * 32 + 32; ++k)
                        dot += arow[k] * brow[k];
                    int ex = (int)ea[m * G + gi] + (int)eb[n * G + gi] - 254;
                    g += ldexp(dot, ex);
                }
                acc[i * N + n] += g;
            }
        }
        free(arow);
    }
    free(bdec);
}

/*
 * ptpc GEMM of one K-slice: one fp32 scale per row of A (per token) and one
 * per row of B (per output channel), the quantisation mode the MORI benchmark
 * runs by default ("A CK-shaped 4-wave GEMM" paragraph of "Negative results":
 * `--quant ptpc`), read as per-token / per-channel:
 *   G[m,n] = (sa[m] * sb[n]) * sum_k a[m,k] b[n,k]
 * sa is [M], sb is [N].  Added into acc as above.
 */
void orc_gemm_ptpc_acc(const uint8_t *A, const float *sa, const uint8_t *B, const float *sb,
                       int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                       double *acc)
{
    if (rows == NULL) nrows = M;
    double *bdec = (double *)malloc(sizeof(double) * (size_t)(N * K));
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N * K; ++i)
        bdec[i] = e4m3_value[B[i]];
#pragma omp parallel
    {
        double *arow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t m = rows ? rows[i] : i;
            for (int64_t k = 0; k < K; ++k)
                arow[k] = e4m3_value[A[m * K + k]];
            for (int64_t n = 0; n < N; ++n) {
                const double *brow = bdec + n * K;
                double dot = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    dot += arow[k] * brow[k];
                acc[i * N + n] += ((double)sa[m] * (double)sb[n]) * dot;
            }
        }
        free(arow);
    }
    free(bdec);
}

/*
 * The whole path for the listed rows: R = sum_{p=0}^{P-1} G_p in fp64, then
 * out = bf16_rn(R) ([PR40757] "What": a block-scale fp8 GEMM followed by the
 * all-reduce of the [M, hidden] result; [MORI] "The fp8 wire": the reduce
 * accumulates in fp32 and the output is bf16 -- here the sum is carried in
 * fp64 and rounded once, the plain definition the fp32 sum approximates).
 * scale_kind 0 = block 128 (sa/sb fp32), 1 = mx 32 (sa/sb ue8m0 bytes),
 * 2 = ptpc (sa [M], sb [N] fp32).
 * ref (optional, [nrows,N] fp64) receives R; out receives bf16 bits.
 */
void orc_gemm_reduce(int P, const uint8_t *const *A, const void *const *sa,
                     const uint8_t *const *B, const void *const *sb, int scale_kind,
                     int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                     double *ref, uint16_t *out)
{
    if (rows == NULL) nrows = M;
    double *acc = ref ? ref : (double *)malloc(sizeof(double) * (size_t)(nrows * N));
    memset(acc, 0, sizeof(double) * (size_t)(nrows * N));
    for (int p = 0; p < P; ++p) {
        if (scale_kind == 0)
            orc_gemm_blockscale_acc(A[p], (const float *)sa[p], B[p], (const float *)sb[p],
                                    M, N, K, rows, nrows, acc);
        else if (scale_kind == 1)
            orc_gemm_mx_acc(A[p], (const uint8_t *)sa[p], B[p], (const uint8_t *)sb[p],
                            M, N, K, rows, nrows, acc);
        else
            orc_gemm_ptpc_acc(A[p], (const float *)sa[p], B[p], (const float *)sb[p],
                              M, N, K, rows, nrows, acc);
    }
    if (out)
        for (int64_t i = 0; i < nrows * N; ++i)
            out[i] = orc_bf16_rn(acc[i]);
    if (!ref) free(acc);
}

/*
 * The row-parallel reduction with the pages' own arithmetic, used to check
 * the reducer bit for bit: partials are fp32, summed in fp32 in the fixed
 * order p = 0, 1, ..., P-1 starting from slice 0, then rounded to bf16
 * ([MORI] "The fp8 wire": "the reduce still accumulates in fp32").
 * W is [P][rows][N] fp32 for one band; out is [rows][N] bf16 bits.
 */
void orc_reduce_f32_ordered(int P, const float *W, int64_t rows, int64_t N, uint16_t *out)
{
    int64_t n = rows * N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float s = W[i];
        for (int p = 1; p < P; ++p)
            s = s + W[(int64_t)p * n + i];
        out[i] = orc_bf16_rn((double)s);
    }
}

/* ------------------------------------------------------------------------ */
/* fp8 wire: per-row e4m3 codec ([MORI] "The fp8 wire": one fp32 scale per  */
/* row; [PR40757] "The optional fp8 gather").                               */
/* ------------------------------------------------------------------------ */

/*
 * Row quantiser: for each row of a row-major [M,N] fp32 matrix,
 * s[m] = fp32(amax_row / 448), q = e4m3(fp32(x / s)); a zero row gives s = 0
 * and +0 codes.  (Identical to orc_quant_block with one group per row.)
 */
void orc_rowquant(const float *x, int64_t M, int64_t N, uint8_t *q, float *s)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const float *row = x + m * N;
        float amax = 0.0f;
        for (int64_t n = 0; n < N; ++n) {
            float v = fabsf(row[n]);
            if (v > amax) amax = v;
        }
        float sc = amax / 448.0f;
        s[m] = sc;
        for (int64_t n = 0; n < N; ++n)
            q[m * N + n] = (sc == 0.0f) ? 0x00 : orc_e4m3_encode(row[n] / sc);
    }
}

/* Row dequantiser: y = bf16_rn(fp32(decode(q) * s[m])). */
void orc_rowdequant(const uint8_t *q, const float *s, int64_t M, int64_t N, uint16_t *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            float v = (float)e4m3_value[q[m * N + n]] * s[m];
            y[m * N + n] = orc_bf16_rn((double)v);
        }
}

/* Convenience for callers that hold bf16 bits: widen to fp32 (exact). */
void orc_bf16_to_f32(const uint16_t *b, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)bf16_bits_to_double(b[i]);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
