/*
 * Plain, slow CPU oracle for the TN matrix multiply-accumulate D = A x B + C.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: it is built next to the CUDA library and used only by the tests,
 * by the package's smoke check and by the CPU-baseline leg of the benchmark.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes, and the passages it follows:
 *
 *   FP16:  D[m][n] = round( C[m][n] + sum_k A[m][k] * B[n][k] )
 *     "CuTe 中 A、B 如何加载到 MMA 寄存器", section 1: D = A x B + C with A
 *     indexed (M,K) and B indexed (N,K), both K-contiguous ("TN"); C and D
 *     are M x N.  Every term and the sum are taken in fp64; round() is one
 *     round-to-nearest-even to fp16, applied once at the end.
 *
 *   Dense, other element types:  D[m][n] = round( C[m][n] + sum_k a[m][k] * b[n][k] )
 *     the same TN multiply-accumulate (section 1 of the CuTe page) with A and B
 *     in BF16, FP8 E4M3 or FP8 E5M2 and C / D in fp16 or bf16; every term and
 *     the sum in fp64, one round-to-nearest-even at the end.
 *
 *   Block-scaled:  A_real[m][k] = A_low[m][k] * SFA[m][k / K_blk]
 *                  B_real[n][k] = B_low[n][k] * SFB[n][k / K_blk]
 *                  D = C + A_real x B_real  (rounded once to bf16)
 *     "数据布局及其记号", section "TMEM 中 Scale Factors 的跨 Warp 广播":
 *     sfk = k // K_blk and the two scaled operands.  NVFP4 = E2M1 data with
 *     one E4M3 scale per 16 K-elements; MXFP8 = E4M3 data with one E8M0
 *     scale per 32 K-elements (same section).  B is stored (N,K): the page
 *     writes B_low[k,n] but names SFB[n, sfk] the scale of column n, so the
 *     element is the same; storage follows section 1's (N,K) indexing.
 *
 * Readings where the pages are silent (each is listed with the design notes):
 *   - The element encodings are not defined on the pages; the decoders below
 *     follow the OCP microscaling / FP8 definitions: E2M1 (1 sign, 2 exponent
 *     bits, bias 1, 1 mantissa bit, no Inf/NaN), E4M3 "fn" (bias 7,
 *     subnormals, S.1111.111 is NaN, no Inf, max 448), E5M2 (bias 15, two
 *     mantissa bits, subnormals, exponent 31 is Inf or NaN as in IEEE 754),
 *     E8M0 (2^(e-127), 0xFF is NaN).  BF16 is the upper half of an IEEE fp32.
 *     E2M1 is decoded by its table of magnitudes; E4M3, E5M2 and E8M0 by 256-entry
 *     tables filled once from those bit-field definitions.
 *   - FP4 packing: element 2j sits in the low nibble of byte j, element 2j+1
 *     in the high nibble (the pages' "lower slot = low 16 bits" packing rule
 *     for two halves in one 32-bit operand, carried over to two nibbles).
 *   - C may be absent (NULL) and then counts as zero.
 *
 * Inputs and outputs are raw bit patterns: fp16 and bf16 as uint16_t, FP8 /
 * scale bytes as uint8_t, FP4 as uint8_t pairs.  Rows of D may be computed for
 * a subset of m (rows != NULL) so that large problems can be spot-checked.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- decoding */

/* fp16 bit pattern -> exact value. */
double oracle_f16_to_f64(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-14 / 2^10 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -v : v;
}

/* bf16 bit pattern -> exact value (bf16 is the top half of an fp32). */
double oracle_bf16_to_f64(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 7) & 0xff, m = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133); /* m * 2^-126 / 2^7 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + m / 128.0, e - 127);
    return s ? -v : v;
}

/* E2M1 magnitudes for the 3 low bits, as listed by the OCP MX definition. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_to_f64(uint8_t code) {
    double v = E2M1_MAG[code & 7];
    return (code & 8) ? -v : v;
}

/* E4M3 ("fn" variant) from its bit fields: bias 7, 3 mantissa bits.  This builds the
 * decode table; the GEMMs look codes up in it (e4m3_table). */
static double e4m3_from_fields(uint8_t code) {
    int s = code >> 7, e = (code >> 3) & 0xf, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* m/8 * 2^-6 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* E5M2 from its bit fields: bias 15, 2 mantissa bits, IEEE-style Inf / NaN (builds
 * the decode table). */
static double e5m2_from_fields(uint8_t code) {
    int sign = code >> 7, exp = (code >> 2) & 0x1f, man = code & 3;
    double v;
    if (exp == 31)
        v = man ? NAN : INFINITY;
    else if (exp == 0)
        v = ldexp((double)man / 4.0, -14);
    else
        v = ldexp(1.0 + (double)man / 4.0, exp - 15);
    return sign ? -v : v;
}

/* E8M0: a pure power of two, 2^(code - 127); 0xFF is NaN (builds the decode table). */
static double e8m0_from_fields(uint8_t code) {
    if (code == 0xff)
        return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* The 8-bit formats are decoded by table: every code's value, filled once from the
 * bit-field definitions above (E2M1 uses its listed magnitudes, E2M1_MAG). */
static double E4M3_TABLE[256], E5M2_TABLE[256], E8M0_TABLE[256];
static int tables_ready = 0;

static void build_tables(void) {
    for (int c = 0; c < 256; ++c) {
        E4M3_TABLE[c] = e4m3_from_fields((uint8_t)c);
        E5M2_TABLE[c] = e5m2_from_fields((uint8_t)c);
        E8M0_TABLE[c] = e8m0_from_fields((uint8_t)c);
    }
    tables_ready = 1;
}

static void ensure_tables(void) {
#pragma omp critical(oracle_tables)
    if (!tables_ready)
        build_tables();
}

double oracle_e4m3_to_f64(uint8_t code) {
    ensure_tables();
    return E4M3_TABLE[code];
}

double oracle_e5m2_to_f64(uint8_t code) {
    ensure_tables();
    return E5M2_TABLE[code];
}

double oracle_e8m0_to_f64(uint8_t code) {
    ensure_tables();
    return E8M0_TABLE[code];
}

/* ---------------------------------------------------------------- rounding */

/*
 * Round a finite or non-finite double once, to nearest with ties to even, onto
 * a binary format with `mbits` stored mantissa bits, exponent bias `bias` and
 * largest biased exponent `emax_biased` for finite numbers (Inf/NaN above).
 * Returns the bit pattern of the 1+ebits+mbits-bit result.
 */
static uint32_t round_binary(double x, int ebits, int mbits, int bias) {
    uint32_t sign = signbit(x) ? 1u : 0u;
    uint32_t exp_all = (1u << ebits) - 1u;
    uint32_t sign_bit = sign << (ebits + mbits);
    if (isnan(x))
        return (exp_all << mbits) | (1u << (mbits - 1)); /* quiet NaN */
    double a = fabs(x);
    if (isinf(a))
        return sign_bit | (exp_all << mbits);
    if (a == 0.0)
        return sign_bit;
    int e2;
    frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1): unbiased exponent e2-1 */
    int unb = e2 - 1;
    int min_unb = 1 - bias; /* smallest normal exponent */
    if (unb < min_unb)
        unb = min_unb;      /* subnormal range shares the smallest quantum */
    double quantum = ldexp(1.0, unb - mbits);
    double n = nearbyint(a / quantum); /* exact division by a power of two; RNE */
    double v = n * quantum;
    if (v == 0.0) /* rounded down to a signed zero */
        return sign_bit;
    /* encode v */
    int ve2;
    frexp(v, &ve2);
    int vunb = ve2 - 1;
    if (vunb < min_unb) { /* subnormal result: mantissa = v / 2^(min_unb - mbits) */
        uint32_t mant = (uint32_t)(v / ldexp(1.0, min_unb - mbits));
        return sign_bit | mant;
    }
    int biased = vunb + bias;
    if (biased >= (int)exp_all) /* overflow to infinity */
        return sign_bit | (exp_all << mbits);
    double frac = v / ldexp(1.0, vunb) - 1.0; /* in [0,1) */
    uint32_t mant = (uint32_t)(frac * (double)(1u << mbits));
    return sign_bit | ((uint32_t)biased << mbits) | mant;
}

uint16_t oracle_f64_to_f16(double x) { return (uint16_t)round_binary(x, 5, 10, 15); }
uint16_t oracle_f64_to_bf16(double x) { return (uint16_t)round_binary(x, 8, 7, 127); }

/* ---------------------------------------------------------------- GEMM */

/*
 * FP16 TN GEMM.  A: fp16[M][K], B: fp16[N][K], C: fp16[M][N] or NULL.
 * rows: the m indices to compute (NULL = all M rows, in order); nrows their
 * count.  D16 (may be NULL): fp16[nrows][N].  D64 (may be NULL): the exact
 * fp64 sums before rounding, double[nrows][N].
 */
void oracle_gemm_f16(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                     const uint16_t *C, const int64_t *rows, int64_t nrows, uint16_t *D16,
                     double *D64) {
    if (rows == NULL)
        nrows = M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t n = 0; n < N; ++n) {
            double acc = C ? oracle_f16_to_f64(C[m * N + n]) : 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_f16_to_f64(A[m * K + k]) * oracle_f16_to_f64(B[n * K + k]);
            if (D64)
                D64[i * N + n] = acc;
            if (D16)
                D16[i * N + n] = oracle_f64_to_f16(acc);
        }
    }
}

/* fmt: 0 = NVFP4 (E2M1 data, E4M3 scale per 16), 1 = MXFP8 (E4M3 data, E8M0 per 32) */
static double low_element(int fmt, const uint8_t *X, int64_t K, int64_t r, int64_t k) {
    if (fmt == 0) {
        uint8_t byte = X[r * (K / 2) + k / 2];
        uint8_t code = (k % 2 == 0) ? (byte & 0xf) : (byte >> 4);
        return oracle_e2m1_to_f64(code);
    }
    return E4M3_TABLE[X[r * K + k]];
}

static double scale_factor(int fmt, const uint8_t *SF, int64_t K, int64_t r, int64_t sfk) {
    int64_t kblk = (fmt == 0) ? 16 : 32;
    uint8_t code = SF[r * (K / kblk) + sfk];
    return (fmt == 0) ? E4M3_TABLE[code] : E8M0_TABLE[code];
}

/*
 * Block-scaled TN GEMM.  A: NVFP4 u8[M][K/2] | MXFP8 u8[M][K];
 * SFA: u8[M][K/K_blk]; B, SFB the same with N rows; C: bf16[M][N] or NULL.
 * D16: bf16[nrows][N] (may be NULL); D64: exact fp64 sums (may be NULL).
 * Returns 0, or -1 when K is not a multiple of K_blk or fmt is unknown.
 */
int oracle_gemm_block_scaled(int fmt, int64_t M, int64_t N, int64_t K, const uint8_t *A,
                             const uint8_t *SFA, const uint8_t *B, const uint8_t *SFB,
                             const uint16_t *C, const int64_t *rows, int64_t nrows,
                             uint16_t *D16, double *D64) {
    if (fmt != 0 && fmt != 1)
        return -1;
    int64_t kblk = (fmt == 0) ? 16 : 32;
    if (K % kblk != 0)
        return -1;
    if (rows == NULL)
        nrows = M;
    ensure_tables();
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t n = 0; n < N; ++n) {
            double acc = C ? oracle_bf16_to_f64(C[m * N + n]) : 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t sfk = k / kblk;
                double a = low_element(fmt, A, K, m, k) * scale_factor(fmt, SFA, K, m, sfk);
                double b = low_element(fmt, B, K, n, k) * scale_factor(fmt, SFB, K, n, sfk);
                acc += a * b;
            }
            if (D64)
                D64[i * N + n] = acc;
            if (D16)
                D16[i * N + n] = oracle_f64_to_bf16(acc);
        }
    }
    return 0;
}

/* Element formats of oracle_gemm_dense. */
enum { FMT_FP16 = 0, FMT_BF16 = 1, FMT_E4M3 = 2, FMT_E5M2 = 3 };

static double dense_element(int fmt, const void *X, int64_t idx) {
    switch (fmt) {
        case FMT_FP16: return oracle_f16_to_f64(((const uint16_t *)X)[idx]);
        case FMT_BF16: return oracle_bf16_to_f64(((const uint16_t *)X)[idx]);
        case FMT_E4M3: return E4M3_TABLE[((const uint8_t *)X)[idx]];
        default: return E5M2_TABLE[((const uint8_t *)X)[idx]];
    }
}

/*
 * Dense TN GEMM for any pair of element formats.  A: a_fmt[M][K], B: b_fmt[N][K]
 * (fp16 / bf16 as uint16_t bit patterns, E4M3 / E5M2 as bytes); C: out_fmt[M][N]
 * or NULL; out_fmt 0 = fp16, 1 = bf16.  rows / nrows / D16 / D64 as for
 * oracle_gemm_f16.  Returns 0, or -1 for an unknown format.
 */
int oracle_gemm_dense(int a_fmt, int b_fmt, int out_fmt, int64_t M, int64_t N, int64_t K, const void *A,
                      const void *B, const uint16_t *C, const int64_t *rows, int64_t nrows, uint16_t *D16,
                      double *D64) {
    if (a_fmt < FMT_FP16 || a_fmt > FMT_E5M2 || b_fmt < FMT_FP16 || b_fmt > FMT_E5M2)
        return -1;
    if (out_fmt != FMT_FP16 && out_fmt != FMT_BF16)
        return -1;
    if (rows == NULL)
        nrows = M;
    ensure_tables();
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t n = 0; n < N; ++n) {
            double acc = C ? dense_element(out_fmt, C, m * N + n) : 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += dense_element(a_fmt, A, m * K + k) * dense_element(b_fmt, B, n * K + k);
            if (D64)
                D64[i * N + n] = acc;
            if (D16)
                D16[i * N + n] = out_fmt == FMT_FP16 ? oracle_f64_to_f16(acc) : oracle_f64_to_bf16(acc);
        }
    }
    return 0;
}

/* Number of OpenMP threads the GEMM loops use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
