/*
 * gemm_oracle.c -- CPU oracle for the dense GEMM.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this file.  The product path (the CUDA library) shares no code,
 * header, table or build flag with it and never calls it.
 *
 * What it computes (plain definition, no blocking, no reordering):
 *
 *   D[i,j] = round_RNE( sum_{k<K} A[i,k] * B'[j,k] )
 *
 *   - "TIRx GEMM on Blackwell" (jq-wei.github.io), section "The short version":
 *     the operation is D = A @ B.T with 16-bit inputs and output and the
 *     partial products accumulated in FP32 on the GPU.  Here B' = B and B is
 *     stored N x K ("A.Bt" layout).
 *   - "Choosing schedules and instructions for a backend" (TileFoundry tutorial),
 *     section 1, the `gemm(a: (M,K), b: (K,N)) -> (M,N)` program: the plain
 *     product with B stored K x N ("A.B" layout), B'[j,k] = B[k,j].
 *   - "TIRx GEMM on Blackwell", Take away 1: tiling, pipelining and scheduling
 *     do not change the arithmetic, only the order of the additions.  So the
 *     oracle is the definition itself: the sum runs over k in increasing order
 *     in IEEE binary64 from the exact 16-bit input values (every product of two
 *     binary16 or two bfloat16 values is exact in binary64), and the result is
 *     rounded ONCE to the output type with round-to-nearest-even.
 *
 * The 16-bit decode and the binary64 -> 16-bit rounding are written here from
 * the IEEE 754-2008 binary16 definition (1 sign, 5 exponent bits with bias 15,
 * 10 fraction bits, subnormals, inf/NaN at exponent 31) and from the bfloat16
 * definition (the upper half of an IEEE binary32: 1 sign, 8 exponent bits with
 * bias 127, 7 fraction bits).
 *
 * The FP8 variant (oracle_gemm_fp8, below) follows the same rule from exact
 * E4M3 / E5M2 inputs, with one FP32 scale applied to the sum; the block-scaled
 * variant (oracle_gemm_mx) adds one power-of-two scale per 32 K elements of
 * each row of A and of B.
 *
 * Parity pins (tests/test_oracle.py): hand-computed products, identity and
 * permutation operands, the transpose invariant (A.Bt)t == B.At, closed forms
 * for all-ones operands, exact small-integer products, agreement of the two
 * layouts, the rounding rule against numpy's independent binary16 conversion,
 * and torch.mm in float64 on small random cases.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1
#define ORACLE_B_NK 0 /* B stored N x K row-major: D = A . B^T */
#define ORACLE_B_KN 1 /* B stored K x N row-major: D = A . B   */

/* ---- decode: 16-bit pattern -> exact binary64 value ---------------------- */

static double f16_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal (or zero): f * 2^-24 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

static double bf16_bits_to_double(uint16_t h) {
    /* bfloat16 is the top half of a binary32 pattern. */
    uint32_t w = ((uint32_t)h) << 16;
    float x;
    memcpy(&x, &w, sizeof x);
    return (double)x;
}

double oracle_to_double(uint16_t bits, int dtype) {
    return dtype == ORACLE_BF16 ? bf16_bits_to_double(bits) : f16_bits_to_double(bits);
}

/* The same decode, tabulated once for all 65536 patterns of each type, so the
 * GEMM loop below does not pay a libm call per operand. */
static double g_decode[2][65536];
static int g_decode_ready = 0;

static void build_decode_tables(void) {
    if (g_decode_ready) return;
    for (uint32_t b = 0; b < 65536u; ++b) {
        g_decode[ORACLE_F16][b] = oracle_to_double((uint16_t)b, ORACLE_F16);
        g_decode[ORACLE_BF16][b] = oracle_to_double((uint16_t)b, ORACLE_BF16);
    }
    g_decode_ready = 1;
}

/* ---- encode: binary64 -> 16-bit pattern, round to nearest, ties to even ---
 *
 * Generic for a format with `ebits` exponent bits and `fbits` fraction bits.
 * Scaling by a power of two is exact in binary64 over the whole range used, so
 * one nearbyint() (default rounding mode = to nearest, ties to even) performs
 * the single rounding step.
 */
static uint16_t round_to_format(double x, int ebits, int fbits) {
    const int bias = (1 << (ebits - 1)) - 1;
    const int emax_field = (1 << ebits) - 1;
    const uint16_t sign = signbit(x) ? (uint16_t)(1u << (ebits + fbits)) : 0;
    const uint16_t inf = (uint16_t)(emax_field << fbits);
    if (isnan(x)) return (uint16_t)(inf | (1u << (fbits - 1)));
    double a = fabs(x);
    if (isinf(a)) return sign | inf;
    const int emin = 1 - bias; /* exponent of the smallest normal */
    if (a < ldexp(1.0, emin)) {
        /* subnormal range: quantum 2^(emin - fbits).  q == 2^fbits encodes
         * the smallest normal, which the bit pattern below already does. */
        double q = nearbyint(ldexp(a, fbits - emin));
        return sign | (uint16_t)q;
    }
    int e2;
    frexp(a, &e2); /* a = m * 2^e2, m in [0.5, 1): unbiased exponent is e2-1 */
    int e = e2 - 1;
    double q = nearbyint(ldexp(a, fbits - e)); /* in [2^fbits, 2^(fbits+1)] */
    if (q == ldexp(1.0, fbits + 1)) { /* rounding carried into the exponent */
        q = ldexp(1.0, fbits);
        e += 1;
    }
    int field = e + bias;
    if (field >= emax_field) return sign | inf; /* overflow rounds to infinity */
    return sign | (uint16_t)(field << fbits) | (uint16_t)((uint32_t)q - (1u << fbits));
}

uint16_t oracle_from_double(double x, int dtype) {
    return dtype == ORACLE_BF16 ? round_to_format(x, 8, 7) : round_to_format(x, 5, 10);
}

/* ---- the GEMM ------------------------------------------------------------
 *
 * Computes rows [i0,i1) x columns [j0,j1) of D.  A is M x K row-major with row
 * stride lda (elements); B is N x K (b_layout 0) or K x N (b_layout 1)
 * row-major with row stride ldb.  Results go to out[(i-i0)*ldo + (j-j0)].
 * `out_f64` (may be NULL) receives the unrounded binary64 sums; `out16`
 * (may be NULL) the rounded 16-bit patterns.
 */
void oracle_gemm(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                 int64_t lda, int64_t ldb, int b_layout, int dtype,
                 int64_t i0, int64_t i1, int64_t j0, int64_t j1,
                 uint16_t* out16, double* out_f64, int64_t ldo) {
    (void)M;
    (void)N;
    build_decode_tables(); /* before the parallel region: written by one thread */
    const double* dec = g_decode[dtype == ORACLE_BF16 ? ORACLE_BF16 : ORACLE_F16];
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = i0; i < i1; ++i) {
        for (int64_t j = j0; j < j1; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = dec[A[i * lda + k]];
                double b = (b_layout == ORACLE_B_NK) ? dec[B[j * ldb + k]] : dec[B[k * ldb + j]];
                acc += a * b;
            }
            int64_t o = (i - i0) * ldo + (j - j0);
            if (out_f64) out_f64[o] = acc;
            if (out16) out16[o] = oracle_from_double(acc, dtype);
        }
    }
}

/* ---- FP8 inputs ------------------------------------------------------------
 *
 * The 8-bit formats, written from the OCP 8-bit floating point specification
 * ("OFP8"), the encodings the tcgen05 kind::f8f6f4 MMA consumes:
 *   E4M3: 1 sign, 4 exponent bits (bias 7), 3 fraction bits; subnormals at
 *         exponent field 0 (f/8 * 2^-6); NO infinities; S.1111.111 is NaN, so
 *         exponent field 15 with fraction 0..6 is an ordinary normal number
 *         (largest finite 1.75 * 2^8 = 448).
 *   E5M2: 1 sign, 5 exponent bits (bias 15), 2 fraction bits, IEEE 754 style:
 *         subnormals f/4 * 2^-14, exponent field 31 is inf (f = 0) or NaN.
 */
#define ORACLE_E4M3 0
#define ORACLE_E5M2 1

double oracle_fp8_to_double(uint8_t b, int fmt) {
    const int sign = (b >> 7) & 1;
    double v;
    if (fmt == ORACLE_E4M3) {
        const int e = (b >> 3) & 0xf, f = b & 7;
        if (e == 15 && f == 7) return NAN;
        v = (e == 0) ? ldexp((double)f, -9) : ldexp((double)(8 + f), e - 10);
    } else {
        const int e = (b >> 2) & 0x1f, f = b & 3;
        if (e == 31) return f ? NAN : (sign ? -INFINITY : INFINITY);
        v = (e == 0) ? ldexp((double)f, -16) : ldexp((double)(4 + f), e - 17);
    }
    return sign ? -v : v;
}

/* D[i,j] = round_RNE( alpha * sum_{k<K} A[i,k] * B[j,k] ), A (M x K) and B
 * (N x K) both K-major ("Choosing schedules and instructions for a backend",
 * the instruction table: fp8e4m3 operands are K-major only).  The products of
 * two 8-bit values are exact in binary64 and the sum runs over k in order;
 * alpha (one scale for the whole product: "TIRx: A Unified Tile Primitive ML
 * Compiler", kernel performance, "scale factors that adjust their numerical
 * range", with one group spanning each tensor) multiplies the sum once, and
 * the result is rounded once to the 16-bit output type. */
void oracle_gemm_fp8(const uint8_t* A, const uint8_t* B, int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int in_fmt, int out_dtype, double alpha,
                     int64_t i0, int64_t i1, int64_t j0, int64_t j1,
                     uint16_t* out16, double* out_f64, int64_t ldo) {
    (void)M;
    (void)N;
    double dec[256];
    for (int c = 0; c < 256; ++c) dec[c] = oracle_fp8_to_double((uint8_t)c, in_fmt);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = i0; i < i1; ++i) {
        for (int64_t j = j0; j < j1; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += dec[A[i * lda + k]] * dec[B[j * ldb + k]];
            const double d = alpha * acc;
            int64_t o = (i - i0) * ldo + (j - j0);
            if (out_f64) out_f64[o] = d;
            if (out16) out16[o] = oracle_from_double(d, out_dtype);
        }
    }
}

/* ---- Block-scaled FP8 inputs (MX) --------------------------------------------
 *
 * "TIRx: A Unified Tile Primitive ML Compiler", kernel performance, names FP8
 * block-scaled matrix multiplication: groups of input values share scale
 * factors that adjust their numerical range.  The page gives neither the group
 * size nor the scale encoding.  Reading taken here: the OCP Microscaling (MX)
 * formats, the block-scaled form that the tcgen05 kind::mxf8f6f4 MMA consumes.
 * Each run of 32 consecutive K elements of a row of A, and of a row of B (both
 * K-major), shares one 8-bit scale X in the UE8M0 encoding: the value is
 * 2^(X - 127), and X = 255 is NaN.  An element's value is its FP8 value times
 * its group's scale, so
 *
 *   D[i,j] = round_RNE( alpha * sum_{k<K} (A[i,k] * 2^(SA[i][k/32] - 127))
 *                                      * (B[j,k] * 2^(SB[j][k/32] - 127)) )
 *
 * Scaling by a power of two is exact in binary64 over the whole UE8M0 range,
 * so every term is exact; the sum runs over k in order and the result is
 * rounded once.  SA is M x ceil(K/32) bytes and SB is N x ceil(K/32) bytes,
 * row-major with row strides ldsa and ldsb.  With every scale equal to 127
 * this is oracle_gemm_fp8.
 */
double oracle_ue8m0_to_double(uint8_t x) {
    if (x == 255) return NAN;
    return ldexp(1.0, (int)x - 127);
}

void oracle_gemm_mx(const uint8_t* A, const uint8_t* B, const uint8_t* SA, const uint8_t* SB,
                    int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldsa,
                    int64_t ldsb, int in_fmt, int out_dtype, double alpha,
                    int64_t i0, int64_t i1, int64_t j0, int64_t j1,
                    uint16_t* out16, double* out_f64, int64_t ldo) {
    (void)M;
    (void)N;
    double dec[256], scale[256];
    for (int c = 0; c < 256; ++c) {
        dec[c] = oracle_fp8_to_double((uint8_t)c, in_fmt);
        scale[c] = oracle_ue8m0_to_double((uint8_t)c);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = i0; i < i1; ++i) {
        for (int64_t j = j0; j < j1; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = dec[A[i * lda + k]] * scale[SA[i * ldsa + k / 32]];
                const double b = dec[B[j * ldb + k]] * scale[SB[j * ldsb + k / 32]];
                acc += a * b;
            }
            const double d = alpha * acc;
            int64_t o = (i - i0) * ldo + (j - j0);
            if (out_f64) out_f64[o] = d;
            if (out16) out16[o] = oracle_from_double(d, out_dtype);
        }
    }
}

/* Number of threads the OpenMP runtime will use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the number of threads later calls use (n >= 1; ignored without OpenMP).
 * Used only to time the oracle on one core. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
