/*
 * oracle.c -- plain CPU oracle for the dense GEMM C = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load or run this file. The
 * product (the CUDA library) never calls it, links it or includes it, and this
 * file includes nothing from the CUDA library. It is deliberately slow and
 * plain: decode every operand exactly to double, multiply, add in FP64, in the
 * order the definition states. No blocking, no fusion, no reordering.
 *
 * Definitions followed:
 *  - BF16 GEMM. "Achieve cuBLAS Performance on NVIDIA GB300 for HGEMM",
 *    introduction: each kernel computes a row-major C = A @ B^T with A: MxK,
 *    B: NxK, C: MxN, BF16 inputs and outputs, FP32 accumulation.
 *    Here C_ref[i][j] = sum_k bf16(A[i][k]) * bf16(B[j][k]) in FP64, which is
 *    the exact real-valued result to ~1e-16 relative (every product of two
 *    BF16 values is exact in FP64). Output rounding to BF16 is round to
 *    nearest, ties to even ("Optimized B200 Matrix Multiplication", section
 *    "5. The Epilogue": FP32 -> BF16 with the _rn conversion), applied
 *    directly to the FP64 value (no intermediate FP32 rounding).
 *  - NVFP4 GEMM. "NVFP4 GEMM on Blackwell", section "NVFP4 Datatype": values
 *    are E2M1 (1 sign, 2 exponent, 1 mantissa bit; the 16 values +-0, +-0.5,
 *    +-1, +-1.5, +-2, +-3, +-4, +-6) and every 16 FP4 values share one FP8
 *    scale factor. C_ref[i][j] = sum_k e2m1(a_ik) * e4m3(SFA[i][k/16]) *
 *    e2m1(b_jk) * e4m3(SFB[j][k/16]) in FP64. Every factor has at most four
 *    significant bits, so every product is exact in FP64 and, for the operand
 *    ranges used (|C| < 2^27, products multiples of 2^-16), so is every sum.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - operands are K-major: A is [M][K], B is [N][K] (the HGEMM page's A @ B^T);
 *  - packed E2M1: byte j of a row holds element 2j in bits 0-3, 2j+1 in bits 4-7;
 *  - scale layout: SFA is [M][K/16], SFB is [N][K/16], row-major bytes;
 *  - the FP8 scale is E4M3 (OCP E4M3FN: bias 7, no infinities, S.1111.111 = NaN).
 *
 * Every function here is pinned by the CPU tests (tests/test_oracle.py)
 * against values the pages print, closed forms, brute force in exact rational
 * arithmetic and independent library routines.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------- exact decoders ---------- */

/* BF16 is the upper half of an IEEE binary32: widen the bits, then to double. */
double oracle_dec_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E2M1: bit 3 sign, bits 2-1 exponent (bias 1), bit 0 mantissa.
 * Exponent 0 is subnormal: value = m * 0.5. Otherwise 2^(e-1) * (1 + m/2). */
double oracle_dec_e2m1(uint8_t code)
{
    unsigned c = code & 0xFu;
    unsigned s = (c >> 3) & 1u, e = (c >> 1) & 3u, m = c & 1u;
    double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -v : v;
}

/* E4M3 (OCP E4M3FN): bit 7 sign, bits 6-3 exponent (bias 7), bits 2-0 mantissa.
 * Exponent 0 is subnormal: (m/8) * 2^-6. Exponent 15 with mantissa 7 is NaN;
 * there are no infinities. */
double oracle_dec_e4m3(uint8_t code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 0xFu, m = code & 7u;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -v : v;
}

/* ---------- output rounding ---------- */

/* Round a double to the nearest BF16 (8 significant bits, binary32 exponent
 * range, subnormals down to 2^-133), ties to even, in one rounding step.
 * Overflow goes to +-inf, NaN stays NaN. */
uint16_t oracle_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e2;
    frexp(a, &e2);                      /* a = f * 2^e2, f in [0.5, 1): floor(log2 a) = e2 - 1 */
    int q = e2 - 1;
    if (q < -126)
        q = -126;                       /* subnormal range keeps the 2^-133 step */
    q -= 7;                             /* exponent of one unit in the last place */
    double scaled = ldexp(a, -q);       /* exact: power-of-two scaling */
    double n = floor(scaled);
    double r = scaled - n;              /* exact: n < 2^9 and scaled has <= 53 bits */
    if (r > 0.5 || (r == 0.5 && fmod(n, 2.0) != 0.0))
        n += 1.0;
    double v = ldexp(n, q);             /* representable in BF16 unless it overflows */
    if (v > 3.3895313892515355e38)      /* largest finite BF16, (2 - 2^-7) * 2^127 */
        return (uint16_t)(sign | 0x7F80);
    float f = (float)v;                 /* exact */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFF));
}

void oracle_round_bf16(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_rne(x[i]);
}

/* ---------- BF16 GEMM: C = A * B^T ---------- */

static double* decode_bf16_rows(const uint16_t* X, int64_t rows, int64_t K)
{
    double* D = (double*)malloc((size_t)(rows * K > 0 ? rows * K : 1) * sizeof(double));
    if (!D)
        return NULL;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t k = 0; k < K; ++k)
            D[i * K + k] = oracle_dec_bf16(X[i * K + k]);
    return D;
}

/* Rows [row0, row1) of C = A * B^T in FP64; C is (row1-row0) x N, row-major.
 * A: M x K BF16 bits, B: N x K BF16 bits, both row-major (K contiguous).
 * Returns 0 on success, -1 if memory could not be allocated. */
int oracle_gemm_bf16(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                     int64_t row0, int64_t row1, double* C)
{
    (void)M;
    int64_t rows = row1 - row0;
    double* Ad = decode_bf16_rows(A + row0 * K, rows, K);
    double* Bd = decode_bf16_rows(B, N, K);
    if (!Ad || !Bd) {
        free(Ad);
        free(Bd);
        return -1;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < rows; ++i) {
        const double* a = Ad + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const double* b = Bd + j * K;
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += a[k] * b[k];
            C[i * N + j] = s;
        }
    }
    free(Ad);
    free(Bd);
    return 0;
}

/* Selected elements C[rows[t]][cols[t]], t < n, each computed on its own. */
void oracle_gemm_bf16_at(const uint16_t* A, const uint16_t* B, int64_t K,
                         const int64_t* rows, const int64_t* cols, int64_t n, double* out)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t* a = A + rows[t] * K;
        const uint16_t* b = B + cols[t] * K;
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += oracle_dec_bf16(a[k]) * oracle_dec_bf16(b[k]);
        out[t] = s;
    }
}

/* ---------- NVFP4 block-scaled GEMM ---------- */

/* Element k of a row of packed E2M1 codes, scaled by its block's E4M3 scale. */
static double nvfp4_elem(const uint8_t* codes_row, const uint8_t* scales_row, int64_t k)
{
    uint8_t byte = codes_row[k >> 1];
    uint8_t code = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
    return oracle_dec_e2m1(code) * oracle_dec_e4m3(scales_row[k >> 4]);
}

static double* decode_nvfp4_rows(const uint8_t* X, const uint8_t* SF, int64_t rows, int64_t K)
{
    double* D = (double*)malloc((size_t)(rows * K > 0 ? rows * K : 1) * sizeof(double));
    if (!D)
        return NULL;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t k = 0; k < K; ++k)
            D[i * K + k] = nvfp4_elem(X + i * (K / 2), SF + i * (K / 16), k);
    return D;
}

/* Rows [row0, row1) of C = A * B^T for NVFP4 operands, in FP64.
 * A: M x K/2 packed codes, SFA: M x K/16 scale bytes, B: N x K/2, SFB: N x K/16.
 * K must be a multiple of 16. Returns 0, or -1 on allocation failure. */
int oracle_gemm_nvfp4(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                      int64_t M, int64_t N, int64_t K, int64_t row0, int64_t row1, double* C)
{
    (void)M;
    int64_t rows = row1 - row0;
    double* Ad = decode_nvfp4_rows(A + row0 * (K / 2), SFA + row0 * (K / 16), rows, K);
    double* Bd = decode_nvfp4_rows(B, SFB, N, K);
    if (!Ad || !Bd) {
        free(Ad);
        free(Bd);
        return -1;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < rows; ++i) {
        const double* a = Ad + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const double* b = Bd + j * K;
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += a[k] * b[k];
            C[i * N + j] = s;
        }
    }
    free(Ad);
    free(Bd);
    return 0;
}

void oracle_gemm_nvfp4_at(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                          int64_t K, const int64_t* rows, const int64_t* cols, int64_t n, double* out)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
        const uint8_t* a = A + rows[t] * (K / 2);
        const uint8_t* sa = SFA + rows[t] * (K / 16);
        const uint8_t* b = B + cols[t] * (K / 2);
        const uint8_t* sb = SFB + cols[t] * (K / 16);
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += nvfp4_elem(a, sa, k) * nvfp4_elem(b, sb, k);
        out[t] = s;
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
