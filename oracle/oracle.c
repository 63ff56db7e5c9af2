/*
 * CPU oracle for the FP16 "TN" GEMM D = A * B^T and the M = 1 GEMV y = x * W^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference leg use it.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (the plain definition that the tiled kernels reach up to
 * rounding order):
 *
 *   D[m][n] = fp16_rne( sum_{k=0}^{K-1} double(A[m][k]) * double(B[n][k]) )
 *   y[n]    = fp16_rne( sum_{k=0}^{K-1} double(x[k])    * double(W[n][k]) )
 *
 *   - A is M x K row-major and B is N x K row-major, both fp16, so both
 *     operands are K-contiguous ("TN"): "使用 TMA 为 GEMM 建立 Pipeline",
 *     step 4 "完整 Kernel" (A: (M, K), B: (N, K), D: (M, N) buffers) and the
 *     Croqtile chapter "高级数据搬运：TMA、Swizzle 与不规则访问", section
 *     "示例：流水线矩阵乘法中的 TMA" (lhs [M, K], rhs [N, K], output [M, N]).
 *   - Accumulation is at least FP32 (the pages accumulate in FP32: step 4's
 *     acc_type float32; "Learning TileLang with GEMV" §01: every kernel
 *     accumulates in FP32).  The oracle accumulates in FP64, k ascending, with
 *     a single rounding to binary16 at the end (round to nearest, ties to
 *     even).
 *   - GEMV: "Learning TileLang with GEMV" §01 GEMV: W is N x K row-major (the
 *     nn.Linear layout) and y[n] is the dot product of x with row n of W.
 *
 * The binary16 codec below is written from the IEEE 754 binary16 format
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits; exponent 0 =
 * zero/subnormal, exponent 31 = inf/NaN).
 *
 * The bfloat16 forms (oracle_gemm_bf16, oracle_gemv_bf16) follow the same
 * definition with bf16 operands and a bf16 result ("TensorCore_GEMM_with_TMA"
 * runs its TN GEMM in bf16 with FP32 accumulation).
 *
 * Parity status: every function here is pinned by the CPU tests (exact
 * rational arithmetic on tiny shapes, integer-valued inputs against an exact
 * integer matmul, identity / rank-1 / unit-vector closed forms, transpose
 * symmetry, the full binary16 decode/encode tables against numpy, and the
 * bf16 codec against float32 bit patterns and exact rationals).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- IEEE 754 binary16 codec ------------------------------------------- */

double oracle_half_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                 /* zero or subnormal */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);  /* 1.f * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a non-negative double holding an exact binary fraction to the nearest
 * integer, ties to even.  q - floor(q) is exact for doubles. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double diff = q - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint16_t oracle_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = q * 2^-24, q in [0, 1024]; q == 1024 is the
         * smallest normal (exponent field 1, fraction 0), which the bit
         * pattern q also encodes. */
        double q = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e2;
    (void)frexp(a, &e2);            /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                 /* 2^e <= a < 2^(e+1) */
    double q = round_half_even(ldexp(a, 10 - e));   /* in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00);   /* overflow -> inf */
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* ---- bfloat16 codec ------------------------------------------------------
 * bfloat16 keeps the top 16 bits of an IEEE binary32: 1 sign bit, 8 exponent
 * bits with bias 127, 7 fraction bits (exponent 0 = zero/subnormal, 255 =
 * inf/NaN).  Decoding and encoding are written from that format, the same
 * way as the binary16 codec above. */

double oracle_bf16_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 7) & 0xff;
    const int frac = h & 0x7f;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -133);                 /* 0.f * 2^-126 */
    } else if (expo == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + frac), expo - 134);   /* 1.f * 2^(e-127) */
    }
    return sign ? -v : v;
}

uint16_t oracle_double_to_bf16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7fc0);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7f80);
    if (a < ldexp(1.0, -126)) {
        /* subnormal range: value = q * 2^-133, q in [0, 128]; q == 128 is the
         * smallest normal, which the bit pattern q also encodes. */
        double q = round_half_even(ldexp(a, 133));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e2;
    (void)frexp(a, &e2);
    int e = e2 - 1;                                 /* 2^e <= a < 2^(e+1) */
    double q = round_half_even(ldexp(a, 7 - e));    /* in [128, 256] */
    if (q == 256.0) { q = 128.0; e += 1; }
    if (e > 127) return (uint16_t)(sign | 0x7f80);  /* overflow -> inf */
    return (uint16_t)(sign | (uint16_t)((e + 127) << 7) | (uint16_t)(q - 128.0));
}

/* ---- decode tables (pure functions of the codecs above) ----------------- */

static double g_lut[65536];
static double g_lut_bf16[65536];
static int g_lut_ready = 0;

static void build_lut(void)
{
    if (g_lut_ready) return;
    for (int h = 0; h < 65536; ++h) {
        g_lut[h] = oracle_half_to_double((uint16_t)h);
        g_lut_bf16[h] = oracle_bf16_to_double((uint16_t)h);
    }
    g_lut_ready = 1;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- one output element: the plain definition -------------------------- */

static double dot_f16(const uint16_t* a, const uint16_t* b, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += g_lut[a[k]] * g_lut[b[k]];
    return acc;
}

static double dot_bf16(const uint16_t* a, const uint16_t* b, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += g_lut_bf16[a[k]] * g_lut_bf16[b[k]];
    return acc;
}

/* D (M x N fp16 bits) = A (M x K) * B (N x K)^T.  If sum64 != NULL it also
 * receives the unrounded FP64 sums (M x N doubles).  nthreads <= 0 means all
 * available threads; threads split the rows of D and do not change any
 * element's arithmetic.  Returns the thread count used. */
int oracle_gemm_f16(int64_t M, int64_t N, int64_t K,
                    const uint16_t* A, const uint16_t* B,
                    uint16_t* D, double* sum64, int nthreads)
{
    build_lut();
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    used = nthreads;
    #pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = dot_f16(A + m * K, B + n * K, K);
            if (sum64) sum64[m * N + n] = s;
            D[m * N + n] = oracle_double_to_half(s);
        }
    }
    return used;
}

/* The same definition evaluated at `count` chosen positions (ms[i], ns[i]):
 * out[i] = D[ms[i]][ns[i]], sum64[i] = its unrounded FP64 sum (if non-NULL).
 * Used to check full-size runs on samples. */
int oracle_gemm_f16_at(int64_t M, int64_t N, int64_t K,
                       const uint16_t* A, const uint16_t* B,
                       int64_t count, const int64_t* ms, const int64_t* ns,
                       uint16_t* out, double* sum64, int nthreads)
{
    build_lut();
    (void)M; (void)N;
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    used = nthreads;
    #pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < count; ++i) {
        double s = dot_f16(A + ms[i] * K, B + ns[i] * K, K);
        if (sum64) sum64[i] = s;
        out[i] = oracle_double_to_half(s);
    }
    return used;
}

/* y (N fp16 bits) = x (K) * W (N x K)^T; optional FP64 sums. */
int oracle_gemv_f16(int64_t N, int64_t K, const uint16_t* x, const uint16_t* W,
                    uint16_t* y, double* sum64, int nthreads)
{
    build_lut();
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    used = nthreads;
    #pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t n = 0; n < N; ++n) {
        double s = dot_f16(x, W + n * K, K);
        if (sum64) sum64[n] = s;
        y[n] = oracle_double_to_half(s);
    }
    return used;
}

/* ---- bfloat16 forms: the same definitions with bf16 operands and output --
 * ("TensorCore_GEMM_with_TMA" runs the same TN GEMM in bf16 with FP32
 * accumulation and a round-to-nearest conversion of the result). */

int oracle_gemm_bf16(int64_t M, int64_t N, int64_t K,
                     const uint16_t* A, const uint16_t* B,
                     uint16_t* D, double* sum64, int nthreads)
{
    build_lut();
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    used = nthreads;
    #pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = dot_bf16(A + m * K, B + n * K, K);
            if (sum64) sum64[m * N + n] = s;
            D[m * N + n] = oracle_double_to_bf16(s);
        }
    }
    return used;
}

int oracle_gemv_bf16(int64_t N, int64_t K, const uint16_t* x, const uint16_t* W,
                     uint16_t* y, double* sum64, int nthreads)
{
    build_lut();
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    used = nthreads;
    #pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int64_t n = 0; n < N; ++n) {
        double s = dot_bf16(x, W + n * K, K);
        if (sum64) sum64[n] = s;
        y[n] = oracle_double_to_bf16(s);
    }
    return used;
}
