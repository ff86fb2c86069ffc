/*
 * oracle.c -- plain, slow, obviously correct CPU reference for the skinny
 * weight-only linear layer  y[M][N] = x[M][K] . dequant(W)^T .
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) may link, load or call this file; only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark use it.  It shares no
 * code, header, table or constant with the CUDA path.
 *
 * What it computes.  The method keeps the weights compressed in memory and
 * expands each small piece to FP16 right before the multiply, with no
 * separate "dequantize the whole model first" pass (page "NVFP4 在 Volta 上！",
 * section "我实际构建了什么"; the NVFP4 format is named as block-wise 4-bit
 * floating point in the v100-skinny ai-manual.ru article, section
 * "Конвертация модели в NVFP4").  The result of that is, up to rounding, the
 * plain product of the FP16 activations with the decoded weights, so this
 * oracle is that product written out:
 *   - every element is decoded from its bit fields into an exact double;
 *   - every product x*w is exact in double (at most 11+2+4+24 = 41 significant
 *     bits for NVFP4, 11+4+24 = 39 for FP8);
 *   - the sum runs over k in ascending order in double.
 *
 * Formats (the pages name them but do not define them; the definitions are
 * the public ones):
 *   - FP16: IEEE 754 binary16.
 *   - E2M1 (FP4): OCP Microscaling Formats v1.0, FP4 element type: sign bit 3,
 *     exponent bits 2..1 with bias 1, mantissa bit 0; exponent 0 is subnormal
 *     (0 or 0.5).
 *   - E4M3: OCP 8-bit floating point (OFP8) "E4M3": sign bit 7, exponent bits
 *     6..3 with bias 7, mantissa bits 2..0; exponent 0 is subnormal; S.1111.111
 *     is NaN; there is no infinity.
 *   - NVFP4 weight tensor: codes u8[N][K/2], two E2M1 codes per byte, the LOW
 *     nibble holding the even k; one E4M3 scale per 16 consecutive k of a row,
 *     scales u8[N][K/16]; one FP32 tensor scale.
 *       w[n][k] = E2M1(code(n,k)) * E4M3(scale[n][k/16]) * gscale
 *   - FP8 weight tensor: codes u8[N][K] (E4M3), FP32 scales per 128x128 block,
 *     scales f32[ceil(N/128)][ceil(K/128)] row-major.
 *       w[n][k] = E4M3(code[n][k]) * scale[n/128][k/128]
 *
 * Besides y, every entry point also returns l1[m][n] = sum_k |x[m][k]*w[n][k]|,
 * which the accuracy contract of the library uses:
 *   |y_gpu - y| <= 1e-3 * l1 + 1e-6   (FP32 output; FP16 adds one FP16 ulp).
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (no -ffast-math: it would change the
 * double arithmetic).  With OpenMP the loop over output columns runs in
 * parallel; each column is still summed in ascending k by one thread, so the
 * result does not depend on the thread count.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, from the bit fields. */
double oracle_f16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                  /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = (m == 0) ? INFINITY : NAN;
    else
        v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return s ? -v : v;
}

/* OCP E2M1 (4-bit) -> double.  Only the low 4 bits of c are used. */
double oracle_e2m1_to_f64(uint8_t c)
{
    int s = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    double v;
    if (e == 0)
        v = 0.5 * (double)m;                        /* subnormal: 0 or 0.5 */
    else
        v = ldexp(1.0 + 0.5 * (double)m, e - 1);
    return s ? -v : v;
}

/* OCP E4M3 ("FN" variant: no infinities, only S.1111.111 is NaN) -> double. */
double oracle_e4m3_to_f64(uint8_t b)
{
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m / 8.0, -6);             /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* One NVFP4 weight, decoded: w[n][k] = E2M1 * E4M3(block scale) * gscale. */
static double nvfp4_weight(const uint8_t *codes, const uint8_t *scales,
                           double gscale, int64_t K, int64_t n, int64_t k)
{
    uint8_t byte = codes[n * (K / 2) + k / 2];
    uint8_t nib = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
    uint8_t sc = scales[n * (K / 16) + k / 16];
    return oracle_e2m1_to_f64(nib) * oracle_e4m3_to_f64(sc) * gscale;
}

/* One FP8 weight, decoded: w[n][k] = E4M3(code) * scale[n/128][k/128]. */
static double fp8_weight(const uint8_t *codes, const float *scales,
                         int64_t K, int64_t n, int64_t k)
{
    int64_t kb = (K + 127) / 128;
    return oracle_e4m3_to_f64(codes[n * K + k]) *
           (double)scales[(n / 128) * kb + (k / 128)];
}

/*
 * y[m][j] and l1[m][j] for output column n = cols[j] (or n = j when cols is
 * NULL, ncols = N).  x is FP16 bits, row-major [M][K].  Outputs are row-major
 * [M][ncols].
 */
void oracle_nvfp4_linear(int64_t M, int64_t N, int64_t K, const uint16_t *x,
                         const uint8_t *codes, const uint8_t *scales,
                         float gscale, const int64_t *cols, int64_t ncols,
                         double *y, double *l1)
{
    (void)N;
    double g = (double)gscale;
    int64_t j;
#pragma omp parallel for schedule(dynamic, 16)
    for (j = 0; j < ncols; j++) {
        int64_t n = cols ? cols[j] : j;
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = oracle_f16_to_f64(x[m * K + k]) *
                           nvfp4_weight(codes, scales, g, K, n, k);
                acc += p;
                mag += fabs(p);
            }
            y[m * ncols + j] = acc;
            l1[m * ncols + j] = mag;
        }
    }
}

void oracle_fp8_linear(int64_t M, int64_t N, int64_t K, const uint16_t *x,
                       const uint8_t *codes, const float *scales,
                       const int64_t *cols, int64_t ncols, double *y, double *l1)
{
    (void)N;
    int64_t j;
#pragma omp parallel for schedule(dynamic, 16)
    for (j = 0; j < ncols; j++) {
        int64_t n = cols ? cols[j] : j;
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = oracle_f16_to_f64(x[m * K + k]) *
                           fp8_weight(codes, scales, K, n, k);
                acc += p;
                mag += fabs(p);
            }
            y[m * ncols + j] = acc;
            l1[m * ncols + j] = mag;
        }
    }
}

/*
 * Greedy pick per row: idx[m] = the lowest n with y[m][n] equal to the row
 * maximum (the greedy / local-argmax proposal of the verify round, page
 * "NVFP4 在 Volta 上！", section "这是一个服务器，不是 GEMM 截图").  NaN entries
 * are skipped; a row of all NaN gives -1.
 */
void oracle_argmax_rows(int64_t M, int64_t N, const double *y, int64_t *idx)
{
    for (int64_t m = 0; m < M; m++) {
        int64_t best = -1;
        for (int64_t n = 0; n < N; n++) {
            double v = y[m * N + n];
            if (isnan(v))
                continue;
            if (best < 0 || v > y[m * N + best])
                best = n;
        }
        idx[m] = best;
    }
}

/*
 * Greedy verification of one speculative round (page "NVFP4 在 Volta 上！":
 * the k = 7 MTP round is verified by the target on eight rows, and a round
 * commits a prefix of the drafts plus one token of the target's own).  Row m
 * of the target holds its greedy pick target[m] for the position after the
 * prefix and the first m drafts; draft[j] (j < M - 1) is the j-th drafted
 * token.  Draft j is accepted while every draft before it was, and it equals
 * target[j].  accept[0] = the number of accepted drafts a; accept[1] =
 * target[a], the token the target itself commits after them.
 */
void oracle_verify(int64_t M, const int64_t *target, const int32_t *draft, int64_t *accept)
{
    int64_t a = 0;
    for (int64_t j = 0; j < M - 1; j++) {
        if ((int64_t)draft[j] != target[j])
            break;
        a = j + 1;
    }
    accept[0] = a;
    accept[1] = target[a];
}

/* Threads for the column loops from now on (n >= 1); used to time the
 * oracle single-threaded next to the OpenMP run.  Results do not depend on it. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
