/*
 * oracle.c -- plain, slow, obviously correct CPU reference of the W4A16
 * group-quantised linear layer  y = x . dequant(W)^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares no source,
 * header, table or helper with the CUDA library: every step below is written
 * out from its definition.
 *
 * What the pages fix, and where:
 *  - "[ROCm][Kernel] Add HybridW4A16LinearKernel: Triton prefill + HIP skinny
 *    decode" (vllm-project/vllm#40977), PR description: one weight tensor
 *    packed [N, K/8] (8 x 4-bit per int32 along K), symmetric weights with a
 *    fixed bias of 8 (uint4b8) or asymmetric weights with per-group zero
 *    points, group sizes 32, 64 or 128.
 *  - "Upstream sync 67/N: merge 382bbd5144 HybridW4A16LinearKernel
 *    (conflict)" (ROCm/vllm#1175), section "Upstream's Python side is kept --
 *    and it does NOT work here": zero points packed as int32 [N/8, groups],
 *    8 x uint4 along dim 0 (N).  Same page, selection example: no act-order
 *    (has_g_idx=False), so groups are contiguous runs of G along K.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - nibble order in a weight word: element k = 8j+i sits in bits [4i, 4i+3]
 *    of word j (sequential);
 *  - zero-point nibble order: row n's zero point is nibble n%8 of word n/8;
 *  - the dequantised weight is w = RN_dtype((q - z) * s): the product is
 *    formed exactly and rounded once, to nearest, ties to even, into the
 *    activation dtype; the GEMM then accumulates x * w in fp64 (no rounding
 *    of y).  The exact-weight product  sum x * (q - z) * s  is also offered
 *    for information.
 *
 * Parity pins (see tests/test_oracle_pins.py): pack/unpack round trip,
 * symmetric == asymmetric with all zero points 8, hand-worked tiny cases,
 * per-group brute force in numpy, exhaustive rounding of (q - z) * s against
 * numpy/torch casts, a numpy float64 matmul of the materialised weights.
 *
 * dtype codes: 0 = fp16 (IEEE binary16), 1 = bf16 (bfloat16).
 * 16-bit floats are carried as their raw uint16 bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- 16-bit float formats ------------------------------------------------
 * binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
 * bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.            */
static void fmt_params(int dtype, int *exp_bits, int *frac_bits) {
    if (dtype == 0) { *exp_bits = 5; *frac_bits = 10; }
    else            { *exp_bits = 8; *frac_bits = 7; }
}

/* Exact value of a 16-bit pattern, as a double (every such value is exactly
 * representable in binary64). */
double oracle_half_to_double(uint16_t bits, int dtype) {
    int eb, fb;
    fmt_params(dtype, &eb, &fb);
    int sign = (bits >> 15) & 1;
    int e = (bits >> fb) & ((1 << eb) - 1);
    int f = bits & ((1 << fb) - 1);
    int bias = (1 << (eb - 1)) - 1;
    double v;
    if (e == (1 << eb) - 1) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)f, 1 - bias - fb);           /* subnormal */
    } else {
        v = ldexp((double)((1 << fb) | f), e - bias - fb);
    }
    return sign ? -v : v;
}

/* Round a double to the 16-bit format: round to nearest, ties to even,
 * overflow to infinity, gradual underflow.  Written from the IEEE-754
 * definition: find the quantum (spacing of representable numbers) at the
 * value's binade, express the value in quanta, round that to an integer. */
uint16_t oracle_double_to_half(double v, int dtype) {
    int eb, fb;
    fmt_params(dtype, &eb, &fb);
    int bias = (1 << (eb - 1)) - 1;
    int emin = 1 - bias;                  /* exponent of the smallest normal */
    int emax = bias;                      /* exponent of the largest finite  */
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    uint16_t exp_all_ones = (uint16_t)(((1 << eb) - 1) << fb);
    if (isnan(v)) return (uint16_t)(exp_all_ones | (1 << (fb - 1)));
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | exp_all_ones);

    int ex;
    (void)frexp(a, &ex);                  /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;                       /* a in [2^e, 2^(e+1))         */
    if (e < emin) e = emin;               /* subnormal: fixed quantum    */
    double quanta = ldexp(a, fb - e);     /* a / 2^(e - fb), exact       */
    double r = floor(quanta);
    double frac = quanta - r;             /* exact: quanta < 2^(fb+2)    */
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) == 1.0)) r += 1.0;
    if (r >= ldexp(1.0, fb + 1)) {        /* rounded up into next binade */
        r = ldexp(1.0, fb);
        e += 1;
    }
    if (e > emax) return (uint16_t)(sign | exp_all_ones);   /* overflow */
    uint32_t ri = (uint32_t)r;
    if (ri < (1u << fb)) {                /* subnormal (only when e == emin) */
        return (uint16_t)(sign | ri);
    }
    uint32_t efield = (uint32_t)(e + bias);
    return (uint16_t)(sign | (efield << fb) | (ri - (1u << fb)));
}

/* ---- packing ---------------------------------------------------------------
 * qweight[n, j] holds q[n, 8j + i] in bits [4i, 4i+3], i = 0..7.         */
void oracle_pack(const uint8_t *q, int N, int K, int32_t *qweight) {
    for (int n = 0; n < N; ++n)
        for (int j = 0; j < K / 8; ++j) {
            uint32_t w = 0;
            for (int i = 0; i < 8; ++i)
                w |= (uint32_t)(q[(size_t)n * K + 8 * j + i] & 0xF) << (4 * i);
            qweight[(size_t)n * (K / 8) + j] = (int32_t)w;
        }
}

void oracle_unpack(const int32_t *qweight, int N, int K, uint8_t *q) {
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            uint32_t w = (uint32_t)qweight[(size_t)n * (K / 8) + k / 8];
            q[(size_t)n * K + k] = (uint8_t)((w >> (4 * (k % 8))) & 0xF);
        }
}

/* qzeros[r, g] holds z[8r + i, g] in bits [4i, 4i+3], i = 0..7. */
void oracle_pack_zeros(const uint8_t *z, int N, int n_groups, int32_t *qzeros) {
    for (int r = 0; r < N / 8; ++r)
        for (int g = 0; g < n_groups; ++g) {
            uint32_t w = 0;
            for (int i = 0; i < 8; ++i)
                w |= (uint32_t)(z[(size_t)(8 * r + i) * n_groups + g] & 0xF) << (4 * i);
            qzeros[(size_t)r * n_groups + g] = (int32_t)w;
        }
}

void oracle_unpack_zeros(const int32_t *qzeros, int N, int n_groups, uint8_t *z) {
    for (int n = 0; n < N; ++n)
        for (int g = 0; g < n_groups; ++g) {
            uint32_t w = (uint32_t)qzeros[(size_t)(n / 8) * n_groups + g];
            z[(size_t)n * n_groups + g] = (uint8_t)((w >> (4 * (n % 8))) & 0xF);
        }
}

/* ---- dequantisation --------------------------------------------------------
 * One weight: q from its word, z = 8 (symmetric) or the packed zero point,
 * s = scales[n, k / G]; w = RN_dtype((q - z) * s), the product taken exactly
 * in binary64 (|q - z| <= 15 and s has at most 11 significant bits).     */
static double exact_weight(const int32_t *qweight, const uint16_t *scales,
                           const int32_t *qzeros, int G, int N, int K,
                           int dtype, int n, int k) {
    (void)N;
    int n_groups = K / G;
    uint32_t w = (uint32_t)qweight[(size_t)n * (K / 8) + k / 8];
    int q = (int)((w >> (4 * (k % 8))) & 0xF);
    int g = k / G;
    int z = 8;
    if (qzeros) {
        uint32_t zw = (uint32_t)qzeros[(size_t)(n / 8) * n_groups + g];
        z = (int)((zw >> (4 * (n % 8))) & 0xF);
    }
    double s = oracle_half_to_double(scales[(size_t)n * n_groups + g], dtype);
    return (double)(q - z) * s;
}

void oracle_dequant(const int32_t *qweight, const uint16_t *scales,
                    const int32_t *qzeros, int G, int N, int K, int dtype,
                    uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            out[(size_t)n * K + k] = oracle_double_to_half(
                exact_weight(qweight, scales, qzeros, G, N, K, dtype, n, k), dtype);
}

/* Rounding table: out[i, j] = RN_dtype(d[i] * s_j) for every 16-bit pattern
 * s_j (j = 0..65535), d[i] an integer.  Used by the exhaustive rounding pin. */
void oracle_round_products(const int *d, int nd, int dtype, uint16_t *out) {
    for (int i = 0; i < nd; ++i)
        for (int j = 0; j < 65536; ++j)
            out[(size_t)i * 65536 + j] = oracle_double_to_half(
                (double)d[i] * oracle_half_to_double((uint16_t)j, dtype), dtype);
}

/* ---- GEMM ------------------------------------------------------------------
 * y[m, n] = sum_k x[m, k] * W_ref[n, k], accumulated in binary64, where
 * W_ref = RN_dtype((q - z) * s) as above.  rows (length n_rows) selects which
 * m to compute (NULL = all M); y has n_rows (or M) rows of N doubles.
 * exact_w != 0 uses the unrounded product (q - z) * s instead (informative). */
void oracle_gemm_rows(const uint16_t *x, int M, int K, const int32_t *qweight,
                      const uint16_t *scales, const int32_t *qzeros, int G,
                      int N, int dtype, const int *rows, int n_rows,
                      int exact_w, double *y) {
    int R = rows ? n_rows : M;
    double *xd = (double *)malloc(sizeof(double) * (size_t)R * K);
    for (int r = 0; r < R; ++r) {
        int m = rows ? rows[r] : r;
        for (int k = 0; k < K; ++k)
            xd[(size_t)r * K + k] = oracle_half_to_double(x[(size_t)m * K + k], dtype);
    }
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int n = 0; n < N; ++n) {
            for (int k = 0; k < K; ++k) {
                double e = exact_weight(qweight, scales, qzeros, G, N, K, dtype, n, k);
                wrow[k] = exact_w ? e
                                  : oracle_half_to_double(oracle_double_to_half(e, dtype), dtype);
            }
            for (int r = 0; r < R; ++r) {
                double acc = 0.0;
                for (int k = 0; k < K; ++k) acc += xd[(size_t)r * K + k] * wrow[k];
                y[(size_t)r * N + n] = acc;
            }
        }
        free(wrow);
    }
    free(xd);
}

void oracle_gemm(const uint16_t *x, int M, int K, const int32_t *qweight,
                 const uint16_t *scales, const int32_t *qzeros, int G, int N,
                 int dtype, double *y) {
    oracle_gemm_rows(x, M, K, qweight, scales, qzeros, G, N, dtype, NULL, 0, 0, y);
}

/* ---- fused epilogues --------------------------------------------------------
 * The steps the layer may fuse after its GEMM, on the unrounded binary64
 * accumulations y [R, N]:
 *  - bias (the optional `bias` operand of the skinny GEMM call in "Upstream
 *    sync 67/N: merge 382bbd5144 HybridW4A16LinearKernel (conflict)",
 *    section "Upstream's Python side is kept"): a[r, n] = y[r, n] + b[n],
 *    b[n] the exact value of the 16-bit bias pattern; no bias: a = y;
 *  - SiLU-and-multiply over a merged gate/up projection (N = 2 I, the gate
 *    rows first): h[r, j] = silu(a[r, j]) * a[r, I + j] with
 *    silu(v) = v / (1 + exp(-v)), every step in binary64.
 * out holds [R, N] (no activation) or [R, N / 2] (SiLU-and-multiply); the
 * library rounds each result once into the activation dtype. */
void oracle_epilogue(const double *y, int R, int N, const uint16_t *bias, int dtype,
                     int silu_mul, double *out) {
    const int I = N / 2;
    for (int r = 0; r < R; ++r) {
        const double *yr = y + (size_t)r * N;
        if (!silu_mul) {
            for (int n = 0; n < N; ++n)
                out[(size_t)r * N + n] = yr[n] + (bias ? oracle_half_to_double(bias[n], dtype) : 0.0);
        } else {
            for (int j = 0; j < I; ++j) {
                double g = yr[j] + (bias ? oracle_half_to_double(bias[j], dtype) : 0.0);
                double u = yr[I + j] + (bias ? oracle_half_to_double(bias[I + j], dtype) : 0.0);
                out[(size_t)r * I + j] = g / (1.0 + exp(-g)) * u;
            }
        }
    }
}

/* Output rounding: RN_dtype of each double (the library's output is the
 * fp32 accumulator rounded once into the activation dtype). */
void oracle_round_array(const double *v, long long n, int dtype, uint16_t *out) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_double_to_half(v[i], dtype);
}

void oracle_half_array_to_double(const uint16_t *bits, long long n, int dtype, double *out) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_half_to_double(bits[i], dtype);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
