/*
 * MXFP4 oracle: a plain, scalar, deliberately slow CPU statement of what the
 * MXFP4 training-GEMM path computes.  TEST INFRASTRUCTURE ONLY: the tests, the
 * smoke check and the benchmark's CPU-baseline leg call it; the product path
 * (the CUDA library) never does, and the two share no code.
 *
 * What the method is, from the pages:
 *   - jax-aiter README, "Supported ops" table, rows "MXFP4 Cast" and
 *     "FP4 GEMM (low-level)": BF16 is cast to MXFP4, i.e. E2M1 elements with
 *     E8M0 block scales, packed two per byte ("fp4x2"), with a row-wise and a
 *     transposed (column-wise) copy.
 *   - same table, row "FP4 GEMM (training)", and "Quick start": forward,
 *     dA (dgrad) and dB (wgrad) all run as FP4 GEMMs with BF16 output;
 *     grad_out is cast with a Hadamard transform.
 * The pages fix no rounding rule, block size, transform size or bit layout.
 * The readings taken here (each one listed in the design notes) are:
 *   - block = 32 consecutive elements along the contraction dimension;
 *   - shared exponent e = floor(log2(amax)) - 2, clamped to [-127, 127],
 *     stored as the byte e + 127 (the OCP MX scale rule); an all-zero block
 *     gets the smallest scale, byte 0x00;
 *   - a block holding a NaN or an infinity gets scale byte 0xFF and codes 0;
 *   - elements are v = x * 2^-e rounded to the nearest E2M1 value
 *     {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even code, |v| > 6 saturating
 *     to 6; the sign is kept, also for results that round to zero;
 *   - element 2j goes to the low nibble of byte j;
 *   - the Hadamard transform is the 32-point orthonormal Sylvester transform,
 *     applied per block before the scale is taken.  Because its output decides
 *     integer codes, it is evaluated in fp32 in one fixed order (butterfly
 *     stages h = 1, 2, 4, 8, 16; pair (j, j+h) with j & h == 0 becomes
 *     (a + b, a - b)), then multiplied once by the fp32 value nearest to
 *     1/sqrt(32); no fused multiply-add anywhere (built with
 *     -ffp-contract=off).
 * Everything else is carried out in fp64, where it is exact.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define BLOCK 32

/* The eight E2M1 magnitudes, indexed by the 3-bit magnitude code. */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

int oracle_abi_version(void) { return 1; }

double oracle_e2m1_value(int code) {
    double m = kE2M1[code & 7];
    return (code & 8) ? -m : m;
}

/* bf16 bit pattern -> float, exactly (a bf16 is the top half of an fp32). */
static float bf16_to_float(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Magnitude code of u >= 0: the grid point at the smallest distance, found by
 * trying all eight; on a tie the candidate with the even code wins.  Anything
 * at or above 6 is the largest code (saturation). */
int oracle_e2m1_magnitude_code(double u) {
    if (u >= 6.0) return 7;
    int best = 0;
    double best_d = fabs(u - kE2M1[0]);
    for (int c = 1; c < 8; ++c) {
        double d = fabs(u - kE2M1[c]);
        if (d < best_d || (d == best_d && (c % 2) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* Shared exponent of a block whose largest magnitude is amax (finite).
 * frexp gives amax = m * 2^p with m in [0.5, 1), so floor(log2 amax) = p - 1. */
int oracle_block_exponent(double amax) {
    if (amax == 0.0) return -127;
    int p = 0;
    (void)frexp(amax, &p);
    int e = (p - 1) - 2;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* 32-point Walsh-Hadamard transform in fp32, natural (Sylvester) order,
 * orthonormal.  The fixed evaluation order is the one stated in the header. */
void oracle_fwht32_f32(float* y) {
    for (int h = 1; h < BLOCK; h <<= 1) {
        for (int j = 0; j < BLOCK; ++j) {
            if (j & h) continue;
            float a = y[j];
            float b = y[j + h];
            y[j] = a + b;
            y[j + h] = a - b;
        }
    }
    const float inv_sqrt32 = (float)(1.0 / sqrt(32.0)); /* rounded once to fp32 */
    for (int j = 0; j < BLOCK; ++j) y[j] = y[j] * inv_sqrt32;
}

/* Quantize one block of 32 fp32 values (already transformed if the transform
 * is on).  Writes 16 code bytes and returns the scale byte. */
static uint8_t quantize_block(const float* y, uint8_t* codes16) {
    int nonfinite = 0;
    double amax = 0.0;
    for (int i = 0; i < BLOCK; ++i) {
        if (isnan(y[i]) || isinf(y[i])) nonfinite = 1;
        double a = fabs((double)y[i]);
        if (a > amax) amax = a;
    }
    if (nonfinite) {
        memset(codes16, 0, BLOCK / 2);
        return 0xFF;
    }
    int e = oracle_block_exponent(amax);
    for (int j = 0; j < BLOCK / 2; ++j) codes16[j] = 0;
    for (int i = 0; i < BLOCK; ++i) {
        double v = ldexp((double)y[i], -e); /* exact: a power-of-two multiply in fp64 */
        int code = oracle_e2m1_magnitude_code(fabs(v));
        if (signbit(y[i])) code |= 8;
        if (i % 2 == 0)
            codes16[i / 2] |= (uint8_t)code;
        else
            codes16[i / 2] |= (uint8_t)(code << 4);
    }
    return (uint8_t)(e + 127);
}

/* Row-wise MXFP4 cast of a bf16 matrix x[rows, cols] (row pitch ldx elements):
 * blocks of 32 consecutive elements of each row.
 *   codes : [rows, cols/2] bytes, row-major, pitch cols/2
 *   scales: [rows, cols/32] bytes, row-major (plain linear layout)
 * hadamard != 0 applies the 32-point transform to every block first.
 * Returns 0, or -1 if cols is not a multiple of 32. */
int oracle_cast_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, int hadamard,
                     uint8_t* codes, uint8_t* scales) {
    if (cols % BLOCK != 0) return -1;
    const int64_t nb = cols / BLOCK;
    float y[BLOCK];
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < BLOCK; ++i) y[i] = bf16_to_float(x[r * ldx + b * BLOCK + i]);
            if (hadamard) oracle_fwht32_f32(y);
            scales[r * nb + b] = quantize_block(y, codes + r * (cols / 2) + b * (BLOCK / 2));
        }
    }
    return 0;
}

/* Column-wise (transposed) cast: the row-wise cast of x^T, whose blocks run
 * down 32 consecutive rows of one column of x.
 *   codes : [cols, rows/2],  scales: [cols, rows/32]
 * Returns -1 if rows is not a multiple of 32. */
int oracle_cast_cols(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, int hadamard,
                     uint8_t* codes, uint8_t* scales) {
    if (rows % BLOCK != 0) return -1;
    const int64_t nb = rows / BLOCK;
    float y[BLOCK];
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < BLOCK; ++i) y[i] = bf16_to_float(x[(b * BLOCK + i) * ldx + c]);
            if (hadamard) oracle_fwht32_f32(y);
            scales[c * nb + b] = quantize_block(y, codes + c * (rows / 2) + b * (BLOCK / 2));
        }
    }
    return 0;
}

/* Dequantize row-wise MXFP4 data: out[r, k] = e2m1(code) * 2^(scale - 127),
 * NaN for scale byte 0xFF.  codes [rows, cols/2], scales [rows, cols/32]. */
int oracle_dequant_rows(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                        double* out) {
    if (cols % BLOCK != 0) return -1;
    const int64_t nb = cols / BLOCK;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t k = 0; k < cols; ++k) {
            uint8_t byte = codes[r * (cols / 2) + k / 2];
            int code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            uint8_t s = scales[r * nb + k / BLOCK];
            out[r * cols + k] = (s == 0xFF) ? NAN : ldexp(oracle_e2m1_value(code), (int)s - 127);
        }
    }
    return 0;
}

/* C[M,N] = A[M,K] * B[N,K]^T in fp64: one dot product per output, k ascending.
 * The straight triple loop.  Rows of C are split over nthreads threads; each
 * output is still the same single sequential sum, so the result does not
 * depend on nthreads. */
typedef struct {
    const double* a;
    const double* b;
    double* c;
    int64_t m0, m1, n, k;
} gemm_job;

static void* gemm_rows(void* p) {
    gemm_job* j = (gemm_job*)p;
    for (int64_t i = j->m0; i < j->m1; ++i) {
        for (int64_t n = 0; n < j->n; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < j->k; ++k) s += j->a[i * j->k + k] * j->b[n * j->k + k];
            j->c[i * j->n + n] = s;
        }
    }
    return NULL;
}

int oracle_gemm_abt_f64(const double* a, const double* b, int64_t m, int64_t n, int64_t k, double* c,
                        int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > m) nthreads = (int)(m > 0 ? m : 1);
    pthread_t tid[256];
    int running[256];
    gemm_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].a = a;
        jobs[t].b = b;
        jobs[t].c = c;
        jobs[t].m0 = m * t / nthreads;
        jobs[t].m1 = m * (t + 1) / nthreads;
        jobs[t].n = n;
        jobs[t].k = k;
    }
    for (int t = 0; t < nthreads; ++t) {
        running[t] = (nthreads > 1) && pthread_create(&tid[t], NULL, gemm_rows, &jobs[t]) == 0;
        if (!running[t]) gemm_rows(&jobs[t]); /* one thread, or no thread to be had: run inline */
    }
    for (int t = 0; t < nthreads; ++t)
        if (running[t]) pthread_join(tid[t], NULL);
    return 0;
}

/*
 * MXFP8 (E4M3 elements, E8M0 block scales): the FP8 alternative for the wgrad
 * operands.  Method: jax-aiter README, "MXFP4 training architecture" (an FP8
 * dB path next to the FP4 one).  The pages fix nothing about it; the readings
 * (listed in the design notes) follow the OCP MX rules as above:
 *   - E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
 *     subnormal (m * 2^-9); magnitude code 0x7F is NaN, so the largest
 *     finite magnitude is 0x7E = 1.75 * 2^8 = 448;
 *   - e = floor(log2(amax)) - 8 (8 = the exponent of E4M3's largest normal),
 *     clamped to [-127, 127], byte e + 127; all-zero block: byte 0x00;
 *     NaN or infinity in the block: byte 0xFF and codes 0;
 *   - v = x * 2^-e rounded to the nearest E4M3 value, ties to the even code,
 *     |v| >= 448 saturating to 448; the sign is kept; one byte per element.
 */

/* Magnitude of the 7-bit E4M3 magnitude code m (0..126); NaN for 127. */
static double e4m3_magnitude(int m) {
    if (m >= 127) return NAN;
    int ex = m >> 3, mant = m & 7;
    if (ex == 0) return ldexp((double)mant, -9);
    return ldexp(1.0 + mant / 8.0, ex - 7);
}

double oracle_e4m3_value(int code) {
    double v = e4m3_magnitude(code & 0x7F);
    return (code & 0x80) ? -v : v;
}

/* Magnitude code of u >= 0: the nearest of the 127 finite magnitudes, found by
 * trying them all; on a tie the even code wins.  u >= 448 gives 0x7E. */
int oracle_e4m3_magnitude_code(double u) {
    if (u >= 448.0) return 0x7E;
    int best = 0;
    double best_d = fabs(u - e4m3_magnitude(0));
    for (int c = 1; c < 127; ++c) {
        double d = fabs(u - e4m3_magnitude(c));
        if (d < best_d || (d == best_d && (c % 2) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* Shared exponent for E4M3 elements: floor(log2 amax) - 8, clamped. */
int oracle_block_exponent_e4m3(double amax) {
    if (amax == 0.0) return -127;
    int p = 0;
    (void)frexp(amax, &p);
    int e = (p - 1) - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* One block of 32 fp32 values -> 32 code bytes; returns the scale byte. */
static uint8_t quantize_block_e4m3(const float* y, uint8_t* codes32) {
    int nonfinite = 0;
    double amax = 0.0;
    for (int i = 0; i < BLOCK; ++i) {
        if (isnan(y[i]) || isinf(y[i])) nonfinite = 1;
        double a = fabs((double)y[i]);
        if (a > amax) amax = a;
    }
    if (nonfinite) {
        memset(codes32, 0, BLOCK);
        return 0xFF;
    }
    int e = oracle_block_exponent_e4m3(amax);
    for (int i = 0; i < BLOCK; ++i) {
        double v = ldexp((double)y[i], -e);
        int code = oracle_e4m3_magnitude_code(fabs(v));
        if (signbit(y[i])) code |= 0x80;
        codes32[i] = (uint8_t)code;
    }
    return (uint8_t)(e + 127);
}

/* Row-wise MXFP8 cast: codes [rows, cols] (one byte per element), scales
 * [rows, cols/32]; hadamard != 0 transforms every block first (fp32, as
 * above).  Returns -1 if cols is not a multiple of 32. */
int oracle_cast_rows_mxfp8(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, int hadamard,
                           uint8_t* codes, uint8_t* scales) {
    if (cols % BLOCK != 0) return -1;
    const int64_t nb = cols / BLOCK;
    float y[BLOCK];
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < BLOCK; ++i) y[i] = bf16_to_float(x[r * ldx + b * BLOCK + i]);
            if (hadamard) oracle_fwht32_f32(y);
            scales[r * nb + b] = quantize_block_e4m3(y, codes + r * cols + b * BLOCK);
        }
    }
    return 0;
}

/* Column-wise (transposed) MXFP8 cast: the row-wise cast of x^T.
 * codes [cols, rows], scales [cols, rows/32]. */
int oracle_cast_cols_mxfp8(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, int hadamard,
                           uint8_t* codes, uint8_t* scales) {
    if (rows % BLOCK != 0) return -1;
    const int64_t nb = rows / BLOCK;
    float y[BLOCK];
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < BLOCK; ++i) y[i] = bf16_to_float(x[(b * BLOCK + i) * ldx + c]);
            if (hadamard) oracle_fwht32_f32(y);
            scales[c * nb + b] = quantize_block_e4m3(y, codes + c * rows + b * BLOCK);
        }
    }
    return 0;
}

/* out[r, k] = e4m3(code) * 2^(scale - 127); NaN for scale byte 0xFF. */
int oracle_dequant_rows_mxfp8(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                              double* out) {
    if (cols % BLOCK != 0) return -1;
    const int64_t nb = cols / BLOCK;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t k = 0; k < cols; ++k) {
            uint8_t s = scales[r * nb + k / BLOCK];
            out[r * cols + k] = (s == 0xFF) ? NAN : ldexp(oracle_e4m3_value(codes[r * cols + k]), (int)s - 127);
        }
    }
    return 0;
}
