/*
 * mxfp4_oracle.c -- plain, slow CPU oracle for H16/H32 + MXFP4 linear-layer GEMMs.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code, header,
 * table or constant with the CUDA path and must never be used as a fallback for it.
 *
 * Sources (web pages, cited by title and section):
 *   [MXFP4-HW]  "Pretraining Large Language Models with MXFP4 on Native FP4 Hardware"
 *               (arXiv:2605.09825): summary ("how it is done"), A.1 "MXFP4 and
 *               micro-scaling", A.2 "Hadamard transform architecture",
 *               C "mathematical cancellation" (C.1 Fprop, C.2 Dgrad, C.3 Wgrad),
 *               D "1D and 2D quantisation strategies".
 *   [DECOMP]    "Decomposing MXFP4 quantization error for LLM reinforcement learning":
 *               "pain point" (E8M0 scale, E2M1 grid), "core insight" (ideal-scale
 *               quantiser), "experiments" (QDQ numerically equal to native MXFP4:
 *               same grid, same E8M0 block scale, FP32 accumulation).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - shared exponent: OCP MX rule e = floor(log2 amax) - 2 (default) or the
 *     ceiling rule "smallest e with 6 * 2^e >= amax" (mode 1), clamped to the
 *     E8M0 range [-127, 127]; amax == 0 gives e = -127;
 *   - Q_FP4 = nearest E2M1 grid value, ties to the code with an even mantissa bit,
 *     magnitudes beyond 6 saturate to 6, the sign of zero is kept;
 *   - the rotation is evaluated in fp32 by the Sylvester recursion
 *     H_2n [a; b] = [H_n a + H_n b ; H_n a - H_n b] (every add rounded to fp32),
 *     followed by one fp32 multiply by 1/sqrt(n); the quantiser consumes fp32;
 *   - Hadamard blocks are contiguous along the rotated dimension, starting at 0.
 *
 * Everything here is written as loops over the definitions; OpenMP only splits
 * independent rows across threads (no reordering inside a computation).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* bf16 is the upper 16 bits of an IEEE binary32. */
static float bf16_to_float(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* E2M1 magnitudes indexed by the 3-bit code (exponent bits, mantissa bit):
 * [DECOMP] "pain point": grid {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6}. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Q_FP4 ([MXFP4-HW] A.1): nearest grid value by exhaustive distance search.
 * Ties go to the code whose mantissa bit (lowest code bit) is 0.  Returns the
 * 4-bit code: sign in bit 3, magnitude index in bits 0..2. */
int oracle_e2m1_code(double u) {
    int sign = signbit(u) ? 1 : 0;
    double a = fabs(u);
    /* saturation: every magnitude beyond the largest grid value maps to it (this also
     * keeps huge |u| away from the distance search, where a - 6 would round to a) */
    if (a >= E2M1_MAG[7]) return (sign << 3) | 7;
    int best = 0;
    double best_d = fabs(a - E2M1_MAG[0]);
    for (int c = 1; c < 8; ++c) {
        double d = fabs(a - E2M1_MAG[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (sign << 3) | best;
}

double oracle_e2m1_value(int code) {
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* Shared block exponent e (E8M0 stores e + 127).
 * mode 0 (OCP floor): e = floor(log2 amax) - 2, i.e. the largest e with
 *                     2^(e+2) <= amax ([MXFP4-HW] A.1, OCP MX convention).
 * mode 1 (ceiling):   smallest e with 6 * 2^e >= amax, so that the E8M0 scale is
 *                     never below the ideal scale amax / 6 ([DECOMP] "core insight").
 * Both clamped to [-127, 127]; amax == 0 gives -127. */
static int shared_exponent_f64(double amax, int mode);

int oracle_shared_exponent(float amax_f, int mode) { return shared_exponent_f64((double)amax_f, mode); }

/* The same rule for any non-negative fp64 amax (the fp32 entry point widens exactly). */
static int shared_exponent_f64(double amax, int mode) {
    if (!(amax > 0.0)) return -127;
    int ex;
    frexp(amax, &ex);              /* amax = f * 2^ex, f in [0.5, 1) */
    int flog2 = ex - 1;            /* floor(log2 amax), exact */
    int e;
    if (mode == 0) {
        e = flog2 - 2;
    } else {
        e = flog2 - 3;
        while (ldexp(6.0, e) < amax) e += 1;
        while (ldexp(6.0, e - 1) >= amax) e -= 1;
    }
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

int oracle_scale_byte(float amax, int mode) { return oracle_shared_exponent(amax, mode) + 127; }

/* ------------------------------------------------------------------------- */
/* Hadamard rotation                                                          */
/* ------------------------------------------------------------------------- */

/* Sylvester construction H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]] written out
 * as an explicit +-1 matrix, row-major n x n ([MXFP4-HW] A.2). */
void oracle_hadamard_pm1(int n, int8_t* h) {
    h[0] = 1;
    for (int m = 1; m < n; m *= 2) {
        for (int i = 0; i < m; ++i)
            for (int j = 0; j < m; ++j) {
                int8_t v = h[i * n + j];
                h[i * n + (j + m)] = v;
                h[(i + m) * n + j] = v;
                h[(i + m) * n + (j + m)] = (int8_t)-v;
            }
    }
}

/* fp32 constant 1/sqrt(n) that normalises H_n so that H H^T = I. */
static float norm_const(int n) {
    if (n == 1) return 1.0f;
    return (float)(1.0 / sqrt((double)n));
}

/* H_n x by the Sylvester recursion, every add/sub rounded to fp32. */
static void sylvester_apply_f32(float* v, int n) {
    if (n == 1) return;
    int h = n / 2;
    sylvester_apply_f32(v, h);
    sylvester_apply_f32(v + h, h);
    for (int i = 0; i < h; ++i) {
        float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
    }
}

/* Canonical fp32 rotation of a contiguous vector of length len (len % n == 0):
 * each block of n is replaced by fl32(fl32(H_n x) * fl32(1/sqrt(n))). n = 1 is
 * the identity ("none"). */
void oracle_rotate_f32(const float* x, int64_t len, int n, float* out) {
    float c = norm_const(n);
    for (int64_t b = 0; b < len; b += n) {
        float blk[64];
        for (int i = 0; i < n; ++i) blk[i] = x[b + i];
        sylvester_apply_f32(blk, n);
        for (int i = 0; i < n; ++i) out[b + i] = blk[i] * c;
    }
}

/* Exact rotation in fp64 by explicit matrix-vector products with the +-1 matrix
 * divided by sqrt(n): used for the cancellation identities and diagnostics. */
void oracle_rotate_f64(const double* x, int64_t len, int n, double* out) {
    int8_t h[32 * 32];
    oracle_hadamard_pm1(n, h);
    double c = 1.0 / sqrt((double)n);
    for (int64_t b = 0; b < len; b += n)
        for (int i = 0; i < n; ++i) {
            double s = 0.0;
            for (int j = 0; j < n; ++j) s += (double)h[i * n + j] * x[b + j];
            out[b + i] = s * c;
        }
}

/* ------------------------------------------------------------------------- */
/* MXFP4 quantisation of 32-element blocks                                    */
/* ------------------------------------------------------------------------- */

/* Quantise one 32-element block of already-rotated fp32 values with exponent e:
 * code_i = Q_FP4(v_i / 2^e) ([MXFP4-HW] A.1 reconstruction formula). */
static void quantize_block(const float* v, int e, uint8_t* codes /*32 nibble codes, one per byte*/) {
    for (int i = 0; i < 32; ++i) {
        double u = ldexp((double)v[i], -e);
        codes[i] = (uint8_t)oracle_e2m1_code(u);
    }
}

static float block_amax(const float* v, int n) {
    float m = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > m) m = a;
    }
    return m;
}

/* Store nibble code c for element index i of a packed row (2 per byte, element
 * 2j in the low nibble of byte j). */
static void put_nibble(uint8_t* row, int64_t i, uint8_t c) {
    uint8_t* b = row + i / 2;
    if (i % 2 == 0) *b = (uint8_t)((*b & 0xF0) | (c & 0xF));
    else *b = (uint8_t)((*b & 0x0F) | ((c & 0xF) << 4));
}

/* Quantise a contiguous vector of len bf16 values (len % 32 == 0) along itself:
 * rotate by H_n blocks, then one E8M0 scale per 32 elements.
 * codes: len/2 bytes; scales: len/32 bytes. */
void oracle_quantize_vec(const uint16_t* x, int64_t stride, int64_t len, int had, int mode,
                         uint8_t* codes, uint8_t* scales) {
    float* xf = (float*)malloc(sizeof(float) * (size_t)len);
    float* v = (float*)malloc(sizeof(float) * (size_t)len);
    for (int64_t i = 0; i < len; ++i) xf[i] = bf16_to_float(x[i * stride]);
    oracle_rotate_f32(xf, len, had, v);
    for (int64_t b = 0; b < len / 32; ++b) {
        const float* blk = v + b * 32;
        int e = oracle_shared_exponent(block_amax(blk, 32), mode);
        uint8_t q[32];
        quantize_block(blk, e, q);
        for (int i = 0; i < 32; ++i) put_nibble(codes, b * 32 + i, q[i]);
        scales[b] = (uint8_t)(e + 127);
    }
    free(xf);
    free(v);
}

/* 1x32 row-wise layout ([MXFP4-HW] D): x is [R, C] (leading dim ld elements);
 * each row is rotated and quantised along C.  codes [R, C/2], scales [R, C/32]. */
void oracle_quantize_row(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                         uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        oracle_quantize_vec(x + r * ld, 1, C, had, mode, codes + r * (C / 2), scales + r * (C / 32));
}

/* 32x1 column-wise layout, stored transposed ([MXFP4-HW] D): output row c is
 * column c of x, rotated and quantised along R.  codes [C, R/2], scales [C, R/32]. */
void oracle_quantize_colT(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                          uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; ++c)
        oracle_quantize_vec(x + c, ld, R, had, mode, codes + c * (R / 2), scales + c * (R / 32));
}

/* 32x32 2D layout ([MXFP4-HW] D): rotation along C, one E8M0 scale per 32x32
 * tile taken from the amax of the tile's rotated values.
 * codes [R, C/2], scales [R/32, C/32]. */
void oracle_quantize_2d(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                        uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t tr = 0; tr < R / 32; ++tr) {
        float* xf = (float*)malloc(sizeof(float) * (size_t)C);
        float* v = (float*)malloc(sizeof(float) * 32 * (size_t)C);
        for (int i = 0; i < 32; ++i) {
            for (int64_t c = 0; c < C; ++c) xf[c] = bf16_to_float(x[(tr * 32 + i) * ld + c]);
            oracle_rotate_f32(xf, C, had, v + (int64_t)i * C);
        }
        for (int64_t tc = 0; tc < C / 32; ++tc) {
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = block_amax(v + (int64_t)i * C + tc * 32, 32);
                if (a > amax) amax = a;
            }
            int e = oracle_shared_exponent(amax, mode);
            scales[tr * (C / 32) + tc] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i) {
                uint8_t q[32];
                quantize_block(v + (int64_t)i * C + tc * 32, e, q);
                uint8_t* row = codes + (tr * 32 + i) * (C / 2);
                for (int j = 0; j < 32; ++j) put_nibble(row, tc * 32 + j, q[j]);
            }
        }
        free(xf);
        free(v);
    }
}

/* Dequantise a row-layout tensor: out[r][k] = 2^e(r, k/32) * value(code). */
void oracle_dequant_row(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t C, double* out) {
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < C; ++k) {
            uint8_t b = codes[r * (C / 2) + k / 2];
            int c = (k % 2 == 0) ? (b & 0xF) : (b >> 4);
            int e = (int)scales[r * (C / 32) + k / 32] - 127;
            out[r * C + k] = ldexp(oracle_e2m1_value(c), e);
        }
}

/* ------------------------------------------------------------------------- */
/* Block-scaled GEMM (QDQ semantics, [DECOMP] "experiments")                 */
/* ------------------------------------------------------------------------- */

static int twice_value(const uint8_t* row, int64_t k) {
    /* 2 * E2M1 value is an integer in [-12, 12]. */
    static const int TW[8] = {0, 1, 2, 3, 4, 6, 8, 12};
    uint8_t b = row[k / 2];
    int c = (k % 2 == 0) ? (b & 0xF) : (b >> 4);
    int m = TW[c & 7];
    return (c & 8) ? -m : m;
}

/* One output element: sum over 32-blocks of 2^(ea+eb) * sum_k qa_k * qb_k.  The
 * inner sum is an exact integer; block terms are summed in fp64 in k order.
 * Also returns s = sum_k |dq a_k| |dq b_k| (fp64) for the tolerance. */
static void dot_one(const uint8_t* ca, const uint8_t* sa, const uint8_t* cb, const uint8_t* sb, int64_t K,
                    double* c_out, double* s_out) {
    double acc = 0.0, sacc = 0.0;
    for (int64_t blk = 0; blk < K / 32; ++blk) {
        long isum = 0, iabs = 0;
        for (int64_t k = blk * 32; k < blk * 32 + 32; ++k) {
            int a = twice_value(ca, k), b = twice_value(cb, k);
            isum += (long)a * b;
            iabs += (long)abs(a) * abs(b);
        }
        int e = ((int)sa[blk] - 127) + ((int)sb[blk] - 127);
        acc += ldexp((double)isum / 4.0, e);
        sacc += ldexp((double)iabs / 4.0, e);
    }
    *c_out = acc;
    if (s_out) *s_out = sacc;
}

/* C[m][n] = sum_k dq(A)[m][k] * dq(B)[n][k] for A [M,K], B [N,K] in row layout with
 * plain scales (codes [rows, K/2], scales [rows, K/32]). */
void oracle_gemm(const uint8_t* ca, const uint8_t* sa, const uint8_t* cb, const uint8_t* sb, int64_t M,
                 int64_t N, int64_t K, double* C, double* S) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            dot_one(ca + m * (K / 2), sa + m * (K / 32), cb + n * (K / 2), sb + n * (K / 32), K, &C[m * N + n],
                    S ? &S[m * N + n] : 0);
}

/* The same for a list of (row of A, row of B) pairs taken from separately
 * quantised single rows: a_rows [P, K/2] codes + [P, K/32] scales, likewise b. */
void oracle_dot_pairs(const uint8_t* ca, const uint8_t* sa, const uint8_t* cb, const uint8_t* sb, int64_t P,
                      int64_t K, double* C, double* S) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < P; ++p)
        dot_one(ca + p * (K / 2), sa + p * (K / 32), cb + p * (K / 2), sb + p * (K / 32), K, &C[p], S ? &S[p] : 0);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------- */
/* Error decomposition ([DECOMP] "core insight", property 1)                 */
/* ------------------------------------------------------------------------- */

/* Round |u| (a real number, given in fp64) to the E2M1 grid with the same rule as
 * oracle_e2m1_code; returns the signed grid value. */
static double grid_round(double u) { return oracle_e2m1_value(oracle_e2m1_code(u)); }

/* For x [R, C] (bf16, ld elements per row), quantised row-wise (rotation along C):
 * per 32-block, with the E8M0 scale s_b of `mode` and the ideal scale s* = amax/6,
 *   Q(x)  = s_b * grid(x / s_b)          (the MXFP4 value)
 *   Q*(x) = s*  * grid(x / s*)           (ideal-scale quantiser)
 *   e_scale = Q - Q*, e_DZ = (Q* - x) on the deadzone |x| < amax/24, e_grid = (Q* - x) off it.
 * out[0..6] = sum e^2, sum e_scale^2, sum e_DZ^2, sum e_grid^2, sum e_scale*e_grid,
 *             number of deadzone elements, number of elements (all in fp64). */
void oracle_error_decomposition(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                                double* out) {
    double acc[7] = {0, 0, 0, 0, 0, 0, 0};
#pragma omp parallel
    {
        double loc[7] = {0, 0, 0, 0, 0, 0, 0};
        float* xf = (float*)malloc(sizeof(float) * (size_t)C);
        float* v = (float*)malloc(sizeof(float) * (size_t)C);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            for (int64_t c = 0; c < C; ++c) xf[c] = bf16_to_float(x[r * ld + c]);
            oracle_rotate_f32(xf, C, had, v);
            for (int64_t b = 0; b < C / 32; ++b) {
                const float* blk = v + b * 32;
                float amax_f = block_amax(blk, 32);
                int e = oracle_shared_exponent(amax_f, mode);
                double amax = (double)amax_f;
                double sstar = amax / 6.0;
                for (int i = 0; i < 32; ++i) {
                    double xv = (double)blk[i];
                    double q = ldexp(grid_round(ldexp(xv, -e)), e);
                    double qs = sstar > 0.0 ? sstar * grid_round(xv / sstar) : 0.0;
                    int dz = fabs(xv) < amax / 24.0;
                    double es = q - qs, ed = dz ? qs - xv : 0.0, eg = dz ? 0.0 : qs - xv, et = q - xv;
                    loc[0] += et * et;
                    loc[1] += es * es;
                    loc[2] += ed * ed;
                    loc[3] += eg * eg;
                    loc[4] += es * eg;
                    loc[5] += dz;
                    loc[6] += 1.0;
                }
            }
        }
#pragma omp critical
        for (int k = 0; k < 7; ++k) acc[k] += loc[k];
        free(xf);
        free(v);
    }
    for (int k = 0; k < 7; ++k) out[k] = acc[k];
}

/* ------------------------------------------------------------------------- */
/* Quantiser fixes ([DECOMP] "three fixes": OF and MBS)                       */
/* ------------------------------------------------------------------------- */

/* Quantise len fp32 values (len % 32 == 0) block by block as they are (no
 * rotation): codes (packed nibbles) and E8M0 bytes. */
static void quantize_f32_vec(const float* v, int64_t len, int mode, uint8_t* codes, uint8_t* scales) {
    for (int64_t b = 0; b < len / 32; ++b) {
        const float* blk = v + b * 32;
        int e = oracle_shared_exponent(block_amax(blk, 32), mode);
        uint8_t q[32];
        quantize_block(blk, e, q);
        for (int i = 0; i < 32; ++i) put_nibble(codes, b * 32 + i, q[i]);
        scales[b] = (uint8_t)(e + 127);
    }
}

/* The same for R rows of C fp32 values: codes [R, C/2], scales [R, C/32]. */
void oracle_quantize_f32_rows(const float* v, int64_t R, int64_t C, int mode, uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) quantize_f32_vec(v + r * C, C, mode, codes + r * (C / 2), scales + r * (C / 32));
}

static void rotated_row(const uint16_t* x, int64_t len, int had, float* xf, float* v) {
    for (int64_t i = 0; i < len; ++i) xf[i] = bf16_to_float(x[i]);
    oracle_rotate_f32(xf, len, had, v);
}

/* Value of nibble code c of element i of a packed row times 2^e, in fp64. */
static double dq_elem(const uint8_t* row, int64_t i, int e) {
    uint8_t b = row[i / 2];
    int c = (i % 2 == 0) ? (b & 0xF) : (b >> 4);
    return ldexp(oracle_e2m1_value(c), e);
}

/* OF ([DECOMP] "OF -- outlier fallback, with residual weight alpha"):
 *   x1 = Q(x),  x2 = Q(x - x1),  x_OF = x1 + alpha * x2,
 * with Q the row quantiser acting on the rotated row (1x32 blocks along C).  The
 * residual x - dq(x1) is formed in fp64; it is exactly representable in fp32 (the
 * return value counts the values for which it was not, expected 0) and the second
 * pass quantises it as an fp32 vector.  alpha = 2^alpha_log2 (alpha_log2 <= 0; the
 * pages settle on 0.5) is carried exactly by the second pass's E8M0 bytes: stored
 * byte = max(byte + alpha_log2, 0), so a block whose residual amax is below 2^-125
 * keeps byte 0 (weight 1 instead of alpha).  Then x_OF = dq(q1) + dq(q2). */
int64_t oracle_quantize_of_row(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                               int alpha_log2, uint8_t* codes1, uint8_t* scales1, uint8_t* codes2,
                               uint8_t* scales2) {
    int64_t inexact = 0;
#pragma omp parallel for schedule(static) reduction(+ : inexact)
    for (int64_t r = 0; r < R; ++r) {
        float* xf = (float*)malloc(sizeof(float) * (size_t)C);
        float* v = (float*)malloc(sizeof(float) * (size_t)C);
        float* res = (float*)malloc(sizeof(float) * (size_t)C);
        uint8_t* c1 = codes1 + r * (C / 2);
        uint8_t* s1 = scales1 + r * (C / 32);
        rotated_row(x + r * ld, C, had, xf, v);
        quantize_f32_vec(v, C, mode, c1, s1);
        for (int64_t i = 0; i < C; ++i) {
            double d = (double)v[i] - dq_elem(c1, i, (int)s1[i / 32] - 127);
            res[i] = (float)d;
            if ((double)res[i] != d) ++inexact;
        }
        uint8_t* s2 = scales2 + r * (C / 32);
        quantize_f32_vec(res, C, mode, codes2 + r * (C / 2), s2);
        for (int64_t b = 0; b < C / 32; ++b) {
            int sb = (int)s2[b] + alpha_log2;
            s2[b] = (uint8_t)(sb < 0 ? 0 : sb);
        }
        free(xf);
        free(v);
        free(res);
    }
    return inexact;
}

/* MBS byte of a macro block with amax A ([DECOMP] "MBS -- macro block scaling":
 * scale 2^e_M * (1 + m), m in [0, 1), 8 bits of mantissa).  Reading (the pages do
 * not say how m is chosen): write A = f * 2^E with f in [1, 2) and let T = 1.5 if
 * f <= 1.5, else 3; k is the largest value in 0..255 with (1 + k/256) * f <= T, i.e.
 * the largest 8-bit correction that does not lift the macro-block maximum above the
 * top grid value 6 of its E8M0 scale.  A == 0 or subnormal: k = 0.  By scanning k. */
int oracle_mbs_byte(float A) {
    if (!(A >= FLT_MIN)) return 0;
    int E;
    double f = frexp((double)A, &E) * 2.0; /* in [1, 2) */
    double T = (f <= 1.5) ? 1.5 : 3.0;
    for (int k = 255; k >= 0; --k)
        if ((1.0 + k / 256.0) * f <= T) return k;
    return 0;
}

/* MBS quantiser, row layout: per macro block of 128 consecutive rotated values (four
 * 32-blocks) one byte k = oracle_mbs_byte(macro amax); the values are prescaled,
 * x' = fl32((1 + k/256) * x), and quantised by Q (32-blocks, `mode`); the
 * reconstruction is dq(q) / (1 + k/256).  codes [R, C/2], scales [R, C/32],
 * mbs [R, C/128]; C % 128 == 0. */
void oracle_quantize_mbs_row(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                             uint8_t* codes, uint8_t* scales, uint8_t* mbs) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        float* xf = (float*)malloc(sizeof(float) * (size_t)C);
        float* v = (float*)malloc(sizeof(float) * (size_t)C);
        rotated_row(x + r * ld, C, had, xf, v);
        for (int64_t mb = 0; mb < C / 128; ++mb) {
            float* blk = v + mb * 128;
            int k = oracle_mbs_byte(block_amax(blk, 128));
            float mul = 1.0f + (float)k / 256.0f;
            for (int i = 0; i < 128; ++i) blk[i] = blk[i] * mul;
            mbs[r * (C / 128) + mb] = (uint8_t)k;
        }
        quantize_f32_vec(v, C, mode, codes + r * (C / 2), scales + r * (C / 32));
        free(xf);
        free(v);
    }
}

/* MBS reconstruction: out[r][i] = dq(code) / (1 + k/256). */
void oracle_dequant_mbs_row(const uint8_t* codes, const uint8_t* scales, const uint8_t* mbs, int64_t R, int64_t C,
                            double* out) {
    for (int64_t r = 0; r < R; ++r)
        for (int64_t i = 0; i < C; ++i) {
            double q = dq_elem(codes + r * (C / 2), i, (int)scales[r * (C / 32) + i / 32] - 127);
            out[r * C + i] = q / (1.0 + mbs[r * (C / 128) + i / 128] / 256.0);
        }
}

/* GEMM over MBS operands ([DECOMP] "MBS": x_hat = Q((1 + m) x) / (1 + m), the postscale
 * applied to each macro block of 128 consecutive elements along the quantised, i.e. the
 * contraction, dimension): C[m][n] = sum over macro blocks kb of
 *   f_A[m][kb] f_B[n][kb] * sum_{k in kb} dq(A)[m][k] dq(B)[n][k],
 * f = 1 / (1 + byte / 256) (f = 1 where mbs_a / mbs_b is NULL: that operand is plain
 * MXFP4).  The inner sums are those of oracle_gemm (exact integers per 32-block); the
 * factors and sums are fp64.  S[m][n] = sum_k |x_hat_a| |x_hat_b|.  K % 128 == 0. */
void oracle_gemm_mbs(const uint8_t* ca, const uint8_t* sa, const uint8_t* mbs_a, const uint8_t* cb,
                     const uint8_t* sb, const uint8_t* mbs_b, int64_t M, int64_t N, int64_t K, double* C, double* S) {
    const int64_t nkb = K / 128;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, sacc = 0.0;
            for (int64_t kb = 0; kb < nkb; ++kb) {
                double part, spart;
                dot_one(ca + m * (K / 2) + kb * 64, sa + m * (K / 32) + kb * 4, cb + n * (K / 2) + kb * 64,
                        sb + n * (K / 32) + kb * 4, 128, &part, &spart);
                const double fa = mbs_a ? 1.0 / (1.0 + mbs_a[m * nkb + kb] / 256.0) : 1.0;
                const double fb = mbs_b ? 1.0 / (1.0 + mbs_b[n * nkb + kb] / 256.0) : 1.0;
                acc += fa * fb * part;
                sacc += fa * fb * spart;
            }
            C[m * N + n] = acc;
            if (S) S[m * N + n] = sacc;
        }
}

/* ------------------------------------------------------------------------- */
/* Randomised baselines ([MXFP4-HW] A.2 and "experiments", table 1: random sign */
/* flips before the Hadamard, stochastic rounding)                             */
/* ------------------------------------------------------------------------- */

/* Stochastic rounding of u (the fp32 value v * 2^-e, |u| < 8) to the E2M1 grid with
 * the uniform 16-bit integer r: below 6 the magnitude a lies in [lo, lo + step) with
 * step 0.5 on [0, 2), 1 on [2, 4), 2 on [4, 6); it rounds up with probability
 * p = (a - lo) / step, i.e. iff r < p * 65536.  a >= 6 saturates to 6.  The sign is
 * kept (a zero keeps its sign).  All of lo, a - lo, p and p * 65536 are exact in
 * fp32, so the decision is the same in any precision.  Returns the 4-bit code. */
int oracle_e2m1_code_sr(float u, uint16_t r) {
    float a = fabsf(u);
    double mag;
    if (a >= 6.0f) {
        mag = 6.0;
    } else {
        double step = a < 2.0f ? 0.5 : (a < 4.0f ? 1.0 : 2.0);
        double lo = floor((double)a / step) * step;
        double p = ((double)a - lo) / step;
        mag = lo + (((double)r < p * 65536.0) ? step : 0.0);
    }
    int code = oracle_e2m1_code(mag); /* mag is a grid value: its own code */
    if (signbit(u)) code |= 8;
    return code;
}

/* Quantise a contiguous vector of len bf16 values (element i at x[i*stride]) along
 * itself, with optional random signs and stochastic rounding:
 *   signs: NULL or a bitmask over the vector's indices (bit i set: x_i negated before
 *          the rotation, the random-sign Hadamard H D x);
 *   sr:    NULL (round to nearest even) or one uniform 16-bit integer per element.
 * The E8M0 scale is taken as in oracle_quantize_vec. */
void oracle_quantize_vec_rand(const uint16_t* x, int64_t stride, int64_t len, int had, int mode, const uint8_t* signs,
                              const uint16_t* sr, uint8_t* codes, uint8_t* scales) {
    float* xf = (float*)malloc(sizeof(float) * (size_t)len);
    float* v = (float*)malloc(sizeof(float) * (size_t)len);
    for (int64_t i = 0; i < len; ++i) {
        xf[i] = bf16_to_float(x[i * stride]);
        if (signs && ((signs[i / 8] >> (i % 8)) & 1)) xf[i] = -xf[i];
    }
    oracle_rotate_f32(xf, len, had, v);
    for (int64_t b = 0; b < len / 32; ++b) {
        const float* blk = v + b * 32;
        int e = oracle_shared_exponent(block_amax(blk, 32), mode);
        for (int i = 0; i < 32; ++i) {
            int c;
            if (sr) {
                float u = (float)ldexp((double)blk[i], -e); /* one rounding: fl32(v * 2^-e) */
                c = oracle_e2m1_code_sr(u, sr[b * 32 + i]);
            } else {
                c = oracle_e2m1_code(ldexp((double)blk[i], -e));
            }
            put_nibble(codes, b * 32 + i, (uint8_t)c);
        }
        scales[b] = (uint8_t)(e + 127);
    }
    free(xf);
    free(v);
}

/* Row layout with the randomised options: col_signs over C, sr [R, C] (row-major). */
void oracle_quantize_row_rand(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                              const uint8_t* col_signs, const uint16_t* sr, uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        oracle_quantize_vec_rand(x + r * ld, 1, C, had, mode, col_signs, sr ? sr + r * C : 0, codes + r * (C / 2),
                                 scales + r * (C / 32));
}

/* Column layout (stored transposed) with row_signs over R and sr [C, R]. */
void oracle_quantize_colT_rand(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                               const uint8_t* row_signs, const uint16_t* sr, uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; ++c)
        oracle_quantize_vec_rand(x + c, ld, R, had, mode, row_signs, sr ? sr + c * R : 0, codes + c * (R / 2),
                                 scales + c * (R / 32));
}

/* ------------------------------------------------------------------------- */
/* Counter-based random numbers for the randomised baselines                  */
/* ------------------------------------------------------------------------- */

/* Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
 * 1, 2, 3", SC'11), written from its published definition.  A 128-bit counter
 * (c0, c1, c2, c3) and a 64-bit key (k0, k1) give four 32-bit outputs after ten rounds.
 * One round: the 64-bit products M0 * c0 and M1 * c2 (M0 = 0xD2511F53,
 * M1 = 0xCD9E8D57) with high words h0, h1 and low words l0, l1 give the new counter
 * (h1 ^ c1 ^ k0, l1, h0 ^ c3 ^ k1, l0).  The key is bumped by the Weyl constants
 * (k0 += 0x9E3779B9, k1 += 0xBB67AE85) between rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c[0];
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
        const uint32_t h0 = (uint32_t)(p0 >> 32), l0 = (uint32_t)p0;
        const uint32_t h1 = (uint32_t)(p1 >> 32), l1 = (uint32_t)p1;
        const uint32_t n0 = h1 ^ c[1] ^ k0, n2 = h0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = l1;
        c[2] = n2;
        c[3] = l0;
    }
    for (int i = 0; i < 4; ++i) out[i] = c[i];
}

/* The random-sign vector of one dimension, from the 64-bit seed of that dimension:
 * sign bit j is bit (j % 32) of output word (j % 128) / 32 of Philox4x32-10 with counter
 * (j / 128, 0, 0, 0) and key (seed low word, seed high word).  bits: (n + 7) / 8 bytes,
 * bit j in bit j % 8 of byte j / 8 (set = negate), the layout of the sign masks above.
 * The operands of a GEMM share the vector of their contraction when they share its seed. */
void oracle_philox_signs(uint64_t seed, int64_t n, uint8_t* bits) {
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    memset(bits, 0, (size_t)((n + 7) / 8));
    for (int64_t j = 0; j < n; ++j) {
        const uint32_t ctr[4] = {(uint32_t)(j / 128), 0u, 0u, 0u};
        uint32_t o[4];
        oracle_philox4x32_10(ctr, key, o);
        if ((o[(j % 128) / 32] >> (j % 32)) & 1u) bits[j / 8] |= (uint8_t)(1u << (j % 8));
    }
}

/* Stochastic-rounding integers of one quantised copy, lines x len of them (line = the
 * row of the stored copy, position = the index along the quantised dimension): the
 * integer of (line l, position i) is 16-bit half (i % 8) of Philox4x32-10 with counter
 * (i / 8, l, copy, 0) and key (seed low, seed high) -- half h is bits 16 (h % 2) ..
 * 16 (h % 2) + 15 of output word h / 2.  copy: 0 the row copy, 1 the transposed copy.
 * out: lines * len uint16, row-major. */
void oracle_philox_sr(uint64_t seed, int64_t lines, int64_t len, uint32_t copy, uint16_t* out) {
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
#pragma omp parallel for schedule(static)
    for (int64_t l = 0; l < lines; ++l)
        for (int64_t i = 0; i < len; ++i) {
            const uint32_t ctr[4] = {(uint32_t)(i / 8), (uint32_t)l, copy, 0u};
            uint32_t o[4];
            oracle_philox4x32_10(ctr, key, o);
            const int h = (int)(i % 8);
            out[l * len + i] = (uint16_t)(o[h / 2] >> (16 * (h % 2)));
        }
}

/* ------------------------------------------------------------------------- */
/* Diagnostic: canonical fp32 rotation against the exact rotation             */
/* ------------------------------------------------------------------------- */

/* The pages fix the rotation only in exact arithmetic ([MXFP4-HW] A.2); the quantiser
 * takes the canonical fp32 order.  For x [R, C] (row layout, blocks of 32 along C) this
 * counts the blocks whose E8M0 byte or codes would change if the exact rotation -- fp64
 * products with the +-1 matrix divided by sqrt(n) -- were quantised instead: amax of
 * the exact values, the same exponent rule, codes of v / 2^e by the same nearest-grid
 * search.  out[0] = blocks that differ, out[1] = blocks whose byte differs,
 * out[2] = blocks.  A diagnostic of the canonical order, not a failure. */
void oracle_rotation_divergence(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                                int64_t* out) {
    int64_t differ = 0, byte_differ = 0;
#pragma omp parallel for schedule(static) reduction(+ : differ, byte_differ)
    for (int64_t r = 0; r < R; ++r) {
        float* xf = (float*)malloc(sizeof(float) * (size_t)C);
        float* v = (float*)malloc(sizeof(float) * (size_t)C);
        double* xd = (double*)malloc(sizeof(double) * (size_t)C);
        double* vd = (double*)malloc(sizeof(double) * (size_t)C);
        for (int64_t c = 0; c < C; ++c) {
            xf[c] = bf16_to_float(x[r * ld + c]);
            xd[c] = (double)xf[c];
        }
        oracle_rotate_f32(xf, C, had, v);
        oracle_rotate_f64(xd, C, had, vd);
        for (int64_t b = 0; b < C / 32; ++b) {
            const float* blk = v + b * 32;
            const double* bd = vd + b * 32;
            const int e = oracle_shared_exponent(block_amax(blk, 32), mode);
            double amax = 0.0;
            for (int i = 0; i < 32; ++i)
                if (fabs(bd[i]) > amax) amax = fabs(bd[i]);
            const int ex = shared_exponent_f64(amax, mode);
            uint8_t q[32];
            quantize_block(blk, e, q);
            int same = ex == e;
            for (int i = 0; i < 32 && same; ++i) same = oracle_e2m1_code(ldexp(bd[i], -ex)) == q[i];
            differ += !same;
            byte_differ += ex != e;
        }
        free(xf);
        free(v);
        free(xd);
        free(vd);
    }
    out[0] = differ;
    out[1] = byte_differ;
    out[2] = R * (C / 32);
}
