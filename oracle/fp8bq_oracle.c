/*
 * Plain CPU oracle for the block-scaled FP8 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * What it follows.  The Puro-2B technical report ("Puro-2B: pretraining for
 * an ordinary lab", section 2 "FP8") says the main linear layers run their
 * matrix multiplications in FP8 following DeepSeek-V3's fine-grained block
 * quantization, with numerically sensitive work left in BF16/FP32; the German
 * write-up of the same report (36kr, FP8 section) says the same.  The pages
 * print no formula, so the numerical contract is the one the project fixes:
 * activations/gradients are quantized per 1x128 tile and weights per 128x128
 * block to E4M3 with an FP32 scale s = amax/448 (s = 1 when amax = 0),
 * round-to-nearest-even with saturation at +-448; the GEMMs accumulate each
 * 128-wide reduction chunk, multiply it by the product of the two scales of
 * that chunk and sum the chunks; the output is BF16.
 *
 * E4M3 itself is the OCP 8-bit floating point format ("FP8 Formats for Deep
 * Learning", Micikevicius et al. 2022): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite
 * magnitude 448, subnormals m * 2^-9.
 *
 * Arithmetic rules: compiled without fast-math, without FMA contraction and
 * without flush-to-zero, so every float operation written here is one
 * correctly rounded IEEE-754 binary32 (or binary64) operation.
 *
 * Every function is deliberately slow and direct.  OpenMP (if enabled at
 * compile time) only splits independent outer loops across cores.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* E4M3 codec                                                               */
/* ------------------------------------------------------------------------ */

/* Decode one E4M3 code straight from the format definition (OCP FP8, E4M3:
 * exponent bias 7, exponent field 0 = subnormal m*2^-9, code x.1111.111 is
 * NaN).  Returns the exact value as a double. */
ORACLE_API double fp8bq_oracle_e4m3_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Encode a binary32 value to E4M3 by brute force: the non-negative finite
 * magnitudes are codes 0x00..0x7E; pick the one nearest to |v|, break an exact
 * tie toward the code whose least significant bit is 0 (round half to even),
 * clamp anything at or above the largest finite value to 448 (saturating
 * conversion), and copy the sign bit of v (so -0 and negative values that
 * round to zero give 0x80).  NaN gives 0x7F with the sign of v. */
ORACLE_API uint8_t fp8bq_oracle_e4m3_encode(float v) {
    uint32_t bits;
    memcpy(&bits, &v, 4);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    if (isnan(v)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(fp8bq_oracle_e4m3_decode((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* A second, independent encoder written from the arithmetic of the format
 * instead of a table search: find the binade of |v| (the subnormal range
 * shares the quantum of the lowest binade), divide by the quantum 2^(E-3),
 * round that integer to nearest with ties to even, and rebuild the code.
 * Used only to cross-check the brute-force encoder. */
ORACLE_API uint8_t fp8bq_oracle_e4m3_encode_arith(float v) {
    uint32_t bits;
    memcpy(&bits, &v, 4);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    if (isnan(v)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int E;
    if (a == 0.0) {
        E = -6;
    } else {
        int ex;
        frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) -> floor(log2 a) = ex - 1 */
        E = ex - 1;
        if (E < -6) E = -6;
    }
    double quantum = ldexp(1.0, E - 3);
    double r = a / quantum;           /* exact: a has 24 significant bits */
    double n = nearbyint(r);          /* default rounding mode: half to even */
    long k = (long)n;
    uint8_t code;
    if (E == -6 && k < 8) {
        code = (uint8_t)k;            /* subnormal: value k * 2^-9 */
    } else {
        int e = E + 7;
        if (k == 16) { k = 8; e += 1; }  /* rounded up into the next binade */
        code = (uint8_t)((e << 3) | (int)(k - 8));
    }
    if (code > 0x7E) code = 0x7E;     /* saturate (cannot exceed 448 here) */
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------------ */
/* Tile quantization                                                        */
/* ------------------------------------------------------------------------ */

/* Element fetch: dtype 0 = BF16 (raw 16-bit patterns, widened exactly by
 * placing them in the top half of a binary32), dtype 1 = FP32. */
static float load_elem(const void* x, int dtype, int64_t idx) {
    if (dtype == 0) {
        uint16_t h = ((const uint16_t*)x)[idx];
        uint32_t w = (uint32_t)h << 16;
        float f;
        memcpy(&f, &w, 4);
        return f;
    }
    return ((const float*)x)[idx];
}

/* The scale rule: s = amax / 448 in binary32, and s = 1 for an all-zero tile. */
ORACLE_API float fp8bq_oracle_tile_scale(float amax) {
    if (amax == 0.0f) return 1.0f;
    return amax / 448.0f;
}

/* Quantize one element of a tile whose scale is s: the quotient x / s is
 * formed as one correctly rounded binary32 division, then encoded. */
static uint8_t quantize_elem(float x, float s) {
    float y = x / s;
    return fp8bq_oracle_e4m3_encode(y);
}

/* Row-wise 1x128 quantization (activations for Fprop, output gradients for
 * Dgrad).  x is [R][C] with row pitch ldx elements; q is [R][C] contiguous;
 * s is [C/128][R]: for tile (r, t) covering x[r][128t .. 128t+127], the scale
 * is s[t*R + r]. */
ORACLE_API void fp8bq_oracle_quantize_rowwise(const void* x, int dtype, int64_t R, int64_t C,
                                              int64_t ldx, uint8_t* q, float* s) {
    int64_t T = C / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t t = 0; t < T; ++t) {
            float amax = 0.0f;
            for (int64_t j = 0; j < 128; ++j) {
                float a = fabsf(load_elem(x, dtype, r * ldx + t * 128 + j));
                if (a > amax) amax = a;
            }
            float sc = fp8bq_oracle_tile_scale(amax);
            s[t * R + r] = sc;
            for (int64_t j = 0; j < 128; ++j)
                q[r * C + t * 128 + j] = quantize_elem(load_elem(x, dtype, r * ldx + t * 128 + j), sc);
        }
    }
}

/* Column-wise 128x1 quantization, emitted transposed (inputs of Wgrad, which
 * reduces over tokens).  x is [M][C] with row pitch ldx; the tile (b, c) is
 * x[128b .. 128b+127][c]; qT is [C][M] with qT[c][m] the code of x[m][c];
 * s is [M/128][C] with s[b*C + c] the scale of tile (b, c). */
ORACLE_API void fp8bq_oracle_quantize_colwise(const void* x, int dtype, int64_t M, int64_t C,
                                              int64_t ldx, uint8_t* qT, float* s) {
    int64_t B = M / 128;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t b = 0; b < B; ++b) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i) {
                float a = fabsf(load_elem(x, dtype, (b * 128 + i) * ldx + c));
                if (a > amax) amax = a;
            }
            float sc = fp8bq_oracle_tile_scale(amax);
            s[b * C + c] = sc;
            for (int64_t i = 0; i < 128; ++i)
                qT[c * M + b * 128 + i] = quantize_elem(load_elem(x, dtype, (b * 128 + i) * ldx + c), sc);
        }
    }
}

/* Weight quantization per 128x128 block.  w is [N][K] (nn.Linear layout) with
 * row pitch ldw; q is [N][K]; qT (optional, may be NULL) is [K][N] holding the
 * same codes transposed; s is [N/128][K/128]. */
ORACLE_API void fp8bq_oracle_quantize_weight_block(const void* w, int dtype, int64_t N, int64_t K,
                                                   int64_t ldw, uint8_t* q, uint8_t* qT, float* s) {
    int64_t NB = N / 128, KB = K / 128;
#pragma omp parallel for schedule(static)
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    float a = fabsf(load_elem(w, dtype, (nb * 128 + i) * ldw + kb * 128 + j));
                    if (a > amax) amax = a;
                }
            float sc = fp8bq_oracle_tile_scale(amax);
            s[nb * KB + kb] = sc;
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    int64_t n = nb * 128 + i, k = kb * 128 + j;
                    uint8_t code = quantize_elem(load_elem(w, dtype, n * ldw + k), sc);
                    q[n * K + k] = code;
                    if (qT) qT[k * N + n] = code;
                }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Block-scaled GEMMs in binary64                                           */
/* ------------------------------------------------------------------------ */
/*
 * Each output is  sum over chunks c of  sA(c) * sB(c) * P_c  with
 * P_c = sum over the 128 reduction indices of chunk c of D(a) * D(b).
 * In binary64 every product of two E4M3 values and every 128-term chunk sum
 * is exact (a product has at most 8 significant bits and the products of one
 * chunk span far fewer than 53 bits), so the only roundings are the scale
 * multiplication and the sum over chunks, each at 2^-53 relative.
 *
 * Besides the value, each routine returns abs_sum = sum over all reduction
 * indices of |sA*D(a) * sB*D(b)|, the magnitude the error bound is scaled by.
 *
 * Outputs are computed only for the requested rows and columns (index lists),
 * so that large problems can be checked on sampled tiles; out_val and out_abs
 * are [n_rows][n_cols].
 */

/* Fprop: Y[m][n] = sum_c sx[c][m] * sw[n/128][c] * sum_{k in c} D(xq[m][k]) D(wq[n][k]).
 * xq [M][K], sx [K/128][M], wq [N][K], sw [N/128][K/128]. */
ORACLE_API void fp8bq_oracle_gemm_fprop(const uint8_t* xq, const float* sx, const uint8_t* wq,
                                        const float* sw, int64_t M, int64_t N, int64_t K,
                                        const int64_t* rows, int64_t n_rows, const int64_t* cols,
                                        int64_t n_cols, double* out_val, double* out_abs) {
    int64_t KC = K / 128;
#pragma omp parallel for schedule(dynamic)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t m = rows[ri];
        for (int64_t ci = 0; ci < n_cols; ++ci) {
            int64_t n = cols[ci];
            double total = 0.0, total_abs = 0.0;
            for (int64_t c = 0; c < KC; ++c) {
                double p = 0.0, pa = 0.0;
                for (int64_t k = c * 128; k < c * 128 + 128; ++k) {
                    double prod = fp8bq_oracle_e4m3_decode(xq[m * K + k]) * fp8bq_oracle_e4m3_decode(wq[n * K + k]);
                    p += prod;
                    pa += fabs(prod);
                }
                double scale = (double)sx[c * M + m] * (double)sw[(n / 128) * KC + c];
                total += scale * p;
                total_abs += scale * pa;
            }
            out_val[ri * n_cols + ci] = total;
            out_abs[ri * n_cols + ci] = total_abs;
        }
    }
}

/* Dgrad: dX[m][k] = sum_c sdy[c][m] * sw[c][k/128] * sum_{n in c} D(dyq[m][n]) D(wq[n][k]).
 * The reduction runs over the output features n; the weight is used in its
 * natural [N][K] layout (its block scale sw[n/128][k/128]).
 * dyq [M][N], sdy [N/128][M], wq [N][K], sw [N/128][K/128]. */
ORACLE_API void fp8bq_oracle_gemm_dgrad(const uint8_t* dyq, const float* sdy, const uint8_t* wq,
                                        const float* sw, int64_t M, int64_t N, int64_t K,
                                        const int64_t* rows, int64_t n_rows, const int64_t* cols,
                                        int64_t n_cols, double* out_val, double* out_abs) {
    int64_t NC = N / 128, KB = K / 128;
#pragma omp parallel for schedule(dynamic)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t m = rows[ri];
        for (int64_t ci = 0; ci < n_cols; ++ci) {
            int64_t k = cols[ci];
            double total = 0.0, total_abs = 0.0;
            for (int64_t c = 0; c < NC; ++c) {
                double p = 0.0, pa = 0.0;
                for (int64_t n = c * 128; n < c * 128 + 128; ++n) {
                    double prod = fp8bq_oracle_e4m3_decode(dyq[m * N + n]) * fp8bq_oracle_e4m3_decode(wq[n * K + k]);
                    p += prod;
                    pa += fabs(prod);
                }
                double scale = (double)sdy[c * M + m] * (double)sw[c * KB + k / 128];
                total += scale * p;
                total_abs += scale * pa;
            }
            out_val[ri * n_cols + ci] = total;
            out_abs[ri * n_cols + ci] = total_abs;
        }
    }
}

/* Wgrad: dW[n][k] = sum_c sdyT[c][n] * sxT[c][k] * sum_{m in c} D(dyqT[n][m]) D(xqT[k][m]).
 * The reduction runs over the tokens m; both operands come from the
 * column-wise (128x1, transposed) quantizer.
 * dyqT [N][M], sdyT [M/128][N], xqT [K][M], sxT [M/128][K]. */
ORACLE_API void fp8bq_oracle_gemm_wgrad(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT,
                                        const float* sxT, int64_t M, int64_t N, int64_t K,
                                        const int64_t* rows, int64_t n_rows, const int64_t* cols,
                                        int64_t n_cols, double* out_val, double* out_abs) {
    int64_t MC = M / 128;
#pragma omp parallel for schedule(dynamic)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t n = rows[ri];
        for (int64_t ci = 0; ci < n_cols; ++ci) {
            int64_t k = cols[ci];
            double total = 0.0, total_abs = 0.0;
            for (int64_t c = 0; c < MC; ++c) {
                double p = 0.0, pa = 0.0;
                for (int64_t m = c * 128; m < c * 128 + 128; ++m) {
                    double prod = fp8bq_oracle_e4m3_decode(dyqT[n * M + m]) * fp8bq_oracle_e4m3_decode(xqT[k * M + m]);
                    p += prod;
                    pa += fabs(prod);
                }
                double scale = (double)sdyT[c * N + n] * (double)sxT[c * K + k];
                total += scale * p;
                total_abs += scale * pa;
            }
            out_val[ri * n_cols + ci] = total;
            out_abs[ri * n_cols + ci] = total_abs;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MX variant: power-of-two scales per 1x32 block                           */
/* ------------------------------------------------------------------------ */
/*
 * The variant replaces the FP32 tile scale by a power of two 2^E shared by 32
 * consecutive elements along the reduction dimension, the block shape and
 * scale type (an 8-bit exponent, "E8M0") of the OCP Microscaling (MX)
 * formats specification, so that the tensor cores can apply the scales inside
 * the MMA.  The exponent rule is this project's reading, kept as close to the
 * layer's amax/448 rule as a power of two allows: E is the smallest integer
 * (not below -127, the smallest E8M0 scale) with amax <= 448 * 2^E, i.e. the
 * scale amax/448 rounded up to a power of two, so that no element saturates
 * and the largest lands in (224, 448].  An all-zero block gets E = -127.
 * Elements: code = E4M3(x * 2^-E), round-half-to-even; the product is exact
 * whenever it is at least 2^-126 in magnitude, and anything smaller encodes
 * to a signed zero either way.
 *
 * Storage: codes exactly like the 1x128 quantizers (row-wise [R][C], or
 * column-wise emitted transposed [C][M]); exponent bytes E + 127 in
 * "chunk-major" order e[C/128][R][4] (row-wise) or e[M/128][C][4]
 * (column-wise): byte t of row r in chunk c covers elements 128c + 32t ..
 * 128c + 32t + 31 of that row.
 */

/* The shared exponent of a block with maximum magnitude amax, found by a
 * plain upward search from -127. */
ORACLE_API int fp8bq_oracle_mx_exponent(float amax) {
    int e = -127;
    while ((double)amax > ldexp(448.0, e)) ++e;
    return e;
}

static uint8_t mx_quantize_elem(float x, int e) {
    double v = ldexp((double)x, -e);   /* exact in binary64 */
    return fp8bq_oracle_e4m3_encode((float)v);
}

/* Row-wise 1x32 MX quantization: x [R][C] (pitch ldx) -> q [R][C],
 * e8 [C/128][R][4]. */
ORACLE_API void fp8bq_oracle_mx_quantize_rowwise(const void* x, int dtype, int64_t R, int64_t C,
                                                 int64_t ldx, uint8_t* q, uint8_t* e8) {
    int64_t NB = C / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < NB; ++b) {
            float amax = 0.0f;
            for (int64_t j = 0; j < 32; ++j) {
                float a = fabsf(load_elem(x, dtype, r * ldx + b * 32 + j));
                if (a > amax) amax = a;
            }
            int e = fp8bq_oracle_mx_exponent(amax);
            e8[((b / 4) * R + r) * 4 + (b % 4)] = (uint8_t)(e + 127);
            for (int64_t j = 0; j < 32; ++j)
                q[r * C + b * 32 + j] = mx_quantize_elem(load_elem(x, dtype, r * ldx + b * 32 + j), e);
        }
    }
}

/* Column-wise 32x1 MX quantization, emitted transposed: x [M][C] (pitch ldx)
 * -> qT [C][M] with qT[c][m] the code of x[m][c], e8 [M/128][C][4]. */
ORACLE_API void fp8bq_oracle_mx_quantize_colwise(const void* x, int dtype, int64_t M, int64_t C,
                                                 int64_t ldx, uint8_t* qT, uint8_t* e8) {
    int64_t NB = M / 32;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t b = 0; b < NB; ++b) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 32; ++i) {
                float a = fabsf(load_elem(x, dtype, (b * 32 + i) * ldx + c));
                if (a > amax) amax = a;
            }
            int e = fp8bq_oracle_mx_exponent(amax);
            e8[((b / 4) * C + c) * 4 + (b % 4)] = (uint8_t)(e + 127);
            for (int64_t i = 0; i < 32; ++i)
                qT[c * M + b * 32 + i] = mx_quantize_elem(load_elem(x, dtype, (b * 32 + i) * ldx + c), e);
        }
    }
}

/* MX GEMM: D[i][j] = sum_k 2^(ea(i,k)) D(a[i][k]) * 2^(eb(j,k)) D(b[j][k]) for
 * two K-major operands a [I][K], b [J][K] with exponent bytes
 * ea [K/128][I][4], eb [K/128][J][4] (value = byte - 127).  Fprop, Dgrad and
 * Wgrad are all this product with the operands the MX quantizers emit.
 * Every term is exact in binary64; the sum rounds at 2^-53 relative. */
ORACLE_API void fp8bq_oracle_mx_gemm(const uint8_t* a, const uint8_t* ea, const uint8_t* b,
                                     const uint8_t* eb, int64_t I, int64_t J, int64_t K,
                                     const int64_t* rows, int64_t n_rows, const int64_t* cols,
                                     int64_t n_cols, double* out_val, double* out_abs) {
#pragma omp parallel for schedule(dynamic)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t i = rows[ri];
        for (int64_t ci = 0; ci < n_cols; ++ci) {
            int64_t j = cols[ci];
            double total = 0.0, total_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t c = k / 128, t = (k / 32) % 4;
                double va = ldexp(fp8bq_oracle_e4m3_decode(a[i * K + k]), (int)ea[(c * I + i) * 4 + t] - 127);
                double vb = ldexp(fp8bq_oracle_e4m3_decode(b[j * K + k]), (int)eb[(c * J + j) * 4 + t] - 127);
                total += va * vb;
                total_abs += fabs(va * vb);
            }
            out_val[ri * n_cols + ci] = total;
            out_abs[ri * n_cols + ci] = total_abs;
        }
    }
}

/* Round a binary64 value to BF16 (8 significant bits, 8 exponent bits,
 * subnormals down to 2^-133) with round-half-to-even, directly from the
 * double (no intermediate binary32 rounding).  Returns the 16-bit pattern. */
ORACLE_API uint16_t fp8bq_oracle_bf16_from_double(double v) {
    if (isnan(v)) return 0x7FC0;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    uint16_t out;
    if (a == 0.0) {
        out = 0;
    } else {
        int ex;
        frexp(a, &ex);
        int E = ex - 1;                 /* floor(log2 a) */
        if (E < -126) E = -126;         /* subnormal range shares the quantum 2^-133 */
        double quantum = ldexp(1.0, E - 7);
        double n = nearbyint(a / quantum); /* exact division by a power of two; ties to even */
        double r = n * quantum;
        if (r > ldexp(255.0 / 128.0, 127) || isinf(r)) {
            /* beyond the largest finite BF16 after rounding */
            out = 0x7F80;
        } else {
            float f = (float)r;         /* exact: r has at most 8 significant bits */
            uint32_t w;
            memcpy(&w, &f, 4);
            out = (uint16_t)(w >> 16);
        }
    }
    return (uint16_t)(out | (neg << 15));
}

/* Array forms of the scalar routines above (plain loops, for the tests). */
ORACLE_API void fp8bq_oracle_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = fp8bq_oracle_e4m3_decode(c[i]);
}
ORACLE_API void fp8bq_oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = fp8bq_oracle_e4m3_encode(v[i]);
}
ORACLE_API void fp8bq_oracle_e4m3_encode_arith_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = fp8bq_oracle_e4m3_encode_arith(v[i]);
}
ORACLE_API void fp8bq_oracle_bf16_from_double_array(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = fp8bq_oracle_bf16_from_double(v[i]);
}

/* Number of OpenMP threads the oracle will use (1 when built without it). */
#ifdef _OPENMP
#include <omp.h>
ORACLE_API int fp8bq_oracle_num_threads(void) { return omp_get_max_threads(); }
ORACLE_API void fp8bq_oracle_set_num_threads(int n) { omp_set_num_threads(n); }
#else
ORACLE_API int fp8bq_oracle_num_threads(void) { return 1; }
ORACLE_API void fp8bq_oracle_set_num_threads(int n) { (void)n; }
#endif
