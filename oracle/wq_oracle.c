/*
 * wq_oracle.c -- plain, slow, f64 CPU oracle for the weight-format contraction
 *
 *     Y[n][m] = epi( X[n][k] . W[m][k]^T )
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA library: everything below is written
 * from the definitions on the pages.
 *
 * Definitions followed (page title, item):
 *   - bf16 pairs: cortiq-engine 0.8.49 src/gpu_wgpu/nemotron_audio.rs, kernel
 *     ae_gemm: word c of a W row holds element 2c in its low half and element
 *     2c+1 in its high half; each half is the top 16 bits of an f32.
 *   - Q8_0: hanzo-ml 0.11.13 src/wgpu_backend.rs, matvec_q8_0_gpu (34-byte
 *     blocks); wavo 0.3.0 src/gpu/mod.rs, upload_linear (scale = bytes 0..1,
 *     data = bytes 2..) and its test quantiser (scale written little-endian):
 *     32 weights per block, value d*q with q a signed byte.
 *   - Q4_0: hanzo-ml 0.11.13, matvec_q4_0_gpu (the blocks read as stored, k a
 *     multiple of 32).  The nibble order is not on the pages; this oracle takes
 *     the Q4_0 workload's definition: 18-byte block = f16 d + 16 bytes, element
 *     t < 16 is the low nibble of byte t, t >= 16 the high nibble of byte t-16,
 *     value d*(q-8).
 *   - epilogue: cortiq-engine ae_put: flag 1 adds bias[c]; flag 2 applies
 *     0.5*v*(1+erf(v/sqrt 2)); flag 4 adds the old Y[r][c]; in that order.
 *     The oracle takes erf exactly (C99 erf in f64); the page's kernel uses the
 *     Abramowitz-Stegun 7.1.26 rational approximation of it.
 *   - more activations: wavo 0.3.0 src/gpu/mod.rs, enum Epilogue and its test
 *     reference epilogue(): Silu v/(1+exp(-v)), Relu max(v, 0), Tanh tanh(v); here
 *     flags 8, 16, 32, in the activation's place (after bias, before residual);
 *     at most one activation per call.
 *   - dual outputs: wavo 0.3.0 src/gpu/mod.rs, Gpu::linear (a bias with `dual`
 *     more values than rows) and its gemm test: the first `dual` outputs are
 *     written again after the others, as the plain sum plus the extra bias values,
 *     with no epilogue.
 *   - MoE: hanzo-ml 0.11.13, moe_matvec_gpu: y[s, r] = sum_k W[ids[s], r, k] x[s, k]
 *     over one bank [E][rows][k]; here x is per token and slot (t, s) reads
 *     token t's row, output [t][s][m].
 *
 * Accumulation: f64, natural k order, one output at a time.  The per-output
 * bound S[i][j] = sum_k |X[i][k]| |W[j][k]| (f64) is returned beside Y.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { O_BF16 = 0, O_Q8_0 = 1, O_Q4_0 = 2, O_F16 = 3, O_F32 = 4 };
enum { O_BIAS = 1u, O_GELU = 2u, O_RESIDUAL = 4u, O_SILU = 8u, O_RELU = 16u, O_TANH = 32u };
#define O_ACTS (O_GELU | O_SILU | O_RELU | O_TANH)

/* IEEE 754 binary16 -> f64, from its bit fields (1 sign, 5 exponent, 10 fraction). */
double oracle_half_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                /* subnormal: f * 2^-24 (and +-0) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);    /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bf16 -> f64, from its bit fields (1 sign, 8 exponent, 7 fraction): the top
 * half of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);               /* subnormal: f * 2^-126 * 2^-7 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);    /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a finite value to the nearest bf16 (8 significant bits, exponent range
 * of binary32), ties to even; used only for the tensor-core check that feeds
 * the oracle X rounded the way the kernel rounds it. */
double oracle_round_bf16(double x) {
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    int ex;
    frexp(x, &ex);                               /* |x| in [2^(ex-1), 2^ex) */
    int q = ex - 8;                              /* exponent of one unit in the last place */
    if (q < -133) q = -133;                      /* subnormal spacing */
    double r = ldexp(rint(ldexp(x, -q)), q);     /* rint: nearest, ties to even */
    double maxv = ldexp(255.0, 120);             /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > maxv) r = copysign(INFINITY, x);
    return r;
}

double oracle_gelu(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }

static size_t row_bytes(int wtype, int k) {
    switch (wtype) {
    case O_BF16: return (size_t)2 * k;
    case O_Q8_0: return (size_t)34 * (k / 32);
    case O_Q4_0: return (size_t)18 * (k / 32);
    case O_F16: return (size_t)2 * k;
    case O_F32: return (size_t)4 * k;
    }
    return 0;
}

/* Dequantise one W row of k weights into f64.  F16 / F32: wavo 0.3.0
 * src/gpu/mod.rs, Linear (pipeline index 0 for F32, 1 for F16 weights) -- plain IEEE
 * binary16 / binary32 elements, little-endian, row after row. */
static void dequant_row(int wtype, const uint8_t *row, int k, double *w) {
    if (wtype == O_F16) {
        for (int t = 0; t < k; ++t)
            w[t] = oracle_half_to_f64((uint16_t)(row[2 * t] | (row[2 * t + 1] << 8)));
        return;
    }
    if (wtype == O_F32) {
        for (int t = 0; t < k; ++t) {
            uint32_t bits = (uint32_t)row[4 * t] | ((uint32_t)row[4 * t + 1] << 8) |
                            ((uint32_t)row[4 * t + 2] << 16) | ((uint32_t)row[4 * t + 3] << 24);
            float f;
            memcpy(&f, &bits, sizeof f);
            w[t] = (double)f;
        }
        return;
    }
    if (wtype == O_BF16) {
        for (int c = 0; c < k / 2; ++c) {
            uint32_t word = (uint32_t)row[4 * c] | ((uint32_t)row[4 * c + 1] << 8) |
                            ((uint32_t)row[4 * c + 2] << 16) | ((uint32_t)row[4 * c + 3] << 24);
            w[2 * c] = oracle_bf16_to_f64((uint16_t)(word & 0xFFFFu));
            w[2 * c + 1] = oracle_bf16_to_f64((uint16_t)(word >> 16));
        }
    } else if (wtype == O_Q8_0) {
        for (int b = 0; b < k / 32; ++b) {
            const uint8_t *blk = row + (size_t)34 * b;
            double d = oracle_half_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int t = 0; t < 32; ++t) w[32 * b + t] = d * (double)(int8_t)blk[2 + t];
        }
    } else {
        for (int b = 0; b < k / 32; ++b) {
            const uint8_t *blk = row + (size_t)18 * b;
            double d = oracle_half_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int t = 0; t < 32; ++t) {
                uint8_t byte = blk[2 + (t % 16)];
                int q = (t < 16) ? (byte & 0x0F) : (byte >> 4);
                w[32 * b + t] = d * (double)(q - 8);
            }
        }
    }
}

static int shape_ok(int wtype, int m, int k) {
    if (m < 0 || k <= 0) return 0;
    if (wtype == O_BF16) return k % 2 == 0;
    if (wtype == O_Q8_0 || wtype == O_Q4_0) return k % 32 == 0;
    if (wtype == O_F16 || wtype == O_F32) return 1;
    return 0;
}

/* out[m][k] = dequantised W. Returns 0, or -1 on a bad shape/type. */
int oracle_dequant(int wtype, int m, int k, const uint8_t *W, double *out) {
    if (!shape_ok(wtype, m, k)) return -1;
    size_t rb = row_bytes(wtype, k);
    for (int j = 0; j < m; ++j) dequant_row(wtype, W + rb * j, k, out + (size_t)k * j);
    return 0;
}

/* One output element from a dequantised W row.  alpha scales the contribution
 * before the residual is added: wavo 0.3.0 src/gpu/mod.rs, Epilogue::Residual(a),
 * "c += a(aW^T + b)" (1 for every other epilogue); the bound scales with |alpha|. */
static void dot_epi(int k, unsigned flags, int round_x, double alpha, const float *x,
                    const double *w, const float *bias_j, const float *res_ij, double *y,
                    double *s) {
    double acc = 0.0, bound = 0.0;
    for (int t = 0; t < k; ++t) {
        double xv = round_x ? oracle_round_bf16((double)x[t]) : (double)x[t];
        acc += xv * w[t];
        bound += fabs(xv) * fabs(w[t]);
    }
    double v = acc;
    if (flags & O_BIAS) v += (double)*bias_j;
    /* the activation: at most one of wavo's Epilogue::{Gelu, Silu, Relu, Tanh} */
    if (flags & O_GELU) v = oracle_gelu(v);
    else if (flags & O_SILU) v = v / (1.0 + exp(-v));
    else if (flags & O_RELU) v = v > 0.0 ? v : 0.0;
    else if (flags & O_TANH) v = tanh(v);
    v *= alpha;
    if (flags & O_RESIDUAL) v += (double)*res_ij;
    *y = v;
    if (s) *s = fabs(alpha) * bound;
}

static int set_threads(int threads) {
#ifdef _OPENMP
    return threads > 0 ? threads : omp_get_max_threads();
#else
    (void)threads;
    return 1;
#endif
}

/*
 * Y[i][j] (f64) for all i < n and output rows j in [j0, j1) of W, with wavo's
 * dual outputs (wavo 0.3.0 src/gpu/mod.rs, Gpu::linear and its gemm test): a bias
 * with `dual` more values has the first `dual` outputs written once more after
 * the m others, as the plain sum plus those values, with no epilogue:
 *   Y[i][j]     = epi(sum_k X[i][k] W[j][k]),         j < m
 *   Y[i][m + j] = sum_k X[i][k] W[j][k] + bias2[j],   j < dual.
 * Y, S and R have rows of m + dual values.  X f32 [n][k]; W byte image
 * [m][row_bytes]; bias f32 [m] (flag 1); R f32 (flag 4, the old Y; its columns
 * m.. are not read); bias2 f32 [dual]; S (optional) gets the bound of each output.
 * round: bit 0 feeds bf16-rounded X, bit 1 bf16-rounded W (each dequantised value
 * d*q, exact in f64, rounded to the nearest bf16, ties to even): the operands of
 * the tensor-core path.  threads <= 0: all.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gemm_dual(int n, int m, int k, int dual, int wtype, unsigned flags, int round,
                     double alpha, const float *X, const uint8_t *W, const float *bias,
                     const float *bias2, const float *R, double *Y, double *S, int j0, int j1,
                     int threads) {
    if (n < 0 || !shape_ok(wtype, m, k) || j0 < 0 || j1 > m || j0 > j1) return -1;
    if (dual < 0 || dual > m || (dual > 0 && !bias2)) return -1;
    if (__builtin_popcount(flags & O_ACTS) > 1) return -1;
    if (((flags & O_BIAS) && !bias) || ((flags & O_RESIDUAL) && !R)) return -1;
    size_t rb = row_bytes(wtype, k);
    size_t ld = (size_t)m + (size_t)dual;
    int nt = set_threads(threads);
    int bad = 0;
    const int round_x = round & 1, round_w = (round >> 1) & 1;
#pragma omp parallel num_threads(nt)
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)k);
        if (!w) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int j = j0; j < j1; ++j) {
                dequant_row(wtype, W + rb * j, k, w);
                if (round_w)
                    for (int t = 0; t < k; ++t) w[t] = oracle_round_bf16(w[t]);
                for (int i = 0; i < n; ++i) {
                    size_t o = (size_t)i * ld + j;
                    dot_epi(k, flags, round_x, alpha, X + (size_t)i * k, w,
                            bias ? bias + j : NULL, R ? R + o : NULL, Y + o, S ? S + o : NULL);
                    if (j < dual) /* the second output: bias only, alpha 1 */
                        dot_epi(k, O_BIAS, round_x, 1.0, X + (size_t)i * k, w, bias2 + j, NULL,
                                Y + o + m, S ? S + o + m : NULL);
                }
            }
            free(w);
        }
    }
    return bad ? -1 : 0;
}

/* Without dual outputs: Y, S and R are [n][m]. */
int oracle_gemm_alpha(int n, int m, int k, int wtype, unsigned flags, int round, double alpha,
                      const float *X, const uint8_t *W, const float *bias, const float *R,
                      double *Y, double *S, int j0, int j1, int threads) {
    return oracle_gemm_dual(n, m, k, 0, wtype, flags, round, alpha, X, W, bias, NULL, R, Y, S,
                            j0, j1, threads);
}

/* The same with alpha = 1 (every epilogue but wavo's Residual(a)). */
int oracle_gemm(int n, int m, int k, int wtype, unsigned flags, int round,
                const float *X, const uint8_t *W, const float *bias, const float *R,
                double *Y, double *S, int j0, int j1, int threads) {
    return oracle_gemm_alpha(n, m, k, wtype, flags, round, 1.0, X, W, bias, R, Y, S, j0, j1,
                             threads);
}

/*
 * MoE routed matvec over one bank Wbank[E][m][row_bytes]:
 *   Y[t][s][j] = epi( X[t] . Wbank[ids[t][s]][j]^T ),  bias[E][m], R[t][s][m].
 * Slots (t, s) with slot index q = t*topk + s are processed in [q0, q1).
 * Returns 0, -1 on a bad argument, -2 on an expert id outside [0, E).
 */
int oracle_moe(int n_tok, int topk, int n_experts, int m, int k, int wtype, unsigned flags,
               const float *X, const uint8_t *Wbank, const int32_t *ids, const float *bias,
               const float *R, double *Y, double *S, int q0, int q1, int threads) {
    if (n_tok < 0 || topk <= 0 || n_experts <= 0 || !shape_ok(wtype, m, k)) return -1;
    if (q0 < 0 || q1 > n_tok * topk || q0 > q1) return -1;
    if (((flags & O_BIAS) && !bias) || ((flags & O_RESIDUAL) && !R)) return -1;
    if (__builtin_popcount(flags & O_ACTS) > 1) return -1;
    for (int q = q0; q < q1; ++q)
        if (ids[q] < 0 || ids[q] >= n_experts) return -2;
    size_t rb = row_bytes(wtype, k);
    int nt = set_threads(threads);
    int bad = 0;
#pragma omp parallel num_threads(nt)
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)k);
        if (!w) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for collapse(2) schedule(dynamic, 8)
            for (int q = q0; q < q1; ++q) {
                for (int j = 0; j < m; ++j) {
                    int e = ids[q];
                    int t = q / topk;
                    dequant_row(wtype, Wbank + rb * ((size_t)e * m + j), k, w);
                    size_t o = (size_t)q * m + j;
                    dot_epi(k, flags, 0, 1.0, X + (size_t)t * k, w,
                            bias ? bias + (size_t)e * m + j : NULL, R ? R + o : NULL, Y + o,
                            S ? S + o : NULL);
                }
            }
            free(w);
        }
    }
    return bad ? -1 : 0;
}

int oracle_max_threads(void) { return set_threads(0); }

/*
 * Row LayerNorm, cortiq-engine 0.8.49 src/gpu_wgpu/nemotron_audio.rs, kernel ae_ln
 * (and wavo 0.3.0's test reference layer_norm): for each row of X f32 [n][k],
 * mean = sum x / k, var = sum (x - mean)^2 / k (two passes), and
 * Y = (x - mean) / sqrt(var + 1e-5) * g + b, in f64.  gb = [g (k) | b (k)].
 */
int oracle_layer_norm(int n, int k, const float *X, const float *gb, double *Y) {
    if (n < 0 || k <= 0 || !X || !gb || !Y) return -1;
    for (int i = 0; i < n; ++i) {
        const float *x = X + (size_t)i * k;
        double mean = 0.0, var = 0.0;
        for (int t = 0; t < k; ++t) mean += (double)x[t];
        mean /= k;
        for (int t = 0; t < k; ++t) var += ((double)x[t] - mean) * ((double)x[t] - mean);
        var /= k;
        const double rstd = 1.0 / sqrt(var + 1e-5);
        for (int t = 0; t < k; ++t)
            Y[(size_t)i * k + t] = ((double)x[t] - mean) * rstd * (double)gb[t] + (double)gb[k + t];
    }
    return 0;
}

/*
 * Embedding row gather, wavo 0.3.0 src/gpu/mod.rs, Recorder::embed (and its test
 * gemv_and_embed): row ids[t] of the weight table W (rows x k, any weight format),
 * dequantised, plus the positional values pos[t][j] and the table's bias[j] for
 * the k columns j, added in that order:
 *   out[t][j] = W[ids[t]][j] + pos[t][j] + bias[j]     (pos / bias optional).
 * f64.  An id outside [0, rows) leaves its row of out as it was and clears
 * valid[t]; valid[t] = 1 otherwise.  Returns 0, or -1 on a bad shape/type.
 */
int oracle_embed(int n_ids, int rows, int k, int wtype, const uint8_t *W, const int32_t *ids,
                 const float *pos, const float *bias, double *out, int *valid) {
    if (n_ids < 0 || rows <= 0 || !shape_ok(wtype, rows, k) || !W || !ids || !out || !valid)
        return -1;
    size_t rb = row_bytes(wtype, k);
    double *w = (double *)malloc(sizeof(double) * (size_t)k);
    if (!w) return -1;
    for (int t = 0; t < n_ids; ++t) {
        const int id = ids[t];
        valid[t] = id >= 0 && id < rows;
        if (!valid[t]) continue;
        dequant_row(wtype, W + rb * (size_t)id, k, w);
        for (int j = 0; j < k; ++j) {
            double v = w[j];
            if (pos) v += (double)pos[(size_t)t * k + j];
            if (bias) v += (double)bias[j];
            out[(size_t)t * k + j] = v;
        }
    }
    free(w);
    return 0;
}
