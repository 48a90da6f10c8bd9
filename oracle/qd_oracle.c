/*
 * qd_oracle.c — the plain, slow CPU oracle for the quantized decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this code.  It shares no code, header,
 * table or constant with the CUDA library: it is written from the pages'
 * statement of each operation, and computes the plain definition of each one:
 * every block is dequantised to f32, and every dot product, norm, softmax and
 * weighted sum is accumulated in double, in index order.  The only
 * parallelism is OpenMP over independent outputs (matrix rows, attention
 * heads), which does not change any output's summation order.
 *
 * Sources (the five pages on quantized decode GEMV):
 *  [llmoxide]  "Running an LLM, then forgetting it" (llmoxide blog):
 *              s1 "A neuron is a dot product", s2 "Layers, and the bend
 *              between them", s3 "Text in, vectors out", s4 "Keeping the numbers
 *              in range", s5 "Attention", s6 "Where things are: RoPE", s7 "The
 *              block, and the residual stream", s10 "Loading weights", s12 "The
 *              KV cache".
 *  [go-llm]    "llm" Go package documentation (go-wasmcontainers/llm v0.1.0):
 *              "Design points", "Oracle tolerances", index entries Argmax,
 *              F16ToF32.
 *  [llamini]   "Building llamini.cpp: a from-scratch llama.cpp core in C99",
 *              section "What I reimplemented" (the Q4_K 6-bit scale unpacker).
 *  [dasLLAMA]  "dasLLAMA-00 - The Problem Statement", 8.7.1.4 "Five small
 *              functions", 8.7.1.6.2 "Attention", 8.7.1.6.3 "Feed-forward",
 *              8.7.1.6.4 "Logits", 8.7.1.7 "Prompting is repeated forward".
 *  [minillm]   minillm-cpp README: "Loader" (BF16 zero-extension), "NEON
 *              kernels" and "Quantization" (per-row symmetric INT8).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - Q4_0 block: f16 d at byte 0, then 16 code bytes; element j (0..15) is the
 *    low nibble of code byte j and element j+16 its high nibble; value (q-8)*d.
 *  - Q4_K super-block: d, dmin (f16), 12 scale bytes, 128 code bytes; code
 *    chunk c (0..3) is bytes 32c..32c+31, whose low nibbles are sub-block 2c
 *    (elements 64c..64c+31) and high nibbles sub-block 2c+1 (elements
 *    64c+32..64c+63); value d*sc*q - dmin*m.
 *  - per-row INT8 tensor bytes: int8 codes [rows][cols], then f32 scale[rows].
 *  - RoPE angle for pair i at position p: p * theta^(-2i/hd), in double.
 *
 * Portable C99 + optional OpenMP; no architecture intrinsics.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_Q4_0 = 0, OR_Q8_0 = 1, OR_Q4_K = 2, OR_I8_ROW = 3, OR_Q4_1 = 4, OR_Q5_0 = 5, OR_Q5_K = 6, OR_Q6_K = 7, OR_F16 = 8,
       OR_I4_ROW = 9 };
enum { OR_ROPE_ADJACENT = 0, OR_ROPE_HALF = 1 };

/* ------------------------------------------------------------------------- */
/* Scalar formats                                                             */
/* ------------------------------------------------------------------------- */

/* IEEE 754 binary16 -> double, exactly (the [go-llm] index entry F16ToF32 is an
 * exact conversion).  Written from the format's definition: 1 sign bit, 5 exponent
 * bits (bias 15), 10 fraction bits. */
double or_f16_to_f64(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1F;
    const int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* zero or subnormal: f * 2^-14 / 1024 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    }
    return sign ? -v : v;
}

/* BF16 -> f32 by zero-extension of the bit pattern ([minillm] "Loader"). */
float or_bf16_to_f32(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* f32 rounded through IEEE binary16 and back ([go-llm] index RoundF16: what an f16 KV
 * cache stores).  Written from the format's definition: the nearest binary16 value, ties
 * to the even significand; magnitudes from 65520 up become infinity; below 2^-14 the
 * spacing is the subnormal one, 2^-24; NaN stays NaN, the sign of zero is kept. */
float or_round_f16(float f) {
    if (isnan(f)) return f;
    const double a = fabs((double)f);
    double r;
    if (a >= 65520.0) {
        r = INFINITY;
    } else {
        int e;
        frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
        int ex = e - 1;               /* a in [2^ex, 2^(ex+1)) */
        if (ex < -14) ex = -14;       /* subnormal range: fixed spacing 2^-24 */
        const double ulp = ldexp(1.0, ex - 10);
        const double q = a / ulp;     /* exact: a has at most 24 significant bits */
        double n = floor(q);
        const double frac = q - n;
        if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
        r = n * ulp;
    }
    return (float)(f < 0.0f || (f == 0.0f && signbit(f)) ? -r : r);
}

/* Array form of the two conversions, writing f32 bit patterns (keeps NaN payloads). */
void or_bf16_to_f32_array(const uint16_t* in, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_bf16_to_f32(in[i]);
}

void or_f16_to_f32_array(const uint16_t* in, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (float)or_f16_to_f64(in[i]);
}

static double f16_at(const uint8_t* p) { return or_f16_to_f64((uint16_t)(p[0] | (p[1] << 8))); }

/* ------------------------------------------------------------------------- */
/* Block dequantisation ([llmoxide] s10 "Loading weights"; [llamini])         */
/* ------------------------------------------------------------------------- */

/* The Q4_K 12-byte field holds eight 6-bit (scale, min) pairs.  Sub-blocks 0-3
 * keep theirs in the low six bits of bytes j and j+4; sub-blocks 4-7 take their
 * low four bits from byte j+4 (scale: low nibble, min: high nibble) and their
 * top two bits from the spare top bits of bytes j-4 (scale) and j (min).
 * ([llamini] "What I reimplemented", the get_scale_min_k4 unpacker.) */
void or_get_scale_min_k4(int j, const uint8_t* q, uint8_t* sc, uint8_t* m) {
    if (j < 4) {
        *sc = q[j] & 63;
        *m = q[j + 4] & 63;
    } else {
        *sc = (uint8_t)((q[j + 4] & 0x0F) | ((q[j - 4] >> 6) << 4));
        *m = (uint8_t)((q[j + 4] >> 4) | ((q[j] >> 6) << 4));
    }
}

static int64_t row_bytes(int fmt, int64_t cols) {
    switch (fmt) {
        case OR_Q4_0: return (cols / 32) * 18;
        case OR_Q8_0: return (cols / 32) * 34;
        case OR_Q4_K: return (cols / 256) * 144;
        case OR_I8_ROW: return cols;
        case OR_Q4_1: return (cols / 32) * 20;
        case OR_Q5_0: return (cols / 32) * 22;
        case OR_Q5_K: return (cols / 256) * 176;
        case OR_Q6_K: return (cols / 256) * 210;
        case OR_F16: return cols * 2;
        case OR_I4_ROW: return cols / 2;
        default: return -1;
    }
}

int or_shape_ok(int fmt, int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    switch (fmt) {
        case OR_Q4_0:
        case OR_Q8_0:
        case OR_Q4_1:
        case OR_Q5_0: return cols % 32 == 0;
        case OR_Q4_K:
        case OR_Q5_K:
        case OR_Q6_K: return cols % 256 == 0;
        case OR_I8_ROW:
        case OR_F16: return 1;
        case OR_I4_ROW: return cols % 2 == 0;
        default: return 0;
    }
}

/* Dequantise row r of a rows x cols tensor (model-file layout) into out[cols],
 * each value rounded once to f32. */
static void dequant_row(int fmt, const uint8_t* w, int64_t rows, int64_t cols, int64_t r, float* out) {
    const uint8_t* row = w + r * row_bytes(fmt, cols);
    if (fmt == OR_Q4_0) {
        for (int64_t b = 0; b < cols / 32; ++b) {
            const uint8_t* blk = row + b * 18;
            const double d = f16_at(blk);
            for (int j = 0; j < 16; ++j) {
                const int lo = blk[2 + j] & 0x0F, hi = blk[2 + j] >> 4;
                out[b * 32 + j] = (float)((lo - 8) * d);
                out[b * 32 + j + 16] = (float)((hi - 8) * d);
            }
        }
    } else if (fmt == OR_Q8_0) {
        /* [llmoxide] s10: d = f16 at byte 0, 32 signed bytes follow. */
        for (int64_t b = 0; b < cols / 32; ++b) {
            const uint8_t* blk = row + b * 34;
            const double d = f16_at(blk);
            for (int j = 0; j < 32; ++j) out[b * 32 + j] = (float)((int8_t)blk[2 + j] * d);
        }
    } else if (fmt == OR_Q4_K) {
        for (int64_t s = 0; s < cols / 256; ++s) {
            const uint8_t* blk = row + s * 144;
            const double d = f16_at(blk), dmin = f16_at(blk + 2);
            const uint8_t* scales = blk + 4;
            const uint8_t* qs = blk + 16;
            for (int c = 0; c < 4; ++c) {
                uint8_t sc0, m0, sc1, m1;
                or_get_scale_min_k4(2 * c, scales, &sc0, &m0);
                or_get_scale_min_k4(2 * c + 1, scales, &sc1, &m1);
                for (int l = 0; l < 32; ++l) {
                    const int lo = qs[32 * c + l] & 0x0F, hi = qs[32 * c + l] >> 4;
                    out[s * 256 + 64 * c + l] = (float)(d * sc0 * lo - dmin * m0);
                    out[s * 256 + 64 * c + 32 + l] = (float)(d * sc1 * hi - dmin * m1);
                }
            }
        }
    } else if (fmt == OR_Q4_1) {
        /* d, m, then 16 bytes of codes as Q4_0; value d*q + m */
        for (int64_t b = 0; b < cols / 32; ++b) {
            const uint8_t* blk = row + b * 20;
            const double d = f16_at(blk), m = f16_at(blk + 2);
            for (int j = 0; j < 16; ++j) {
                out[b * 32 + j] = (float)(d * (blk[4 + j] & 0x0F) + m);
                out[b * 32 + j + 16] = (float)(d * (blk[4 + j] >> 4) + m);
            }
        }
    } else if (fmt == OR_Q5_0) {
        /* d, a 32-bit word of fifth bits (bit j for element j), low nibbles as Q4_0;
         * value (q - 16) * d */
        for (int64_t b = 0; b < cols / 32; ++b) {
            const uint8_t* blk = row + b * 22;
            const double d = f16_at(blk);
            const uint32_t qh = (uint32_t)blk[2] | ((uint32_t)blk[3] << 8) | ((uint32_t)blk[4] << 16) |
                                ((uint32_t)blk[5] << 24);
            for (int j = 0; j < 16; ++j) {
                const int lo = (blk[6 + j] & 0x0F) | (int)(((qh >> j) & 1u) << 4);
                const int hi = (blk[6 + j] >> 4) | (int)(((qh >> (j + 16)) & 1u) << 4);
                out[b * 32 + j] = (float)((lo - 16) * d);
                out[b * 32 + j + 16] = (float)((hi - 16) * d);
            }
        }
    } else if (fmt == OR_Q5_K) {
        /* Q4_K's header, then 32 bytes of fifth bits and 128 bytes of low nibbles: chunk c
         * of 64 takes bit 2c of byte l for element l and bit 2c+1 for element 32+l */
        for (int64_t s = 0; s < cols / 256; ++s) {
            const uint8_t* blk = row + s * 176;
            const double d = f16_at(blk), dmin = f16_at(blk + 2);
            const uint8_t* scales = blk + 4;
            const uint8_t* qh = blk + 16;
            const uint8_t* qs = blk + 48;
            for (int c = 0; c < 4; ++c) {
                uint8_t sc0, m0, sc1, m1;
                or_get_scale_min_k4(2 * c, scales, &sc0, &m0);
                or_get_scale_min_k4(2 * c + 1, scales, &sc1, &m1);
                for (int l = 0; l < 32; ++l) {
                    const int lo = (qs[32 * c + l] & 0x0F) + (((qh[l] >> (2 * c)) & 1) ? 16 : 0);
                    const int hi = (qs[32 * c + l] >> 4) + (((qh[l] >> (2 * c + 1)) & 1) ? 16 : 0);
                    out[s * 256 + 64 * c + l] = (float)(d * sc0 * lo - dmin * m0);
                    out[s * 256 + 64 * c + 32 + l] = (float)(d * sc1 * hi - dmin * m1);
                }
            }
        }
    } else if (fmt == OR_Q6_K) {
        /* 128 bytes of low nibbles, 64 bytes of two-bit high parts, 16 signed scales, d.
         * Each half of 128 elements uses 64 low-nibble bytes and 32 high-part bytes: byte l
         * of the half's high parts carries, two bits each, the high parts of elements l,
         * 32+l, 64+l and 96+l; low-nibble bytes l and 32+l give elements l, 32+l (low
         * nibbles) and 64+l, 96+l (high nibbles).  Scale i covers elements 16i..16i+15.
         * value d * scale * (q - 32) */
        for (int64_t s = 0; s < cols / 256; ++s) {
            const uint8_t* blk = row + s * 210;
            const double d = f16_at(blk + 208);
            const int8_t* sc = (const int8_t*)(blk + 192);
            for (int h = 0; h < 2; ++h) {
                const uint8_t* ql = blk + 64 * h;
                const uint8_t* qh = blk + 128 + 32 * h;
                float* o = out + s * 256 + 128 * h;
                for (int l = 0; l < 32; ++l) {
                    const int q0 = (ql[l] & 0x0F) | ((qh[l] & 3) << 4);
                    const int q1 = (ql[32 + l] & 0x0F) | (((qh[l] >> 2) & 3) << 4);
                    const int q2 = (ql[l] >> 4) | (((qh[l] >> 4) & 3) << 4);
                    const int q3 = (ql[32 + l] >> 4) | (((qh[l] >> 6) & 3) << 4);
                    o[l] = (float)(d * sc[8 * h + (l / 16)] * (q0 - 32));
                    o[32 + l] = (float)(d * sc[8 * h + 2 + (l / 16)] * (q1 - 32));
                    o[64 + l] = (float)(d * sc[8 * h + 4 + (l / 16)] * (q2 - 32));
                    o[96 + l] = (float)(d * sc[8 * h + 6 + (l / 16)] * (q3 - 32));
                }
            }
        }
    } else if (fmt == OR_F16) {
        for (int64_t c = 0; c < cols; ++c) out[c] = (float)f16_at(row + 2 * c);
    } else if (fmt == OR_I4_ROW) {
        /* [minillm] "Quantization": symmetric per-row INT4, one scale per output row; codes
         * two per byte (element 2i in the low nibble), two's complement, then the f32 row
         * scales after all codes */
        float sc;
        memcpy(&sc, w + rows * (cols / 2) + 4 * r, sizeof sc);
        for (int64_t c = 0; c < cols; ++c) {
            const int nib = (row[c / 2] >> (4 * (c & 1))) & 0x0F;
            const int q = nib >= 8 ? nib - 16 : nib;
            out[c] = (float)((double)sc * q);
        }
    } else { /* OR_I8_ROW ([minillm] "Quantization": one scale per output row) */
        float s;
        memcpy(&s, w + rows * cols + 4 * r, sizeof s);
        const int8_t* q = (const int8_t*)row;
        for (int64_t c = 0; c < cols; ++c) out[c] = (float)((double)s * q[c]);
    }
}

/* Dequantise rows [row0, row0+nrows) into out[nrows][cols]. */
int or_dequant(int fmt, const uint8_t* w, int64_t rows, int64_t cols, int64_t row0, int64_t nrows, float* out) {
    if (!or_shape_ok(fmt, rows, cols) || row0 < 0 || nrows < 0 || row0 + nrows > rows) return -1;
#pragma omp parallel for schedule(static) if (nrows * cols > 262144)
    for (int64_t r = 0; r < nrows; ++r) dequant_row(fmt, w, rows, cols, row0 + r, out + r * cols);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Matrix-vector product ([llmoxide] s1; [dasLLAMA] 8.7.1.4 matmul)          */
/* y[b][r] = sum_c deq(W)[r][c] * x[b][c], W row-major [out][in].             */
/* ------------------------------------------------------------------------- */

static void gemv_rows_d(int fmt, const uint8_t* w, int64_t rows, int64_t cols, const double* x, int batch,
                        int64_t x_stride, double* y, int64_t y_stride, int64_t row0, int64_t nrows) {
#pragma omp parallel if (nrows * cols > 65536)
    {
        float* deq = (float*)malloc(sizeof(float) * (size_t)cols);
#pragma omp for schedule(static)
        for (int64_t i = 0; i < nrows; ++i) {
            const int64_t r = row0 + i;
            dequant_row(fmt, w, rows, cols, r, deq);
            for (int b = 0; b < batch; ++b) {
                double acc = 0.0;
                const double* xb = x + (int64_t)b * x_stride;
                for (int64_t c = 0; c < cols; ++c) acc += (double)deq[c] * xb[c];
                y[(int64_t)b * y_stride + i] = acc;
            }
        }
        free(deq);
    }
}

/* Public GEMV over f32 activations: x[batch][cols] (f32), y[batch][nrows]
 * (double) for rows [row0, row0+nrows). */
/* The same product over double activations x[batch][cols] (the decode step's own
 * intermediate vectors are double). */
int or_gemv_xd(int fmt, const uint8_t* w, int64_t rows, int64_t cols, const double* x, int batch, int64_t row0,
               int64_t nrows, double* y) {
    if (!or_shape_ok(fmt, rows, cols) || batch <= 0 || row0 < 0 || nrows < 0 || row0 + nrows > rows) return -1;
    gemv_rows_d(fmt, w, rows, cols, x, batch, cols, y, nrows, row0, nrows);
    return 0;
}

int or_gemv(int fmt, const uint8_t* w, int64_t rows, int64_t cols, const float* x, int batch, int64_t row0,
            int64_t nrows, double* y) {
    if (!or_shape_ok(fmt, rows, cols) || batch <= 0 || row0 < 0 || nrows < 0 || row0 + nrows > rows) return -1;
    double* xd = (double*)malloc(sizeof(double) * (size_t)(cols * batch));
    if (!xd) return -2;
    for (int64_t i = 0; i < cols * batch; ++i) xd[i] = x[i];
    gemv_rows_d(fmt, w, rows, cols, xd, batch, cols, y, nrows, row0, nrows);
    free(xd);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* RMSNorm ([llmoxide] s4 rms_norm_mul; [dasLLAMA] 8.7.1.6.2 rmsnorm):        */
/* out = x * g / sqrt(mean(x^2) + eps), eps inside the root.                  */
/* ------------------------------------------------------------------------- */

void or_rmsnorm_d(const double* x, const float* g, int n, double eps, double* out) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    const double scale = 1.0 / sqrt(ss / n + eps);
    for (int i = 0; i < n; ++i) out[i] = x[i] * scale * (double)g[i];
}

int or_rmsnorm(const float* x, const float* g, int n, int batch, double eps, double* out) {
    if (n <= 0 || batch <= 0) return -1;
    double* xd = (double*)malloc(sizeof(double) * (size_t)n);
    if (!xd) return -2;
    for (int b = 0; b < batch; ++b) {
        for (int i = 0; i < n; ++i) xd[i] = x[(int64_t)b * n + i];
        or_rmsnorm_d(xd, g, n, eps, out + (int64_t)b * n);
    }
    free(xd);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* RoPE ([llmoxide] s6 rope; [dasLLAMA] 8.7.1.6.2 rope)                      */
/* Pair i of a head of width hd turns by pos * theta^(-2i/hd).  Pairs are     */
/* (2i, 2i+1) ("adjacent", llama files) or (i, i+hd/2) ("half", NeoX/Qwen).   */
/* ------------------------------------------------------------------------- */

static double rope_angle(int pos, int i, int hd, double theta) {
    return (double)pos * pow(theta, -2.0 * (double)i / (double)hd);
}

void or_rope_head_d(double* v, int hd, int pos, int pairing, double theta) {
    const int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        const double a = rope_angle(pos, i, hd, theta);
        const double c = cos(a), s = sin(a);
        const int ia = (pairing == OR_ROPE_ADJACENT) ? 2 * i : i;
        const int ib = (pairing == OR_ROPE_ADJACENT) ? 2 * i + 1 : i + half;
        const double x0 = v[ia], x1 = v[ib];
        v[ia] = x0 * c - x1 * s;
        v[ib] = x0 * s + x1 * c;
    }
}

/* Rotate n_heads heads of v (f32 in, double out) at position pos. */
int or_rope(const float* v, int n_heads, int hd, int pos, int pairing, double theta, double* out) {
    if (n_heads <= 0 || hd <= 0 || (hd & 1) || pos < 0) return -1;
    for (int64_t i = 0; i < (int64_t)n_heads * hd; ++i) out[i] = v[i];
    for (int h = 0; h < n_heads; ++h) or_rope_head_d(out + (int64_t)h * hd, hd, pos, pairing, theta);
    return 0;
}

/* cos/sin table [ctx][hd/2][2] rounded to f32 ([go-llm] "Design points": RoPE
 * angles computed on the CPU in double precision). */
int or_rope_table(double theta, int hd, int ctx, float* out) {
    if (hd <= 0 || (hd & 1) || ctx <= 0) return -1;
    for (int p = 0; p < ctx; ++p)
        for (int i = 0; i < hd / 2; ++i) {
            const double a = rope_angle(p, i, hd, theta);
            out[((int64_t)p * (hd / 2) + i) * 2 + 0] = (float)cos(a);
            out[((int64_t)p * (hd / 2) + i) * 2 + 1] = (float)sin(a);
        }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Causal GQA decode attention ([llmoxide] s5; [dasLLAMA] 8.7.1.6.2)          */
/* For q head h: kvh = h / (hq/hk); score[p] = q.k_p / sqrt(hd), p=0..n_pos-1;*/
/* softmax with the max subtracted; out = sum_p w_p v_p.                      */
/* Cache for one layer and one sequence: k[kvh][ctx][hd], v likewise (f32).   */
/* ------------------------------------------------------------------------- */

void or_attention_d(const double* q, const float* k, const float* v, int hq, int hk, int hd, int n_pos,
                    int64_t ctx, double* out) {
    const int group = hq / hk;
#pragma omp parallel if ((int64_t)hq * n_pos * hd > 262144)
    {
        double* sc = (double*)malloc(sizeof(double) * (size_t)n_pos);
#pragma omp for schedule(static)
        for (int h = 0; h < hq; ++h) {
            const int kvh = h / group;
            const double* qh = q + (int64_t)h * hd;
            const float* kb = k + (int64_t)kvh * ctx * hd;
            const float* vb = v + (int64_t)kvh * ctx * hd;
            for (int p = 0; p < n_pos; ++p) {
                double dot = 0.0;
                for (int i = 0; i < hd; ++i) dot += qh[i] * (double)kb[(int64_t)p * hd + i];
                sc[p] = dot / sqrt((double)hd);
            }
            /* softmax: [dasLLAMA] 8.7.1.6.2 softmax */
            double mx = sc[0];
            for (int p = 1; p < n_pos; ++p) mx = sc[p] > mx ? sc[p] : mx;
            double sum = 0.0;
            for (int p = 0; p < n_pos; ++p) {
                sc[p] = exp(sc[p] - mx);
                sum += sc[p];
            }
            for (int p = 0; p < n_pos; ++p) sc[p] /= sum;
            double* oh = out + (int64_t)h * hd;
            for (int i = 0; i < hd; ++i) oh[i] = 0.0;
            for (int p = 0; p < n_pos; ++p)
                for (int i = 0; i < hd; ++i) oh[i] += sc[p] * (double)vb[(int64_t)p * hd + i];
        }
        free(sc);
    }
}

int or_attention(const float* q, const float* k, const float* v, int hq, int hk, int hd, int n_pos, int64_t ctx,
                 double* out) {
    if (hq <= 0 || hk <= 0 || hq % hk || hd <= 0 || n_pos <= 0 || n_pos > ctx) return -1;
    double* qd = (double*)malloc(sizeof(double) * (size_t)hq * hd);
    if (!qd) return -2;
    for (int64_t i = 0; i < (int64_t)hq * hd; ++i) qd[i] = q[i];
    or_attention_d(qd, k, v, hq, hk, hd, n_pos, ctx, out);
    free(qd);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* SwiGLU ([llmoxide] s2; [dasLLAMA] 8.7.1.6.3): silu(g) * u with              */
/* silu(z) = z / (1 + exp(-z)).                                               */
/* ------------------------------------------------------------------------- */

double or_silu(double z) { return z / (1.0 + exp(-z)); }

int or_swiglu(const float* g, const float* u, int64_t n, double* out) {
    if (n <= 0) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = or_silu((double)g[i]) * (double)u[i];
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Load-time per-row INT8 quantisation of BF16 weights ([minillm] "Direct INT8 */
/* loading": each matrix quantised row by row from the BF16 file; "Quantization":*/
/* symmetric, one scale per output row).  The pages do not print the rule; the  */
/* reading taken: s = max|w| / 127 in f32, q = w / s (f32) rounded to nearest   */
/* with ties away from zero (C roundf), clamped to [-127, 127].  A row of zeros  */
/* gets s = 0 and codes 0; a row holding a non-finite value gets codes 0 and a   */
/* NaN scale.  Output: the per-row INT8 tensor bytes (codes [rows][cols], then   */
/* f32 scales [rows]).                                                          */
/* ------------------------------------------------------------------------- */

int or_quantize_i8_rows(const uint16_t* w, int64_t rows, int64_t cols, int8_t* codes, float* scales) {
    if (rows < 1 || cols < 1) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* wr = w + r * cols;
        int8_t* qr = codes + r * cols;
        float m = 0.0f;
        int finite = 1;
        for (int64_t c = 0; c < cols; ++c) {
            const float v = or_bf16_to_f32(wr[c]);
            if (!isfinite(v))
                finite = 0;
            else if (fabsf(v) > m)
                m = fabsf(v);
        }
        if (!finite || m == 0.0f) {
            scales[r] = finite ? 0.0f : NAN;
            for (int64_t c = 0; c < cols; ++c) qr[c] = 0;
            continue;
        }
        const float s = m / 127.0f;
        scales[r] = s;
        for (int64_t c = 0; c < cols; ++c) {
            float q = roundf(or_bf16_to_f32(wr[c]) / s);
            if (q > 127.0f) q = 127.0f;
            if (q < -127.0f) q = -127.0f;
            qr[c] = (int8_t)q;
        }
    }
    return 0;
}

/* Per-row symmetric INT4 of BF16 weights ([minillm] "Quantization": INT8 and INT4, one
 * scale per output row).  The page prints no rule; the one implemented mirrors the INT8
 * one with the 4-bit code range: s = max|w| / 7 (f32), q = w / s (f32) rounded to nearest
 * with ties away from zero (C roundf), clamped to +-7; a row of zeros gets s = 0 and codes
 * 0, a row holding a non-finite value codes 0 and a NaN scale.  codes: [rows][cols / 2]
 * bytes, element 2i in the low nibble (two's complement). */
int or_quantize_i4_rows(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* codes, float* scales) {
    if (rows < 1 || cols < 2 || cols % 2) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* wr = w + r * cols;
        uint8_t* qr = codes + r * (cols / 2);
        float m = 0.0f;
        int finite = 1;
        for (int64_t c = 0; c < cols; ++c) {
            const float v = or_bf16_to_f32(wr[c]);
            if (!isfinite(v))
                finite = 0;
            else if (fabsf(v) > m)
                m = fabsf(v);
        }
        for (int64_t c = 0; c < cols / 2; ++c) qr[c] = 0;
        if (!finite || m == 0.0f) {
            scales[r] = finite ? 0.0f : NAN;
            continue;
        }
        const float s = m / 7.0f;
        scales[r] = s;
        for (int64_t c = 0; c < cols; ++c) {
            float q = roundf(or_bf16_to_f32(wr[c]) / s);
            if (q > 7.0f) q = 7.0f;
            if (q < -7.0f) q = -7.0f;
            qr[c / 2] |= (uint8_t)(((int)q & 0x0F) << (4 * (c & 1)));
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* ggml-exact activations ([go-llm] type CPU, "ExactGGML": activations are      */
/* quantised to Q8_0 -- Q8_1 for Q4_1 weights -- before every quantised matrix  */
/* product).  The page prints no rule; the one implemented, per 32-element      */
/* block: d = max|x| / 127 (f32), q = x / d (f32) rounded to nearest with ties  */
/* away from zero (C roundf), clamped to +-127; the block keeps d rounded to    */
/* binary16 and, for Q8_1, s = d * sum(q) (f32) rounded to binary16.  A zero    */
/* block has d = 0 and codes 0; a block holding a non-finite value codes 0 and  */
/* d = s = NaN.  d16 / s16 receive the binary16 values (s16 may be NULL).       */
/* ------------------------------------------------------------------------- */
int or_quantize_q8(const float* x, int64_t n, int8_t* q, float* d16, float* s16) {
    if (n < 1 || n % 32) return -1;
    for (int64_t b = 0; b < n / 32; ++b) {
        const float* xb = x + 32 * b;
        int8_t* qb = q + 32 * b;
        float m = 0.0f;
        int finite = 1;
        for (int j = 0; j < 32; ++j) {
            if (!isfinite(xb[j]))
                finite = 0;
            else if (fabsf(xb[j]) > m)
                m = fabsf(xb[j]);
        }
        if (!finite || m == 0.0f) {
            for (int j = 0; j < 32; ++j) qb[j] = 0;
            d16[b] = finite ? 0.0f : NAN;
            if (s16) s16[b] = d16[b];
            continue;
        }
        const float d = m / 127.0f;
        int sum = 0;
        for (int j = 0; j < 32; ++j) {
            float v = roundf(xb[j] / d);
            if (v > 127.0f) v = 127.0f;
            if (v < -127.0f) v = -127.0f;
            qb[j] = (int8_t)v;
            sum += qb[j];
        }
        d16[b] = or_round_f16(d);
        if (s16) s16[b] = or_round_f16(d * (float)sum);
    }
    return 0;
}

/* The product over quantised activations, in the block's own integers ([llamini]
 * "Optimizing for CPU, and finding out what was actually true": ggml's dot products
 * multiply the packed bytes directly and convert to float only for the scaled sum): y[b][r] = sum over blocks k of row r of
 *   Q8_0: d_w d_x sum_j q_w q_x;   Q4_0: d_w d_x sum_j (q_w - 8) q_x;
 *   Q4_1: d_w d_x sum_j q_w q_x + m_w s_x,
 * with x's binary16 d and s; accumulated in double. */
int or_gemv_q8act(int fmt, const uint8_t* w, int64_t rows, int64_t cols, const int8_t* xq, const float* xd,
                  const float* xs, int batch, int64_t row0, int64_t nrows, double* y) {
    if ((fmt != OR_Q8_0 && fmt != OR_Q4_0 && fmt != OR_Q4_1) || !or_shape_ok(fmt, rows, cols) || batch < 1 ||
        row0 < 0 || nrows < 0 || row0 + nrows > rows || (fmt == OR_Q4_1 && !xs))
        return -1;
    const int64_t nb = cols / 32, rb = row_bytes(fmt, cols);
#pragma omp parallel for schedule(static) if (nrows * cols * batch > 262144)
    for (int64_t r = 0; r < nrows; ++r) {
        const uint8_t* row = w + (row0 + r) * rb;
        for (int bt = 0; bt < batch; ++bt) {
            double acc = 0.0;
            for (int64_t k = 0; k < nb; ++k) {
                const int8_t* qx = xq + (int64_t)bt * cols + 32 * k;
                const double dx = xd[(int64_t)bt * nb + k];
                long sumi = 0;
                if (fmt == OR_Q8_0) {
                    const uint8_t* blk = row + k * 34;
                    for (int j = 0; j < 32; ++j) sumi += (long)(int8_t)blk[2 + j] * qx[j];
                    acc += f16_at(blk) * dx * (double)sumi;
                } else if (fmt == OR_Q4_0) {
                    const uint8_t* blk = row + k * 18;
                    for (int j = 0; j < 16; ++j)
                        sumi += (long)((blk[2 + j] & 0x0F) - 8) * qx[j] + (long)((blk[2 + j] >> 4) - 8) * qx[16 + j];
                    acc += f16_at(blk) * dx * (double)sumi;
                } else {
                    const uint8_t* blk = row + k * 20;
                    for (int j = 0; j < 16; ++j)
                        sumi += (long)(blk[4 + j] & 0x0F) * qx[j] + (long)(blk[4 + j] >> 4) * qx[16 + j];
                    acc += f16_at(blk) * dx * (double)sumi + f16_at(blk + 2) * (double)xs[(int64_t)bt * nb + k];
                }
            }
            y[(int64_t)bt * nrows + r] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Greedy argmax: the largest value, the first index on ties ([go-llm] index, */
/* Argmax; [dasLLAMA] 8.7.1.6.4 most_likely: strict '>' from index 0).        */
/* ------------------------------------------------------------------------- */

int64_t or_argmax_f32(const float* v, int64_t n) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

int64_t or_argmax_f64(const double* v, int64_t n) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

/* ------------------------------------------------------------------------- */
/* One decode step of a llama-style model for one sequence                    */
/* ([llmoxide] s7 "The block, and the residual stream"; [dasLLAMA] 8.7.1.6    */
/* forward):                                                                  */
/*   x = embed(token)                                                         */
/*   per layer: x += Wo . attn(rope(Wq xn), rope(Wk xn), Wv xn),              */
/*              xn = rmsnorm(x) * attn_norm;                                  */
/*              x += Wd . (silu(Wg xn) * (Wu xn)), xn = rmsnorm(x) * ffn_norm */
/*   logits = W_out . (rmsnorm(x) * out_norm); next = argmax(logits)           */
/* The new k, v are appended to the f32 cache at pos before attending over    */
/* positions 0..pos ([llmoxide] s12; [dasLLAMA] 8.7.1.6.2); with kv_f16 they  */
/* are rounded through binary16 first (the cache then holds f16 values).     */
/*                                                                            */
/* tensors[] (host pointers, model-file layouts):                             */
/*   [0] token embedding (emb_fmt, vocab x dim)  [1] out_norm f32[dim]        */
/*   [2] output head (emb_fmt, vocab x dim) or NULL when tied to [0]          */
/*   then for each layer l, at 3 + 9l: attn_norm, wq, wk, wv, wo, ffn_norm,   */
/*   wg, wu, wd.                                                              */
/* k_cache, v_cache: this sequence's cache, element (l, kvh, p, i) at         */
/*   l*layer_stride + (kvh*max_ctx + p)*hd + i.                               */
/* ------------------------------------------------------------------------- */

typedef struct {
    int layers, dim, ffn, n_heads, n_kv_heads, head_dim, vocab, max_ctx;
    double rope_theta, eps;
    int pairing, w_fmt, emb_fmt;
    int kv_f16; /* 1: the cache stores k and v rounded through binary16 ([go-llm] RoundF16) */
    int act_q8; /* 1: every quantised product takes its activations (rounded to f32) as Q8_0
                 * -- Q8_1 for Q4_1 weights -- and multiplies in integers ([go-llm]
                 * "ExactGGML"; or_quantize_q8, or_gemv_q8act) */
    /* the format of each class of layer matrix: wq, wk, wv; wo; wg, wu; wd (model files
     * mix formats by tensor: [llamini] "Quants", [go-llm] package overview).  w_fmt is the
     * format of a model that does not mix; the caller sets all four to it then. */
    int qkv_fmt, wo_fmt, gate_up_fmt, down_fmt;
} or_config;

int or_quantize_q8(const float* x, int64_t n, int8_t* q, float* d16, float* s16);
int or_gemv_q8act(int fmt, const uint8_t* w, int64_t rows, int64_t cols, const int8_t* xq, const float* xd,
                  const float* xs, int batch, int64_t row0, int64_t nrows, double* y);

/* Teacher-forcing slots of the Q8 activations (act_q8): one per quantised input of the
 * step, in order -- per layer l the QKV input (4l), the attention output (4l + 1), the
 * feed-forward input (4l + 2), the SwiGLU output (4l + 3) -- and the head's input (4L). */
typedef struct {
    const int8_t* q_given; /* [slots][slot_cols] codes to use instead of quantising, or NULL */
    const float* d_given;  /* [slots][slot_cols / 32] their (binary16) block scales          */
    float* x_out;          /* [slots][slot_cols] the f32 inputs the step formed, or NULL     */
    int64_t slot_cols;     /* row length of the three arrays                                 */
} or_q8_tf;

/* y[0..rows) = W x for one activation vector: over the f32-rounded activations' Q8 blocks
 * (act_q8) or, otherwise, the plain double product.  With act_q8, slot `slot` of tf (when
 * given) receives the f32 input, and supplies the codes and scales to multiply instead of
 * the quantisation of that input (Q4_0 / Q8_0 weights only: Q4_1 would also need the
 * Q8_1 sums). */
static int product(const or_config* c, int fmt, const uint8_t* w, int64_t rows, int64_t cols, const double* x,
                   double* y, const or_q8_tf* tf, int slot) {
    if (!c->act_q8) {
        gemv_rows_d(fmt, w, rows, cols, x, 1, cols, y, rows, 0, rows);
        return 0;
    }
    if (tf && tf->q_given && (fmt == OR_Q4_1 || !tf->d_given || cols > tf->slot_cols)) return -1;
    float* xf = (float*)malloc(sizeof(float) * (size_t)cols);
    int8_t* q = (int8_t*)malloc((size_t)cols);
    float* d = (float*)malloc(sizeof(float) * (size_t)(cols / 32));
    float* sm = (float*)malloc(sizeof(float) * (size_t)(cols / 32));
    int rc = -2;
    if (xf && q && d && sm) {
        for (int64_t i = 0; i < cols; ++i) xf[i] = (float)x[i];
        if (tf && tf->x_out) memcpy(tf->x_out + (int64_t)slot * tf->slot_cols, xf, sizeof(float) * (size_t)cols);
        if (tf && tf->q_given) {
            memcpy(q, tf->q_given + (int64_t)slot * tf->slot_cols, (size_t)cols);
            memcpy(d, tf->d_given + (int64_t)slot * (tf->slot_cols / 32), sizeof(float) * (size_t)(cols / 32));
            rc = 0;
        } else {
            rc = or_quantize_q8(xf, cols, q, d, sm);
        }
        if (!rc) rc = or_gemv_q8act(fmt, w, rows, cols, q, d, sm, 1, 0, rows, y);
    }
    free(xf); free(q); free(d); free(sm);
    return rc;
}

/* The step with test hooks for teacher forcing against another implementation; the
 * arithmetic is the step's own.
 *   kv_given = 1: the cache already holds this step's k and v at pos (the other
 *     implementation's values); the step attends over the cache as it is and does not
 *     write it.
 *   kv_out (or NULL): receives the k and v the step formed, rounded to f32 but before any
 *     binary16 rounding, as [layer][2][n_kv_heads * head_dim] (k, then v).
 *   head_x (or NULL): receives the head's input, the final normed x rounded to f32.
 *   tf (or NULL; act_q8 only): per quantised input, the f32 values formed and the codes
 *     and scales to multiply instead (or_q8_tf above). */
int or_decode_step_tf(const or_config* c, const void* const* tensors, float* k_cache, float* v_cache,
                      int64_t layer_stride, int pos, int token, double* logits, int64_t* next_token, int kv_given,
                      float* kv_out, float* head_x, const or_q8_tf* tf) {
    if (!c || pos < 0 || pos >= c->max_ctx || token < 0 || token >= c->vocab) return -1;
    if (c->n_heads % c->n_kv_heads) return -1;
    const int D = c->dim, F = c->ffn, hd = c->head_dim, hq = c->n_heads, hk = c->n_kv_heads;
    const int QD = hq * hd, KD = hk * hd;
    double* x = (double*)calloc((size_t)D, sizeof(double));
    double* xn = (double*)calloc((size_t)D, sizeof(double));
    double* q = (double*)calloc((size_t)QD, sizeof(double));
    double* k = (double*)calloc((size_t)KD, sizeof(double));
    double* v = (double*)calloc((size_t)KD, sizeof(double));
    double* att = (double*)calloc((size_t)QD, sizeof(double));
    double* t = (double*)calloc((size_t)(D > F ? D : F), sizeof(double));
    double* g = (double*)calloc((size_t)F, sizeof(double));
    double* u = (double*)calloc((size_t)F, sizeof(double));
    float* erow = (float*)calloc((size_t)D, sizeof(float));
    int rc = 0;
    if (!x || !xn || !q || !k || !v || !att || !t || !g || !u || !erow) {
        rc = -2;
        goto done;
    }
    /* embedding: row `token` of the table ([llmoxide] s3) */
    dequant_row(c->emb_fmt, (const uint8_t*)tensors[0], c->vocab, D, token, erow);
    for (int i = 0; i < D; ++i) x[i] = erow[i];

    for (int l = 0; l < c->layers; ++l) {
        const void* const* L = tensors + 3 + 9 * l;
        float* kl = k_cache + (int64_t)l * layer_stride;
        float* vl = v_cache + (int64_t)l * layer_stride;
        /* attention block */
        or_rmsnorm_d(x, (const float*)L[0], D, c->eps, xn);
        if ((rc = product(c, c->qkv_fmt, (const uint8_t*)L[1], QD, D, xn, q, tf, 4 * l)) ||
            (rc = product(c, c->qkv_fmt, (const uint8_t*)L[2], KD, D, xn, k, tf, 4 * l)) ||
            (rc = product(c, c->qkv_fmt, (const uint8_t*)L[3], KD, D, xn, v, tf, 4 * l)))
            goto done;
        for (int h = 0; h < hq; ++h) or_rope_head_d(q + (int64_t)h * hd, hd, pos, c->pairing, c->rope_theta);
        for (int h = 0; h < hk; ++h) or_rope_head_d(k + (int64_t)h * hd, hd, pos, c->pairing, c->rope_theta);
        for (int h = 0; h < hk; ++h)
            for (int i = 0; i < hd; ++i) {
                float kf = (float)k[h * hd + i], vf = (float)v[h * hd + i];
                if (kv_out) {
                    kv_out[(int64_t)l * 2 * KD + h * hd + i] = kf;
                    kv_out[(int64_t)l * 2 * KD + KD + h * hd + i] = vf;
                }
                if (c->kv_f16) {
                    kf = or_round_f16(kf);
                    vf = or_round_f16(vf);
                }
                if (!kv_given) {
                    kl[((int64_t)h * c->max_ctx + pos) * hd + i] = kf;
                    vl[((int64_t)h * c->max_ctx + pos) * hd + i] = vf;
                }
            }
        or_attention_d(q, kl, vl, hq, hk, hd, pos + 1, c->max_ctx, att);
        if ((rc = product(c, c->wo_fmt, (const uint8_t*)L[4], D, QD, att, t, tf, 4 * l + 1))) goto done;
        for (int i = 0; i < D; ++i) x[i] += t[i];
        /* feed-forward block */
        or_rmsnorm_d(x, (const float*)L[5], D, c->eps, xn);
        if ((rc = product(c, c->gate_up_fmt, (const uint8_t*)L[6], F, D, xn, g, tf, 4 * l + 2)) ||
            (rc = product(c, c->gate_up_fmt, (const uint8_t*)L[7], F, D, xn, u, tf, 4 * l + 2)))
            goto done;
        for (int i = 0; i < F; ++i) g[i] = or_silu(g[i]) * u[i];
        if ((rc = product(c, c->down_fmt, (const uint8_t*)L[8], D, F, g, t, tf, 4 * l + 3))) goto done;
        for (int i = 0; i < D; ++i) x[i] += t[i];
    }
    or_rmsnorm_d(x, (const float*)tensors[1], D, c->eps, xn);
    if (head_x)
        for (int i = 0; i < D; ++i) head_x[i] = (float)xn[i];
    {
        const uint8_t* head = (const uint8_t*)(tensors[2] ? tensors[2] : tensors[0]);
        if ((rc = product(c, c->emb_fmt, head, c->vocab, D, xn, logits, tf, 4 * c->layers))) goto done;
    }
    if (next_token) *next_token = or_argmax_f64(logits, c->vocab);
done:
    free(x); free(xn); free(q); free(k); free(v); free(att); free(t); free(g); free(u); free(erow);
    return rc;
}

int or_decode_step(const or_config* c, const void* const* tensors, float* k_cache, float* v_cache,
                   int64_t layer_stride, int pos, int token, double* logits, int64_t* next_token) {
    return or_decode_step_tf(c, tensors, k_cache, v_cache, layer_stride, pos, token, logits, next_token, 0, NULL,
                             NULL, NULL);
}

int or_abi_version(void) { return 1; }

/* Threads for the OpenMP loops above (1 = single-threaded; the per-output summation order
 * does not depend on it, so results are identical).  Returns the count now in use. */
int or_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}
