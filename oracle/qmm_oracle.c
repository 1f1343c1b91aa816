/*
 * qmm_oracle.c -- CPU oracle for the block-quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check in __graft_entry__.py
 * and the CPU-baseline leg of bench.py may load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Plain, slow, obviously-correct restatement of what the method computes.
 * Floating point is fp64 except where the q8_1 format itself fixes fp32/fp16
 * (the activation quantizer), which is written out in fp32 exactly as defined.
 *
 * Sources (web pages on block-quantized matmul):
 *   [MMQ]   "llama.cpp 源码完全拆解(十五): 量化 GEMM 的矩阵编队 -- MMQ 如何把 MoE 与预填充塞满 GPU"
 *   [P0007] "Patch 0007: an fp16 matrix-vector path for GP100" (p100-llama-cpp, docs/fp16-mmvq.md)
 *   [QMM]   "QTensor 与 QMatMul" (candle 0.11.0 notes, rustineverything.app)
 *
 * Readings taken where the pages are silent or garbled:
 *   - q8_1 block = {fp16 d, fp16 s, int8 q[32]} (36 B); d = amax/127 in fp32,
 *     q = roundf(x/d) with IEEE fp32 division (ties away from zero),
 *     stored d_h = fp16_rne(d), s_h = fp16_rne(d_h * sum(q)); if the fp32 d is 0
 *     the whole block is zero.  [MMQ] section "dp4a 路径的 Q4_K" names s = d*sum(q).
 *   - Q4_K block = {fp16 d, fp16 dmin, 12 B packed 6-bit scales/mins, 128 B nibbles};
 *     scale/min packing is the GGUF rule that [MMQ] section
 *     "Q4_K: 在加载期就把两层 scale 合并成 half2" refers to (its own sentence is garbled).
 *     Nibbles: 4 chunks of 32 bytes; in chunk c byte l holds weight 64c+l in its low
 *     nibble and weight 64c+32+l in its high nibble ([MMQ] "dp4a 路径的 Q4_K":
 *     sub-block i of a 32-bit word takes nibble i).
 *   - Q5_K block = {fp16 d, fp16 dmin, 12 B packed 6-bit scales/mins, qh[32], qs[128]}
 *     (176 B).  [MMQ] section "Q4_K: 在加载期就把两层 scale 合并成 half2" says Q4_K and
 *     Q5_K share the 12-byte scale/min rule; the rest is read as Q4_K plus one bit plane:
 *     qs holds the low 4 bits in Q4_K's nibble order, and the fifth bit of weight 32j + l
 *     (sub-block j, l = 0..31) is bit j of qh[l]; value d*sc*q - dmin*m with q in 0..31.
 *   - Q6_K block = {ql[128], qh[64], int8 sc[16], fp16 d}; bit placement as pinned by
 *     the index arithmetic in [MMQ] "Q6_K: 6 位数据要多占一半的共享内存"; code - 32.
 *   - Q8_0 block = {fp16 d, int8 q[32]}.
 *   - Q4_0 block = {fp16 d, 16 B nibbles} (18 B per 32 weights, [MMQ] sections
 *     "tile_x_sizes" and "Q4_0: 一个 get_int_b2 搬进 8 个 4-bit"): byte i holds weight i
 *     in its low nibble and weight 16+i in its high nibble (the load side splits the
 *     nibbles of a word into the front and back halves of the block); the value is
 *     d*(q - 8), and the dot takes the offset codes q - 8 in -8..7 as its integers,
 *     as the load side does with __vsub4 before the dot.
 *
 * Parity status: every exported function is pinned by tests under tests/ against
 * closed forms, library routines, brute force or the pages' printed sizes
 * (see test_oracle_*.py); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_API __attribute__((visibility("default")))

enum { OT_Q4_0 = 2, OT_Q8_0 = 8, OT_Q4_K = 12, OT_Q5_K = 13, OT_Q6_K = 14 };

/* ---------------------------------------------------------------- fp16 */

/* IEEE binary16 -> double (exact). */
ORACLE_API double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* fp32 -> IEEE binary16, round to nearest, ties to even.  Written from the
 * definition: scale to the fp16 quantum of the binade, rint (ties-to-even in
 * the default rounding mode), re-encode. */
ORACLE_API uint16_t oracle_float_to_half(float xf) {
    double x = (double)xf;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(a)) return (uint16_t)(sign | 0x7e00);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);  /* rounds to infinity */
    if (a < ldexp(1.0, -14)) {                           /* subnormal binade (and zero) */
        double q = rint(ldexp(a, 24));                   /* multiples of 2^-24; q <= 1024 */
        return (uint16_t)(sign | (uint16_t)q);           /* q == 1024 encodes 2^-14 */
    }
    int e;
    frexp(a, &e);                                        /* a in [2^(e-1), 2^e) */
    int E = e - 1;
    double q = rint(ldexp(a, 10 - E));                   /* in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)q - 1024));
}

static double h2d(const uint8_t *p) {
    uint16_t h = (uint16_t)(p[0] | (p[1] << 8));
    return oracle_half_to_double(h);
}

static void put_half(uint8_t *p, uint16_t h) {
    p[0] = (uint8_t)(h & 0xff);
    p[1] = (uint8_t)(h >> 8);
}

/* ---------------------------------------------------------------- q8_1 */

/* x: fp32 [m][k] row-major; out: [m][k/32] blocks of 36 bytes.
 * Returns 0, or -1 if k is not a multiple of 32. */
ORACLE_API int oracle_quantize_q8_1(const float *x, int64_t m, int64_t k, uint8_t *out) {
    if (k % 32) return -1;
    int64_t nb = k / 32;
    for (int64_t r = 0; r < m; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + r * k + 32 * b;
            uint8_t *ob = out + (r * nb + b) * 36;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;                     /* IEEE fp32 division */
            int S = 0;
            for (int i = 0; i < 32; ++i) {
                int q = 0;
                if (d != 0.0f) q = (int)roundf(xb[i] / d);  /* fp32 divide, round half away */
                ob[4 + i] = (uint8_t)(int8_t)q;
                S += q;
            }
            uint16_t dh = oracle_float_to_half(d);
            float dhf = (float)oracle_half_to_double(dh);
            uint16_t sh = oracle_float_to_half(dhf * (float)S);  /* exact fp32 product, one rounding */
            if (d == 0.0f) { dh = 0; sh = 0; }
            put_half(ob + 0, dh);
            put_half(ob + 2, sh);
        }
    }
    return 0;
}

/* fp64 values d_h * q of q8_1 blocks: out [m][k]. */
ORACLE_API int oracle_dequant_q8_1(const uint8_t *xq, int64_t m, int64_t k, double *out) {
    if (k % 32) return -1;
    int64_t nb = k / 32;
    for (int64_t r = 0; r < m; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = xq + (r * nb + b) * 36;
            double d = h2d(blk);
            for (int i = 0; i < 32; ++i) out[r * k + 32 * b + i] = d * (double)(int8_t)blk[4 + i];
        }
    return 0;
}

/* ---------------------------------------------------------------- weight blocks */

static int block_elems(int type) { return type == OT_Q8_0 || type == OT_Q4_0 ? 32 : 256; }
static int block_bytes(int type) {
    switch (type) {
    case OT_Q4_K: return 144;
    case OT_Q5_K: return 176;
    case OT_Q6_K: return 210;
    case OT_Q8_0: return 34;
    case OT_Q4_0: return 18;
    default: return -1;
    }
}

ORACLE_API int oracle_block_bytes(int type) { return block_bytes(type); }
ORACLE_API int oracle_block_elems(int type) { return block_bytes(type) < 0 ? -1 : block_elems(type); }

/* Q4_K sub-block j (0..7): 6-bit scale and min from the 12 packed bytes. */
static void q4k_scale_min(const uint8_t *s12, int j, int *sc, int *mn) {
    if (j < 4) {
        *sc = s12[j] & 63;
        *mn = s12[j + 4] & 63;
    } else {
        *sc = (s12[j + 4] & 0x0f) | ((s12[j - 4] >> 6) << 4);
        *mn = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
    }
}

/* Q4_K weight i (0..255): its 4-bit code. */
static int q4k_code(const uint8_t *blk, int i) {
    const uint8_t *qs = blk + 16;
    int c = i / 64, t = i % 64;
    return t < 32 ? (qs[32 * c + t] & 0x0f) : (qs[32 * c + t - 32] >> 4);
}

/* Q5_K weight i (0..255): its 5-bit code, the Q4_K-ordered nibble of qs plus bit i/32 of
 * qh[i%32] as the fifth bit. */
static int q5k_code(const uint8_t *blk, int i) {
    const uint8_t *qh = blk + 16, *qs = blk + 48;
    int c = i / 64, t = i % 64;
    int low = t < 32 ? (qs[32 * c + t] & 0x0f) : (qs[32 * c + t - 32] >> 4);
    int high = (qh[i % 32] >> (i / 32)) & 1;
    return low | (high << 4);
}

/* Q6_K weight i (0..255): its code minus 32, in -32..31. */
static int q6k_value(const uint8_t *blk, int i) {
    const uint8_t *ql = blk, *qh = blk + 128;
    int h = i / 128, r = i % 128, t = r / 32, l = r % 32;
    int low = (ql[64 * h + l + 32 * (t & 1)] >> (4 * (t >> 1))) & 0x0f;
    int high = (qh[32 * h + l] >> (2 * t)) & 3;
    return (low | (high << 4)) - 32;
}

/* Q4_0 weight i (0..31): its offset code q - 8, in -8..7. */
static int q40_value(const uint8_t *blk, int i) {
    const uint8_t *qs = blk + 2;
    return (i < 16 ? (qs[i] & 0x0f) : (qs[i - 16] >> 4)) - 8;
}

/* Decoded fields of one Q4_K block, for tests. */
ORACLE_API int oracle_q4_K_fields(const uint8_t *blk, double *d, double *dmin, int *sc8, int *mn8, int *q256) {
    *d = h2d(blk);
    *dmin = h2d(blk + 2);
    for (int j = 0; j < 8; ++j) q4k_scale_min(blk + 4, j, &sc8[j], &mn8[j]);
    for (int i = 0; i < 256; ++i) q256[i] = q4k_code(blk, i);
    return 0;
}

ORACLE_API int oracle_q5_K_fields(const uint8_t *blk, double *d, double *dmin, int *sc8, int *mn8, int *q256) {
    *d = h2d(blk);
    *dmin = h2d(blk + 2);
    for (int j = 0; j < 8; ++j) q4k_scale_min(blk + 4, j, &sc8[j], &mn8[j]);
    for (int i = 0; i < 256; ++i) q256[i] = q5k_code(blk, i);
    return 0;
}

ORACLE_API int oracle_q6_K_fields(const uint8_t *blk, double *d, int *sc16, int *q256) {
    *d = h2d(blk + 208);
    for (int j = 0; j < 16; ++j) sc16[j] = (int8_t)blk[192 + j];
    for (int i = 0; i < 256; ++i) q256[i] = q6k_value(blk, i);
    return 0;
}

/* fp64 dequantized weight rows: W [n][k/QK blocks] -> out [n][k]. */
ORACLE_API int oracle_dequant(int type, const uint8_t *W, int64_t n, int64_t k, double *out) {
    int bb = block_bytes(type), qk;
    if (bb < 0) return -2;
    qk = block_elems(type);
    if (k % qk) return -1;
    int64_t nb = k / qk;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = W + (r * nb + b) * bb;
            double *o = out + r * k + b * qk;
            if (type == OT_Q4_K || type == OT_Q5_K) {
                double d = h2d(blk), dmin = h2d(blk + 2);
                for (int i = 0; i < 256; ++i) {
                    int sc, mn;
                    q4k_scale_min(blk + 4, i / 32, &sc, &mn);
                    int q = type == OT_Q4_K ? q4k_code(blk, i) : q5k_code(blk, i);
                    o[i] = d * sc * q - dmin * mn;
                }
            } else if (type == OT_Q6_K) {
                double d = h2d(blk + 208);
                for (int i = 0; i < 256; ++i) o[i] = d * (int8_t)blk[192 + i / 16] * q6k_value(blk, i);
            } else if (type == OT_Q4_0) {
                double d = h2d(blk);
                for (int i = 0; i < 32; ++i) o[i] = d * q40_value(blk, i);
            } else {
                double d = h2d(blk);
                for (int i = 0; i < 32; ++i) o[i] = d * (int8_t)blk[2 + i];
            }
        }
    return 0;
}

/* ---------------------------------------------------------------- the fold */

/* One output element y[c][r] = sum over the row's sub-blocks of
 * (exact integer sub-block dot) x (block scales), in fp64, plus
 * T = sum of |each block term| (both terms separately for Q4_K).
 *
 * Q4_K ([MMQ] "dp4a 路径的 Q4_K"): per 32-wide sub-block b of a superblock,
 *     d*sc_b*d8_b*sumi_b - dmin*m_b*s8_b.
 * Q5_K: the same with the 5-bit codes.
 * Q6_K ([MMQ] "Q6_K: 子块尺度与 q8_1 块长错位"): per 16-wide sub-block j,
 *     d*sc_j*d8_{j/2}*sumi_j.
 * Q8_0: per 32-block, d_w*d8*sumi.
 * Q4_0: per 32-block, d_w*d8*sumi with sumi over the offset codes q - 8.
 */
static void fold_one(int type, const uint8_t *wrow, const uint8_t *xrow, int64_t k, double *y, double *T) {
    double acc = 0.0, tabs = 0.0;
    if (type == OT_Q4_K || type == OT_Q5_K) {
        const int bb = type == OT_Q4_K ? 144 : 176;
        for (int64_t s = 0; s < k / 256; ++s) {
            const uint8_t *blk = wrow + s * bb;
            double d = h2d(blk), dmin = h2d(blk + 2);
            for (int b = 0; b < 8; ++b) {
                const uint8_t *xb = xrow + (s * 8 + b) * 36;
                double d8 = h2d(xb), s8 = h2d(xb + 2);
                int sc, mn;
                q4k_scale_min(blk + 4, b, &sc, &mn);
                int64_t sumi = 0;
                for (int i = 0; i < 32; ++i) {
                    int q = type == OT_Q4_K ? q4k_code(blk, 32 * b + i) : q5k_code(blk, 32 * b + i);
                    sumi += (int64_t)q * (int8_t)xb[4 + i];
                }
                double t1 = d * sc * d8 * (double)sumi;
                double t2 = dmin * mn * s8;
                acc += t1 - t2;
                tabs += fabs(t1) + fabs(t2);
            }
        }
    } else if (type == OT_Q6_K) {
        for (int64_t s = 0; s < k / 256; ++s) {
            const uint8_t *blk = wrow + s * 210;
            double d = h2d(blk + 208);
            for (int j = 0; j < 16; ++j) {
                const uint8_t *xb = xrow + (s * 8 + j / 2) * 36;
                double d8 = h2d(xb);
                int64_t sumi = 0;
                for (int i = 0; i < 16; ++i) {
                    int w = 16 * j + i;
                    sumi += (int64_t)q6k_value(blk, w) * (int8_t)xb[4 + (w % 32)];
                }
                double t = d * (int8_t)blk[192 + j] * d8 * (double)sumi;
                acc += t;
                tabs += fabs(t);
            }
        }
    } else if (type == OT_Q4_0) {
        for (int64_t b = 0; b < k / 32; ++b) {
            const uint8_t *blk = wrow + b * 18;
            const uint8_t *xb = xrow + b * 36;
            int64_t sumi = 0;
            for (int i = 0; i < 32; ++i) sumi += (int64_t)q40_value(blk, i) * (int8_t)xb[4 + i];
            double t = h2d(blk) * h2d(xb) * (double)sumi;
            acc += t;
            tabs += fabs(t);
        }
    } else {
        for (int64_t b = 0; b < k / 32; ++b) {
            const uint8_t *blk = wrow + b * 34;
            const uint8_t *xb = xrow + b * 36;
            int64_t sumi = 0;
            for (int i = 0; i < 32; ++i) sumi += (int64_t)(int8_t)blk[2 + i] * (int8_t)xb[4 + i];
            double t = h2d(blk) * h2d(xb) * (double)sumi;
            acc += t;
            tabs += fabs(t);
        }
    }
    *y = acc;
    if (T) *T = tabs;
}

static int check_shape(int type, int64_t k) {
    int bb = block_bytes(type);
    if (bb < 0) return -2;
    if (k % block_elems(type) || k % 32) return -1;
    return 0;
}

/* y[m][n] = sum_k x[m,k] * dequant(W)[n,k], computed as the fold above.
 * W: [n] rows of k/QK blocks; xq: [m][k/32] q8_1 blocks.  y, T: fp64 [m][n]. */
ORACLE_API int oracle_mul_mat(int type, const uint8_t *W, int64_t n, int64_t k, const uint8_t *xq, int64_t m,
                              double *y, double *T) {
    int rc = check_shape(type, k);
    if (rc) return rc;
    int64_t rb = (k / block_elems(type)) * block_bytes(type);
    int64_t xb = (k / 32) * 36;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int64_t c = 0; c < m; ++c)
            fold_one(type, W + r * rb, xq + c * xb, k, &y[c * n + r], T ? &T[c * n + r] : NULL);
    return 0;
}

/* The same fold for a list of (row, col) output positions: y[i] = y[cols[i]][rows[i]]. */
ORACLE_API int oracle_mul_mat_at(int type, const uint8_t *W, int64_t n, int64_t k, const uint8_t *xq, int64_t m,
                                 const int64_t *rows, const int64_t *cols, int64_t count, double *y, double *T) {
    int rc = check_shape(type, k);
    if (rc) return rc;
    int64_t rb = (k / block_elems(type)) * block_bytes(type);
    int64_t xb = (k / 32) * 36;
    for (int64_t i = 0; i < count; ++i)
        if (rows[i] < 0 || rows[i] >= n || cols[i] < 0 || cols[i] >= m) return -3;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i)
        fold_one(type, W + rows[i] * rb, xq + cols[i] * xb, k, &y[i], T ? &T[i] : NULL);
    return 0;
}

/* Brute force on tiny shapes: y_B[m][n] = sum_i w_fp64[n,i] * (d_h*q)[m,i]. */
ORACLE_API int oracle_brute(int type, const uint8_t *W, int64_t n, int64_t k, const uint8_t *xq, int64_t m, double *y) {
    int rc = check_shape(type, k);
    if (rc) return rc;
    double *w = (double *)malloc(sizeof(double) * n * k);
    double *x = (double *)malloc(sizeof(double) * m * k);
    if (!w || !x) { free(w); free(x); return -4; }
    oracle_dequant(type, W, n, k, w);
    oracle_dequant_q8_1(xq, m, k, x);
    for (int64_t c = 0; c < m; ++c)
        for (int64_t r = 0; r < n; ++r) {
            double acc = 0.0;
            for (int64_t i = 0; i < k; ++i) acc += w[r * k + i] * x[c * k + i];
            y[c * n + r] = acc;
        }
    free(w);
    free(x);
    return 0;
}

/* ---------------------------------------------------------------- MoE */

/* Expert bucketing ([MMQ] "专家边界: 在 GPU 上做分段"): a stable counting sort of
 * the (token, slot) pairs by expert id.  bounds[e]..bounds[e+1] is expert e's
 * range in perm; perm[i] = token*top_k + slot.  Pairs whose id is outside
 * [0, n_experts) are left out; returns their count. */
ORACLE_API int64_t oracle_bucket(const int32_t *ids, int64_t n_tokens, int64_t top_k, int64_t n_experts,
                                 int32_t *bounds, int32_t *perm) {
    int64_t bad = 0, pos = 0;
    for (int64_t e = 0; e < n_experts; ++e) {
        bounds[e] = (int32_t)pos;
        for (int64_t i = 0; i < n_tokens * top_k; ++i)
            if (ids[i] == e) perm[pos++] = (int32_t)i;
    }
    bounds[n_experts] = (int32_t)pos;
    for (int64_t i = 0; i < n_tokens * top_k; ++i)
        if (ids[i] < 0 || ids[i] >= n_experts) ++bad;
    return bad;
}

/* mul_mat_id: y[t][s][n] = mul_mat(W_experts[ids[t][s]], x row)[n], the x row being
 * t (shared by a token's slots) or, with x_per_slot, t*top_k + s (one row per slot, as
 * in a MoE down projection).  Invalid ids give a zero output row (and T = 0).  Returns
 * the number of invalid ids, or a negative error. */
static int64_t mul_mat_id_rows(int type, const uint8_t *W, int64_t n_experts, int64_t n, int64_t k,
                               const uint8_t *xq, int x_per_slot, const int32_t *ids, int64_t top_k,
                               int64_t n_tokens, double *y, double *T) {
    int rc = check_shape(type, k);
    if (rc) return rc;
    int64_t rb = (k / block_elems(type)) * block_bytes(type);
    int64_t xb = (k / 32) * 36;
    int64_t bad = 0;
    for (int64_t i = 0; i < n_tokens * top_k; ++i)
        if (ids[i] < 0 || ids[i] >= n_experts) ++bad;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n_tokens * top_k; ++i) {
        int64_t xrow = x_per_slot ? i : i / top_k;
        int32_t e = ids[i];
        for (int64_t r = 0; r < n; ++r) {
            double *yy = &y[i * n + r];
            double *tt = T ? &T[i * n + r] : NULL;
            if (e < 0 || e >= n_experts) {
                *yy = 0.0;
                if (tt) *tt = 0.0;
            } else {
                fold_one(type, W + ((int64_t)e * n + r) * rb, xq + xrow * xb, k, yy, tt);
            }
        }
    }
    return bad;
}

ORACLE_API int64_t oracle_mul_mat_id(int type, const uint8_t *W, int64_t n_experts, int64_t n, int64_t k,
                                     const uint8_t *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens,
                                     double *y, double *T) {
    return mul_mat_id_rows(type, W, n_experts, n, k, xq, 0, ids, top_k, n_tokens, y, T);
}

ORACLE_API int64_t oracle_mul_mat_id_slot(int type, const uint8_t *W, int64_t n_experts, int64_t n, int64_t k,
                                          const uint8_t *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens,
                                          double *y, double *T) {
    return mul_mat_id_rows(type, W, n_experts, n, k, xq, 1, ids, top_k, n_tokens, y, T);
}

/* ---------------------------------------------------------------- threads */

ORACLE_API int oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
