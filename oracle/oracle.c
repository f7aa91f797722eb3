/*
 * oracle.c — plain CPU reference of the routed-MoE block (test
 * infrastructure; see oracle.h).  Plain C11, built with -ffp-contract=off so
 * every fp32 expression below is rounded exactly as written; OpenMP only
 * spreads independent output rows over threads (each row is still summed by
 * one thread in index order).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t rd32(const uint8_t *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

float oracle_fp16_to_f32(uint16_t h) {
    /* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, man = h & 1023;
    float v;
    if (ex == 0)
        v = ldexpf((float)man, -24); /* subnormal: man * 2^-24 */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexpf((float)(man | 1024), ex - 25); /* 1.man * 2^(ex-15) */
    return sign ? -v : v;
}

uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40); /* quiet nan */
    /* round to nearest, ties to even: add 0x7fff plus the lsb that stays */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

int oracle_block_bytes(int qtype) {
    switch (qtype) {
    case ORACLE_IQ2_XXS: return 66; /* uint16 d; uint16 qs[32]           */
    case ORACLE_Q2_K: return 84;    /* scales[16]; qs[64]; d; dmin       */
    case ORACLE_Q4_K: return 144;   /* d; dmin; scales[12]; qs[128]      */
    default: return 0;
    }
}

/* IQ2_XXS block ([P5] §2.3 block_iq2_xxs: fp16 d, then 64 bytes of codes).
 * Reading of the inner layout (GGUF convention): 8 sub-blocks of 32 weights;
 * sub-block b owns code bytes 8b..8b+7.  Bytes 0..3 are four grid-row indices
 * (each row = 8 weights, [P5] §2.4), bytes 4..7 a little-endian word v whose
 * bits 7l..7l+6 are the sign bits of row l (the 8th sign is the parity of the
 * 7, so an even number of weights is negative) and whose top nibble ls scales
 * the sub-block: db = d * (0.5 + ls) * 0.25. */
static void deq_iq2_xxs_block(const uint8_t *blk, const uint8_t *grid, float *y) {
    const float d = oracle_fp16_to_f32(rd16(blk));
    const uint8_t *q = blk + 2;
    for (int b = 0; b < 8; ++b) {
        const uint8_t *s = q + 8 * b;
        const uint32_t v = rd32(s + 4);
        const float db = (d * (0.5f + (float)(v >> 28))) * 0.25f;
        for (int l = 0; l < 4; ++l) {
            const uint8_t *row = grid + 8 * (int)s[l];
            const uint32_t s7 = (v >> (7 * l)) & 127u;
            int par = 0;
            for (int i = 0; i < 7; ++i) par ^= (int)((s7 >> i) & 1u);
            const uint32_t signs = s7 | ((uint32_t)par << 7);
            for (int j = 0; j < 8; ++j) {
                int g = (int)row[j];
                if ((signs >> j) & 1u) g = -g;
                y[32 * b + 8 * l + j] = db * (float)g;
            }
        }
    }
}

/* Q2_K block ([P5] §2.3 block_q2_K: scales[16], qs[64], fp16 d, fp16 dmin).
 * Reading: weight n = 128h + 32j + l takes the 2-bit field j of byte
 * qs[32h + l]; its 16-weight sub-block is 8h + 2j + (l >= 16); a scale byte
 * holds sc (low nibble) and m (high nibble); w = d*sc*q - dmin*m with the
 * multiply-subtract as one fused rounding. */
static void deq_q2_k_block(const uint8_t *blk, float *y) {
    const uint8_t *sc = blk, *qs = blk + 16;
    const float d = oracle_fp16_to_f32(rd16(blk + 80));
    const float dmin = oracle_fp16_to_f32(rd16(blk + 82));
    for (int n = 0; n < 256; ++n) {
        const int h = n / 128, j = (n % 128) / 32, l = n % 32;
        const int q = (qs[32 * h + l] >> (2 * j)) & 3;
        const int sb = 8 * h + 2 * j + (l >= 16 ? 1 : 0);
        const int s = sc[sb] & 15, m = sc[sb] >> 4;
        y[n] = fmaf(d * (float)s, (float)q, -(dmin * (float)m));
    }
}

/* Q4_K block (fp16 d, fp16 dmin, 12 bytes of 6-bit scale/min pairs, 128
 * bytes of nibbles).  Reading: sub-block i (32 weights) has
 *   i < 4: sc = s[i] & 63, m = s[i+4] & 63
 *   i >= 4: sc = (s[i+4] & 15) | ((s[i-4] >> 6) << 4),
 *           m  = (s[i+4] >> 4) | ((s[i] >> 6) << 4)
 * and weight 64c + l (l < 32) is the low nibble of qs[32c + l] (sub-block 2c),
 * weight 64c + 32 + l the high nibble (sub-block 2c + 1). */
static void deq_q4_k_block(const uint8_t *blk, float *y) {
    const float d = oracle_fp16_to_f32(rd16(blk));
    const float dmin = oracle_fp16_to_f32(rd16(blk + 2));
    const uint8_t *s = blk + 4, *qs = blk + 16;
    int scv[8], mv[8];
    for (int i = 0; i < 8; ++i) {
        if (i < 4) {
            scv[i] = s[i] & 63;
            mv[i] = s[i + 4] & 63;
        } else {
            scv[i] = (s[i + 4] & 15) | ((s[i - 4] >> 6) << 4);
            mv[i] = (s[i + 4] >> 4) | ((s[i] >> 6) << 4);
        }
    }
    for (int n = 0; n < 256; ++n) {
        const int c = n / 64, r = n % 64;
        int q, sb;
        if (r < 32) {
            q = qs[32 * c + r] & 15;
            sb = 2 * c;
        } else {
            q = qs[32 * c + r - 32] >> 4;
            sb = 2 * c + 1;
        }
        y[n] = fmaf(d * (float)scv[sb], (float)q, -(dmin * (float)mv[sb]));
    }
}

int oracle_dequant_row(int qtype, const uint8_t *row_blocks, int cols,
                       const uint8_t *grid, float *out) {
    if (!row_blocks || !out || cols <= 0 || cols % 256) return -1;
    const int bb = oracle_block_bytes(qtype);
    if (!bb) return -1;
    if (qtype == ORACLE_IQ2_XXS && !grid) return -1;
    for (int b = 0; b < cols / 256; ++b) {
        const uint8_t *blk = row_blocks + (size_t)b * bb;
        if (qtype == ORACLE_IQ2_XXS) deq_iq2_xxs_block(blk, grid, out + 256 * b);
        else if (qtype == ORACLE_Q2_K) deq_q2_k_block(blk, out + 256 * b);
        else deq_q4_k_block(blk, out + 256 * b);
    }
    return 0;
}

int oracle_dequantize(int qtype, const void *gguf, int rows, int cols,
                      const uint8_t *grid, float *out_f32, uint16_t *out_bf16) {
    if (!gguf || rows <= 0 || (!out_f32 && !out_bf16)) return -1;
    const int bb = oracle_block_bytes(qtype);
    if (!bb || cols <= 0 || cols % 256) return -1;
    float *row = (float *)malloc(sizeof(float) * (size_t)cols);
    if (!row) return -1;
    int rc = 0;
    for (int r = 0; r < rows && rc == 0; ++r) {
        rc = oracle_dequant_row(qtype, (const uint8_t *)gguf + (size_t)r * (cols / 256) * bb,
                                cols, grid, row);
        for (int c = 0; c < cols; ++c) {
            if (out_f32) out_f32[(size_t)r * cols + c] = row[c];
            if (out_bf16) out_bf16[(size_t)r * cols + c] = oracle_f32_to_bf16(row[c]);
        }
    }
    free(row);
    return rc;
}

/* ---------------------------------------------------------------- router */

typedef struct {
    double key;
    int e;
} key_id;

/* Larger key first; equal keys -> lower expert id first. */
static int cmp_key_id(const void *a, const void *b) {
    const key_id *x = (const key_id *)a, *y = (const key_id *)b;
    if (x->key > y->key) return -1;
    if (x->key < y->key) return 1;
    return (x->e > y->e) - (x->e < y->e);
}

/* Router ([P1] §3.2 "Router 计算专家选择", [P5] §2.1 six experts used).
 * Readings (pages silent): sigmoid score, bias added only for selection,
 * weights = selected unbiased scores / their sum, no extra scale. */
int oracle_route(const float *hidden, int T, int H, int E, int K,
                 const float *router, const float *bias, int32_t *ids,
                 float *w, double *keys_out, double *margin_out) {
    if (!hidden || !router || !bias || !ids || !w || T < 1 || H < 1 || E < 1 ||
        K < 1 || K > E)
        return -1;
    key_id *kv = (key_id *)malloc(sizeof(key_id) * (size_t)E);
    double *s = (double *)malloc(sizeof(double) * (size_t)E);
    if (!kv || !s) {
        free(kv);
        free(s);
        return -1;
    }
    for (int t = 0; t < T; ++t) {
        const float *x = hidden + (size_t)t * H;
        for (int e = 0; e < E; ++e) {
            double logit = 0.0;
            for (int j = 0; j < H; ++j) logit += (double)x[j] * (double)router[(size_t)e * H + j];
            s[e] = 1.0 / (1.0 + exp(-logit));
            kv[e].key = s[e] + (double)bias[e];
            kv[e].e = e;
            if (keys_out) keys_out[(size_t)t * E + e] = kv[e].key;
        }
        qsort(kv, (size_t)E, sizeof(key_id), cmp_key_id);
        double ssum = 0.0;
        for (int k = 0; k < K; ++k) ssum += s[kv[k].e];
        for (int k = 0; k < K; ++k) {
            ids[(size_t)t * K + k] = kv[k].e;
            w[(size_t)t * K + k] = (float)(s[kv[k].e] / ssum);
        }
        if (margin_out) margin_out[t] = (K < E) ? kv[K - 1].key - kv[K].key : INFINITY;
    }
    free(kv);
    free(s);
    return 0;
}

/* ---------------------------------------------------------------- bucket */

int oracle_bucket(const int32_t *ids, int T, int K, int E, int32_t *counts,
                  int32_t *offsets, int32_t *perm, int32_t *inv) {
    if (!ids || !counts || !offsets || !perm || !inv || T < 1 || K < 1 || E < 1) return -1;
    const int n = T * K;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E) return -2;
        counts[ids[i]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    if (!fill) return -1;
    for (int i = 0; i < n; ++i) { /* entries visited in (t,k) order: stable */
        const int e = ids[i];
        const int pos = offsets[e] + fill[e]++;
        perm[pos] = i;
        inv[i] = pos;
    }
    free(fill);
    return 0;
}

void oracle_rmsnorm(const float *x, int T, int n, double eps, float *y) {
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int j = 0; j < n; ++j) ss += (double)x[(size_t)t * n + j] * (double)x[(size_t)t * n + j];
        const double r = 1.0 / sqrt(ss / n + eps);
        for (int j = 0; j < n; ++j) y[(size_t)t * n + j] = (float)((double)x[(size_t)t * n + j] * r);
    }
}

/* ------------------------------------------------------------ expert MLP */

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* out[r] = sum_c M[r][c] * v[c] for a GGUF-format or bf16 matrix [rows][cols],
 * each row dequantised to fp32 first, then summed in fp64 in index order. */
static int matvec(int qtype, const void *M, int rows, int cols, const uint8_t *grid,
                  const double *v, double *out, int nthreads) {
    if (!M) return -2;
    const int bb = qtype == ORACLE_BF16 ? 512 : oracle_block_bytes(qtype);
    if (!bb) return -1;
    int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads()) reduction(| : bad)
    {
        float *row = (float *)malloc(sizeof(float) * (size_t)cols);
        if (!row) bad = 1;
#pragma omp for schedule(static)
        for (int r = 0; r < rows; ++r) {
            if (!row) continue;
            if (qtype == ORACLE_BF16) {
                const uint16_t *src = (const uint16_t *)M + (size_t)r * cols;
                for (int c = 0; c < cols; ++c) row[c] = bf16_to_f32(src[c]);
            } else {
                oracle_dequant_row(qtype, (const uint8_t *)M + (size_t)r * (cols / 256) * bb, cols,
                                   grid, row);
            }
            double acc = 0.0;
            for (int c = 0; c < cols; ++c) acc += (double)row[c] * v[c];
            out[r] = acc;
        }
        free(row);
    }
    return bad ? -1 : 0;
}

static int expert_mlp_d(const double *x, int H, int F, int gut, int dt, const void *G,
                        const void *U, const void *D, const uint8_t *grid, double *y,
                        int nthreads) {
    double *g = (double *)malloc(sizeof(double) * (size_t)F);
    double *u = (double *)malloc(sizeof(double) * (size_t)F);
    int rc = (!g || !u) ? -1 : 0;
    if (!rc) rc = matvec(gut, G, F, H, grid, x, g, nthreads);
    if (!rc) rc = matvec(gut, U, F, H, grid, x, u, nthreads);
    if (!rc) {
        for (int i = 0; i < F; ++i) g[i] = silu(g[i]) * u[i]; /* SwiGLU, no clamp */
        rc = matvec(dt, D, H, F, grid, g, y, nthreads);
    }
    free(g);
    free(u);
    return rc;
}

int oracle_expert_mlp(const float *x, int H, int F, int gate_up_type, int down_type,
                      const void *G, const void *U, const void *D, const uint8_t *grid,
                      double *y, int nthreads) {
    if (!x || !y || H % 256 || F % 256 || H <= 0 || F <= 0) return -1;
    double *xd = (double *)malloc(sizeof(double) * (size_t)H);
    if (!xd) return -1;
    for (int j = 0; j < H; ++j) xd[j] = (double)x[j];
    const int rc = expert_mlp_d(xd, H, F, gate_up_type, down_type, G, U, D, grid, y, nthreads);
    free(xd);
    return rc;
}

/* The block ([P1] §3.2 moe_forward: router result -> only the routed experts
 * -> shared expert -> merge):
 *   out[t] = Sd(silu(Sg x) * Su x) + sum_k w[t][k] * D_e(silu(G_e x) * U_e x) */
int oracle_moe_forward(const float *hidden, int T, int H, int F, int E, int K,
                       int gate_up_type, int down_type, const void *const *gate,
                       const void *const *up, const void *const *down,
                       const uint16_t *sh_gate, const uint16_t *sh_up,
                       const uint16_t *sh_down, const uint8_t *grid, const int32_t *ids,
                       const float *w, float *out, int nthreads) {
    if (!hidden || !gate || !up || !down || !sh_gate || !sh_up || !sh_down || !ids || !w ||
        !out || T < 1 || K < 1 || E < 1 || H % 256 || F % 256 || H <= 0 || F <= 0)
        return -1;
    double *x = (double *)malloc(sizeof(double) * (size_t)H);
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    int rc = (!x || !acc || !y) ? -1 : 0;
    for (int t = 0; t < T && rc == 0; ++t) {
        for (int j = 0; j < H; ++j) x[j] = (double)hidden[(size_t)t * H + j];
        for (int j = 0; j < H; ++j) acc[j] = 0.0;
        for (int k = 0; k < K && rc == 0; ++k) {
            const int e = ids[(size_t)t * K + k];
            if (e < 0 || e >= E || !gate[e] || !up[e] || !down[e]) {
                rc = -2;
                break;
            }
            rc = expert_mlp_d(x, H, F, gate_up_type, down_type, gate[e], up[e], down[e], grid, y,
                              nthreads);
            const double wk = (double)w[(size_t)t * K + k];
            for (int j = 0; j < H; ++j) acc[j] += wk * y[j];
        }
        if (rc) break;
        rc = expert_mlp_d(x, H, F, ORACLE_BF16, ORACLE_BF16, sh_gate, sh_up, sh_down, NULL, y,
                          nthreads);
        for (int j = 0; j < H; ++j) out[(size_t)t * H + j] = (float)(y[j] + acc[j]);
    }
    free(x);
    free(acc);
    free(y);
    return rc;
}

/* ------------------------------------------------------------ q8 path */

int oracle_quantize_q8(const float *x, int n, int8_t *q, float *d) {
    if (!x || !q || !d || n <= 0 || n % 256) return -1;
    for (int b = 0; b < n / 256; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 256; ++i) {
            const float a = fabsf(x[256 * b + i]);
            if (a > amax) amax = a;
        }
        const float db = amax / 127.0f;
        d[b] = db;
        for (int i = 0; i < 256; ++i) {
            int v = 0;
            if (db > 0.0f) {
                const float r = rintf(x[256 * b + i] / db); /* default mode: nearest, ties to even */
                v = r > 127.0f ? 127 : r < -127.0f ? -127 : (int)r;
            }
            q[256 * b + i] = (int8_t)v;
        }
    }
    return 0;
}

/* The pages' dot of 16 int8 grid values (two grid rows) against 16 int8
 * activations (chenxutan ds4 article §2.4, dot_iq2_pair_16), restated. */
static int32_t dot16_i8(const int8_t *g0, const int8_t *g1, const int8_t *q) {
    int32_t s = 0;
    for (int i = 0; i < 8; ++i) s += (int32_t)g0[i] * q[i] + (int32_t)g1[i] * q[i + 8];
    return s;
}

/* One IQ2_XXS row [cols] on q8 activations (q, dx per 256 columns). */
static double iq2_row_dot_q8(const uint8_t *row_blocks, int cols, const uint8_t *grid, const int8_t *q,
                             const float *dx) {
    double acc = 0.0;
    for (int b = 0; b < cols / 256; ++b) {
        const uint8_t *blk = row_blocks + (size_t)b * 66;
        const float d = oracle_fp16_to_f32(rd16(blk));
        for (int sb = 0; sb < 8; ++sb) {
            const uint8_t *c = blk + 2 + 8 * sb;
            const uint32_t v = rd32(c + 4);
            const float db = (d * (0.5f + (float)(v >> 28))) * 0.25f;
            int8_t gs[4][8]; /* signed grid values of the sub-block's four rows */
            for (int l = 0; l < 4; ++l) {
                const uint32_t s7 = (v >> (7 * l)) & 127u;
                uint32_t sg = s7;
                int par = 0;
                for (int k = 0; k < 7; ++k) par ^= (int)((s7 >> k) & 1u);
                sg |= (uint32_t)par << 7;
                for (int i = 0; i < 8; ++i) {
                    const int g = grid[8 * c[l] + i];
                    gs[l][i] = (int8_t)(((sg >> i) & 1u) ? -g : g);
                }
            }
            const int8_t *qs = q + 256 * b + 32 * sb;
            const int32_t S = dot16_i8(gs[0], gs[1], qs) + dot16_i8(gs[2], gs[3], qs + 16);
            acc += (double)db * (double)dx[b] * (double)S;
        }
    }
    return acc;
}

static int expert_mlp_q8(const double *x, const int8_t *q, const float *dx, int H, int F, int dt, const void *G,
                         const void *U, const void *D, const uint8_t *grid, double *y, int nthreads) {
    double *g = (double *)malloc(sizeof(double) * (size_t)F);
    double *u = (double *)malloc(sizeof(double) * (size_t)F);
    int rc = (!g || !u || !G || !U) ? -1 : 0;
    if (!rc) {
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : omp_get_max_threads()) schedule(static)
        for (int r = 0; r < F; ++r) {
            g[r] = iq2_row_dot_q8((const uint8_t *)G + (size_t)r * (H / 256) * 66, H, grid, q, dx);
            u[r] = iq2_row_dot_q8((const uint8_t *)U + (size_t)r * (H / 256) * 66, H, grid, q, dx);
        }
        for (int i = 0; i < F; ++i) g[i] = silu(g[i]) * u[i];
        rc = matvec(dt, D, H, F, grid, g, y, nthreads);
    }
    (void)x;
    free(g);
    free(u);
    return rc;
}

int oracle_moe_forward_q8(const float *hidden, int T, int H, int F, int E, int K,
                          int gate_up_type, int down_type, const void *const *gate,
                          const void *const *up, const void *const *down,
                          const uint16_t *sh_gate, const uint16_t *sh_up,
                          const uint16_t *sh_down, const uint8_t *grid, const int32_t *ids,
                          const float *w, float *out, int nthreads) {
    if (!hidden || !gate || !up || !down || !sh_gate || !sh_up || !sh_down || !ids || !w || !grid ||
        !out || T < 1 || K < 1 || E < 1 || H % 256 || F % 256 || H <= 0 || F <= 0 ||
        gate_up_type != ORACLE_IQ2_XXS)
        return -1;
    double *x = (double *)malloc(sizeof(double) * (size_t)H);
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    int8_t *q = (int8_t *)malloc((size_t)H);
    float *dx = (float *)malloc(sizeof(float) * (size_t)(H / 256));
    int rc = (!x || !acc || !y || !q || !dx) ? -1 : 0;
    for (int t = 0; t < T && rc == 0; ++t) {
        const float *xt = hidden + (size_t)t * H;
        for (int j = 0; j < H; ++j) x[j] = (double)xt[j];
        for (int j = 0; j < H; ++j) acc[j] = 0.0;
        rc = oracle_quantize_q8(xt, H, q, dx);
        for (int k = 0; k < K && rc == 0; ++k) {
            const int e = ids[(size_t)t * K + k];
            if (e < 0 || e >= E || !gate[e] || !up[e] || !down[e]) {
                rc = -2;
                break;
            }
            rc = expert_mlp_q8(x, q, dx, H, F, down_type, gate[e], up[e], down[e], grid, y, nthreads);
            const double wk = (double)w[(size_t)t * K + k];
            for (int j = 0; j < H; ++j) acc[j] += wk * y[j];
        }
        if (rc) break;
        rc = expert_mlp_d(x, H, F, ORACLE_BF16, ORACLE_BF16, sh_gate, sh_up, sh_down, NULL, y, nthreads);
        for (int j = 0; j < H; ++j) out[(size_t)t * H + j] = (float)(y[j] + acc[j]);
    }
    free(x);
    free(acc);
    free(y);
    free(q);
    free(dx);
    return rc;
}
