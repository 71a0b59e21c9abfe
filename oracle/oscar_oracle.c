/*
 * OSCAR oracle: plain, slow, obviously correct CPU reference of the INT2 KV-cache
 * decode path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library; the product path never
 * does, and this file shares no code with the CUDA library.
 *
 * Sources (web pages on OSCAR; cited by title and section):
 *   [news]   OSCAR news article, m.kljzs.com mirror: paragraph on the online
 *            layout ("sink token 和 recent window 维持 BF16 ... 每 4 个 2-bit 值
 *            打包进 1 个 byte ... online softmax merge").
 *   [tai]    "Together AI 開源 OSCAR" (news.chathome.org): sections
 *            "OSCAR 的不同之處" (key error identity, C_Q, C_S, R = U·H·P_br) and
 *            "服務系統：混合精度快取佈局" (64 sink + 256 recent in BF16).
 *   [notes]  "OSCAR — 离线转个方向，把 KV Cache 压到 2-bit" (estelledc study
 *            notes): "核心要点" items 2-3 (R = U·H_Had·P_br, layout
 *            [BF16 sink] || [INT2 history] || [BF16 recent], c_K ~ 0.96,
 *            c_V ~ 0.92 in "案例 2").
 *
 * Conventions fixed by the workload definition where the pages are silent:
 *   - row vectors: x_rot = x · R, so q_rot·k_rot = q·k and o = (sum p v_rot) · R_V^T;
 *   - asymmetric INT2 per group of g channels: lo = c·min, hi = c·max
 *     (min/max of the group's fp32 values, a signed zero read as +0),
 *     zero = bf16(lo), scale = bf16((hi - lo)/3),
 *     code = clamp(rint((x - zero)/scale), 0, 3) using the STORED bf16 zero/scale,
 *     code 0 when scale == 0;
 *   - 4 codes per byte, element i at bits 2·(i mod 4) of byte i/4.
 *
 * Precision: every "definition" routine is fp64.  The routines that decide an
 * integer (rotation feeding the quantizer, the quantizer itself) and the fold
 * that must match bit for bit (ora_merge_f32, ora_exp2f) are fp32 with every
 * operation spelled out; build with -ffp-contract=off so that the compiler
 * fuses nothing the source does not say.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 -- */

/* bf16 is the upper half of an IEEE binary32. */
double ora_bf16_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static float bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a binary32 to bf16, round-to-nearest, ties to even (NaN stays NaN). */
uint16_t ora_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);           /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    uint32_t rounded = u + 0x7fffu + lsb;                  /* half-way goes to even */
    return (uint16_t)(rounded >> 16);
}

/* -------------------------------------------------------------- rotation -- */

/*
 * y = x · R for one bf16 row x[D] and a row-major fp32 R[D][D], in fp32:
 * y_j = fma(x_{D-1}, R[D-1][j], ... fma(x_1, R[1][j], fma(x_0, R[0][j], 0))).
 * This is the precision in which the quantizer's decisions are taken, so the
 * order (ascending i, one fused multiply-add per term) is part of the contract.
 * [tai] "OSCAR 的不同之處": the rotation applied before quantization.
 */
void ora_rotate_f32(const uint16_t *x, const float *R, int D, float *y) {
    for (int j = 0; j < D; ++j) {
        float acc = 0.0f;
        for (int i = 0; i < D; ++i)
            acc = fmaf(bf16_to_f32(x[i]), R[(size_t)i * D + j], acc);
        y[j] = acc;
    }
}

/* Same product in fp64 (the mathematical definition; used to pin the fp32 one). */
void ora_rotate_f64(const uint16_t *x, const float *R, int D, double *y) {
    for (int j = 0; j < D; ++j) {
        double acc = 0.0;
        for (int i = 0; i < D; ++i)
            acc += ora_bf16_to_f64(x[i]) * (double)R[(size_t)i * D + j];
        y[j] = acc;
    }
}

/* ------------------------------------------------------------- quantizer -- */

/*
 * Asymmetric INT2 with clipping, one row of D fp32 values, groups of g
 * consecutive channels (in the rotated order).  [news] layout paragraph
 * ("rotate/clip/quantize/pack"), [notes] "核心要点" item 2 (clip ratio c fixed
 * offline, c_K ~ 0.96, c_V ~ 0.92), INT2 = 4 levels restored by scale/zero.
 */
void ora_quantize_row(const float *xr, int D, int g, float clip,
                      uint8_t *codes, uint16_t *zero_out, uint16_t *scale_out) {
    for (int g0 = 0; g0 < D; g0 += g) {
        float mn = xr[g0], mx = xr[g0];
        for (int i = g0 + 1; i < g0 + g; ++i) {
            if (xr[i] < mn) mn = xr[i];
            if (xr[i] > mx) mx = xr[i];
        }
        mn = mn + 0.0f;                       /* a signed zero is read as +0 */
        mx = mx + 0.0f;
        float lo = clip * mn;                 /* clipped range c·[min, max] */
        float hi = clip * mx;
        float diff = hi - lo;
        float step = diff / 3.0f;             /* 4 levels: 3 steps */
        uint16_t zb = ora_f32_to_bf16(lo);
        uint16_t sb = ora_f32_to_bf16(step);
        zero_out[g0 / g] = zb;
        scale_out[g0 / g] = sb;
        float z = bf16_to_f32(zb);
        float s = bf16_to_f32(sb);
        for (int i = g0; i < g0 + g; ++i) {
            int c = 0;
            if (s != 0.0f) {
                float t = (xr[i] - z) / s;
                float r = rintf(t);           /* nearest, ties to even */
                if (r >= 3.0f) c = 3;
                else if (r >= 0.0f) c = (int)r;
                else c = 0;                   /* also NaN */
            }
            codes[i] = (uint8_t)c;
        }
    }
}

/* 4 codes per byte, element i at bits 2*(i mod 4) of byte i/4. [news], [notes]. */
void ora_pack_row(const uint8_t *codes, int D, uint8_t *packed) {
    for (int j = 0; j < D / 4; ++j) {
        unsigned b = 0;
        for (int k = 0; k < 4; ++k)
            b |= (unsigned)(codes[4 * j + k] & 3u) << (2 * k);
        packed[j] = (uint8_t)b;
    }
}

void ora_unpack_row(const uint8_t *packed, int D, uint8_t *codes) {
    for (int i = 0; i < D; ++i)
        codes[i] = (uint8_t)((packed[i / 4] >> (2 * (i % 4))) & 3u);
}

/*
 * Non-uniform 4-level codebook (OSCAR news article, closing paragraph: the latest codebase
 * brings a Lloyd-Max codebook to the attention-aware rotation).  The pages give no levels and
 * no formula; the reading taken here keeps the uniform quantizer's per-group normalisation
 * (zero = bf16(c*min), scale = bf16((c*max - c*min)/3), so u = (x - zero)/scale puts the
 * clipped range on [0, 3]) and replaces the levels 0, 1, 2, 3 of that axis by a codebook
 * lv[0] < lv[1] < lv[2] < lv[3] designed offline by Lloyd's algorithm (oracle/__init__.py,
 * lloyd_max).  A value takes the nearest level: with the fp32 midpoints
 * t_k = (lv[k] + lv[k+1]) * 0.5, code = [u >= t_0] + [u >= t_1] + [u >= t_2] (a value on a
 * midpoint takes the upper level; NaN, or scale 0, gives code 0), and it is restored as
 * zero + lv[code] * scale.  lv == NULL selects the uniform quantizer above.
 */
void ora_quantize_row_cb(const float *xr, int D, int g, float clip, const float *lv,
                         uint8_t *codes, uint16_t *zero_out, uint16_t *scale_out) {
    if (!lv) {
        ora_quantize_row(xr, D, g, clip, codes, zero_out, scale_out);
        return;
    }
    float t[3];
    for (int k = 0; k < 3; ++k) t[k] = (lv[k] + lv[k + 1]) * 0.5f;
    for (int g0 = 0; g0 < D; g0 += g) {
        float mn = xr[g0], mx = xr[g0];
        for (int i = g0 + 1; i < g0 + g; ++i) {
            if (xr[i] < mn) mn = xr[i];
            if (xr[i] > mx) mx = xr[i];
        }
        mn = mn + 0.0f;
        mx = mx + 0.0f;
        float lo = clip * mn;
        float hi = clip * mx;
        float step = (hi - lo) / 3.0f;
        uint16_t zb = ora_f32_to_bf16(lo);
        uint16_t sb = ora_f32_to_bf16(step);
        zero_out[g0 / g] = zb;
        scale_out[g0 / g] = sb;
        float z = bf16_to_f32(zb);
        float s = bf16_to_f32(sb);
        for (int i = g0; i < g0 + g; ++i) {
            int c = 0;
            if (s != 0.0f) {
                float u = (xr[i] - z) / s;
                c = (u >= t[0]) + (u >= t[1]) + (u >= t[2]);
            }
            codes[i] = (uint8_t)c;
        }
    }
}

/* x_hat_i = zero + code_i * scale, in fp64 ("scale/zero point 还原"). */
void ora_dequant_row(const uint8_t *packed, const uint16_t *zero, const uint16_t *scale,
                     int D, int g, double *out) {
    for (int i = 0; i < D; ++i) {
        int c = (packed[i / 4] >> (2 * (i % 4))) & 3;
        out[i] = ora_bf16_to_f64(zero[i / g]) + (double)c * ora_bf16_to_f64(scale[i / g]);
    }
}

/* The same with a codebook: x_hat_i = zero + lv[code_i] * scale in fp64 (lv NULL: uniform). */
void ora_dequant_row_cb(const uint8_t *packed, const uint16_t *zero, const uint16_t *scale,
                        int D, int g, const float *lv, double *out) {
    if (!lv) {
        ora_dequant_row(packed, zero, scale, D, g, out);
        return;
    }
    for (int i = 0; i < D; ++i) {
        int c = (packed[i / 4] >> (2 * (i % 4))) & 3;
        out[i] = ora_bf16_to_f64(zero[i / g]) + (double)lv[c] * ora_bf16_to_f64(scale[i / g]);
    }
}

/*
 * Demotion of n rows that share one rotation: rotate (fp32, as above), then
 * clip/quantize/pack.  rot_out may be NULL.
 */
void ora_demote_rows_cb(const uint16_t *x, const float *R, int n, int D, int g, float clip, const float *lv,
                        float *rot_out, uint8_t *packed, uint16_t *zero, uint16_t *scale);

void ora_demote_rows(const uint16_t *x, const float *R, int n, int D, int g, float clip,
                     float *rot_out, uint8_t *packed, uint16_t *zero, uint16_t *scale) {
    ora_demote_rows_cb(x, R, n, D, g, clip, NULL, rot_out, packed, zero, scale);
}

/* ora_demote_rows with a codebook (lv NULL: uniform). */
void ora_demote_rows_cb(const uint16_t *x, const float *R, int n, int D, int g, float clip, const float *lv,
                        float *rot_out, uint8_t *packed, uint16_t *zero, uint16_t *scale) {
    float *y = (float *)malloc(sizeof(float) * (size_t)D);
    uint8_t *c = (uint8_t *)malloc((size_t)D);
    for (int r = 0; r < n; ++r) {
        ora_rotate_f32(x + (size_t)r * D, R, D, y);
        if (rot_out) memcpy(rot_out + (size_t)r * D, y, sizeof(float) * (size_t)D);
        ora_quantize_row_cb(y, D, g, clip, lv, c, zero + (size_t)r * (D / g), scale + (size_t)r * (D / g));
        ora_pack_row(c, D, packed + (size_t)r * (D / 4));
    }
    free(y);
    free(c);
}

/* Quantize n fp32 rows that are already rotated (the codec alone; lv NULL: uniform). */
void ora_quantize_rows(const float *xr, int n, int D, int g, float clip, const float *lv,
                       uint8_t *packed, uint16_t *zero, uint16_t *scale) {
    uint8_t *c = (uint8_t *)malloc((size_t)D);
    for (int r = 0; r < n; ++r) {
        ora_quantize_row_cb(xr + (size_t)r * D, D, g, clip, lv, c,
                            zero + (size_t)r * (D / g), scale + (size_t)r * (D / g));
        ora_pack_row(c, D, packed + (size_t)r * (D / 4));
    }
    free(c);
}

/* ------------------------------------------------------------- attention -- */

/*
 * One kv head's cache for one request, logical (unpaged) token-major arrays:
 *   k, v   : bf16 [T][D]   (read only at BF16 positions p < sink or p >= h_end)
 *   ck, cv : packed codes [T][D/4]  (read only at history positions)
 *   zk, sk, zv, sv : bf16 [T][D/g]
 * Region split [tai] "服務系統": first `sink` tokens and the last tokens from
 * h_end on are BF16 and unrotated; [sink, h_end) is rotated INT2 history.
 */
typedef struct {
    int D, T, sink, h_end, g;
    const uint16_t *k, *v;
    const uint8_t *ck, *cv;
    const uint16_t *zk, *sk, *zv, *sv;
    const float *lk, *lv;             /* key / value codebooks, NULL: uniform */
} ora_cache_t;

static int is_history(const ora_cache_t *c, int p) { return p >= c->sink && p < c->h_end; }

/* logit (before sm_scale) and value row of position p; value in the basis it is stored in. */
static double logit_at(const ora_cache_t *c, int p, const double *q, const double *q_rot, double *tmp) {
    double s = 0.0;
    if (is_history(c, p)) {
        ora_dequant_row_cb(c->ck + (size_t)p * (c->D / 4), c->zk + (size_t)p * (c->D / c->g),
                           c->sk + (size_t)p * (c->D / c->g), c->D, c->g, c->lk, tmp);
        for (int d = 0; d < c->D; ++d) s += q_rot[d] * tmp[d];
    } else {
        for (int d = 0; d < c->D; ++d) s += q[d] * ora_bf16_to_f64(c->k[(size_t)p * c->D + d]);
    }
    return s;
}

static void value_at(const ora_cache_t *c, int p, double *out) {
    if (is_history(c, p)) {
        ora_dequant_row_cb(c->cv + (size_t)p * (c->D / 4), c->zv + (size_t)p * (c->D / c->g),
                           c->sv + (size_t)p * (c->D / c->g), c->D, c->g, c->lv, out);
    } else {
        for (int d = 0; d < c->D; ++d) out[d] = ora_bf16_to_f64(c->v[(size_t)p * c->D + d]);
    }
}

/*
 * Full decode attention of one query head against its kv head, fp64:
 *   logits: q·k for BF16 positions, (q·R_K)·k_hat for history positions;
 *   p = softmax(sm_scale · logits) over all T positions;
 *   o = sum_BF16 p v + (sum_hist p v_hat) · R_V^T.
 * out[D]; *lse = log sum exp(sm_scale · logits) (natural log).
 * [news] layout paragraph, [notes] "核心要点" item 3 (BF16 and INT2 segments
 * combined into the full attention).
 */
void ora_attend_head_f64(int D, int T, int sink, int h_end, int g, double sm_scale,
                         const uint16_t *q, const float *RK, const float *RV,
                         const uint16_t *k, const uint16_t *v,
                         const uint8_t *ck, const uint8_t *cv,
                         const uint16_t *zk, const uint16_t *sk,
                         const uint16_t *zv, const uint16_t *sv, const float *lk, const float *lv,
                         double *out, double *lse) {
    ora_cache_t c = {D, T, sink, h_end, g, k, v, ck, cv, zk, sk, zv, sv, lk, lv};
    double *qd = (double *)malloc(sizeof(double) * D);
    double *qr = (double *)malloc(sizeof(double) * D);
    double *tmp = (double *)malloc(sizeof(double) * D);
    double *s = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
    double *acc_b = (double *)calloc(D, sizeof(double));
    double *acc_h = (double *)calloc(D, sizeof(double));
    for (int d = 0; d < D; ++d) qd[d] = ora_bf16_to_f64(q[d]);
    for (int j = 0; j < D; ++j) {
        double a = 0.0;
        for (int i = 0; i < D; ++i) a += qd[i] * (double)RK[(size_t)i * D + j];
        qr[j] = a;
    }
    double m = -INFINITY;
    for (int p = 0; p < T; ++p) {
        s[p] = sm_scale * logit_at(&c, p, qd, qr, tmp);
        if (s[p] > m) m = s[p];
    }
    double L = 0.0;
    for (int p = 0; p < T; ++p) {
        double w = exp(s[p] - m);
        L += w;
        value_at(&c, p, tmp);
        double *acc = is_history(&c, p) ? acc_h : acc_b;
        for (int d = 0; d < D; ++d) acc[d] += w * tmp[d];
    }
    for (int j = 0; j < D; ++j) {
        double a = 0.0;                                   /* (acc_h · R_V^T)_j */
        for (int i = 0; i < D; ++i) a += acc_h[i] * (double)RV[(size_t)j * D + i];
        out[j] = (acc_b[j] + a) / L;
    }
    if (lse) *lse = m + log(L);
    free(qd); free(qr); free(tmp); free(s); free(acc_b); free(acc_h);
}

/*
 * Partial of a flash-decoding split in the base-2 domain, fp64.  Positions
 * [lo[r], hi[r]) for r < n_ranges; every position must lie in one region kind:
 * history (int2 = 1, value accumulated in the ROTATED basis, no R_V^T) or BF16
 * (int2 = 0).  With t_p = sm_scale·logit_p·log2(e):
 *   m2 = max t_p, l = sum 2^(t_p - m2), acc = sum 2^(t_p - m2)·value_p.
 * An empty split gives m2 = -inf, l = 0, acc = 0.
 */
void ora_partial_f64(int D, int T, int sink, int h_end, int g, double sm_scale,
                     const uint16_t *q, const float *RK,
                     const uint16_t *k, const uint16_t *v,
                     const uint8_t *ck, const uint8_t *cv,
                     const uint16_t *zk, const uint16_t *sk,
                     const uint16_t *zv, const uint16_t *sv, const float *lk, const float *lv,
                     int n_ranges, const int *lo, const int *hi,
                     double *m2_out, double *l_out, double *acc_out) {
    ora_cache_t c = {D, T, sink, h_end, g, k, v, ck, cv, zk, sk, zv, sv, lk, lv};
    const double log2e = 1.0 / log(2.0);
    double *qd = (double *)malloc(sizeof(double) * D);
    double *qr = (double *)malloc(sizeof(double) * D);
    double *tmp = (double *)malloc(sizeof(double) * D);
    for (int d = 0; d < D; ++d) qd[d] = ora_bf16_to_f64(q[d]);
    for (int j = 0; j < D; ++j) {
        double a = 0.0;
        for (int i = 0; i < D; ++i) a += qd[i] * (double)RK[(size_t)i * D + j];
        qr[j] = a;
    }
    double m2 = -INFINITY;
    for (int r = 0; r < n_ranges; ++r)
        for (int p = lo[r]; p < hi[r]; ++p) {
            double t = sm_scale * logit_at(&c, p, qd, qr, tmp) * log2e;
            if (t > m2) m2 = t;
        }
    double l = 0.0;
    for (int d = 0; d < D; ++d) acc_out[d] = 0.0;
    for (int r = 0; r < n_ranges; ++r)
        for (int p = lo[r]; p < hi[r]; ++p) {
            double w = exp2(sm_scale * logit_at(&c, p, qd, qr, tmp) * log2e - m2);
            l += w;
            value_at(&c, p, tmp);
            for (int d = 0; d < D; ++d) acc_out[d] += w * tmp[d];
        }
    *m2_out = m2;
    *l_out = l;
    free(qd); free(qr); free(tmp);
}

/*
 * Online-softmax merge, fp64 definition.  Partials 0..S-1 are history splits
 * (rotated basis), partial S is the BF16 one (unrotated).  If RV is NULL no
 * partial is rotated (an all-BF16 cache).
 *   M = max m_i, L = sum l_i 2^(m_i - M), A = sum acc_i 2^(m_i - M),
 *   o = (A_hist · R_V^T + A_bf16) / L,  lse = (M + log2 L)·ln 2.
 * [news] "online softmax merge", [notes] "核心要点" item 3.
 */
void ora_merge_f64(int D, int S, const double *m2, const double *l, const double *acc,
                   const float *RV, double *out, double *lse) {
    double M = -INFINITY;
    for (int i = 0; i <= S; ++i) if (l[i] > 0.0 && m2[i] > M) M = m2[i];
    double L = 0.0;
    double *ah = (double *)calloc(D, sizeof(double));
    double *ab = (double *)calloc(D, sizeof(double));
    for (int i = 0; i <= S; ++i) {
        if (!(l[i] > 0.0)) continue;
        double w = exp2(m2[i] - M);
        L += l[i] * w;
        double *a = (i < S && RV) ? ah : ab;
        for (int d = 0; d < D; ++d) a[d] += acc[(size_t)i * D + d] * w;
    }
    for (int j = 0; j < D; ++j) {
        double r = 0.0;
        if (RV)
            for (int i = 0; i < D; ++i) r += ah[i] * (double)RV[(size_t)j * D + i];
        out[j] = (r + ab[j]) / L;
    }
    if (lse) *lse = (M + log2(L)) * log(2.0);
    free(ah); free(ab);
}

/* ------------------------------------------------- fp32 merge, bit exact -- */

/*
 * 2^x in fp32 by Cody-Waite range reduction and a Taylor polynomial:
 *   n = rint(x), f = x - n in [-1/2, 1/2] (exact),
 *   2^f = sum_{k=0}^{7} (f ln 2)^k / k!   evaluated by Horner with fmaf,
 *   2^x = 2^f * 2^n.
 * Coefficients are the binary32 roundings of (ln 2)^k / k!, computed here
 * from ln 2 in double precision.  x < -125 (including -inf) gives 0.
 * Truncation error of the series < 6e-9 on [-1/2, 1/2].
 */
static float taylor_c[8];
static int taylor_ready = 0;

static void taylor_init(void) {
    double ln2 = log(2.0), t = 1.0;
    for (int k = 0; k < 8; ++k) {
        taylor_c[k] = (float)t;
        t = t * ln2 / (double)(k + 1);
    }
    taylor_ready = 1;
}

float ora_exp2f(float x) {
    if (!taylor_ready) taylor_init();
    if (!(x >= -125.0f)) return 0.0f;            /* also -inf and NaN */
    if (x > 127.0f) return INFINITY;
    float n = rintf(x);
    float f = x - n;
    float p = taylor_c[7];
    for (int k = 6; k >= 0; --k) p = fmaf(p, f, taylor_c[k]);
    uint32_t e = (uint32_t)((int)n + 127) << 23;   /* 2^n, n in [-125, 127] */
    float two_n;
    memcpy(&two_n, &e, 4);
    return p * two_n;
}

/*
 * The merge as an ordered fp32 computation, the exact sequence of roundings
 * that the CUDA merge kernel must reproduce (a fixed order of the online-
 * softmax combination: global maximum first, so that the weights are
 * independent of each other):
 *   M = max of m_i over the non-empty partials (l_i > 0), i = 0..S
 *   w_i = 2^(m_i - M)
 *   L = 0, A = 0; for i = 0..S-1 with l_i > 0 (history splits, ascending):
 *       L = fma(l_i, w_i, L);  A_d = fma(acc_i,d, w_i, A_d)
 *   if RV: A'_j = fma-chain over i ascending of A_i * RV[j][i] (A · R_V^T), else A' = A
 *   BF16 partial (index S), if l_S > 0: L = fma(l_S, w_S, L); A'_d = fma(acc_S,d, w_S, A'_d)
 *   o_j = A'_j / L (IEEE division), out_bf16 = bf16_rne(o_j)
 * 2^x is ora_exp2f.  If every l is 0 the output is 0.
 */
void ora_merge_f32(int D, int S, const float *m2, const float *l, const float *acc,
                   const float *RV, float *out_f32, uint16_t *out_bf16) {
    float M = -INFINITY, L = 0.0f;
    float *A = (float *)calloc(D, sizeof(float));
    float *Ar = (float *)calloc(D, sizeof(float));
    for (int i = 0; i <= S; ++i)
        if (l[i] > 0.0f && m2[i] > M) M = m2[i];
    for (int i = 0; i < S; ++i) {
        if (!(l[i] > 0.0f)) continue;
        float w = ora_exp2f(m2[i] - M);
        L = fmaf(l[i], w, L);
        for (int d = 0; d < D; ++d) A[d] = fmaf(acc[(size_t)i * D + d], w, A[d]);
    }
    if (RV) {
        for (int j = 0; j < D; ++j) {
            float r = 0.0f;
            for (int i = 0; i < D; ++i) r = fmaf(A[i], RV[(size_t)j * D + i], r);
            Ar[j] = r;
        }
    } else {
        memcpy(Ar, A, sizeof(float) * D);
    }
    if (l[S] > 0.0f) {
        float w = ora_exp2f(m2[S] - M);
        L = fmaf(l[S], w, L);
        for (int d = 0; d < D; ++d) Ar[d] = fmaf(acc[(size_t)S * D + d], w, Ar[d]);
    }
    for (int j = 0; j < D; ++j) {
        float o = (L > 0.0f) ? Ar[j] / L : 0.0f;
        if (out_f32) out_f32[j] = o;
        if (out_bf16) out_bf16[j] = ora_f32_to_bf16(o);
    }
    free(A); free(Ar);
}

/* ------------------------------------------------------ layout accounting -- */

/*
 * Effective bits per KV element of one request of T tokens: history tokens
 * cost 2 bits of code plus 2 bf16 numbers (scale, zero) per group of g, the
 * sink + recent tokens cost 16 bits.  [news] "2.28 effective bits per KV
 * element", [notes] "是什么" (about 2.28 bits including scale/zero and the BF16
 * windows), [tai] "服務系統" (BF16 windows are 0.24% of tokens at 128K).
 */
double ora_bits_per_element(long long T, int g, int sink, int recent) {
    long long bf = (long long)sink + recent;
    if (bf > T) bf = T;
    long long hist = T - bf;
    double bits = (double)hist * (2.0 + 32.0 / (double)g) + (double)bf * 16.0;
    return bits / (double)T;
}
