/*
 * oracle.c -- plain fp64 CPU oracle of the deterministic MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): loaded by the tests, the package smoke check and
 * the benchmark's CPU-baseline leg; never by the CUDA path, with which it shares no code.
 *
 * Each function follows the plain definition of its step; the passages are cited in
 * oracle.h. Parallelism is over independent tokens (or independent experts) only, so
 * every sum keeps the order its definition states.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- routing */

void oracle_route(int64_t T, int32_t E, int32_t K, const double *logits, int32_t *idx,
                  double *w)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double *l = logits + t * (int64_t)E;
        char *taken = (char *)calloc((size_t)E, 1);
        /* selection in the order (logit descending, expert ascending): a strictly larger
         * logit wins, so among equal logits the lower expert id stays chosen; the double
         * comparison treats -0 and +0 as equal. */
        for (int32_t k = 0; k < K; ++k) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])
                    best = e;
            }
            taken[best] = 1;
            idx[t * K + k] = best;
        }
        free(taken);
        /* softmax over the K chosen logits, shifted by the largest one */
        const double m = l[idx[t * K]];
        double den = 0.0;
        for (int32_t k = 0; k < K; ++k)
            den += exp(l[idx[t * K + k]] - m);
        for (int32_t k = 0; k < K; ++k)
            w[t * K + k] = exp(l[idx[t * K + k]] - m) / den;
    }
}

/* ---------------------------------------------------------------- schedule */

int oracle_schedule(int64_t R, int32_t E, int64_t MB, const int32_t *idx, int32_t *counts,
                    int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *segs,
                    int64_t seg_cap, int32_t *n_segs)
{
    for (int32_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t f = 0; f < R; ++f)
        counts[idx[f]] += 1;
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    /* stable counting sort: flat ids visited in ascending order */
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t f = 0; f < R; ++f) {
        const int32_t e = idx[f];
        const int32_t row = offsets[e] + fill[e];
        fill[e] += 1;
        perm[row] = (int32_t)f;
        inv[f] = row;
    }
    free(fill);
    /* expert ranges cut at minibatch boundaries */
    int64_t n = 0;
    for (int32_t e = 0; e < E; ++e) {
        int64_t b = offsets[e];
        const int64_t end = offsets[e + 1];
        while (b < end) {
            int64_t mb_end = (b / MB + 1) * MB;
            int64_t se = end < mb_end ? end : mb_end;
            if (n >= seg_cap) {
                *n_segs = (int32_t)n;
                return -1;
            }
            segs[3 * n + 0] = e;
            segs[3 * n + 1] = (int32_t)b;
            segs[3 * n + 2] = (int32_t)se;
            ++n;
            b = se;
        }
    }
    *n_segs = (int32_t)n;
    return 0;
}

/* ---------------------------------------------------------------- MXFP8 */

uint8_t oracle_e4m3_encode(double v)
{
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v))
        return 0x7F;
    double a = fabs(v);
    if (a >= 448.0)
        return sign | 0x7E; /* saturate to the largest finite magnitude */
    if (a == 0.0)
        return sign;
    /* grid spacing in the binade [2^e, 2^(e+1)) is 2^(e-3); below 2^-6 (subnormals) it is
     * 2^-9. Scaling a by the spacing is exact, nearbyint rounds ties to even, and an even
     * grid index is an even mantissa. */
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    if (e < -6)
        e = -6;
    const double r = nearbyint(ldexp(a, 3 - e));
    const double mag = ldexp(r, e - 3);
    if (mag == 0.0)
        return sign;
    if (mag < ldexp(1.0, -6)) /* subnormal: mag = m * 2^-9, m = 1..7 */
        return sign | (uint8_t)ldexp(mag, 9);
    frexp(mag, &ex);
    const int E = ex - 1; /* -6..8 */
    const int mant = (int)ldexp(mag, 3 - E) - 8;
    return sign | (uint8_t)(((E + 7) << 3) | mant);
}

double oracle_e4m3_decode(uint8_t code)
{
    const double s = (code & 0x80) ? -1.0 : 1.0;
    const int ef = (code >> 3) & 0xF;
    const int m = code & 0x7;
    if (ef == 0xF && m == 0x7)
        return NAN;
    if (ef == 0)
        return s * ldexp((double)m, -9);
    return s * ldexp(8.0 + m, ef - 7 - 3);
}

void oracle_mxfp8_quantize(int64_t rows, int64_t cols, const double *src, uint8_t *q,
                           uint8_t *scale)
{
    const int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const double *v = src + r * cols + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i)
                if (fabs(v[i]) > amax)
                    amax = fabs(v[i]);
            int sexp = -127;
            if (amax > 0.0) {
                int ex;
                frexp(amax, &ex);
                sexp = (ex - 1) - 8; /* floor(log2 amax) minus the E4M3 max exponent */
                if (sexp < -127)
                    sexp = -127;
                if (sexp > 127)
                    sexp = 127;
            }
            scale[r * nb + b] = (uint8_t)(sexp + 127);
            for (int i = 0; i < 32; ++i)
                q[r * cols + b * 32 + i] = oracle_e4m3_encode(ldexp(v[i], -sexp));
        }
    }
}

void oracle_mxfp8_dequantize(int64_t rows, int64_t cols, const uint8_t *q, const uint8_t *scale,
                             double *out)
{
    const int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = ldexp(oracle_e4m3_decode(q[r * cols + c]),
                                      (int)scale[r * nb + c / 32] - 127);
}

void oracle_mxfp8_quantize_bf16(int64_t rows, int64_t cols, const uint16_t *src, uint8_t *q,
                                uint8_t *scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double v[32];
        for (int64_t b = 0; b < cols / 32; ++b) {
            for (int i = 0; i < 32; ++i) {
                uint32_t u = (uint32_t)src[r * cols + b * 32 + i] << 16;
                float f;
                memcpy(&f, &u, 4);
                v[i] = (double)f;
            }
            oracle_mxfp8_quantize(1, 32, v, q + r * cols + b * 32, scale + r * (cols / 32) + b);
        }
    }
}

/* element i of a weight tensor stored as `kind`, widened exactly to double */
static double wget(int32_t kind, const void *data, const uint8_t *scale, int64_t row_len,
                   int64_t i)
{
    if (kind == ORACLE_W_F64)
        return ((const double *)data)[i];
    if (kind == ORACLE_W_BF16) {
        uint32_t u = (uint32_t)((const uint16_t *)data)[i] << 16;
        float f;
        memcpy(&f, &u, 4);
        return (double)f;
    }
    const int64_t row = i / row_len, col = i % row_len;
    return ldexp(oracle_e4m3_decode(((const uint8_t *)data)[i]),
                 (int)scale[row * (row_len / 32) + col / 32] - 127);
}

/* element [e][r][col] of a weight given as the MXFP8 codes q [E][ncol][nrow] and scales
 * s [E][ncol][nrow/32] of its transpose, quantized along the transposed rows (that is,
 * along r in 32-blocks) */
static double wq_t(const uint8_t *q, const uint8_t *s, int64_t e, int64_t ncol, int64_t nrow,
                   int64_t r, int64_t col)
{
    const int64_t row_t = e * ncol + col;
    return ldexp(oracle_e4m3_decode(q[row_t * nrow + r]),
                 (int)s[row_t * (nrow / 32) + r / 32] - 127);
}

double oracle_round_bf16(double v)
{
    if (v == 0.0 || isnan(v) || isinf(v))
        return v;
    /* 8 significant bits in the binade of v; below 2^-126 the spacing stays 2^-133 */
    int ex;
    frexp(fabs(v), &ex);
    int e = ex - 1;
    if (e < -126)
        e = -126;
    return ldexp(nearbyint(ldexp(v, 7 - e)), e - 7);
}

static void qdq_row(int64_t n, double *v)
{
    uint8_t *q = (uint8_t *)malloc((size_t)n);
    uint8_t *s = (uint8_t *)malloc((size_t)(n / 32));
    oracle_mxfp8_quantize(1, n, v, q, s);
    oracle_mxfp8_dequantize(1, n, q, s, v);
    free(q);
    free(s);
}

/* ---------------------------------------------------------------- rounding slack
 * A rounding decision taken on a value that the GPU computes in fp32 (with a relative
 * error of a few fp32 ulps) and the oracle in fp64 can fall on either side of a rounding
 * midpoint when the exact value is that close to it; both outcomes are then correct
 * results of the definition. The slack of a decision is the distance between its two
 * possible results when the exact value lies within ORACLE_SLACK_REL of a midpoint (or, for
 * an MXFP8 block, of a scale-exponent boundary), and 0 otherwise. */

double oracle_bf16_slack(double v, double err)
{
    if (!isfinite(v))
        return 0.0;
    /* the roundings of the extreme values the kernel may hold, v - E and v + E, nudged
     * outward so that a tie on either end counts as the farther neighbour; rounding is
     * monotone, so every other outcome lies between them */
    const double E = err + ORACLE_SLACK_REL * fabs(v);
    const double r = oracle_round_bf16(v);
    const double hi = v + E, lo = v - E;
    const double up = fabs(oracle_round_bf16(hi + fabs(hi) * 0x1p-50) - r);
    const double dn = fabs(oracle_round_bf16(lo - fabs(lo) * 0x1p-50) - r);
    return up > dn ? up : dn;
}

/* E4M3 quantize-dequantize of a scaled value (saturating at 448) */
static double e4m3_qdq(double u) { return oracle_e4m3_decode(oracle_e4m3_encode(u)); }

/* distance from the code chosen for u to the farthest code that a scaled value within
 * err_u of u may take (the same interval rule as oracle_bf16_slack) */
static double e4m3_slack(double u, double err_u)
{
    const double E = err_u + ORACLE_SLACK_REL * fabs(u);
    const double r = e4m3_qdq(u);
    const double hi = u + E, lo = u - E;
    const double up = fabs(e4m3_qdq(hi + fabs(hi) * 0x1p-50) - r);
    const double dn = fabs(e4m3_qdq(lo - fabs(lo) * 0x1p-50) - r);
    return up > dn ? up : dn;
}

/* E8M0 exponent of a 32-element block with maximum magnitude amax: floor(log2 amax) - 8,
 * clamped to [-127, 127]; -127 for an all-zero block */
static int mx_block_exp(double amax)
{
    if (amax <= 0.0)
        return -127;
    int ex;
    frexp(amax, &ex);
    int s = (ex - 1) - 8;
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

void oracle_mxfp8_qdq_slack(int64_t n, const double *v, const double *err, double *out,
                            double *slack, uint8_t *q, uint8_t *scale)
{
    for (int64_t b = 0; b < n / 32; ++b) {
        const double *blk = v + b * 32, *eb = err + b * 32;
        double *ob = out + b * 32, *sl = slack + b * 32;
        double amax = 0.0, emax = 0.0;
        for (int i = 0; i < 32; ++i) {
            if (fabs(blk[i]) > amax)
                amax = fabs(blk[i]);
            if (eb[i] > emax)
                emax = eb[i];
        }
        const int sx = mx_block_exp(amax);
        /* the shared exponent is floor(log2 amax) - 8: a block whose amax lies within its
         * error of the power of two below (or above) it may take the exponent one lower (or
         * one higher) */
        int other = 0;
        if (amax > 0.0) {
            int ex;
            frexp(amax, &ex);
            const double p_lo = ldexp(1.0, ex - 1), p_hi = ldexp(1.0, ex);
            const double tol = emax + ORACLE_SLACK_REL * amax;
            if (sx > -127 && amax - p_lo <= tol)
                other = -1;
            else if (sx < 127 && p_hi - amax <= tol)
                other = +1;
        }
        uint8_t qb[32], sb;
        oracle_mxfp8_quantize(1, 32, blk, qb, &sb);
        oracle_mxfp8_dequantize(1, 32, qb, &sb, ob);
        for (int i = 0; i < 32; ++i)
            sl[i] = ldexp(e4m3_slack(ldexp(blk[i], -sx), ldexp(eb[i], -sx)), sx);
        if (other != 0) {
            /* the other exponent's result, itself possibly one code away */
            const int s2 = sx + other;
            for (int i = 0; i < 32; ++i) {
                const double u = ldexp(blk[i], -s2), E = ldexp(eb[i], -s2) +
                                                       ORACLE_SLACK_REL * fabs(u);
                const double hi = u + E, lo = u - E;
                const double alt[3] = {e4m3_qdq(u), e4m3_qdq(hi + fabs(hi) * 0x1p-50),
                                       e4m3_qdq(lo - fabs(lo) * 0x1p-50)};
                for (int m = 0; m < 3; ++m) {
                    const double d = fabs(ldexp(alt[m], s2) - ob[i]);
                    if (d > sl[i])
                        sl[i] = d;
                }
            }
        }
        if (q)
            memcpy(q + b * 32, qb, 32);
        if (scale)
            scale[b] = sb;
    }
}

/* A value v that a kernel computes to within err (its fp32 arithmetic) and that earlier
 * decisions may move by up to up, rounded to bf16: returns the rounding and sets *slack to
 * the distance within which a correct result lies from it. */
double oracle_dot_rel_rows(int64_t n)
{
    return n > 2048 ? ORACLE_DOT_REL * sqrt((double)n / 2048.0) : ORACLE_DOT_REL;
}

static double round_bf16_with_slack(double v, double err, double up, double *slack)
{
    *slack = up + oracle_bf16_slack(v, err + up);
    return oracle_round_bf16(v);
}

/* ---------------------------------------------------------------- forward */

static double silu(double g) { return g / (1.0 + exp(-g)); }
static double dsilu(double g)
{
    const double sg = 1.0 / (1.0 + exp(-g));
    return sg * (1.0 + g * (1.0 - sg));
}
/* how far h = silu(a_g) a_u can move when a_g and a_u move by up to ug and uu: by the
 * mean-value theorem, with the second derivative of silu at most 1/2 in magnitude,
 * (|silu'(a_g)| + ug / 2) ug (|a_u| + uu) + |silu(a_g)| uu, where sl = silu(a_g) */
static double dh_of_a(double ag, double au, double sl, double ug, double uu)
{
    return (fabs(dsilu(ag)) + 0.5 * ug) * ug * (fabs(au) + uu) + fabs(sl) * uu;
}

static double d2silu(double g)
{
    const double sg = 1.0 / (1.0 + exp(-g));
    return sg * (1.0 - sg) * (2.0 + g * (1.0 - 2.0 * sg));
}

void oracle_forward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const double *x,
                    const int32_t *idx, const double *w, int32_t wkind, const void *w13,
                    const uint8_t *w13_s, const void *w2, const uint8_t *w2_s, int32_t mode,
                    int32_t store, double *y, double *slack, oracle_rows *rows)
{
    (void)E;
    const int rnd = mode != ORACLE_EXACT;            /* operand rounding */
    const int sto = rnd && store == ORACLE_STORE_BF16; /* storage rounding */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *a = (double *)malloc(sizeof(double) * 2 * (size_t)I);
        double *aa = (double *)malloc(sizeof(double) * 2 * (size_t)I); /* sum |W13||x| */
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        double *hr = (double *)malloc(sizeof(double) * (size_t)I);     /* h as rounded */
        double *hs = (double *)calloc((size_t)I, sizeof(double));      /* its slack */
        double *he = (double *)malloc(sizeof(double) * (size_t)I);     /* error bound of h */
        double *o = (double *)malloc(sizeof(double) * (size_t)H);
        double *om = (double *)malloc(sizeof(double) * (size_t)H);     /* sum |W2||h| */
        double *ou = (double *)malloc(sizeof(double) * (size_t)H);     /* slack of o */
        double *ym = (double *)calloc((size_t)H, sizeof(double));      /* sum_k |w o| */
        double *sy = (double *)calloc((size_t)H, sizeof(double));      /* slack of the sum */
        uint8_t *hq = (uint8_t *)malloc((size_t)I);
        uint8_t *hsc = (uint8_t *)malloc((size_t)(I / 32 + 1));
        double *yt = y + t * (int64_t)H;
        /* an output added to an existing one: no slot, the fp32 error of each o and of the
         * additions carried into the final rounding */
        const double *y0 = (rows && rows->y_in) ? rows->y_in + t * (int64_t)H : NULL;
        double *ye = (double *)calloc((size_t)H, sizeof(double));
        memcpy(xt, x + t * (int64_t)H, sizeof(double) * (size_t)H);
        if (mode == ORACLE_MXFP8)
            qdq_row(H, xt);
        for (int32_t c = 0; c < H; ++c) {
            yt[c] = y0 ? y0[c] : 0.0;
            ym[c] = y0 ? fabs(y0[c]) : 0.0;
        }
        for (int32_t k = 0; k < K; ++k) {
            const int64_t f = t * K + k;
            const int64_t e = idx[f];
            const int64_t b13 = e * 2 * (int64_t)I * H, b2 = e * (int64_t)H * I;
            for (int32_t j = 0; j < 2 * I; ++j) {
                double acc = 0.0, mag = 0.0;
                for (int32_t c = 0; c < H; ++c) {
                    const double wv = wget(wkind, w13, w13_s, H, b13 + (int64_t)j * H + c);
                    acc += wv * xt[c];
                    mag += fabs(wv * xt[c]);
                }
                a[j] = acc;
                aa[j] = mag;
            }
            for (int32_t i = 0; i < I; ++i) {
                h[i] = silu(a[i]) * a[I + i];
                /* how far a kernel's fp32 h can be from this one */
                he[i] = fabs(dsilu(a[i]) * a[I + i]) * ORACLE_DOT_REL * aa[i] +
                        fabs(silu(a[i])) * ORACLE_DOT_REL * aa[I + i];
                hr[i] = h[i];
                hs[i] = 0.0;
            }
            if (mode == ORACLE_MXFP8) {
                oracle_mxfp8_qdq_slack(I, h, he, hr, hs, hq, hsc);
            } else if (mode == ORACLE_BF16) {
                for (int32_t i = 0; i < I; ++i)
                    hr[i] = round_bf16_with_slack(h[i], he[i], 0.0, &hs[i]);
            }
            if (rows) {
                if (rows->a)
                    memcpy(rows->a + f * 2 * I, a, sizeof(double) * 2 * (size_t)I);
                if (rows->a_mag)
                    memcpy(rows->a_mag + f * 2 * I, aa, sizeof(double) * 2 * (size_t)I);
                if (rows->h)
                    memcpy(rows->h + f * I, hr, sizeof(double) * (size_t)I);
                if (rows->h_slack)
                    memcpy(rows->h_slack + f * I, hs, sizeof(double) * (size_t)I);
                if (mode == ORACLE_MXFP8 && rows->h_q)
                    memcpy(rows->h_q + f * I, hq, (size_t)I);
                if (mode == ORACLE_MXFP8 && rows->h_scale)
                    memcpy(rows->h_scale + f * (I / 32), hsc, (size_t)(I / 32));
            }
            if (rows && rows->h_in) { /* the given h enters the down GEMM */
                memcpy(hr, rows->h_in + f * I, sizeof(double) * (size_t)I);
                memset(hs, 0, sizeof(double) * (size_t)I);
            }
            /* o = W2 h: its dot-product bound, and the slack carried in from h */
            for (int32_t c = 0; c < H; ++c) {
                double acc = 0.0, mag = 0.0;
                for (int32_t i = 0; i < I; ++i) {
                    const double wv = wget(wkind, w2, w2_s, I, b2 + (int64_t)c * I + i);
                    acc += wv * hr[i];
                    mag += fabs(wv * hr[i]);
                }
                o[c] = acc;
                om[c] = mag;
                ou[c] = 0.0;
            }
            if (rnd)
                for (int32_t i = 0; i < I; ++i) {
                    if (hs[i] == 0.0)
                        continue;
                    for (int32_t c = 0; c < H; ++c)
                        ou[c] += fabs(wget(wkind, w2, w2_s, I, b2 + (int64_t)c * I + i)) * hs[i];
                }
            const double s = w[f];
            for (int32_t c = 0; c < H; ++c) {
                double so = ou[c];
                if (sto && !y0) /* the (token, k) slot holds bf16(o) */
                    o[c] = round_bf16_with_slack(o[c], ORACLE_DOT_REL * om[c], ou[c], &so);
                if (y0)
                    ye[c] += fabs(s) * ORACLE_DOT_REL * om[c];
                yt[c] += s * o[c];
                ym[c] += fabs(s * o[c]);
                sy[c] += fabs(s) * so;
            }
        }
        for (int32_t c = 0; c < H; ++c) {
            double sc = sy[c];
            if (sto) /* y = bf16 of the fixed-order fp32 k-sum */
                yt[c] = round_bf16_with_slack(yt[c], (K + (y0 ? 1 : 0)) * ORACLE_SUM_ULP * ym[c] +
                                                         ye[c],
                                              sy[c], &sc);
            if (slack)
                slack[t * (int64_t)H + c] = sc;
        }
        free(ye);
        free(xt);
        free(a);
        free(aa);
        free(h);
        free(hr);
        free(hs);
        free(he);
        free(o);
        free(om);
        free(ou);
        free(ym);
        free(sy);
        free(hq);
        free(hsc);
    }
}

/* ---------------------------------------------------------------- backward */

void oracle_backward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const double *x,
                     const int32_t *idx, const double *w, int32_t wkind, const void *w13,
                     const uint8_t *w13_s, const void *w2, const double *dy, int32_t mode,
                     int32_t store, const uint8_t *w13d_q, const uint8_t *w13d_s,
                     const uint8_t *w2g_q, const uint8_t *w2g_s, double *dx,
                     double *dw13, double *dw2, double *dtopk, double *sdx, double *sdw13,
                     double *sdw2, oracle_rows *rows)
{
    const int64_t R = T * K;
    const int mx = mode == ORACLE_MXFP8;
    const int rnd = mode != ORACLE_EXACT;
    const int sto = rnd && store == ORACLE_STORE_BF16;
    /* per routed row: da = dL/da [2I] and sh = w * h [I] as the weight gradients read them
     * (bf16 in the rounding modes), with the slack of those values */
    double *da_all = (double *)malloc(sizeof(double) * (size_t)(R * 2 * I));
    double *sh_all = (double *)malloc(sizeof(double) * (size_t)(R * I));
    double *das_all = (double *)calloc((size_t)(R * 2 * I), sizeof(double));
    double *shs_all = (double *)calloc((size_t)(R * I), sizeof(double));

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        const double *xt = x + t * (int64_t)H;
        const double *dyt = dy + t * (int64_t)H;
        double *dxt = dx + t * (int64_t)H;
        double *a = (double *)malloc(sizeof(double) * 2 * (size_t)I);
        double *ea = (double *)malloc(sizeof(double) * 2 * (size_t)I); /* fp32 error of a */
        double *ua = (double *)malloc(sizeof(double) * 2 * (size_t)I); /* slack of a */
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *gg = (double *)malloc(sizeof(double) * (size_t)I);     /* sum |W2||dy| */
        double *dae = (double *)malloc(sizeof(double) * 2 * (size_t)I);
        double *dau = (double *)malloc(sizeof(double) * 2 * (size_t)I);
        double *xs = (double *)malloc(sizeof(double) * (size_t)H);     /* one slot's dgrad */
        double *xm = (double *)malloc(sizeof(double) * (size_t)H);
        double *xu = (double *)malloc(sizeof(double) * (size_t)H);
        double *dxm = (double *)calloc((size_t)H, sizeof(double));
        double *sdt = (double *)calloc((size_t)H, sizeof(double));
        /* MXFP8: the forward's quantized x (operand of the recomputed A), dy quantized along
         * H (operand of G), and dA quantized along 2I with its slack (operand of dgrad) */
        double *xq = mx ? (double *)malloc(sizeof(double) * (size_t)H) : NULL;
        double *dyq = mx ? (double *)malloc(sizeof(double) * (size_t)H) : NULL;
        double *daq = mx ? (double *)malloc(sizeof(double) * 2 * (size_t)I) : NULL;
        double *daqs = mx ? (double *)malloc(sizeof(double) * 2 * (size_t)I) : NULL;
        double *daqe = mx ? (double *)malloc(sizeof(double) * 2 * (size_t)I) : NULL;
        uint8_t *daqc = mx ? (uint8_t *)malloc(2 * (size_t)I) : NULL;
        uint8_t *daqb = mx ? (uint8_t *)malloc(2 * (size_t)I / 32 + 1) : NULL;
        if (mx) {
            memcpy(xq, xt, sizeof(double) * (size_t)H);
            qdq_row(H, xq);
            memcpy(dyq, dyt, sizeof(double) * (size_t)H);
            qdq_row(H, dyq);
        }
        const double *xa = mx ? xq : xt, *dyg = mx ? dyq : dyt;
        /* a dx added to an existing one: no slots, each dgrad result's fp32 error and the
         * additions' carried into the final rounding */
        const double *dx0 = (rows && rows->dx_in) ? rows->dx_in + t * (int64_t)H : NULL;
        double *dxe = (double *)calloc((size_t)H, sizeof(double));
        for (int32_t c = 0; c < H; ++c) {
            dxt[c] = dx0 ? dx0[c] : 0.0;
            dxm[c] = dx0 ? fabs(dx0[c]) : 0.0;
        }
        for (int32_t k = 0; k < K; ++k) {
            const int64_t f = t * K + k;
            const int64_t e = idx[f];
            const int64_t b13 = e * 2 * (int64_t)I * H, b2 = e * (int64_t)H * I;
            const double s = w[f];
            double *da = da_all + f * 2 * I;
            double *sh = sh_all + f * I;
            double *das = das_all + f * 2 * I;
            double *shs = shs_all + f * I;
            for (int32_t j = 0; j < 2 * I; ++j) {
                double acc = 0.0, mag = 0.0;
                for (int32_t c = 0; c < H; ++c) {
                    const double wv = wget(wkind, w13, w13_s, H, b13 + (int64_t)j * H + c);
                    acc += wv * xa[c];
                    mag += fabs(wv * xa[c]);
                }
                /* the saved A: bf16 under bf16 storage (its only uncertainty is then the
                 * slack of that rounding), else the kernel's fp32 value; or the given A */
                if (rows && rows->a_in) {
                    a[j] = rows->a_in[f * 2 * I + j];
                    ua[j] = 0.0;
                    ea[j] = sto ? 0.0 : ORACLE_DOT_REL * mag;
                } else if (sto) {
                    a[j] = round_bf16_with_slack(acc, ORACLE_DOT_REL * mag, 0.0, &ua[j]);
                    ea[j] = 0.0;
                } else {
                    a[j] = acc;
                    ua[j] = 0.0;
                    ea[j] = ORACLE_DOT_REL * mag;
                }
            }
            if (rows) {
                if (rows->a)
                    memcpy(rows->a + f * 2 * I, a, sizeof(double) * 2 * (size_t)I);
                if (rows->a_slack)
                    memcpy(rows->a_slack + f * 2 * I, ua, sizeof(double) * 2 * (size_t)I);
            }
            /* g = W2^T dy */
            for (int32_t i = 0; i < I; ++i) {
                double acc = 0.0, mag = 0.0;
                for (int32_t c = 0; c < H; ++c) {
                    const double wv = mx ? wq_t(w2g_q, w2g_s, e, I, H, c, i)
                                         : wget(wkind, w2, NULL, I, b2 + (int64_t)c * I + i);
                    acc += wv * dyg[c];
                    mag += fabs(wv * dyg[c]);
                }
                g[i] = acc;
                gg[i] = mag;
            }
            double dS = 0.0, sdS = 0.0;
            for (int32_t i = 0; i < I; ++i) {
                const double ag = a[i], au = a[I + i];
                const double sig = 1.0 / (1.0 + exp(-ag));
                const double sl = ag * sig;
                const double hi = sl * au;
                dS += g[i] * hi;
                /* h moves with the stored A's decisions (mean-value bound, dh_of_a) */
                sdS += fabs(g[i]) * dh_of_a(ag, au, sl, ua[i], ua[I + i]);
                const double dh = s * g[i];
                /* silu'(g) = sig * (1 + g * (1 - sig)) */
                da[i] = dh * au * sig * (1.0 + ag * (1.0 - sig));
                da[I + i] = dh * sl;
                sh[i] = s * hi;
                /* how far a kernel's values can be from these, to first order: its fp32 error
                 * (dot-product bounds of g and, with fp32 storage, of a) and the slack of a */
                const double d1 = dsilu(ag), d2 = d2silu(ag);
                const double eg = ORACLE_DOT_REL * gg[i];
                const double as = fabs(s);
                /* silu'(a_g) = sig * (1 + a_g * (1 - sig)) cancels near a_g = -1.28: the
                 * kernel's fp32 evaluation is off by a few ulps of the terms, not of the
                 * result, so its absolute error is bounded by ORACLE_SLACK_REL * sig *
                 * (1 + |a_g|) */
                const double e_d1 = ORACLE_SLACK_REL * sig * (1.0 + fabs(ag));
                dae[i] = as * (fabs(au * d1) * eg + fabs(g[i] * d1) * ea[I + i] +
                               fabs(g[i] * au * d2) * ea[i] + fabs(g[i] * au) * e_d1);
                /* slack carried from the stored A, by the mean-value theorem over the
                 * flipped interval, with the second and third derivatives of silu at
                 * most 1/2 in magnitude everywhere */
                dau[i] = as * fabs(g[i]) * (fabs(d1) * ua[I + i] +
                                            (fabs(au) + ua[I + i]) *
                                                (fabs(d2) + 0.5 * ua[i]) * ua[i]);
                dae[I + i] = as * (fabs(sl) * eg + fabs(g[i] * d1) * ea[i]);
                dau[I + i] = as * fabs(g[i]) * (fabs(d1) + 0.5 * ua[i]) * ua[i];
                if (rnd) {
                    const double e_sh = as * (fabs(d1 * au) * ea[i] + fabs(sl) * ea[I + i]);
                    const double u_sh = as * dh_of_a(ag, au, sl, ua[i], ua[I + i]);
                    sh[i] = round_bf16_with_slack(sh[i], e_sh, u_sh, &shs[i]);
                }
            }
            if (mx) { /* dgrad operand: dA quantized in 32-blocks along 2I */
                for (int32_t j = 0; j < 2 * I; ++j)
                    daqe[j] = dae[j] + dau[j];
                oracle_mxfp8_qdq_slack(2 * (int64_t)I, da, daqe, daq, daqs, daqc, daqb);
                for (int32_t j = 0; j < 2 * I; ++j)
                    daqs[j] += dau[j];
            }
            if (rnd)
                for (int32_t j = 0; j < 2 * I; ++j)
                    da[j] = round_bf16_with_slack(da[j], dae[j], dau[j], &das[j]);
            dtopk[f] = dS;
            if (rows && rows->dtopk_slack)
                rows->dtopk_slack[f] = sdS;
            if (rows) {
                if (rows->da)
                    memcpy(rows->da + f * 2 * I, da, sizeof(double) * 2 * (size_t)I);
                if (rows->da_slack)
                    memcpy(rows->da_slack + f * 2 * I, das, sizeof(double) * 2 * (size_t)I);
                if (rows->sh)
                    memcpy(rows->sh + f * I, sh, sizeof(double) * (size_t)I);
                if (rows->sh_slack)
                    memcpy(rows->sh_slack + f * I, shs, sizeof(double) * (size_t)I);
                if (mx && rows->da_q)
                    memcpy(rows->da_q + f * 2 * I, daqc, 2 * (size_t)I);
                if (mx && rows->da_scale)
                    memcpy(rows->da_scale + f * (2 * I / 32), daqb, (size_t)(2 * I / 32));
                if (mx && rows->daq_slack)
                    memcpy(rows->daq_slack + f * 2 * I, daqs, sizeof(double) * 2 * (size_t)I);
            }
            if (rows && rows->da_in) { /* the given operands of the following GEMMs */
                memcpy(da, rows->da_in + f * 2 * I, sizeof(double) * 2 * (size_t)I);
                memset(das, 0, sizeof(double) * 2 * (size_t)I);
            }
            if (rows && rows->sh_in) {
                memcpy(sh, rows->sh_in + f * I, sizeof(double) * (size_t)I);
                memset(shs, 0, sizeof(double) * (size_t)I);
            }
            if (mx && rows && rows->daq_in) {
                memcpy(daq, rows->daq_in + f * 2 * I, sizeof(double) * 2 * (size_t)I);
                memset(daqs, 0, sizeof(double) * 2 * (size_t)I);
            }
            /* this slot's dgrad result W13^T da (MXFP8: W13 quantized along 2I times dA
             * quantized along 2I), summed over j ascending for every column */
            const double *dad = mx ? daq : da;
            const double *dads = mx ? daqs : das;
            for (int32_t c = 0; c < H; ++c) {
                xs[c] = 0.0;
                xm[c] = 0.0;
                xu[c] = 0.0;
            }
            for (int32_t j = 0; j < 2 * I; ++j) {
                const double dj = dad[j], sj = dads[j];
                for (int32_t c = 0; c < H; ++c) {
                    const int64_t o = b13 + (int64_t)j * H + c;
                    const double wv = mx ? wq_t(w13d_q, w13d_s, e, H, 2 * (int64_t)I, j, c)
                                         : wget(wkind, w13, w13_s, H, o);
                    xs[c] += wv * dj;
                    xm[c] += fabs(wv * dj);
                    xu[c] += fabs(wv) * sj;
                }
            }
            for (int32_t c = 0; c < H; ++c) {
                double sx = xu[c];
                if (sto && !dx0) /* the slot holds bf16 of its dgrad result */
                    xs[c] = round_bf16_with_slack(xs[c], ORACLE_DOT_REL * xm[c], xu[c], &sx);
                if (dx0)
                    dxe[c] += ORACLE_DOT_REL * xm[c];
                dxt[c] += xs[c];
                dxm[c] += fabs(xs[c]);
                sdt[c] += sx;
            }
        }
        for (int32_t c = 0; c < H; ++c) {
            double sc = sdt[c];
            if (sto) /* dx = bf16 of the fixed-order fp32 k-sum */
                dxt[c] = round_bf16_with_slack(
                    dxt[c], (K + (dx0 ? 1 : 0)) * ORACLE_SUM_ULP * dxm[c] + dxe[c], sdt[c], &sc);
            if (sdx)
                sdx[t * (int64_t)H + c] = sc;
        }
        free(dxe);
        free(a);
        free(ea);
        free(ua);
        free(g);
        free(gg);
        free(dae);
        free(dau);
        free(xs);
        free(xm);
        free(xu);
        free(dxm);
        free(sdt);
        free(xq);
        free(dyq);
        free(daq);
        free(daqs);
        free(daqe);
        free(daqc);
        free(daqb);
    }

    if (dw13 != NULL && dw2 != NULL) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int32_t e = 0; e < E; ++e) {
            const int64_t n13 = 2 * (int64_t)I * H, n2 = (int64_t)H * I;
            double *DW13 = dw13 + (int64_t)e * n13;
            double *DW2 = dw2 + (int64_t)e * n2;
            /* per element: the sum of absolute terms (dot-product bound) and the slack
             * carried in from dA and w*h */
            double *M13 = (double *)calloc((size_t)n13, sizeof(double));
            double *M2 = (double *)calloc((size_t)n2, sizeof(double));
            double *U13 = (double *)calloc((size_t)n13, sizeof(double));
            double *U2 = (double *)calloc((size_t)n2, sizeof(double));
            memset(DW13, 0, sizeof(double) * (size_t)n13);
            memset(DW2, 0, sizeof(double) * (size_t)n2);
            int64_t ne = 0; /* the expert's rows: the length of its weight-gradient sums */
            for (int64_t f = 0; f < R; ++f) {
                if (idx[f] != e)
                    continue;
                ++ne;
                const int64_t t = f / K;
                const double *xt = x + t * (int64_t)H;
                const double *dyt = dy + t * (int64_t)H;
                const double *da = da_all + f * 2 * I, *das = das_all + f * 2 * I;
                const double *sh = sh_all + f * I, *shs = shs_all + f * I;
                for (int32_t j = 0; j < 2 * I; ++j)
                    for (int32_t c = 0; c < H; ++c) {
                        const int64_t o = (int64_t)j * H + c;
                        DW13[o] += da[j] * xt[c];
                        M13[o] += fabs(da[j] * xt[c]);
                        U13[o] += das[j] * fabs(xt[c]);
                    }
                for (int32_t c = 0; c < H; ++c)
                    for (int32_t i = 0; i < I; ++i) {
                        const int64_t o = (int64_t)c * I + i;
                        DW2[o] += dyt[c] * sh[i];
                        M2[o] += fabs(dyt[c] * sh[i]);
                        U2[o] += fabs(dyt[c]) * shs[i];
                    }
            }
            double *S13 = sdw13 ? sdw13 + (int64_t)e * n13 : NULL;
            double *S2 = sdw2 ? sdw2 + (int64_t)e * n2 : NULL;
            const double rel = oracle_dot_rel_rows(ne);
            for (int64_t o = 0; o < n13; ++o) {
                double sl = U13[o];
                if (sto) /* dW = bf16 of the sum over the expert's rows */
                    DW13[o] = round_bf16_with_slack(DW13[o], rel * M13[o], U13[o], &sl);
                if (S13)
                    S13[o] = sl;
            }
            for (int64_t o = 0; o < n2; ++o) {
                double sl = U2[o];
                if (sto)
                    DW2[o] = round_bf16_with_slack(DW2[o], rel * M2[o], U2[o], &sl);
                if (S2)
                    S2[o] = sl;
            }
            free(M13);
            free(M2);
            free(U13);
            free(U2);
        }
    }
    free(da_all);
    free(sh_all);
    free(das_all);
    free(shs_all);
}

void oracle_router_grad(int64_t T, int32_t E, int32_t K, const int32_t *idx, const double *w,
                        const double *dtopk, double *dlogits)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double *dl = dlogits + t * (int64_t)E;
        for (int32_t e = 0; e < E; ++e)
            dl[e] = 0.0;
        double sw = 0.0;
        for (int32_t k = 0; k < K; ++k)
            sw += w[t * K + k] * dtopk[t * K + k];
        for (int32_t k = 0; k < K; ++k)
            dl[idx[t * K + k]] = w[t * K + k] * (dtopk[t * K + k] - sw);
    }
}

void oracle_router_grad_slack(int64_t T, int32_t E, int32_t K, const int32_t *idx,
                              const double *w, const double *sdtopk, double *sdlogits)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double *sl = sdlogits + t * (int64_t)E;
        for (int32_t e = 0; e < E; ++e)
            sl[e] = 0.0;
        double sw = 0.0;
        for (int32_t k = 0; k < K; ++k)
            sw += fabs(w[t * K + k]) * sdtopk[t * K + k];
        for (int32_t k = 0; k < K; ++k)
            sl[idx[t * K + k]] = fabs(w[t * K + k]) * (sdtopk[t * K + k] + sw);
    }
}
