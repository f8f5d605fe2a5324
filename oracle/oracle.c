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
    if (v == 0.0 || !isfinite(v))
        return 0.0;
    int ex;
    frexp(fabs(v), &ex);
    int e = ex - 1;
    if (e < -126)
        e = -126;
    const double ulp = ldexp(1.0, e - 7);
    const double q = fabs(v) / ulp;
    const double dist = fabs((q - floor(q)) - 0.5) * ulp;
    return dist <= err + ORACLE_SLACK_REL * fabs(v) ? ulp : 0.0;
}

/* slack of the E4M3 code of a scaled value u known to within err_u (saturation at 448 is
 * one-sided: none) */
static double e4m3_slack(double u, double err_u)
{
    const double a = fabs(u);
    if (a == 0.0 || a >= 448.0)
        return 0.0;
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    if (e < -6)
        e = -6;
    const double sp = ldexp(1.0, e - 3);
    const double q = a / sp;
    const double dist = fabs((q - floor(q)) - 0.5) * sp;
    return dist <= err_u + ORACLE_SLACK_REL * a ? sp : 0.0;
}

/* MXFP8 quantize-dequantize of one row along its 32-element blocks, with each element's
 * slack: the code decision's slack, and when the block's amax is that close to a power of
 * two (the shared exponent could go either way) the difference to the other exponent's
 * result as well. */
static void qdq_row_slack(int64_t n, double *v, const double *err, double *slack)
{
    double alt[32];
    for (int64_t b = 0; b < n / 32; ++b) {
        double *blk = v + b * 32, *sl = slack + b * 32;
        const double *eb = err + b * 32;
        double amax = 0.0, emax = 0.0;
        for (int i = 0; i < 32; ++i) {
            if (fabs(blk[i]) > amax)
                amax = fabs(blk[i]);
            if (eb[i] > emax)
                emax = eb[i];
        }
        int ex = 0;
        if (amax > 0.0)
            frexp(amax, &ex);
        const int sexp = amax > 0.0 ? (ex - 1) - 8 : -127;
        /* the nearer power of two decides which other exponent is possible */
        const double p_lo = ldexp(1.0, ex - 1), p_hi = ldexp(1.0, ex);
        int other = 0;
        const double tol = emax + ORACLE_SLACK_REL * amax;
        if (amax > 0.0 && sexp > -127 && amax - p_lo <= tol)
            other = -1;
        else if (amax > 0.0 && p_hi - amax <= tol)
            other = +1;
        const int sx = sexp < -127 ? -127 : sexp;
        for (int i = 0; i < 32; ++i)
            sl[i] = ldexp(e4m3_slack(ldexp(blk[i], -sx), ldexp(eb[i], -sx)), sx);
        if (other != 0) {
            int s2 = sexp + other;
            if (s2 < -127)
                s2 = -127;
            for (int i = 0; i < 32; ++i)
                alt[i] = ldexp(oracle_e4m3_decode(oracle_e4m3_encode(ldexp(blk[i], -s2))), s2);
        }
        uint8_t q[32], sc;
        oracle_mxfp8_quantize(1, 32, blk, q, &sc);
        oracle_mxfp8_dequantize(1, 32, q, &sc, blk);
        if (other != 0)
            for (int i = 0; i < 32; ++i) {
                const double d = fabs(alt[i] - blk[i]);
                if (d > sl[i])
                    sl[i] = d;
            }
    }
}

/* ---------------------------------------------------------------- forward */

static double silu(double g) { return g / (1.0 + exp(-g)); }
static double dsilu(double g)
{
    const double sg = 1.0 / (1.0 + exp(-g));
    return sg * (1.0 + g * (1.0 - sg));
}
static double d2silu(double g)
{
    const double sg = 1.0 / (1.0 + exp(-g));
    return sg * (1.0 - sg) * (2.0 + g * (1.0 - 2.0 * sg));
}

void oracle_forward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const double *x,
                    const int32_t *idx, const double *w, int32_t wkind, const void *w13,
                    const uint8_t *w13_s, const void *w2, const uint8_t *w2_s, int32_t mode,
                    double *y, double *slack)
{
    (void)E;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *a = (double *)malloc(sizeof(double) * 2 * (size_t)I);
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        double *hs = (double *)calloc((size_t)I, sizeof(double));
        double *aa = (double *)malloc(sizeof(double) * 2 * (size_t)I); /* sum |W13||x| */
        double *he = (double *)malloc(sizeof(double) * (size_t)I);     /* error bound of h */
        double *yt = y + t * (int64_t)H;
        double *st = slack ? slack + t * (int64_t)H : NULL;
        memcpy(xt, x + t * (int64_t)H, sizeof(double) * (size_t)H);
        if (mode == ORACLE_MXFP8)
            qdq_row(H, xt);
        for (int32_t c = 0; c < H; ++c)
            yt[c] = 0.0;
        if (st)
            for (int32_t c = 0; c < H; ++c)
                st[c] = 0.0;
        for (int32_t k = 0; k < K; ++k) {
            const int64_t e = idx[t * K + k];
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
            }
            if (mode == ORACLE_MXFP8) {
                qdq_row_slack(I, h, he, hs);
            } else if (mode == ORACLE_BF16) {
                for (int32_t i = 0; i < I; ++i) {
                    hs[i] = oracle_bf16_slack(h[i], he[i]);
                    h[i] = oracle_round_bf16(h[i]);
                }
            }
            const double s = w[t * K + k];
            for (int32_t c = 0; c < H; ++c) {
                double o = 0.0;
                for (int32_t i = 0; i < I; ++i)
                    o += wget(wkind, w2, w2_s, I, b2 + (int64_t)c * I + i) * h[i];
                yt[c] += s * o;
            }
            /* slack of y: the h decisions that could go either way, through |W2| */
            if (st && mode != ORACLE_EXACT)
                for (int32_t i = 0; i < I; ++i) {
                    if (hs[i] == 0.0)
                        continue;
                    for (int32_t c = 0; c < H; ++c)
                        st[c] += fabs(s * wget(wkind, w2, w2_s, I, b2 + (int64_t)c * I + i)) *
                                 hs[i];
                }
        }
        free(xt);
        free(a);
        free(h);
        free(hs);
        free(aa);
        free(he);
    }
}

/* ---------------------------------------------------------------- backward */

void oracle_backward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const double *x,
                     const int32_t *idx, const double *w, int32_t wkind, const void *w13,
                     const uint8_t *w13_s, const void *w2, const double *dy, int32_t mode,
                     const double *w13d, const double *w2g, double *dx, double *dw13,
                     double *dw2, double *dtopk, double *sdx, double *sdw13, double *sdw2)
{
    const int64_t R = T * K;
    const int mx = mode == ORACLE_MXFP8;
    const int want_slack = (sdx != NULL) && mode != ORACLE_EXACT;
    /* per routed row: da = dL/da [2I] and sh = w * h [I], kept for the weight gradients,
     * and the slack of their bf16 decisions */
    double *da_all = (double *)malloc(sizeof(double) * (size_t)(R * 2 * I));
    double *sh_all = (double *)malloc(sizeof(double) * (size_t)(R * I));
    double *das_all = want_slack ? (double *)calloc((size_t)(R * 2 * I), sizeof(double)) : NULL;
    double *shs_all = want_slack ? (double *)calloc((size_t)(R * I), sizeof(double)) : NULL;
    if (sdx != NULL)
        memset(sdx, 0, sizeof(double) * (size_t)(T * (int64_t)H));

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        const double *xt = x + t * (int64_t)H;
        const double *dyt = dy + t * (int64_t)H;
        double *dxt = dx + t * (int64_t)H;
        double *a = (double *)malloc(sizeof(double) * 2 * (size_t)I);
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *aa = (double *)malloc(sizeof(double) * 2 * (size_t)I); /* sum |W13||x| */
        double *gg = (double *)malloc(sizeof(double) * (size_t)I);     /* sum |W2||dy| */
        /* MXFP8: the forward's quantized x (operand of the recomputed A), dy quantized along
         * H (operand of G), and dA quantized along 2I with its slack (operand of dgrad) */
        double *xq = mx ? (double *)malloc(sizeof(double) * (size_t)H) : NULL;
        double *dyq = mx ? (double *)malloc(sizeof(double) * (size_t)H) : NULL;
        double *daq = mx ? (double *)malloc(sizeof(double) * 2 * (size_t)I) : NULL;
        double *dae = mx ? (double *)malloc(sizeof(double) * 2 * (size_t)I) : NULL;
        double *daqs = mx ? (double *)malloc(sizeof(double) * 2 * (size_t)I) : NULL;
        if (mx) {
            memcpy(xq, xt, sizeof(double) * (size_t)H);
            qdq_row(H, xq);
            memcpy(dyq, dyt, sizeof(double) * (size_t)H);
            qdq_row(H, dyq);
        }
        const double *xa = mx ? xq : xt, *dyg = mx ? dyq : dyt;
        for (int32_t c = 0; c < H; ++c)
            dxt[c] = 0.0;
        for (int32_t k = 0; k < K; ++k) {
            const int64_t f = t * K + k;
            const int64_t e = idx[f];
            const int64_t b13 = e * 2 * (int64_t)I * H, b2 = e * (int64_t)H * I;
            const double s = w[f];
            double *da = da_all + f * 2 * I;
            double *sh = sh_all + f * I;
            for (int32_t j = 0; j < 2 * I; ++j) {
                double acc = 0.0, mag = 0.0;
                for (int32_t c = 0; c < H; ++c) {
                    const double wv = wget(wkind, w13, w13_s, H, b13 + (int64_t)j * H + c);
                    acc += wv * xa[c];
                    mag += fabs(wv * xa[c]);
                }
                a[j] = acc;
                aa[j] = mag;
            }
            /* g = W2^T dy */
            for (int32_t i = 0; i < I; ++i) {
                double acc = 0.0, mag = 0.0;
                for (int32_t c = 0; c < H; ++c) {
                    const double wv = mx ? w2g[b2 + (int64_t)c * I + i]
                                         : wget(wkind, w2, NULL, I, b2 + (int64_t)c * I + i);
                    acc += wv * dyg[c];
                    mag += fabs(wv * dyg[c]);
                }
                g[i] = acc;
                gg[i] = mag;
            }
            double dS = 0.0;
            for (int32_t i = 0; i < I; ++i) {
                const double ag = a[i], au = a[I + i];
                const double sig = 1.0 / (1.0 + exp(-ag));
                const double sl = ag * sig;
                const double hi = sl * au;
                dS += g[i] * hi;
                const double dh = s * g[i];
                /* silu'(g) = sig * (1 + g * (1 - sig)) */
                da[i] = dh * au * sig * (1.0 + ag * (1.0 - sig));
                da[I + i] = dh * sl;
                sh[i] = s * hi;
            }
            if (mode != ORACLE_EXACT) {
                if (want_slack || mx)
                    for (int32_t i = 0; i < I; ++i) {
                        /* how far a kernel's fp32 values can be from these: first-order
                         * propagation of the dot products' error bounds */
                        const double ag = a[i], au = a[I + i], gi = g[i];
                        const double eag = ORACLE_DOT_REL * aa[i];
                        const double eau = ORACLE_DOT_REL * aa[I + i];
                        const double eg = ORACLE_DOT_REL * gg[i];
                        const double sl = silu(ag), d1 = dsilu(ag), d2 = d2silu(ag);
                        const double e_dag = fabs(s) * (fabs(au * d1) * eg + fabs(gi * d1) * eau +
                                                         fabs(gi * au * d2) * eag);
                        const double e_dau = fabs(s) * (fabs(sl) * eg + fabs(gi * d1) * eag);
                        const double e_sh = fabs(s) * (fabs(d1 * au) * eag + fabs(sl) * eau);
                        if (mx) {
                            dae[i] = e_dag;
                            dae[I + i] = e_dau;
                        }
                        if (want_slack) {
                            das_all[f * 2 * I + i] = oracle_bf16_slack(da[i], e_dag);
                            das_all[f * 2 * I + I + i] = oracle_bf16_slack(da[I + i], e_dau);
                            shs_all[f * I + i] = oracle_bf16_slack(sh[i], e_sh);
                        }
                    }
                if (mx) { /* dgrad operand: dA quantized in 32-blocks along 2I */
                    memcpy(daq, da, sizeof(double) * 2 * (size_t)I);
                    qdq_row_slack(2 * (int64_t)I, daq, dae, daqs);
                }
                for (int32_t j = 0; j < 2 * I; ++j)
                    da[j] = oracle_round_bf16(da[j]);
                for (int32_t i = 0; i < I; ++i)
                    sh[i] = oracle_round_bf16(sh[i]);
            }
            dtopk[f] = dS;
            /* dx += W13^T da (MXFP8: W13 quantized along 2I times dA quantized along 2I) */
            const double *dad = mx ? daq : da;
            for (int32_t c = 0; c < H; ++c) {
                double acc = 0.0;
                for (int32_t j = 0; j < 2 * I; ++j) {
                    const int64_t o = b13 + (int64_t)j * H + c;
                    acc += (mx ? w13d[o] : wget(wkind, w13, w13_s, H, o)) * dad[j];
                }
                dxt[c] += acc;
            }
            if (want_slack)
                for (int32_t j = 0; j < 2 * I; ++j) {
                    const double sj = mx ? daqs[j] : das_all[f * 2 * I + j];
                    if (sj == 0.0)
                        continue;
                    for (int32_t c = 0; c < H; ++c) {
                        const int64_t o = b13 + (int64_t)j * H + c;
                        sdx[t * (int64_t)H + c] +=
                            fabs(mx ? w13d[o] : wget(wkind, w13, w13_s, H, o)) * sj;
                    }
                }
        }
        free(a);
        free(g);
        free(aa);
        free(gg);
        free(xq);
        free(dyq);
        free(daq);
        free(dae);
        free(daqs);
    }

    if (dw13 == NULL || dw2 == NULL) {
        free(da_all);
        free(sh_all);
        free(das_all);
        free(shs_all);
        return;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t e = 0; e < E; ++e) {
        double *DW13 = dw13 + (int64_t)e * 2 * I * H;
        double *DW2 = dw2 + (int64_t)e * H * I;
        memset(DW13, 0, sizeof(double) * (size_t)(2 * (int64_t)I * H));
        memset(DW2, 0, sizeof(double) * (size_t)((int64_t)H * I));
        double *S13 = sdw13 ? sdw13 + (int64_t)e * 2 * I * H : NULL;
        double *S2 = sdw2 ? sdw2 + (int64_t)e * H * I : NULL;
        if (S13)
            memset(S13, 0, sizeof(double) * (size_t)(2 * (int64_t)I * H));
        if (S2)
            memset(S2, 0, sizeof(double) * (size_t)((int64_t)H * I));
        for (int64_t f = 0; f < R; ++f) {
            if (idx[f] != e)
                continue;
            const int64_t t = f / K;
            const double *xt = x + t * (int64_t)H;
            const double *dyt = dy + t * (int64_t)H;
            const double *da = da_all + f * 2 * I;
            const double *sh = sh_all + f * I;
            for (int32_t j = 0; j < 2 * I; ++j)
                for (int32_t c = 0; c < H; ++c)
                    DW13[(int64_t)j * H + c] += da[j] * xt[c];
            for (int32_t c = 0; c < H; ++c)
                for (int32_t i = 0; i < I; ++i)
                    DW2[(int64_t)c * I + i] += dyt[c] * sh[i];
            if (want_slack && S13 && S2) {
                for (int32_t j = 0; j < 2 * I; ++j) {
                    const double sj = das_all[f * 2 * I + j];
                    if (sj != 0.0)
                        for (int32_t c = 0; c < H; ++c)
                            S13[(int64_t)j * H + c] += sj * fabs(xt[c]);
                }
                for (int32_t i = 0; i < I; ++i) {
                    const double si = shs_all[f * I + i];
                    if (si != 0.0)
                        for (int32_t c = 0; c < H; ++c)
                            S2[(int64_t)c * I + i] += fabs(dyt[c]) * si;
                }
            }
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
