/*
 * oracle.h -- plain, slow, fp64 CPU oracle of the deterministic MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg may load this library. It shares no code, header, table or helper with
 * the CUDA path, and the CUDA path never calls it.
 *
 * Pages cited (by title and section):
 *   [arex]     "Cursor 放出 MoK：NVL72 训练提速 2.37 倍" (arex-research.com)
 *   [aigwx]    "Cursor 开源 MoK：面向 GB300 NVL72 的确定性 MoE 训练内核，性能提升 2.37 倍" (aigwx.org)
 *   [alphalab] "Mixture-of-Kittens" analysis (alphalab.site)
 *
 * Every floating-point value is a double. Inputs stored as bf16/fp32 are widened exactly
 * by the caller. No step is blocked, fused or reordered beyond its plain definition.
 */
#ifndef MOK_ORACLE_H
#define MOK_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Top-k routing over router logits ([alphalab] section 四: top-k over Gaussian logits).
 * For each token t the pairs (logit, e) are ordered by logit descending, then expert id
 * ascending; the first K are taken in that order. w = softmax over the K chosen logits
 * (routing function read from the workload description; the pages name none). */
void oracle_route(int64_t T, int32_t E, int32_t K, const double *logits, int32_t *idx,
                  double *w);

/* Expert schedule ([arex] section "pull 代替 push": one schedule table serves dispatch,
 * combine and their backward twins). Flat routed ids f = t*K + k are stably sorted by
 * expert: perm[row] = f, inv[f] = row, counts[e], offsets[E+1] (exclusive scan).
 * Segments are the non-empty intersections of each expert's row range with the minibatch
 * row ranges [m*MB, (m+1)*MB), in increasing row order, as (expert, row_begin, row_end).
 * Returns 0, or -1 when more than seg_cap segments would be written. */
int oracle_schedule(int64_t R, int32_t E, int64_t MB, const int32_t *idx, int32_t *counts,
                    int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *segs,
                    int64_t seg_cap, int32_t *n_segs);

/* OFP8 E4M3 (bias 7, no infinities, max finite 448): round to nearest, ties to even,
 * saturating finite overflow to +-448, sign of zero kept. */
uint8_t oracle_e4m3_encode(double v);
double oracle_e4m3_decode(uint8_t code);

/* MXFP8 block quantization along rows: 32-element blocks share an E8M0 scale
 * 2^(floor(log2 amax) - 8), clamped to [2^-127, 2^127]; amax == 0 gives scale byte 0.
 * cols must be a multiple of 32. q is [rows][cols], scale is [rows][cols/32]. */
void oracle_mxfp8_quantize(int64_t rows, int64_t cols, const double *src, uint8_t *q,
                           uint8_t *scale);
void oracle_mxfp8_dequantize(int64_t rows, int64_t cols, const uint8_t *q, const uint8_t *scale,
                             double *out);

/* Weight storage read by the forward and backward. Every element is widened exactly to a
 * double when it is read; nothing else differs between the kinds. */
enum { ORACLE_W_F64 = 0, ORACLE_W_BF16 = 1, ORACLE_W_MXFP8 = 2 };

/* MXFP8 quantization of bf16 bit patterns (same definition as oracle_mxfp8_quantize). */
void oracle_mxfp8_quantize_bf16(int64_t rows, int64_t cols, const uint16_t *src, uint8_t *q,
                                uint8_t *scale);

/* bf16 rounding of a real value: nearest, ties to even, with bf16 subnormals. */
double oracle_round_bf16(double v);

/* Rounding slack. A kernel computes the value it rounds (h, dA, w*h, a stored result) in
 * fp32 from fp32 dot products, so its value may differ from the exact one by up to
 * ORACLE_DOT_REL times the sum of the dot products' absolute terms (propagated through the
 * SwiGLU formulas), plus ORACLE_SLACK_REL of the value for the elementwise operations
 * (of the terms, where a formula cancels: silu'(g) = sig (1 + g (1 - sig)) near its root). A
 * fixed-order fp32 sum of n terms (the k-sums of the combine and of dx) is within
 * n * 2^-24 of the sum of its absolute terms (the textbook bound for recursive summation
 * with unit roundoff 2^-24). When the exact value lies within its bound of a rounding
 * midpoint, the kernel may round to the other neighbour and both results are correct. The
 * slack of such a decision is the distance between its two possible results (for MXFP8
 * also when the block's amax lies that close to a power of two, which decides the shared
 * exponent); otherwise it is 0. A value that depends on earlier decisions carries their
 * slack (propagated linearly through |weights|, |x|, |dy| and the SwiGLU derivatives), and
 * that slack widens the window in which its own rounding is ambiguous. Parity tests
 * subtract the resulting per-element slack before comparing.
 *
 * ORACLE_DOT_REL is a measured property of the hardware, not of the pages: on GB300 tensor
 * cores (bf16 operands, fp32 accumulation, K = 320 .. 4096, random-sign terms) the largest
 * |fp32 result - exact| / sum|terms| seen over 4-8 million outputs per GEMM was 2^-20.2
 * (median 2^-24); the block-scaled MXFP8 path stayed below 2^-22.5. The oracle takes 2^-19. */
#define ORACLE_SLACK_REL 9.5367431640625e-07 /* 2^-20 */
#define ORACLE_DOT_REL 1.9073486328125e-06   /* 2^-19 */
#define ORACLE_SUM_ULP 5.9604644775390625e-08 /* 2^-24: fp32 unit roundoff */

/* The weight gradients are dot products over an expert's routed rows, whose number n runs
 * from 0 to T, and a dot product's fp32 error grows with its length. Measured on GB300
 * (dW13 of the experts of one Zipf-routed workload, 64 x 4096 outputs each, against the
 * exact sums of the GPU's own bf16 operands), the largest |fp32 result - exact| / sum|terms|
 * was 2^-21.3 at n = 318, 2^-20.0 at 1897, 2^-19.2 at 3975, 2^-19.1 at 8829, 2^-18.6 at
 * 16218 and 2^-18.0 at 34469 and 65535: growth of about sqrt(n), as for the accumulation
 * of random-sign terms. The oracle takes ORACLE_DOT_REL * max(1, sqrt(n / 2048)) for a
 * weight gradient over n rows, at least 1.6x above every value seen. */
double oracle_dot_rel_rows(int64_t n);
double oracle_bf16_slack(double v, double err);

/* MXFP8 quantize-dequantize of n values (n a multiple of 32) in 32-element blocks, each
 * value known to within err[i]: out = the dequantized values, slack = the distance to the
 * other correct result of each decision (see above), q / scale = the codes and E8M0 bytes
 * (both nullable). */
void oracle_mxfp8_qdq_slack(int64_t n, const double *v, const double *err, double *out,
                            double *slack, uint8_t *q, uint8_t *scale);

/* Precision modes ([arex] section "pull 代替 push": the layer has a BF16 and an MXFP8
 * mode; in MXFP8 mode activations are quantized where they enter the GEMMs, at dispatch
 * and at SwiGLU). Read here as: the operands of every expert GEMM carry the mode's type.
 *   ORACLE_EXACT: no rounding anywhere (the layer's real-valued definition);
 *   ORACLE_BF16:  h is rounded to bf16 before the down GEMM (backward: dA and w*h are
 *                 rounded to bf16 before the dgrad and weight-gradient GEMMs);
 *   ORACLE_MXFP8: x is MXFP8-quantized along H before the gate/up GEMM and h along I
 *                 before the down GEMM (backward: see oracle_backward). */
enum { ORACLE_EXACT = 0, ORACLE_BF16 = 1, ORACLE_MXFP8 = 2 };

/* Storage of the values that are only stored, never multiplied on the tensor cores: the
 * expert output of each (token, k) slot, the layer outputs y, dx, dW13, dW2, the saved
 * gate/up pre-activations A read by the backward, and the per-slot dgrad results.
 *   ORACLE_STORE_F32:  kept unrounded (a kernel keeps them in fp32);
 *   ORACLE_STORE_BF16: each is rounded to bf16 where it is stored. [alphalab] section
 *                      三 benchmarks the layer as a BF16 (or MXFP8) layer and checks its
 *                      outputs and gradients against a reference within a tolerance; the
 *                      pages fix no storage type, and the reading here is that such a
 *                      layer hands bf16 tensors between its steps: o -> bf16 before the
 *                      weighted k-sum, y = bf16(sum), A -> bf16 before the backward reads
 *                      it, each slot's dgrad result -> bf16 before the k-sum, dx =
 *                      bf16(sum), dW = bf16(sum over rows).
 * In ORACLE_EXACT mode nothing is rounded whatever the storage. */
enum { ORACLE_STORE_F32 = 0, ORACLE_STORE_BF16 = 1 };

/* Optional per-routed-row intermediates (row f = t*K + k), each pointer nullable:
 *   a        [R][2I] forward: the exact gate/up pre-activations; backward: A as the
 *                    backward reads it (bf16 under ORACLE_STORE_BF16)
 *   a_mag    [R][2I] forward: sum over c of |W13[e][j][c] x[t][c]| (the dot-product bound)
 *   a_slack  [R][2I] backward: slack of the stored A
 *   h, h_slack [R][I] forward: h as it enters the down GEMM (bf16 or MXFP8 value)
 *   h_q [R][I], h_scale [R][I/32]  forward, MXFP8: the codes and scale bytes of h
 *   da, da_slack [R][2I]  backward: dA rounded to bf16 (the weight-gradient operand)
 *   sh, sh_slack [R][I]   backward: w*h rounded to bf16
 *   da_q [R][2I], da_scale [R][2I/32], daq_slack [R][2I]  backward, MXFP8: dA quantized
 *                    along 2I (the dgrad operand) and the slack of its dequantized value
 *   dtopk_slack [R]  backward: slack of dS = <g, h> carried in from the stored A's
 *                    decisions (h moves with A); dS itself is not rounded
 * and optional given values, which replace the oracle's own at the point where they enter
 * the next step (each with zero slack). They let a test check one step at a time: the
 * step's own rounding decisions on the values a kernel actually fed it.
 *   h_in   [R][I]  forward: h as it enters the down GEMM
 *   a_in   [R][2I] backward: A as the backward reads it
 *   da_in  [R][2I], sh_in [R][I]  backward: the bf16 dA and w*h of the weight-gradient
 *                  GEMMs (and, in BF16 mode, dA of the dgrad GEMM)
 *   daq_in [R][2I] backward, MXFP8: the dequantized dA of the dgrad GEMM
 * and, for an expert whose output is added to an existing output (a shared expert):
 *   y_in   [T][H] forward: y starts from y_in[t], and each k's weighted expert output is
 *                  added to it directly in fp32 (no slot in between); only the final y is
 *                  stored (bf16 under ORACLE_STORE_BF16)
 *   dx_in  [T][H] backward: likewise, dx starts from dx_in[t] and each k's dgrad result is
 *                  added directly */
typedef struct oracle_rows {
    double *a, *a_mag, *a_slack;
    double *h, *h_slack;
    uint8_t *h_q, *h_scale;
    double *da, *da_slack, *sh, *sh_slack;
    uint8_t *da_q, *da_scale;
    double *daq_slack;
    double *dtopk_slack;
    const double *h_in, *a_in, *da_in, *sh_in, *daq_in;
    const double *y_in, *dx_in;
} oracle_rows;

/* Forward of the layer, per token, with no schedule and no permutation:
 *   a = W13[e] x  (gate rows 0..I-1, up rows I..2I-1), h = silu(a_g) * a_u,
 *   o = W2[e] h,  y_t = sum over k ascending of w[t,k] * o_k,
 * with the operand rounding of `mode` (ORACLE_*) and the storage rounding of `store`
 * (ORACLE_STORE_*). Weights are stored as `wkind` (ORACLE_W_*); for ORACLE_W_MXFP8, w13_s
 * and w2_s hold the E8M0 scales along each weight row. x [T][H], idx/w [T][K],
 * w13 [E][2I][H], w2 [E][H][I], y [T][H]; slack [T][H] and rows are nullable. */
void oracle_forward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const double *x,
                    const int32_t *idx, const double *w, int32_t wkind, const void *w13,
                    const uint8_t *w13_s, const void *w2, const uint8_t *w2_s, int32_t mode,
                    int32_t store, double *y, double *slack, oracle_rows *rows);

/* Backward of the layer by the chain rule, given dy [T][H]:
 *   g = W2[e]^T dy_t, dS[t,k] = <g, h>, dh = w g,
 *   da_g = dh * a_u * silu'(a_g), da_u = dh * silu(a_g),
 *   dx_t = sum_k W13[e]^T da, dW13[e] = sum da x^T, dW2[e] = sum dy (w h)^T
 * ([arex] section "pull 代替 push": router-weight gradient computed with the SwiGLU
 * backward; [alphalab] section 一: expert gradient computation). Sums over routed rows run
 * in ascending flat id, sums over k in ascending k. a and h are those of the forward (a
 * rounded to bf16 first under ORACLE_STORE_BF16, as the backward reads the saved A). mode
 * is ORACLE_EXACT, ORACLE_BF16 (dA and w*h rounded to bf16 where they enter the dgrad and
 * weight-gradient GEMMs) or ORACLE_MXFP8 ([arex] section "pull 代替 push": MXFP8
 * activations and pre-quantized weights): A is recomputed from the forward's quantized
 * operands (x quantized along H, W13 given as ORACLE_W_MXFP8 with w13_s), G = W2g^T Q(dy)
 * with dy quantized along H and W2g = W2 quantized along H, dx = W13d^T Q(dA) with dA
 * quantized in 32-blocks along 2I and W13d = W13 quantized along 2I; the weight gradients
 * take dA and w*h rounded to bf16 as in ORACLE_BF16. W13d and W2g are given as the codes
 * and scales of the transposed weights quantized along their rows: w13d_q [E][H][2I] with
 * w13d_s [E][H][2I/32] (W13d[e][j][c] from code [e][c][j]) and w2g_q [E][I][H] with w2g_s
 * [E][I][H/32] (W2g[e][c][i] from code [e][i][c]). store is ORACLE_STORE_*. Weights are
 * ORACLE_W_F64 or ORACLE_W_BF16 (ORACLE_W_MXFP8 for w13 in MXFP8 mode; the w13d and w2g
 * arrays are NULL otherwise).
 * Outputs: dx [T][H], dw13 [E][2I][H], dw2 [E][H][I], dtopk [T][K] (= dS); dw13/dw2 may be
 * NULL (skipped); the slacks sdx, sdw13, sdw2 and rows are nullable. */
void oracle_backward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const double *x,
                     const int32_t *idx, const double *w, int32_t wkind, const void *w13,
                     const uint8_t *w13_s, const void *w2, const double *dy, int32_t mode,
                     int32_t store, const uint8_t *w13d_q, const uint8_t *w13d_s,
                     const uint8_t *w2g_q, const uint8_t *w2g_s, double *dx,
                     double *dw13, double *dw2, double *dtopk, double *sdx, double *sdw13,
                     double *sdw2, oracle_rows *rows);

/* Router-logit gradient through the top-k softmax: for a chosen expert j = idx[t,k],
 * dlogits[t,j] = w_k (dS_k - sum_m w_m dS_m); every other logit gets 0. */
void oracle_router_grad(int64_t T, int32_t E, int32_t K, const int32_t *idx, const double *w,
                        const double *dtopk, double *dlogits);

/* The slack of those logit gradients given the slack sdtopk [T][K] of each dS: for a chosen
 * expert j = idx[t,k], w_k (sdtopk[t,k] + sum_m w_m sdtopk[t,m]); 0 elsewhere. */
void oracle_router_grad_slack(int64_t T, int32_t E, int32_t K, const int32_t *idx,
                              const double *w, const double *sdtopk, double *sdlogits);

#ifdef __cplusplus
}
#endif
#endif
