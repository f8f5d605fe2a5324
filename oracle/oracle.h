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

/* Rounding slack. A kernel computes the value it rounds (h, dA, w*h) in fp32 from fp32 dot
 * products, so its value may differ from the exact one by about ORACLE_DOT_REL times the
 * sum of the dot products' absolute terms (propagated through the SwiGLU formulas), plus
 * ORACLE_SLACK_REL of the value for the elementwise operations. When the exact value lies
 * within that bound of a rounding midpoint, the kernel may round to the other neighbour
 * and both results are correct. The slack of such a decision is the distance between its
 * two possible results (for MXFP8 also when the block's amax lies that close to a power of
 * two, which decides the shared exponent); otherwise it is 0. The forward and backward
 * propagate these slacks linearly (through |weights|, |x|, |dy|) to bounds on how far a
 * correct result may lie from the oracle's; parity tests subtract them before comparing. */
#define ORACLE_SLACK_REL 9.5367431640625e-07 /* 2^-20 */
#define ORACLE_DOT_REL 2.384185791015625e-07 /* 2^-22 */
double oracle_bf16_slack(double v, double err);

/* Precision modes ([arex] section "pull 代替 push": the layer has a BF16 and an MXFP8
 * mode; in MXFP8 mode activations are quantized where they enter the GEMMs, at dispatch
 * and at SwiGLU). Read here as: the operands of every expert GEMM carry the mode's type.
 *   ORACLE_EXACT: no rounding anywhere (the layer's real-valued definition);
 *   ORACLE_BF16:  h is rounded to bf16 before the down GEMM (backward: dA and w*h are
 *                 rounded to bf16 before the dgrad and weight-gradient GEMMs);
 *   ORACLE_MXFP8: x is MXFP8-quantized along H before the gate/up GEMM and h along I
 *                 before the down GEMM (forward only). */
enum { ORACLE_EXACT = 0, ORACLE_BF16 = 1, ORACLE_MXFP8 = 2 };

/* Forward of the layer, per token, with no schedule and no permutation:
 *   a = W13[e] x  (gate rows 0..I-1, up rows I..2I-1), h = silu(a_g) * a_u,
 *   o = W2[e] h,  y_t = sum over k ascending of w[t,k] * o_k,
 * with the operand rounding of `mode` (ORACLE_*). Weights are stored as `wkind`
 * (ORACLE_W_*); for ORACLE_W_MXFP8, w13_s and w2_s hold the E8M0 scales along each
 * weight row. x [T][H], idx/w [T][K], w13 [E][2I][H], w2 [E][H][I], y [T][H]. */
void oracle_forward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const double *x,
                    const int32_t *idx, const double *w, int32_t wkind, const void *w13,
                    const uint8_t *w13_s, const void *w2, const uint8_t *w2_s, int32_t mode,
                    double *y, double *slack /* nullable [T][H] */);

/* Backward of the BF16 layer by the chain rule, given dy [T][H]:
 *   g = W2[e]^T dy_t, dS[t,k] = <g, h>, dh = w g,
 *   da_g = dh * a_u * silu'(a_g), da_u = dh * silu(a_g),
 *   dx_t = sum_k W13[e]^T da, dW13[e] = sum da x^T, dW2[e] = sum dy (w h)^T
 * ([arex] section "pull 代替 push": router-weight gradient computed with the SwiGLU
 * backward; [alphalab] section 一: expert gradient computation). Sums over routed rows run
 * in ascending flat id. mode is ORACLE_EXACT, ORACLE_BF16 (dA and w*h rounded to bf16
 * where they enter the dgrad and weight-gradient GEMMs) or ORACLE_MXFP8 ([arex] section
 * "pull 代替 push": MXFP8 activations and pre-quantized weights): A is recomputed from the
 * forward's quantized operands (x quantized along H, W13 given as ORACLE_W_MXFP8 with
 * w13_s), G = W2g^T Q(dy) with dy quantized along H and W2g = W2 quantized along H
 * (w2g [E][H][I], dequantized), dx = W13d^T Q(dA) with dA quantized in 32-blocks along 2I
 * and W13d = W13 quantized along 2I (w13d [E][2I][H], dequantized); the weight gradients
 * take dA and w*h rounded to bf16 as in ORACLE_BF16. Weights are ORACLE_W_F64 or
 * ORACLE_W_BF16 (ORACLE_W_MXFP8 for w13 in MXFP8 mode; w13d, w2g are NULL otherwise).
 * Outputs: dx [T][H], dw13 [E][2I][H], dw2 [E][H][I], dtopk [T][K] (= dS); dw13/dw2 may be
 * NULL (skipped). */
void oracle_backward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const double *x,
                     const int32_t *idx, const double *w, int32_t wkind, const void *w13,
                     const uint8_t *w13_s, const void *w2, const double *dy, int32_t mode,
                     const double *w13d, const double *w2g, double *dx, double *dw13,
                     double *dw2, double *dtopk, double *sdx, double *sdw13, double *sdw2);

/* Router-logit gradient through the top-k softmax: for a chosen expert j = idx[t,k],
 * dlogits[t,j] = w_k (dS_k - sum_m w_m dS_m); every other logit gets 0. */
void oracle_router_grad(int64_t T, int32_t E, int32_t K, const int32_t *idx, const double *w,
                        const double *dtopk, double *dlogits);

#ifdef __cplusplus
}
#endif
#endif
