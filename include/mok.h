/*
 * mok.h -- C ABI of the deterministic MoE layer core for one GB300 (sm_103a).
 *
 * The layer: top-k routing over router logits, a deterministic expert schedule, a
 * pull-style gather of token rows into expert order, an expert-grouped SwiGLU FFN
 * (gate/up GEMM, SwiGLU, down GEMM), a push-style scatter of expert outputs back to
 * (token, k) slots and a fixed-order router-weighted reduction; plus the matching
 * backward pass. Every expert lives on this one GPU, so dispatch and combine are HBM
 * gathers and scatters.
 *
 * Pages cited (by title and section):
 *   [arex]     "Cursor 放出 MoK：NVL72 训练提速 2.37 倍" (arex-research.com)
 *   [aigwx]    "Cursor 开源 MoK：面向 GB300 NVL72 的确定性 MoE 训练内核，性能提升 2.37 倍" (aigwx.org)
 *   [alphalab] "Mixture-of-Kittens" analysis (alphalab.site)
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, 16-byte aligned,
 *    row-major and densely packed. The library allocates no device memory: scratch
 *    space comes from the caller's workspace (sized by mok_workspace_size).
 *  - Work is enqueued on `stream` and returns without waiting for the GPU. Only
 *    mok_read_device_status synchronises.
 *  - Arguments are validated on the host before anything is enqueued; a non-OK status
 *    means nothing was enqueued. Problems the GPU detects (an index out of range, a
 *    bounded wait that ran out) are recorded in a device status word that
 *    mok_read_device_status returns; the kernel that found them skips the bad access.
 *  - Same inputs give bitwise-identical outputs, run to run: no floating-point sum
 *    depends on thread or block scheduling ([alphalab] section 二: operator-level
 *    run-to-run bitwise determinism through a fixed floating-point operation order).
 *  - Only compute capability 10.3 is accepted ([alphalab] section 四: the functional API
 *    rejects anything but SM103); other devices get MOK_ERR_UNSUPPORTED.
 *
 * Shapes: T tokens, H hidden, I expert intermediate, E experts, K experts per token,
 * R = T*K routed rows. Limits: 1 <= K <= min(E, 32), E <= 1024, H and I multiples of 128,
 * H <= 16384, I <= 8192, R < 2^31.
 */
#ifndef MOK_H
#define MOK_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOK_ABI_VERSION 2u

typedef enum mok_status {
    MOK_OK = 0,
    MOK_ERR_INVALID_ARG = 1,      /* shape, pointer, alignment or null-pointer error */
    MOK_ERR_UNSUPPORTED = 2,      /* device is not compute capability 10.3 */
    MOK_ERR_WORKSPACE = 3,        /* workspace missing or smaller than mok_workspace_size */
    MOK_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
    MOK_ERR_TIMEOUT = 5,          /* (device) a bounded wait inside a kernel ran out */
    MOK_ERR_DEVICE_INVARIANT = 6, /* (device) an index or count was out of range */
    MOK_ERR_ABI = 7               /* cfg->abi_version != MOK_ABI_VERSION */
} mok_status;

typedef enum mok_precision {
    MOK_BF16 = 0, /* bf16 operands, fp32 accumulation */
    MOK_MXFP8 = 1 /* E4M3 operands with an E8M0 scale per 32 elements along K */
} mok_precision;

/* mok_config.flags */
/* Keep every value that is only stored, never fed to a tensor-core GEMM, in fp32 instead of
 * bf16: the expert output of each (token, k) slot, the outputs y, dx, dw13, dw2 (and the
 * shared expert's), the saved pre-activations and the per-slot dgrad results. Without the
 * flag they are bf16 (round to nearest even of the fp32 accumulation), the storage a BF16
 * layer hands between its steps ([alphalab] section 三: the layer is benchmarked as a BF16
 * or MXFP8 layer and checked against a reference within a tolerance). Every accumulation
 * is fp32 either way; the flag changes what is stored and what later steps read. */
#define MOK_FLAG_FP32_STORAGE 1u
/* Which kernels compute the BF16 expert GEMMs. Each has two forms: one gives each output
 * tile to one SM; the other gives it to a pair of SMs that share their operand tiles (the
 * two-SM tensor-core MMA), so each SM loads fewer operand bytes per FLOP. The results are
 * the same bit for bit ([alphalab] section 五: warp specialization and PTX). By default the
 * gate/up GEMM and the routed experts' down and dx GEMMs run on pairs; the weight gradients
 * (dw13, dw2) run on pairs when an expert averages at least 512 rows (T*K/E; T for the
 * shared expert) and on one SM below that, where the pair measured slower; the shared
 * expert's down and dx GEMMs, which add into y and dx, run on one SM. The MXFP8 GEMMs
 * always run on one SM. MOK_FLAG_ONE_SM_GEMMS forces one SM per tile,
 * MOK_FLAG_SM_PAIR_GEMMS forces pairs for every BF16 GEMM; setting both is
 * MOK_ERR_INVALID_ARG. */
#define MOK_FLAG_ONE_SM_GEMMS 2u
#define MOK_FLAG_SM_PAIR_GEMMS 4u

typedef enum mok_workspace_kind {
    MOK_WS_SCHEDULE = 0,
    MOK_WS_FORWARD = 1,
    MOK_WS_BACKWARD = 2,
    MOK_WS_BACKWARD_RECOMPUTE = 3, /* backward without saved pre-activations */
    MOK_WS_SHARED = 4,             /* shared-expert forward */
    MOK_WS_SHARED_BACKWARD = 5     /* shared-expert backward */
} mok_workspace_kind;

/* Layer configuration. minibatch and ring_capacity are two of the pages' tunables
 * ([alphalab] section 四: forward/backward communication SMs, minibatch, macrobatch and
 * schedule capacity; the communication-SM knobs have no meaning on one GPU). */
typedef struct mok_config {
    uint32_t abi_version; /* MOK_ABI_VERSION */
    int32_t T, H, I, E, K;
    /* Routed rows (of the expert-sorted stream) per minibatch, >= 1. The pages suggest a
     * size that fills at least two SM waves per grouped GEMM ([arex] section "pull 代替
     * push", point 3: about 2,368 tokens for one shape). */
    int32_t minibatch;
    /* Rows of the fixed-size ring ("macrobatch", [arex] section "pull 代替 push", point 2).
     * 0, or any value >= R, means the ring holds every routed row: the forward gathers all
     * of them, then runs each GEMM over every tile. Otherwise ring_capacity >= minibatch is
     * required and the forward is one persistent launch in which sorted row r passes
     * through row r mod ring_capacity of two rings: gather units pull their tokens' x rows
     * into the x ring, gate/up units read them and write h into the h ring, down units
     * read h back and push to the slots; a ring row is rewritten only after the units
     * that read its previous row have finished. Results are the same bit for bit for
     * every ring setting. No routed row is ever dropped. */
    int32_t ring_capacity;
    int32_t prec;   /* mok_precision of the forward; the backward is MOK_BF16 */
    uint32_t flags; /* MOK_FLAG_* (0: bf16 storage) */
} mok_config;

/* The schedule table ([arex] section "pull 代替 push": one schedule serves dispatch,
 * combine, reverse-combine and reverse-dispatch). All device arrays, caller-owned:
 *   counts  [E]      routed rows per expert
 *   offsets [E+1]    exclusive prefix sum of counts (offsets[E] = R)
 *   perm    [R]      sorted row -> flat routed id f = t*K + k; rows are grouped by expert,
 *                    and within an expert ordered by ascending f (a stable sort)
 *   inv     [R]      flat id f -> sorted row (inverse of perm)
 *   segs    [cap][3] (expert, row_begin, row_end): the non-empty intersections of each
 *                    expert's rows with the minibatch ranges [m*MB, (m+1)*MB), in
 *                    increasing row order; cap = mok_segment_capacity(cfg)
 *   n_segs  [1]      number of valid segs entries */
typedef struct mok_schedule {
    int32_t *counts;
    int32_t *offsets;
    int32_t *perm;
    int32_t *inv;
    int32_t *segs;
    int32_t *n_segs;
} mok_schedule;

/* ---- helpers (host only, no GPU work) ---------------------------------------------- */

uint32_t mok_abi_version(void);
const char *mok_status_string(mok_status s);

/* Validates a configuration (shapes, limits, ABI version) without touching the GPU. */
mok_status mok_check_config(const mok_config *cfg);

/* Upper bound on the number of schedule segments: E + ceil(R / minibatch) - 1 (at least 1). */
int64_t mok_segment_capacity(const mok_config *cfg);

/* Bytes of device workspace that mok_build_schedule / mok_forward / mok_backward need
 * (which = mok_workspace_kind). Returns 0 for an invalid configuration. The workspace
 * must be 256-byte aligned; its contents on entry do not matter. */
size_t mok_workspace_size(const mok_config *cfg, int which);

/* Intermediates a call leaves in its workspace, for inspection and testing (the pages have
 * no counterpart; the layer's own outputs never need them). Rows are sorted rows (the
 * schedule's order) in the forward, padded rows in the backward (expert e owns rows
 * [poff[e], poff[e+1]), its counts[e] real rows first, poff[e] = sum over experts before e
 * of counts rounded up to 16). After a forward through a ring that holds every routed row
 * the ring rows are the R sorted rows; through a smaller ring of C rows, ring row j holds
 * the last sorted row r with r mod C = j.
 *   MOK_ITEM_X_RING       forward: gathered x [ring rows][H], bf16 or (MXFP8) E4M3
 *   MOK_ITEM_X_RING_SCALE forward, MXFP8: its E8M0 scales [R][H/32] (ring of every row);
 *                         through a smaller ring, x is quantized once per token and this
 *                         is [T][H/32], the scales of x's token rows
 *   MOK_ITEM_H_RING       forward: h entering the down GEMM [ring rows][I], bf16 or E4M3
 *   MOK_ITEM_H_RING_SCALE forward, MXFP8: its E8M0 scales [ring rows][I/32]
 *   MOK_ITEM_RING_TILES   forward, smaller ring: the tiles (int32 expert, first row, end
 *                         row, 0) of sorted rows cut at expert boundaries, at multiples of
 *                         the ring capacity and at the tile height; int32 [4] header whose
 *                         first word is the tile count, then the tiles
 *   MOK_ITEM_RING_ORDER   forward, smaller ring: the units in the order they are claimed,
 *                         8 int32 each: tile, kind << 16 | weight block, expert, first
 *                         row, end row, first and last tile one ring lap back whose ring
 *                         rows the unit's tile overwrites (last < first: none), 0. Kind 0
 *                         is a gate/up unit (one per 128 features of I), 1 a down unit (one
 *                         per 256 features of H), 2 the tile's gather (block 0)
 *   MOK_ITEM_SLOTS        forward: expert output of each flat id t*K + k [R][H] (bf16, or
 *                         fp32 under MOK_FLAG_FP32_STORAGE); backward: the per-slot dgrad
 *                         results, likewise
 *   MOK_ITEM_PAD_OFFSETS  backward: poff [E+1] int32
 *   MOK_ITEM_DA           backward: dA = dL/d(gate, up) [padded rows][2I] bf16
 *   MOK_ITEM_WH           backward: topk_w * h [padded rows][I] bf16
 *   MOK_ITEM_DA_Q         backward, MXFP8: dA quantized along 2I [padded rows][2I] E4M3
 *   MOK_ITEM_DA_SCALE     backward, MXFP8: its E8M0 scales [padded rows][2I/32]
 *   MOK_ITEM_DY_Q         backward, MXFP8: dy quantized along H [padded rows][H] E4M3
 *   MOK_ITEM_DY_SCALE     backward, MXFP8: its E8M0 scales [padded rows][H/32]
 * For the shared expert (MOK_WS_SHARED / MOK_WS_SHARED_BACKWARD) the rows are token rows:
 *   MOK_ITEM_H_RING (bf16 h [T][I], or E4M3 with MOK_ITEM_H_RING_SCALE), MOK_ITEM_X_RING /
 *   MOK_ITEM_X_RING_SCALE (MXFP8 x [T][H]); backward MOK_ITEM_DA, MOK_ITEM_WH (rows padded
 *   to a multiple of 16), MOK_ITEM_DA_Q / _SCALE, MOK_ITEM_DY_Q / _SCALE.
 * Sets *offset (bytes from the workspace start) and *bytes. Host only. MOK_ERR_INVALID_ARG
 * for an invalid configuration, workspace kind or item, or an item that kind (or that
 * precision) does not hold. */
typedef enum mok_ws_item {
    MOK_ITEM_X_RING = 0,
    MOK_ITEM_X_RING_SCALE = 1,
    MOK_ITEM_H_RING = 2,
    MOK_ITEM_H_RING_SCALE = 3,
    MOK_ITEM_SLOTS = 4,
    MOK_ITEM_PAD_OFFSETS = 5,
    MOK_ITEM_DA = 6,
    MOK_ITEM_WH = 7,
    MOK_ITEM_DA_Q = 8,
    MOK_ITEM_DA_SCALE = 9,
    MOK_ITEM_DY_Q = 10,
    MOK_ITEM_DY_SCALE = 11,
    MOK_ITEM_RING_TILES = 12,
    MOK_ITEM_RING_ORDER = 13
} mok_ws_item;
mok_status mok_workspace_item(const mok_config *cfg, int which, int item, size_t *offset,
                              size_t *bytes);

/* ---- the hot path --------------------------------------------------------------- */

/* Top-k routing ([alphalab] section 四: top-k over router logits).
 * logits   [T][E] fp32.
 * topk_idx [T][K] int32 out: the K largest logits of each token, ordered by logit
 *          descending; equal logits (with -0 equal to +0) go to the lower expert id.
 * topk_w   [T][K] fp32 out: softmax over the K chosen logits (fp32 arithmetic).
 * Logits must be finite; NaN or infinite logits give unspecified (but in-range) ids. */
mok_status mok_route_topk(const mok_config *cfg, const float *logits, int32_t *topk_idx,
                          float *topk_w, cudaStream_t stream);

/* Deterministic expert schedule from topk_idx [T][K] (values in [0, E); an id out of range
 * is counted nowhere and raises MOK_ERR_DEVICE_INVARIANT in the device status). Fills
 * every array of *sched. Bit-exact and run-to-run identical. */
mok_status mok_build_schedule(const mok_config *cfg, const int32_t *topk_idx,
                              const mok_schedule *sched, void *ws, size_t ws_bytes,
                              cudaStream_t stream);

/* The schedule builder for callers that cannot allocate device memory. The pages have no
 * counterpart to this entry point; it is a deployment convenience of this library.
 * mok_build_schedule needs a workspace from the caller. Some callers cannot allocate one:
 * code running under a device-memory budget that another component owns (a framework or
 * server that hands out all GPU memory from its own pool and forbids raw cudaMalloc), or a
 * time-critical loop that cannot pay cudaMalloc's latency and implicit synchronisation.
 * This variant computes exactly what mok_build_schedule computes (same kernels, same
 * outputs, bit for bit) but keeps its scratch in a fixed array inside the library: a
 * file-scope __device__ array of MOK_NOALLOC_SCHEDULE_SCRATCH_BYTES bytes that every GPU
 * loading the library holds until the process exits. It calls no cudaMalloc or cudaFree.
 *   - The first call on a device, with that device current, looks up the array's device
 *     address (cudaGetSymbolAddress) and caches it; make that first call before any stream
 *     capture.
 *   - Configurations whose schedule workspace, mok_workspace_size(cfg, MOK_WS_SCHEDULE),
 *     exceeds MOK_NOALLOC_SCHEDULE_SCRATCH_BYTES are rejected with MOK_ERR_WORKSPACE before
 *     anything is enqueued (with E = 512 that is more than 2,097,152 routed rows).
 *   - Every call shares the one array and leaves its contents behind; nothing in it needs
 *     to start at zero. Calls whose work overlaps on the GPU (other streams, other host
 *     threads) race on the array and give undefined results: order them on one stream.
 *   - While profiling is on (mok_profile_enable), its kernels are timed under the same kind
 *     as mok_build_schedule's. */
#define MOK_NOALLOC_SCHEDULE_SCRATCH_BYTES (4u << 20)
mok_status mok_build_schedule_noalloc(const mok_config *cfg, const int32_t *topk_idx,
                                      const mok_schedule *sched, cudaStream_t stream);

/* Layer forward: gather -> gate/up GEMM + SwiGLU -> down GEMM -> scatter -> reduction
 * ([alphalab] section 一: pull dispatch, expert FFN/SwiGLU, push combine; section 二: the
 * final router-weighted reduction; section 三: that is the timed layer).
 *   x       [T][H] bf16 token activations.
 *   topk_w  [T][K] fp32 routing weights (from mok_route_topk).
 *   BF16:  w13 [E][2I][H] bf16 (rows 0..I-1 gate, I..2I-1 up), w2 [E][H][I] bf16,
 *          w13_scale = w2_scale = NULL. h = silu(gate)*up is rounded to bf16, the down
 *          GEMM's operand type.
 *   MXFP8: w13 [E][2I][H] E4M3 bytes with w13_scale [E][2I][H/32] E8M0 bytes, and
 *          w2 [E][H][I] E4M3 with w2_scale [E][H][I/32] (as made by mok_quantize_mxfp8);
 *          x is quantized to MXFP8 along H inside the gather and h along I inside the
 *          gate/up GEMM's epilogue ([arex] section "pull 代替 push": weights pre-quantized,
 *          activation quantization fused into dispatch, GEMM and SwiGLU).
 *   y       [T][H] bf16 out (fp32 under MOK_FLAG_FP32_STORAGE): y[t] = sum over
 *           k = 0..K-1, in that order, of topk_w[t,k] * o[t,k] in fp32, rounded once at the
 *           end; o[t,k] is the down GEMM's fp32 result stored in the (t, k) slot as bf16
 *           (fp32 under the flag).
 *   saved_preact  NULL, or [R][2I] bf16 out (fp32 under the flag): the gate/up GEMM result
 *           a = W13[e] x of sorted row r (needed by mok_backward, or by mok_backward_mxfp8
 *           after an MXFP8 forward, with the same flags). Each row holds I pairs, one per
 *           feature i: the gate value a[i] at 2i and the up value a[I+i] at 2i+1, so that
 *           the backward reads both halves of a feature with one access.
 * GEMMs accumulate in fp32; values that are only stored (expert outputs, saved
 * pre-activations, y) take the storage type of cfg->flags.
 * A ring smaller than R rows (cfg->ring_capacity) makes the forward one persistent launch
 * (one CTA per SM) that takes units from a device-side counter in a fixed order and waits,
 * before loading a unit's operands, for the units it depends on (a gate/up unit on its
 * tile's gather, a down unit on its tile's gate/up units; a gather or gate/up unit on the
 * units that read, one lap back, the ring rows it overwrites). The order makes every wait
 * one on an earlier unit, so the launch always completes; each wait is still bounded (2 s),
 * after which MOK_ERR_TIMEOUT is recorded in
 * the device status word and the launch returns early with y undefined. In MXFP8, x is
 * quantized along H once per token before that launch. Everything runs on `stream`. */
mok_status mok_forward(const mok_config *cfg, const void *x, const mok_schedule *sched,
                       const float *topk_w, const void *w13, const uint8_t *w13_scale,
                       const void *w2, const uint8_t *w2_scale, void *y, void *saved_preact,
                       void *ws, size_t ws_bytes, cudaStream_t stream);

/* Layer backward (BF16): reverse-combine gather of dy -> G = dy W2 with the SwiGLU
 * backward and the router-weight gradient in its epilogue -> dgrad and reverse-dispatch
 * scatter with a fixed-order k-sum -> weight gradients ([arex] section "pull 代替 push":
 * pull reverse-combine, push reverse-dispatch, router-weight gradient fused into the
 * SwiGLU backward; [alphalab] section 一: expert gradient computation).
 *   x, topk_w, w13, w2 as in mok_forward (BF16), dy [T][H] bf16 upstream gradient.
 *   saved_preact  [R][2I] from mok_forward (bf16, or fp32 under MOK_FLAG_FP32_STORAGE; the
 *            flags must match the forward's), or NULL: the backward then recomputes
 *            the gate/up GEMM from x and W13 ([alphalab] section 一, the backward's
 *            recompute of forward activations), with the same tiles and accumulation order
 *            as the forward, so the results are those of the saved-A path. The workspace
 *            must then be of size mok_workspace_size(cfg, MOK_WS_BACKWARD_RECOMPUTE),
 *            which adds an [R][2I] buffer for the recomputed pre-activations (stored as
 *            a saved one would be).
 *   dx       [T][H] bf16 out (fp32 under the flag): the fp32 sum over k in order of the
 *            per-slot dgrad results, each stored as bf16 (fp32 under the flag), rounded once.
 *   dw13     [E][2I][H], dw2 [E][H][I] bf16 out (fp32 under the flag): fp32 sums over each
 *            expert's rows in ascending flat id, rounded once (experts with no rows get 0).
 *   d_topk_w [T][K] fp32 out: dL/dtopk_w.
 *   d_logits NULL or [T][E] fp32 out: gradient through the top-k softmax (0 for logits
 *            that were not chosen).
 * The GEMM operands dA = dL/d(gate,up) and topk_w*h are rounded to bf16. */
mok_status mok_backward(const mok_config *cfg, const void *x, const mok_schedule *sched,
                        const float *topk_w, const void *saved_preact, const void *w13,
                        const void *w2, const void *dy, void *dx, void *dw13, void *dw2,
                        float *d_topk_w, float *d_logits, void *ws, size_t ws_bytes,
                        cudaStream_t stream);

/* Layer backward, MXFP8 ([arex] section "pull 代替 push": pre-quantized weights, MXFP8
 * activations): as mok_backward, with cfg->prec == MOK_MXFP8, after an MXFP8 mok_forward
 * that saved its pre-activations (required here). The G GEMM contracts over H with dy and
 * W2 quantized along H; the dgrad GEMM over 2I with dA and W13 quantized along 2I (dA is
 * quantized in the G GEMM's epilogue). The weight-gradient GEMMs stay BF16 (dA and w*h
 * rounded to bf16), as in mok_backward.
 *   w13t_q [E][H][2I] E4M3, w13t_s [E][H][2I/32]: W13 quantized along 2I, transposed;
 *   w2t_q  [E][I][H] E4M3,  w2t_s  [E][I][H/32]:  W2 quantized along H, transposed (both as
 *          made by mok_quantize_mxfp8_transposed from the bf16 weights).
 *   Other arguments and outputs as for mok_backward; the workspace is
 *   mok_workspace_size(cfg, MOK_WS_BACKWARD) for this (MXFP8) configuration. */
mok_status mok_backward_mxfp8(const mok_config *cfg, const void *x, const mok_schedule *sched,
                              const float *topk_w, const void *saved_preact,
                              const uint8_t *w13t_q, const uint8_t *w13t_s,
                              const uint8_t *w2t_q, const uint8_t *w2t_s, const void *dy,
                              void *dx, void *dw13, void *dw2, float *d_topk_w,
                              float *d_logits, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Shared expert, forward ([alphalab] "Mixture-of-Kittens" (alphalab.site), section 一: the
 * forward runs the FFN/SwiGLU of the shared and of the routed experts). Every token passes
 * through one more SwiGLU expert, with weight one and no routing, and its output is added
 * to y after the routed combine:
 *   y[t] += W2s (silu(W13s[0:I] x_t) * W13s[I:2I] x_t)      (one writer per element)
 * The shared expert has the routed experts' shape (H, I of cfg) and the mode's operand
 * rounding (h to bf16 before the down GEMM).
 *   x              [T][H] bf16, as for mok_forward.
 *   w13_s          [2I][H] bf16 (gate rows, then up rows); w2_s [H][I] bf16.
 *   y              [T][H], in and out (typically mok_forward's result): bf16, the fp32
 *                  down-GEMM result added to it in fp32 and rounded once (fp32 storage
 *                  under MOK_FLAG_FP32_STORAGE).
 *   saved_preact_s NULL, or [T][2I] out (bf16, or fp32 under the flag): the shared
 *                  expert's gate/up GEMM result, in the (gate, up) pair layout of
 *                  mok_forward's saved_preact.
 *   ws             at least mok_workspace_size(cfg, MOK_WS_SHARED) bytes.
 * BF16 (cfg->prec == MOK_BF16, else MOK_ERR_UNSUPPORTED; MXFP8 configurations use
 * mok_shared_expert_forward_mxfp8). Asynchronous on `stream`. */
mok_status mok_shared_expert_forward(const mok_config *cfg, const void *x, const void *w13_s,
                                     const void *w2_s, void *y, void *saved_preact_s, void *ws,
                                     size_t ws_bytes, cudaStream_t stream);

/* Shared expert, forward, MXFP8 (cfg->prec == MOK_MXFP8): as mok_shared_expert_forward with
 * the MXFP8 mode's operands ([arex] section "pull 代替 push"): x quantized along H, h along
 * I inside the gate/up GEMM's epilogue, pre-quantized weights.
 *   w13s_q [2I][H] E4M3 with w13s_scale [2I][H/32], w2s_q [H][I] E4M3 with w2s_scale
 *   [H][I/32] (as made by mok_quantize_mxfp8 from the bf16 shared weights).
 *   Other arguments as for mok_shared_expert_forward; ws at least
 *   mok_workspace_size(cfg, MOK_WS_SHARED) for this (MXFP8) configuration. */
mok_status mok_shared_expert_forward_mxfp8(const mok_config *cfg, const void *x,
                                           const uint8_t *w13s_q, const uint8_t *w13s_scale,
                                           const uint8_t *w2s_q, const uint8_t *w2s_scale,
                                           void *y, void *saved_preact_s, void *ws,
                                           size_t ws_bytes, cudaStream_t stream);

/* Shared expert, backward: the gradients of y += W2s (silu(W13s[0:I] x) * W13s[I:2I] x)
 * for every token, by the chain rule of mok_backward with one expert, weight one and no
 * router gradient ([alphalab] section 一: the backward's expert gradient computation):
 *   dx[t] += W13s^T dA_t                                    (added after the routed dx)
 *   dw13_s = sum_t dA_t x_t^T, dw2_s = sum_t dy_t h_t^T      (sums over t ascending)
 * with G = W2s^T dy_t, dA = (G * u * silu'(g), G * silu(g)) from the saved gate/up result
 * (g, u), and dA and h rounded to bf16 where they enter GEMMs, as in mok_backward.
 *   x, w13_s, w2_s as for mok_shared_expert_forward; saved_preact_s [T][2I] from it
 *   (required, same flags); dy [T][H] bf16.
 *   dx      [T][H], in and out (typically mok_backward's result): bf16, the fp32 dgrad
 *           result added in fp32 and rounded once (fp32 under MOK_FLAG_FP32_STORAGE).
 *   dw13_s  [2I][H] out; dw2_s [H][I] out (bf16, or fp32 under the flag).
 *   ws      at least mok_workspace_size(cfg, MOK_WS_SHARED_BACKWARD) bytes.
 * BF16 (cfg->prec == MOK_BF16, else MOK_ERR_UNSUPPORTED; MXFP8 configurations use
 * mok_shared_expert_backward_mxfp8). Asynchronous on `stream`. */
mok_status mok_shared_expert_backward(const mok_config *cfg, const void *x, const void *w13_s,
                                      const void *w2_s, const void *saved_preact_s,
                                      const void *dy, void *dx, void *dw13_s, void *dw2_s,
                                      void *ws, size_t ws_bytes, cudaStream_t stream);

/* Shared expert, backward, MXFP8 (cfg->prec == MOK_MXFP8): as mok_shared_expert_backward
 * with the operands of mok_backward_mxfp8 — the G GEMM on dy and W2s quantized along H, the
 * dgrad GEMM on dA and W13s quantized along 2I, the weight gradients on bf16 operands.
 *   w13st_q [H][2I] E4M3 with w13st_scale [H][2I/32]; w2st_q [I][H] E4M3 with w2st_scale
 *   [I][H/32] (mok_quantize_mxfp8_transposed of W13s with batch 1, rows 2I, cols H, and of
 *   W2s with rows H, cols I).
 *   saved_preact_s [T][2I] as written by mok_shared_expert_forward_mxfp8: required.
 *   Other arguments as for mok_shared_expert_backward; ws at least
 *   mok_workspace_size(cfg, MOK_WS_SHARED_BACKWARD) for this (MXFP8) configuration. */
mok_status mok_shared_expert_backward_mxfp8(const mok_config *cfg, const void *x,
                                            const uint8_t *w13st_q, const uint8_t *w13st_scale,
                                            const uint8_t *w2st_q, const uint8_t *w2st_scale,
                                            const void *saved_preact_s, const void *dy,
                                            void *dx, void *dw13_s, void *dw2_s, void *ws,
                                            size_t ws_bytes, cudaStream_t stream);

/* MXFP8 quantization of a bf16 matrix along its rows ([arex] section "pull 代替 push":
 * pre-quantized weights). src [rows][cols] bf16 -> q [rows][cols] E4M3, scale
 * [rows][cols/32] E8M0: per 32-element block, scale = 2^(floor(log2 amax) - 8) clamped to
 * [2^-127, 2^127] (byte 0 for an all-zero block); q = E4M3(value / scale), round to
 * nearest even, saturating at +-448. cols must be a multiple of 32. */
mok_status mok_quantize_mxfp8(const void *src_bf16, int64_t rows, int32_t cols, uint8_t *q,
                              uint8_t *scale, cudaStream_t stream);

/* MXFP8 quantization of a batch of bf16 matrices along their ROWS, stored transposed: the
 * pre-quantized weights of the MXFP8 backward ([arex] section "pull 代替 push"), whose G
 * and dgrad GEMMs contract over W2's H and W13's 2I. src [batch][rows][cols] bf16 ->
 * q [batch][cols][rows] E4M3, scale [batch][cols][rows/32] E8M0, each 32-element block of
 * a column (rows 32j..32j+31) quantized by the rule of mok_quantize_mxfp8. For the
 * backward: W2 [E][H][I] -> W2t [E][I][H]; W13 [E][2I][H] -> W13t [E][H][2I]. rows must be
 * a multiple of 32. */
mok_status mok_quantize_mxfp8_transposed(const void *src_bf16, int64_t batch, int32_t rows,
                                         int32_t cols, uint8_t *q, uint8_t *scale,
                                         cudaStream_t stream);

/* ---- instrumentation ------------------------------------------------------------ */

/* Per-kernel timing. While enabled (on != 0), each kernel (or fixed group of kernels) that
 * the entry points launch is bracketed by a pair of CUDA events recorded on the caller's
 * stream; enabling clears the record. Host-side only, off by default, not thread-safe. */
mok_status mok_profile_enable(int on);

/* Waits for the recorded events and reports, for up to `max` kernel kinds that launched at
 * least once since mok_profile_enable(1): the kind's name (static storage), its number of
 * kernel launches and the summed milliseconds of its event pairs. *n_kinds receives the
 * number of such kinds (it may exceed max). */
mok_status mok_profile_read(int32_t max, int32_t *n_kinds, const char **names,
                            int64_t *launches, double *ms);

/* Waits for the device, returns the first device-side error recorded since the last
 * clear (MOK_OK if none) in *out, and returns MOK_ERR_CUDA if the wait itself failed. */
mok_status mok_read_device_status(mok_status *out);
mok_status mok_clear_device_status(void);

/* A check of the device-side failure path that faults and hangs nothing. One thread waits,
 * through the same bounded wait every tensor-core GEMM role uses (a timeout records
 * MOK_ERR_TIMEOUT and the kernel returns), on an mbarrier that nothing completes, with a
 * limit of limit_us microseconds (1 .. 1000000) instead of the GEMMs' 2 s. After it the
 * device status word reads MOK_ERR_TIMEOUT and the context stays usable.
 * Asynchronous on `stream`; MOK_ERR_INVALID_ARG for a limit out of range. */
mok_status mok_selftest_bounded_wait(uint32_t limit_us, cudaStream_t stream);

/* The same check for the ring forward's waits (mok_forward through a ring smaller than R):
 * one thread waits, through the bounded spin its producers use, on a device counter that
 * nothing raises, with a limit of limit_us microseconds (1 .. 1000000) instead of 2 s.
 * If the status word already holds a problem the wait gives up at once (as a producer does
 * once another CTA has given up). Afterwards the status word reads MOK_ERR_TIMEOUT (or the
 * earlier problem) and the context stays usable. Asynchronous on `stream`;
 * MOK_ERR_INVALID_ARG for a limit out of range. */
mok_status mok_selftest_bounded_count_wait(uint32_t limit_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOK_H */
