// mok_internal.h -- host-side launchers shared between the entry points and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mok.h"

namespace mok {

// ---------------------------------------------------------------- instrumentation
enum KernelKind {
    KK_ROUTE = 0, KK_SCHEDULE, KK_TILES, KK_GATHER, KK_GEMM_UP, KK_GEMM_DOWN, KK_COMBINE,
    KK_QUANTIZE, KK_PAD, KK_GATHER_BWD, KK_GEMM_G, KK_ROUTER_GRAD, KK_GEMM_DGRAD,
    KK_DX_REDUCE, KK_WGRAD13, KK_WGRAD2, KK_SCALE_ATOMS, KK_SHARED_UP, KK_SHARED_DOWN,
    KK_SHARED_BWD, KK_RING_FWD, KK_COUNT
};
// while profiling is on: brackets the launches between begin and end with events
void prof_begin(int kind, cudaStream_t s);
void prof_end(int kind, cudaStream_t s, int n_kernels);
bool prof_on();

// the entry points' device check (compute capability 10.3) and the device's status word
mok_status current_device_status_word(int **status);

// devices a process may use (per-device caches are arrays of this size)
constexpr int MAX_DEV = 64;

// streaming multiprocessors of the current device (queried once per device), for sizing
// grids in whole waves; 1 if the query fails
int device_sm_count();

// ---------------------------------------------------------------- routing / schedule
cudaError_t launch_route_topk(const float *logits, int64_t T, int E, int K, int32_t *idx,
                              float *w, int *status, cudaStream_t s);

struct ScheduleWs {
    int32_t *hist;   // [n_chunks][E] per-chunk expert counts, then per-chunk bases
    int64_t n_chunks;
};
size_t schedule_ws_bytes(int64_t R, int E);
ScheduleWs schedule_ws_carve(void *ws, int64_t R, int E);
cudaError_t launch_build_schedule(const int32_t *idx, int64_t R, int E, int MB,
                                  const mok_schedule &sch, const ScheduleWs &ws, int *status,
                                  cudaStream_t s);

// ---------------------------------------------------------------- tile lists
// A tile is (expert, row_begin, row_end) over sorted rows; lists are built on the device
// from the schedule's offsets for a row window [p0, p1), cutting each expert's rows into
// chunks of at most `chunk` rows. Layout: int32 [cap][4], count at list[-4].
int64_t tile_list_cap(int64_t rows, int E, int chunk);
cudaError_t launch_build_tiles(const int32_t *offsets, int E, int64_t p0, int64_t p1, int chunk,
                               int32_t *list, int64_t cap, int *status, cudaStream_t s);

// ---------------------------------------------------------------- dispatch / combine
// offsets of a single expert owning rows [0, rows): off[0] = 0, off[1] = rows
cudaError_t launch_single_expert_offsets(int32_t *off, int64_t rows, cudaStream_t s);
// one thread waits, through the GEMM roles' bounded wait, on an mbarrier nothing completes
cudaError_t launch_bounded_wait_probe(int *status, uint64_t limit_ns, cudaStream_t s);
// one thread waits, through the ring forward's bounded counter wait, on a counter nothing
// raises
cudaError_t launch_bounded_count_probe(int *status, uint64_t limit_ns, cudaStream_t s);
// the backward's view of a single expert owning every token in token order: offsets
// [0, T], padded offsets [0, T rounded up to 16], counts [T], weight one and row r -> r
cudaError_t launch_single_expert_bwd_setup(int32_t *offsets, int32_t *poff, int32_t *counts,
                                           float *ones, int32_t *perm, int64_t T,
                                           cudaStream_t s);
// token-major gathers, for a ring that holds every row: ring[inv[t*K + k]] = x[t]
cudaError_t launch_gather_tok_bf16(const uint16_t *x, const int32_t *inv, int64_t T, int K,
                                   int H, uint16_t *ring, cudaStream_t s);
cudaError_t launch_gather_tok_mxfp8(const uint16_t *x, const int32_t *inv, int64_t T, int K,
                                    int H, uint8_t *ring_q, uint8_t *ring_s, cudaStream_t s);
cudaError_t launch_quantize_mxfp8(const uint16_t *src, int64_t rows, int cols, uint8_t *q,
                                  uint8_t *scale, cudaStream_t s);
// along rows, stored transposed: src [batch][rows][cols] -> q [batch][cols][rows]
cudaError_t launch_quantize_mxfp8_transposed(const uint16_t *src, int64_t batch, int rows,
                                             int cols, uint8_t *q, uint8_t *scale,
                                             cudaStream_t s);
// y[t] = sum_k w[t,k] * slots[t*K+k] in fp32 (w == nullptr: plain sum), k ascending;
// slots and y are fp32 when f32, else bf16 (y rounded once, after the sum)
cudaError_t launch_combine(const void *slots, const float *w, int64_t T, int K, int H,
                           void *y, bool f32, cudaStream_t s);

// backward: padded row offsets (each expert's rows rounded up to 16) and gathers
cudaError_t launch_pad_offsets(const int32_t *counts, int E, int32_t *poff, cudaStream_t s);
// prow (nullable) receives the padded row of every flat id; with dy_q/dy_s (MXFP8) dy is
// also quantized along H into the padded layout
cudaError_t launch_gather_bwd(const uint16_t *dy, const uint16_t *x, const int32_t *inv,
                              const int32_t *counts, const int32_t *offsets,
                              const int32_t *poff, int E, int64_t T, int K, int H,
                              uint16_t *dy_perm, uint16_t *x_perm, int32_t *prow, uint8_t *dy_q,
                              uint8_t *dy_s, cudaStream_t s);
cudaError_t launch_router_grad(const float *dS_part, int n_parts, const int32_t *inv,
                               const int32_t *offsets, const float *w, int64_t T, int K, int E,
                               float *d_topk, float *d_logits, cudaStream_t s);

// ---------------------------------------------------------------- grouped GEMMs
// Ring map parameters (see RingMap in common.cuh).
struct Ring {
    int64_t R;
    int32_t MB;
    int32_t n_slots;
};

// Forward gate/up GEMM with the SwiGLU epilogue, per tile (e, r0, r1):
//   a[r][j] = sum_c W13[e][j][c] * xring[ring(r)][c]   (j < 2I)
//   h[ring(r)][i] = silu(a[r][i]) * a[r][I+i]          (bf16, or MXFP8 along I)
//   preact[r] = a[r] (fp32 if preact_f32, else bf16) when preact != nullptr, in the saved
//   layout of (gate, up) pairs: preact[r][2i] = a[r][i], preact[r][2i+1] = a[r][I+i]
struct GemmUpArgs {
    const int32_t *tiles;
    int64_t tiles_cap;
    const void *xring;
    const uint8_t *xring_s;
    const void *w13;
    const uint8_t *w13_s;
    void *hring;
    uint8_t *hring_s;
    void *preact;
    int H, I, E;
    bool mxfp8;
    Ring ring;
    int *status;
    bool preact_f32;
};

// Forward down GEMM with the push scatter, per tile (e, r0, r1):
//   slots[perm[r]][c] = sum_i W2[e][c][i] * hring[ring(r)][i]   (fp32 if out_f32, else bf16)
struct GemmDownArgs {
    const int32_t *tiles;
    int64_t tiles_cap;
    const void *hring;
    const uint8_t *hring_s;
    const void *w2;
    const uint8_t *w2_s;
    const int32_t *perm;  // slot of each sorted row; nullptr: row r -> output row r
    void *slots;
    int H, I, E;
    bool mxfp8;
    Ring ring;
    int *status;
    bool accumulate;      // add into the output rows instead of storing
    bool out_f32;
};
// The GEMMs run on the tensor cores (gemm_tc.cu). Tiles are cut at gemm_tc_tile_rows()
// rows; ring_rows / rpad_cap are the rows of the buffers the TMA maps cover.
int gemm_tc_tile_rows(bool mxfp8);
int gemm_tc_dS_parts(int I);
cudaError_t launch_gemm_up_tc(const GemmUpArgs &a, int64_t ring_rows, cudaStream_t s);
// The gate/up GEMM again, for a backward without saved pre-activations: B is the gathered
// x in the padded expert layout (row poff[e] + r - offsets[e] holds sorted row r), and only
// the pre-activations of each sorted row are written (fp32 if preact_f32, else bf16).
cudaError_t launch_gemm_up_recompute_tc(const int32_t *tiles, int64_t tiles_cap,
                                        const uint16_t *x_perm, int64_t rpad_cap,
                                        const void *w13, const int32_t *offsets,
                                        const int32_t *poff, void *preact, bool preact_f32,
                                        int H, int I, int E, int *status, cudaStream_t s);
cudaError_t launch_gemm_down_tc(const GemmDownArgs &a, int64_t ring_rows, cudaStream_t s);
// MXFP8: E4M3 operands with scale atoms (see launch_scale_atoms_*): sf_w for the weights,
// sf_x / sf_h for the token tiles
cudaError_t launch_gemm_up_tc_mx(const GemmUpArgs &a, int64_t ring_rows, const uint8_t *sf_w,
                                 const uint8_t *sf_x, cudaStream_t s);
cudaError_t launch_gemm_down_tc_mx(const GemmDownArgs &a, int64_t ring_rows, const uint8_t *sf_w,
                                   const uint8_t *sf_h, cudaStream_t s);
// MXFP8 scales, plain [rows][K/32] -> the tensor cores' 128-row x 4-block atoms: per 128
// weight rows, or per token tile of the list (one atom per tile and K block)
cudaError_t launch_scale_atoms_rows(const uint8_t *src, int64_t rows, int K, uint8_t *dst,
                                    cudaStream_t s);
cudaError_t launch_scale_atoms_tiles(const int32_t *tiles, int64_t cap, const uint8_t *src,
                                     int64_t R, int MB, int n_slots, int K, uint8_t *dst,
                                     cudaStream_t s);
// the same for the backward's padded layout: sorted row r at poff[e] + r - offsets[e]
cudaError_t launch_scale_atoms_tiles_padded(const int32_t *tiles, int64_t cap,
                                            const uint8_t *src, const int32_t *offsets,
                                            const int32_t *poff, int K, uint8_t *dst,
                                            cudaStream_t s);

// The forward through a partial ring (capacity C < R) in one persistent launch
// (ring_fwd.cu): tiles cut at expert boundaries, at multiples of C and at `chunk` rows;
// gather units copy the x rows of their tokens (MXFP8: x quantized token-major, xs its
// scales) into x ring rows r mod C, gate/up units read them and write h into h ring rows
// r mod C, down units read those and push to the slots. In half rows, a tile's gather is
// ordered `lag_gather` before its gate/up units and its down units `lag` after them;
// 1 <= lag_gather, lag <= 2 (C - chunk) + 1 keeps every wait on an earlier claim.
struct RingFwdArgs {
    const int32_t *offsets;  // schedule offsets [E+1]
    const int32_t *perm;     // flat id of each sorted row
    int32_t *tiles;          // flat tile list (count at [-4]), tiles_cap entries
    int64_t tiles_cap;
    void *units;             // [tiles_cap * (gather_pieces + I/128 + H/256)] 32-byte unit
                             // records in claim order
    int32_t *hdr;            // [2] unit count, claim counter
    int32_t *done_up, *done_dn, *done_g;  // [tiles_cap] per-tile completion counters
    const void *x;           // bf16 x [T][H], or (MXFP8) E4M3 x quantized along H
    const uint8_t *xs;       // MXFP8: x's scales [T][H/32]
    void *xring;             // [C][H] bf16 or E4M3
    const void *w13, *w2;
    const uint8_t *sf_w13, *sf_w2;  // MXFP8: weight scale atoms
    uint8_t *sf_x, *sf_h;    // MXFP8: per-tile scale atoms of x and h ([tiles_cap][K/128][512])
    void *hring;             // [C][I] bf16 or E4M3
    uint8_t *hring_s;        // MXFP8: [C][I/32]
    void *preact;            // saved pre-activations (nullable)
    bool preact_f32;
    void *slots;             // [R][H]
    bool out_f32;
    int64_t T, R, C;
    int chunk;
    int gather_pieces;       // gather units per tile (ring_gather_pieces)
    int64_t lag_gather, lag;
    int H, I, E, K;
    bool mx;
    int *status;
};
// tile rows of the ring forward, its lags and its tile-list capacity
int ring_tile_rows(bool mxfp8, int64_t C);
void ring_lags(bool mxfp8, int64_t C, int64_t *lag_gather, int64_t *lag);
int ring_stage_rows(bool mxfp8, int H);
int ring_gather_pieces(bool mxfp8, int64_t C, int H);
int64_t ring_tiles_cap(int64_t R, int E, int64_t C, int chunk);
cudaError_t launch_ring_forward(const RingFwdArgs &a, cudaStream_t s);

// Backward G GEMM with the SwiGLU backward and router-weight gradient epilogue, per tile
// (e, r0, r1) over sorted rows; p(r) = poff[e] + r - offsets[e] is the padded row:
//   g[r][i] = sum_c W2[e][c][i] * dy_perm[p(r)][c]
//   dS_part[r][part] = fixed-order partial sums of g * h over feature blocks
//   dA[p(r)][i] = w g a_u silu'(a_g), dA[p(r)][I+i] = w g silu(a_g), sh[p(r)][i] = w h
// Pad rows of the tile (up to the next multiple of 16) get zeros in dA and sh.
struct GemmGArgs {
    const int32_t *tiles;
    int64_t tiles_cap;
    const int32_t *offsets;
    const int32_t *poff;
    const uint16_t *w2;
    const uint16_t *dy_perm;
    const void *preact;  // fp32 if preact_f32, else bf16
    const int32_t *perm;
    const float *topk_w;
    uint16_t *dA;
    uint16_t *sh;
    float *dS_part;
    int H, I;
    int *status;
    // MXFP8 (w2 and dy_perm unused): W2 quantized along H and stored as W2t [E*I][H],
    // dy quantized along H [rpad][H]; the scale atoms of W2t and of the dy tiles; dA also
    // quantized along 2I into dA_q [rpad][2I] / dA_s [rpad][2I/32]
    bool mxfp8 = false;
    const uint8_t *w2t_q = nullptr, *sf_w2t = nullptr, *dy_q = nullptr, *sf_dy = nullptr;
    uint8_t *dA_q = nullptr, *dA_s = nullptr;
    bool preact_f32 = false;
};

// Backward dgrad GEMM with the reverse-dispatch scatter, per tile (e, r0, r1):
//   dx_slots[perm[r]][c] = sum_j W13[e][j][c] * dA[p(r)][j]   (fp32 if out_f32, else bf16)
struct GemmDgradArgs {
    const int32_t *tiles;
    int64_t tiles_cap;
    const int32_t *offsets;
    const int32_t *poff;
    const uint16_t *w13;
    const uint16_t *dA;
    const int32_t *perm;
    void *dx_slots;
    int H, I;
    int *status;
    // MXFP8 (w13 and dA unused): W13 quantized along 2I and stored as W13t [E*H][2I], dA
    // quantized along 2I [rpad][2I]; the scale atoms of W13t and of the dA tiles
    bool mxfp8 = false;
    const uint8_t *w13t_q = nullptr, *sf_w13t = nullptr, *dA_q = nullptr, *sf_dA = nullptr;
    bool accumulate = false;  // add into the output rows (the shared expert adds into dx)
    bool out_f32 = false;
};
cudaError_t launch_gemm_g_tc(const GemmGArgs &a, int E, int64_t rpad_cap, cudaStream_t s);
cudaError_t launch_gemm_dgrad_tc(const GemmDgradArgs &a, int E, int64_t rpad_cap,
                                 cudaStream_t s);
// BF16 expert GEMMs on pairs of SMs sharing their operand tiles (tcgen05 cta_group::2),
// bit for bit equal to the one-SM launchers: gate/up and dgrad over tiles of <=
// PAIR_TILE_ROWS rows, down over tiles of <= gemm_tc_tile_rows(false) rows
constexpr int PAIR_TILE_ROWS = 256;
cudaError_t launch_gemm_up_pair_tc(const GemmUpArgs &a, int64_t ring_rows, cudaStream_t s);
cudaError_t launch_gemm_down_pair_tc(const GemmDownArgs &a, int64_t ring_rows, cudaStream_t s);
cudaError_t launch_gemm_dgrad_pair_tc(const GemmDgradArgs &a, int E, int64_t rpad_cap,
                                      cudaStream_t s);
// out [E][N][M] = per expert e, sum over its padded rows p of A[p][m] * B[p][n]
// (fp32 if out_f32, else bf16)
cudaError_t launch_wgrad_tc(const int32_t *counts, const int32_t *poff, const uint16_t *A,
                            const uint16_t *Bm, void *out, bool out_f32, int E, int M, int N,
                            int64_t rows_a, int64_t rows_b, int *status, cudaStream_t s);
// the same on pairs of SMs sharing their operand tiles (tcgen05 cta_group::2), bit for bit
// equal; needs N % 128 == 0 (wgrad_pair_supported)
bool wgrad_pair_supported(int M, int N);
cudaError_t launch_wgrad_pair_tc(const int32_t *counts, const int32_t *poff, const uint16_t *A,
                                 const uint16_t *Bm, void *out, bool out_f32, int E, int M,
                                 int N, int64_t rows_a, int64_t rows_b, int *status,
                                 cudaStream_t s);

}  // namespace mok
