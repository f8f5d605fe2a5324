// gemm_tc.cu -- the expert-grouped GEMMs of the layer on the 5th-generation tensor cores.
//
// [alphalab] "Mixture-of-Kittens" (alphalab.site), section 一: routed experts run a SwiGLU
// FFN (gate/up GEMM, SwiGLU, down GEMM) and the backward computes expert gradients between
// reverse-combine and reverse-dispatch; section 五: warp specialization and PTX.
// [arex] "Cursor 放出 MoK" (arex-research.com), section "pull 代替 push": expert-grouped
// GEMMs fed by pull dispatch, results pushed back to their (token, k) slots, and the
// router-weight gradient computed inside the SwiGLU backward.
//
// One persistent kernel template, 320 threads per CTA, one CTA per SM:
//   warp 0     TMA producer: two 128-row A tiles and one 128-row B tile per 64-wide K
//              block into a 4-stage shared-memory ring, in as few boxes as the operand
//              layout allows (each box costs the copy engine a fixed overhead)
//   warp 1     TMEM owner and MMA issuer: D0 += A0 B^T, D1 += A1 B^T (M=128, N<=128,
//              K=16 per instruction) into one of two fp32 accumulator sets in TMEM
//   warps 2-9  epilogue: TMEM -> registers -> fused epilogue -> global memory; two warps
//              per TMEM lane quadrant, taking alternate 16-column chunks of a unit
// The two accumulator sets alternate between consecutive units of a CTA, so the epilogue
// of one unit runs while the tensor cores compute the next.
//
// Scheduling: one CTA is launched per work unit, but a running CTA does not exit after its
// unit. Near the end of each unit its producer thread asks Cluster Launch Control to cancel
// the launch of a CTA that has not started yet and takes over that CTA's unit, so about one
// CTA per SM runs and units go, in launch order, to whichever CTA frees up first. (The G
// GEMM instead strides statically over its units with one CTA per SM; see BwdGT.) The
// producer passes each unit index to the MMA thread and the epilogue warps through a small
// shared-memory queue. CTAs whose index is past the device-side unit count return at once.
// A problem policy supplies the work-unit decomposition, the operand majors and the
// epilogue:
//   FwdUp     A = W13 (K-major), B = x ring (K-major)      -> SwiGLU, h (bf16 / MXFP8)
//   FwdDown   A = W2 (K-major),  B = h ring (K-major)      -> push scatter to slots
//   BwdG      A = W2^T (MN-major), B = dy_perm (K-major)   -> SwiGLU backward, dA, w*h, dS
//             (MXFP8: A = W2t K-major, B = quantized dy; dA also quantized)
//   BwdDgrad  A = W13^T (MN-major), B = dA (K-major)       -> reverse-dispatch scatter
//             (MXFP8: A = W13t K-major, B = quantized dA)
//   Wgrad     A, B MN-major over an expert's padded rows   -> dW
// Values that are only stored (saved pre-activations, slots, dx slots, dW) are bf16, or fp32
// when the caller asks for fp32 storage; every accumulation is fp32.
// Every GEMM puts the weight (or output-contiguous) dimension on M and the routed rows on
// N or K, so ragged experts cost at most 15 padding rows. Every output element is one
// fixed-order fp32 dot product, independent of which CTA computes its unit.
#include "gemm_tc_core.cuh"

namespace mok {
namespace {

// backward G GEMM: g[r][i] = sum_c W2[e][c][i] dy_perm[p(r)][c]; A0/A1 = features
// [mb*256, +128) and [mb*256+128, +128) of W2^T (MN-major: W2 rows are c).
// MXFP8: A = W2t [E*I][H] E4M3 (W2 quantized along H, stored transposed: K-major), B = dy
// quantized along H; the epilogue also quantizes dA along 2I for the MXFP8 dgrad.
template <bool MXv, bool PF32 = false>
struct BwdGT {
    static constexpr bool A_MN = !MXv, B_MN = false, MX = MXv;
    static constexpr int A_MODE = MXv ? A_ROWS256 : A_MN4;
    // static striding: the four units of a token tile (one per 256-feature block) then run
    // in lockstep on neighbouring CTAs, so their epilogues read the pre-activation rows
    // together; under Cluster Launch Control they drift apart and this epilogue-bound
    // kernel measured 16% slower
    static constexpr bool CLC = false;
    static constexpr bool FUSED = false;  // the engine's own producer
    TileUnits tu;
    int H, I;
    const int32_t *offsets, *poff, *perm;
    const void *preact;  // [R][2I], fp32 if PF32, else bf16
    const float *topk_w;
    uint16_t *dA, *sh;
    float *dS_part;
    int n_parts;
    int *status;
    const uint8_t *sf_a, *sf_b;  // MXFP8: scale atoms of W2t and of the dy tiles
    uint8_t *dA_q, *dA_s;        // MXFP8: dA quantized along 2I [rpad][2I], [rpad][2I/32]

    MOK_DEV int64_t n_units() const { return tu.count(); }
    MOK_DEV Geom geom(int64_t u) const {
        int e, mb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &mb);
        Geom g;
        if (MX) {
            g.ax0 = 0;
            g.ay0 = e * I + mb * 256;  // rows of W2t: features mb*256 .. +256 of expert e
            g.ax1 = 0;
            g.ay1 = g.ay0 + 128;
            g.k_steps = H / 32;
            const int64_t kg = H / 128;
            g.sfa0 = (int64_t)(g.ay0 / 128) * kg * 512;
            // when I is not a multiple of 256 the last block's A1 lies past this expert
            g.sfa1 = mb * 256 + 128 < I ? (int64_t)(g.ay1 / 128) * kg * 512 : g.sfa0;
            g.sfb = (u / tu.n_mblocks) * kg * 512;
        } else {
            g.ax0 = mb * 256;
            g.ay0 = e * H;
            g.ax1 = g.ax0 + 128;
            g.ay1 = e * H;
            g.k_steps = H / 16;
        }
        g.bx = 0;
        g.by = (int32_t)(poff[e] + (r0 - offsets[e]));
        g.n_mma = (int)((r1 - r0 + 15) & ~15);
        g.nbox = 1;
        return g;
    }
    template <class LD>
    MOK_DEV void epilogue(int64_t u, const LD &ld, EpiScratch &es, int q, int half,
                          int lane) const {
        int e, mb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &mb);
        const int nr = (int)(r1 - r0);
        const int n_mma = (nr + 15) & ~15;
        const int64_t pb = poff[e] + (r0 - offsets[e]);
        const bool last = r1 == offsets[e + 1];
        const int i0 = mb * 256 + q * 32 + lane;
        // the routing weight of every column of the unit, loaded once
        for (int n = lane; n < nr; n += 32) es.col[n] = topk_w[perm[r0 + n]];
        __syncwarp();
        for (int n0 = 16 * half; n0 < n_mma; n0 += 32) {
            float d[2][16];
            ld(n0, d[0], d[1]);
            // issue every pre-activation load of the chunk before using any
            // the pre-activation pairs (gate, up) of the lane's features, every load of the
            // chunk issued before the first is used: a 32-bit word of two bf16, or two fp32
            float2 pg[2][16];
            uint32_t pw[2][16];
            uint32_t my_sb = 0;  // MXFP8: the block scale this lane stores for its 4-row group
            const int64_t row0 = (r0 + n0) * (int64_t)I;
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int i = i0 + a * 128;
                    const bool ok = (n0 + j < nr) && i < I;
                    const int64_t o = row0 + (int64_t)j * I + i;
                    if (PF32)
                        pg[a][j] = ok ? static_cast<const float2 *>(preact)[o]
                                      : make_float2(0.f, 0.f);
                    else
                        pw[a][j] = ok ? static_cast<const uint32_t *>(preact)[o] : 0u;
                }
            auto gate_of = [&](int a, int j) { return PF32 ? pg[a][j].x : bf16_lo(pw[a][j]); };
            auto up_of = [&](int a, int j) { return PF32 ? pg[a][j].y : bf16_hi(pw[a][j]); };
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int n = n0 + j;
                const int64_t p = pb + n;
                float gh_sum = 0.f;
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    const int i = i0 + a * 128;
                    if (i >= I) continue;
                    if (n < nr) {
                        const float s = es.col[n];
                        const float g = d[a][j];
                        const float agv = gate_of(a, j), auv = up_of(a, j);
                        const float sig = 1.0f / (1.0f + expf(-agv));
                        const float sl = agv * sig;
                        const float h = sl * auv;
                        const float dh = s * g;
                        const float dag = dh * auv * sig * (1.0f + agv * (1.0f - sig));
                        const float dau = dh * sl;
                        dA[p * 2 * I + i] = f32_to_bf16(dag);
                        dA[p * 2 * I + I + i] = f32_to_bf16(dau);
                        sh[p * I + i] = f32_to_bf16(s * h);
                        gh_sum += g * h;
                        if (MX) {
                            // the warp's 32 lanes hold one 32-feature block of the gate
                            // half and one of the up half of row p; the block maxima of
                            // the magnitudes come from one integer reduction each (the bit
                            // patterns of non-negative floats order like the floats)
                            const float mg = __uint_as_float(__reduce_max_sync(
                                0xFFFFFFFFu, __float_as_uint(fabsf(dag))));
                            const float mu = __uint_as_float(__reduce_max_sync(
                                0xFFFFFFFFu, __float_as_uint(fabsf(dau))));
                            const uint32_t sbg = mx_scale_byte(mg), sbu = mx_scale_byte(mu);
                            const uint32_t c2 =
                                e4m3x2(dag * mx_inv_scale(sbg), dau * mx_inv_scale(sbu));
                            const int pc = ((j & 3) * 2 + a) * 2;  // staged pieces of the row
                            es.stage[pc * 32 + lane] = (uint8_t)(c2 & 0xFFu);
                            es.stage[(pc + 1) * 32 + lane] = (uint8_t)(c2 >> 8);
                            if (lane == pc) my_sb = sbg;
                            if (lane == pc + 1) my_sb = sbu;
                        }
                    } else if (last) {  // zero pad rows up to the next multiple of 16
                        dA[p * 2 * I + i] = 0;
                        dA[p * 2 * I + I + i] = 0;
                        sh[p * I + i] = 0;
                        if (MX) {
                            const int pc = ((j & 3) * 2 + a) * 2;
                            es.stage[pc * 32 + lane] = 0;
                            es.stage[(pc + 1) * 32 + lane] = 0;
                            if (lane == pc || lane == pc + 1) my_sb = 0;
                        }
                    }
                }
                es.red[j][lane] = gh_sum;
                if (MX && (j & 3) == 3) {
                    // MXFP8 codes of the last 4 rows: 16 pieces of 32 bytes (row, feature
                    // half a, gate or up) staged; one 16-byte store per lane, and the 16
                    // block scales from lanes 0-15
                    __syncwarp();
                    const int pl = lane >> 1, hb = lane & 1;
                    const int nl = n0 + j - 3 + (pl >> 2);
                    const int ibl = mb * 256 + q * 32 + ((pl >> 1) & 1) * 128;
                    if (ibl < I && (nl < nr || last))
                        *reinterpret_cast<uint4 *>(dA_q + (pb + nl) * 2 * I + ((pl & 1) ? I : 0) +
                                                   ibl + hb * 16) =
                            *reinterpret_cast<const uint4 *>(es.stage + lane * 16);
                    if (lane < 16) {
                        const int ns = n0 + j - 3 + (lane >> 2);
                        const int ibs = mb * 256 + q * 32 + ((lane >> 1) & 1) * 128;
                        if (ibs < I && (ns < nr || last))
                            dA_s[(pb + ns) * (2 * I / 32) + (((lane & 1) ? I : 0) + ibs) / 32] =
                                (uint8_t)my_sb;
                    }
                    __syncwarp();
                }
            }
            __syncwarp();
            // one partial per (row, weight block, warp): lanes summed in lane order; the
            // router-gradient kernel adds the partials in index order
            if (lane < 16 && n0 + lane < nr) {
                float v = 0.f;
                for (int l = 0; l < 32; ++l) v += es.red[lane][l];
                dS_part[(r0 + n0 + lane) * n_parts + mb * 4 + q] = v;
            }
            __syncwarp();
        }
    }
};

// backward dgrad: dx_slots[perm[r]][c] = sum_j W13[e][j][c] dA[p(r)][j]; A = W13^T
// (MN-major: W13 rows are j). MXFP8: A = W13t [E*H][2I] E4M3 (W13 quantized along 2I,
// stored transposed: K-major), B = dA quantized along 2I.
template <bool MXv>
struct BwdDgradT {
    static constexpr bool A_MN = !MXv, B_MN = false, MX = MXv;
    static constexpr int A_MODE = MXv ? A_ROWS256 : A_MN4;
    static constexpr bool CLC = true;
    static constexpr bool FUSED = false;  // the engine's own producer
    TileUnits tu;
    int H, I;
    const int32_t *offsets, *poff, *perm;
    void *dx_slots;              // [rows][H], fp32 if out_f32, else bf16
    bool out_f32;
    int *status;
    const uint8_t *sf_a, *sf_b;  // MXFP8: scale atoms of W13t and of the dA tiles
    bool accumulate;             // add into the output rows (the shared expert adds into dx)

    MOK_DEV int64_t n_units() const { return tu.count(); }
    MOK_DEV Geom geom(int64_t u) const {
        int e, mb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &mb);
        Geom g;
        if (MX) {
            g.ax0 = 0;
            g.ay0 = e * H + mb * 256;  // rows of W13t: columns mb*256 .. +256 of expert e
            g.ax1 = 0;
            g.ay1 = g.ay0 + 128;
            g.k_steps = 2 * I / 32;
            const int64_t kg = 2 * I / 128;
            g.sfa0 = (int64_t)(g.ay0 / 128) * kg * 512;
            g.sfa1 = mb * 256 + 128 < H ? (int64_t)(g.ay1 / 128) * kg * 512 : g.sfa0;
            g.sfb = (u / tu.n_mblocks) * kg * 512;
        } else {
            g.ax0 = mb * 256;
            g.ay0 = e * 2 * I;
            g.ax1 = g.ax0 + 128;
            g.ay1 = e * 2 * I;
            g.k_steps = 2 * I / 16;
        }
        g.bx = 0;
        g.by = (int32_t)(poff[e] + (r0 - offsets[e]));
        g.n_mma = (int)((r1 - r0 + 15) & ~15);
        g.nbox = 1;
        return g;
    }
    template <class LD>
    MOK_DEV void epilogue(int64_t u, const LD &ld, EpiScratch &es, int q, int half,
                          int lane) const {
        int e, mb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &mb);
        const int nr = (int)(r1 - r0);
        const int n_mma = (nr + 15) & ~15;
        const int c = mb * 256 + q * 32 + lane;
        int *fcol = reinterpret_cast<int *>(es.col);  // slot of each column
        for (int n = lane; n < nr; n += 32) fcol[n] = perm[r0 + n];
        __syncwarp();
        const bool has1 = c + 128 < H;
        for (int n0 = 16 * half; n0 < n_mma; n0 += 32) {
            float d0[16], d1[16];
            ld(n0, d0, d1);
            if (accumulate) {  // every load of the chunk before any store (see FwdDownT)
                float a0[16], a1[16];
                if (out_f32)
                    load_rows16<true>(dx_slots, fcol, n0, nr, H, c, has1, a0, a1);
                else
                    load_rows16<false>(dx_slots, fcol, n0, nr, H, c, has1, a0, a1);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    d0[j] += a0[j];
                    d1[j] += a1[j];
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int n = n0 + j;
                if (n < nr) {
                    const int64_t f = fcol[n];
                    st_val(dx_slots, f * H + c, d0[j], out_f32);
                    if (has1) st_val(dx_slots, f * H + c + 128, d1[j], out_f32);
                }
            }
        }
        __syncwarp();
    }
};

// weight gradient of one expert: out[e][n][m] = sum over its padded rows p of
// A[p][m] * B[p][n]; A, B row-major [rows][M] / [rows][N] (both MN-major operands).
struct Wgrad {
    static constexpr bool A_MN = true, B_MN = true, MX = false;
    static constexpr int A_MODE = A_MN4;
    static constexpr bool CLC = true;
    static constexpr bool FUSED = false;  // the engine's own producer
    static constexpr const uint8_t *sf_a = nullptr, *sf_b = nullptr;
    const int32_t *counts, *poff;
    void *out;       // fp32 if out_f32, else bf16
    bool out_f32;
    int E, M, N;     // out is [E][N][M]
    int nmb, nnb;    // ceil(M/256), ceil(N/128)
    int *status;

    MOK_DEV int64_t n_units() const { return (int64_t)E * nmb * nnb; }
    MOK_DEV void get(int64_t u, int *e, int *mb, int *nb) const {
        *e = (int)(u / ((int64_t)nmb * nnb));
        const int rest = (int)(u % ((int64_t)nmb * nnb));
        *nb = rest / nmb;
        *mb = rest % nmb;
    }
    MOK_DEV Geom geom(int64_t u) const {
        int e, mb, nb;
        get(u, &e, &mb, &nb);
        Geom g;
        g.ax0 = mb * 256;
        g.ay0 = poff[e];
        g.ax1 = g.ax0 + 128;
        g.ay1 = poff[e];
        g.bx = nb * TILE_ROWS;
        g.by = poff[e];
        const int nn = N - nb * TILE_ROWS < TILE_ROWS ? N - nb * TILE_ROWS : TILE_ROWS;
        g.n_mma = nn;
        g.nbox = nn / 64;
        g.k_steps = ((counts[e] + 15) & ~15) / 16;
        return g;
    }
    template <class LD>
    MOK_DEV void epilogue(int64_t u, const LD &ld, EpiScratch &, int q, int half,
                          int lane) const {
        int e, mb, nb;
        get(u, &e, &mb, &nb);
        const int nn = N - nb * TILE_ROWS < TILE_ROWS ? N - nb * TILE_ROWS : TILE_ROWS;
        const bool any = counts[e] > 0;
        const int m = mb * 256 + q * 32 + lane;
        const int64_t base = (int64_t)e * N * M;
        for (int n0 = 16 * half; n0 < nn; n0 += 32) {
            float d0[16], d1[16];
            ld(n0, d0, d1);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int64_t row = base + (int64_t)(nb * TILE_ROWS + n0 + j) * M;
                st_val(out, row + m, any ? d0[j] : 0.f, out_f32);
                if (m + 128 < M) st_val(out, row + m + 128, any ? d1[j] : 0.f, out_f32);
            }
        }
    }
};

}  // namespace

int gemm_tc_tile_rows(bool mxfp8) { return mxfp8 ? TILE_ROWS_MX : TILE_ROWS; }

cudaError_t launch_gemm_up_tc(const GemmUpArgs &a, int64_t ring_rows, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W13 gate/up block pairs; B: the x ring [ring_rows][H]
    if ((e = make_map_w13_pairs(&ma, a.w13, a.E, a.I, a.H, false)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, a.xring, ring_rows, a.H, KBOX_ROWS)) != cudaSuccess) return e;
    FwdUpT<false> p{TileUnits{a.tiles, a.tiles_cap, a.I / 128}, a.H, a.I, a.ring, a.hring,
                    a.hring_s, a.preact, a.preact_f32, false, a.status, nullptr, nullptr,
                    nullptr, nullptr};
    return launch(ma, mb, p, a.tiles_cap * (a.I / 128),
                  (ring_rows + TILE_ROWS - 1) / TILE_ROWS * (a.I / 128), s);
}

cudaError_t launch_gemm_up_recompute_tc(const int32_t *tiles, int64_t tiles_cap,
                                        const uint16_t *x_perm, int64_t rpad_cap,
                                        const void *w13, const int32_t *offsets,
                                        const int32_t *poff, void *preact, bool preact_f32,
                                        int H, int I, int E, int *status, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W13 gate/up block pairs; B: x in the padded layout [rpad][H]
    if ((e = make_map_w13_pairs(&ma, w13, E, I, H, false)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, x_perm, rpad_cap, H, KBOX_ROWS)) != cudaSuccess) return e;
    FwdUpT<false> p{TileUnits{tiles, tiles_cap, I / 128}, H, I, Ring{1, 1, 0}, nullptr,
                    nullptr, preact, preact_f32, false, status, nullptr, nullptr, offsets, poff};
    // the padded rows overestimate the real ones by at most 15 per expert
    return launch(ma, mb, p, tiles_cap * (I / 128),
                  (rpad_cap + TILE_ROWS - 1) / TILE_ROWS * (I / 128), s);
}

cudaError_t launch_gemm_down_tc(const GemmDownArgs &a, int64_t ring_rows, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W2 as [E*H][I], 256-row boxes; B: the h ring [ring_rows][I]
    if ((e = make_map_bf16(&ma, a.w2, (int64_t)a.E * a.H, a.I, 256)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, a.hring, ring_rows, a.I, KBOX_ROWS)) != cudaSuccess) return e;
    const int nmb = (a.H + 255) / 256;
    FwdDownT<false> p{TileUnits{a.tiles, a.tiles_cap, nmb}, a.H, a.I, a.ring, a.perm, a.slots,
                      a.out_f32, a.status, nullptr, nullptr, a.accumulate};
    return launch(ma, mb, p, a.tiles_cap * nmb, (ring_rows + TILE_ROWS - 1) / TILE_ROWS * nmb, s);
}

cudaError_t launch_gemm_up_tc_mx(const GemmUpArgs &a, int64_t ring_rows, const uint8_t *sf_w,
                                 const uint8_t *sf_x, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W13 E4M3 gate/up block pairs; B: the quantized x ring
    if ((e = make_map_w13_pairs(&ma, a.w13, a.E, a.I, a.H, true)) != cudaSuccess) return e;
    if ((e = make_map_u8(&mb, a.xring, ring_rows, a.H, KBOX_ROWS)) != cudaSuccess) return e;
    FwdUpT<true> p{TileUnits{a.tiles, a.tiles_cap, a.I / 128}, a.H, a.I, a.ring, a.hring,
                   a.hring_s, a.preact, a.preact_f32, true, a.status, sf_w, sf_x, nullptr,
                   nullptr};
    return launch(ma, mb, p, a.tiles_cap * (a.I / 128),
                  (ring_rows + TILE_ROWS_MX - 1) / TILE_ROWS_MX * (a.I / 128), s);
}

cudaError_t launch_gemm_down_tc_mx(const GemmDownArgs &a, int64_t ring_rows, const uint8_t *sf_w,
                                   const uint8_t *sf_h, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W2 E4M3 [E*H][I], 256-row boxes; B: the quantized h ring
    if ((e = make_map_u8(&ma, a.w2, (int64_t)a.E * a.H, a.I, 256)) != cudaSuccess) return e;
    if ((e = make_map_u8(&mb, a.hring, ring_rows, a.I, KBOX_ROWS)) != cudaSuccess) return e;
    const int nmb = (a.H + 255) / 256;
    FwdDownT<true> p{TileUnits{a.tiles, a.tiles_cap, nmb}, a.H, a.I, a.ring, a.perm, a.slots,
                     a.out_f32, a.status, sf_w, sf_h, a.accumulate};
    return launch(ma, mb, p, a.tiles_cap * nmb,
                  (ring_rows + TILE_ROWS_MX - 1) / TILE_ROWS_MX * nmb, s);
}

// the G GEMM with its epilogue's operand types fixed at compile time; static striding
template <bool MX, bool PF32>
cudaError_t launch_g(const CUtensorMap &ma, const CUtensorMap &mb, const GemmGArgs &a, int nmb,
                     cudaStream_t s) {
    BwdGT<MX, PF32> p{TileUnits{a.tiles, a.tiles_cap, nmb}, a.H, a.I, a.offsets, a.poff,
                      a.perm, a.preact, a.topk_w, a.dA, a.sh, a.dS_part, 4 * nmb, a.status,
                      MX ? a.sf_w2t : nullptr, MX ? a.sf_dy : nullptr,
                      MX ? a.dA_q : nullptr, MX ? a.dA_s : nullptr};
    return launch(ma, mb, p, a.tiles_cap * nmb, a.tiles_cap * nmb, s);
}

cudaError_t launch_gemm_g_tc(const GemmGArgs &a, int E, int64_t rpad_cap, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W2 as [E*H][I] read MN-major; B: dy_perm [rpad][H]
    if (!a.mxfp8) {
        if ((e = make_map_bf16(&ma, a.w2, (int64_t)E * a.H, a.I, 64)) != cudaSuccess) return e;
        if ((e = make_map_bf16(&mb, a.dy_perm, rpad_cap, a.H, KBOX_ROWS)) != cudaSuccess)
            return e;
    }
    const int nmb = (a.I + 255) / 256;
    if (a.mxfp8) {
        // A: W2t E4M3 [E*I][H], 256-row boxes; B: quantized dy [rpad][H]
        if ((e = make_map_u8(&ma, a.w2t_q, (int64_t)E * a.I, a.H, 256)) != cudaSuccess) return e;
        if ((e = make_map_u8(&mb, a.dy_q, rpad_cap, a.H, KBOX_ROWS)) != cudaSuccess) return e;
        if (a.preact_f32)
            return launch_g<true, true>(ma, mb, a, nmb, s);
        return launch_g<true, false>(ma, mb, a, nmb, s);
    }
    if (a.preact_f32) return launch_g<false, true>(ma, mb, a, nmb, s);
    return launch_g<false, false>(ma, mb, a, nmb, s);
}

int gemm_tc_dS_parts(int I) { return 4 * ((I + 255) / 256); }

cudaError_t launch_gemm_dgrad_tc(const GemmDgradArgs &a, int E, int64_t rpad_cap,
                                 cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W13 as [E*2I][H] read MN-major; B: dA [rpad][2I]
    const int nmb = (a.H + 255) / 256;
    if (a.mxfp8) {
        // A: W13t E4M3 [E*H][2I], 256-row boxes; B: quantized dA [rpad][2I]
        if ((e = make_map_u8(&ma, a.w13t_q, (int64_t)E * a.H, 2 * a.I, 256)) != cudaSuccess)
            return e;
        if ((e = make_map_u8(&mb, a.dA_q, rpad_cap, 2 * a.I, KBOX_ROWS)) != cudaSuccess)
            return e;
        BwdDgradT<true> p{TileUnits{a.tiles, a.tiles_cap, nmb}, a.H, a.I, a.offsets, a.poff,
                          a.perm, a.dx_slots, a.out_f32, a.status, a.sf_w13t, a.sf_dA,
                          a.accumulate};
        return launch(ma, mb, p, a.tiles_cap * nmb,
                      (rpad_cap + TILE_ROWS_MX - 1) / TILE_ROWS_MX * nmb, s);
    }
    if ((e = make_map_bf16(&ma, a.w13, (int64_t)E * 2 * a.I, a.H, 64)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, a.dA, rpad_cap, 2 * a.I, KBOX_ROWS)) != cudaSuccess) return e;
    BwdDgradT<false> p{TileUnits{a.tiles, a.tiles_cap, nmb}, a.H, a.I, a.offsets, a.poff,
                       a.perm, a.dx_slots, a.out_f32, a.status, nullptr, nullptr, a.accumulate};
    return launch(ma, mb, p, a.tiles_cap * nmb, (rpad_cap + TILE_ROWS - 1) / TILE_ROWS * nmb, s);
}

// out [E][N][M] = per expert sum over padded rows of A[p][m] B[p][n]
cudaError_t launch_wgrad_tc(const int32_t *counts, const int32_t *poff, const uint16_t *A,
                            const uint16_t *Bm, void *out, bool out_f32, int E, int M, int N,
                            int64_t rows_a, int64_t rows_b, int *status, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // rows past an operand's own rows read the copy engine's zero fill
    if ((e = make_map_bf16(&ma, A, rows_a, M, 64)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, Bm, rows_b, N, 64)) != cudaSuccess) return e;
    const int nmb = (M + 255) / 256, nnb = (N + TILE_ROWS - 1) / TILE_ROWS;
    Wgrad p{counts, poff, out, out_f32, E, M, N, nmb, nnb, status};
    return launch(ma, mb, p, (int64_t)E * nmb * nnb, (int64_t)E * nmb * nnb, s);  // exact
}

}  // namespace mok