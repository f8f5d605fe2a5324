// gemm_pair.cu -- expert GEMMs on pairs of SMs that share their operand tiles.
//
// [alphalab] "Mixture-of-Kittens" (alphalab.site), section 一: the backward computes the
// expert gradients dW13 = dA^T x and dW2 = (w*h)^T dy per expert over its routed rows, and
// reverse-dispatches dx = dA W13; section 五: warp specialization and PTX.
// [arex] "Cursor 放出 MoK" (arex-research.com), section "pull 代替 push": the backward's dx
// rows are pushed back to their (token, k) slots.
//
// A cluster of two CTAs on two SMs computes one output tile with the two-SM MMA (tcgen05
// cta_group::2, M = 256): rank r holds rows [128r, +128) of the tile's 256 M rows as its A
// half and loads half of the tile's N columns as its B half; the MMA gives each CTA its 128
// M rows against all N columns. Per 64-element K block a SM loads 128 A rows and N/2 B rows
// for 128 x N outputs, where the one-SM engine loads 256 A rows and N B rows (N <= 128) for
// 256 x N: at N = 256 the operand feed per FLOP falls by a third, the weight tiles' by half.
// (A policy with two MMAs per K step loads 256 A rows for 256 x N, N <= 128.)
// Each output element is the same fixed-order fp32 dot product as in the one-SM engine (K
// in 16-element steps from the first), so the results are the same bit for bit.
//
// Per CTA, 320 threads:
//   warp 0     TMA producer (both ranks): its own halves of the unit's operands (boxes per
//              policy) into a ring of 5-6 stages; the copies of both ranks complete on rank
//              0's full barrier of the stage, whose expected bytes rank 0 sets
//   warp 1     TMEM owner (both ranks: the pair allocates together); on rank 0 the MMA
//              issuer, whose commits arrive on the stage-free and accumulator-full barriers
//              of both CTAs
//   warps 2-9  epilogue (both ranks): TMEM -> the policy's epilogue; each warp then arrives
//              on rank 0's accumulator-free barrier
// Two accumulator sets of 256 columns alternate between consecutive units (a set holds
// one accumulator of N <= 256 columns, or two of N <= 128 at columns 0 and 128). The clusters
// take the units in a static stride; consecutive units share operand tiles, so the clusters
// running at one time share them in L2.
//
// Problems (policies):
//   WgradPair  A, B MN-major over an expert's padded rows -> dW (output rows on M)
//   DgradPair  A = W13^T (MN-major), B = dA (K-major) in token tiles of <= 256 rows
//              -> reverse-dispatch scatter to the dx slots (features on M)
//   UpPair     A = 64 gate + 64 up rows of W13 per CTA (K-major), B = x ring rows in tiles
//              of <= 256 -> SwiGLU, with gate and up values of a feature handed between
//              two epilogue warps through shared memory
//   DownPair   A = two 128-row blocks of W2 per CTA (K-major, two MMAs per K step), B = h
//              ring rows in tiles of <= 128 -> push scatter to the slots
//
// Every wait is bounded (2 s); a CTA that gives up records MOK_ERR_TIMEOUT and leaves its
// loops, and both CTAs meet at a cluster barrier before TMEM is freed.
#include "gemm_tc_core.cuh"

namespace mok {
namespace {

constexpr int PAIR_BOX = 64 * 128;           // one 64 x 64 bf16 box (8 KB)
constexpr uint32_t PAIR_SET_COLS = 256;      // TMEM columns of one accumulator set
constexpr int PAIR_TILE = 256;               // max N of a unit (token rows or dW columns)
constexpr int PAIR_MAX_STAGES = 6;

struct PairSmem {
    uint64_t full[PAIR_MAX_STAGES];   // rank 0: both CTAs' copies of the stage have landed
    uint64_t empty[PAIR_MAX_STAGES];  // each CTA: the MMAs that read the stage are done
    uint64_t tmem_full[2];            // each CTA: accumulator set b holds a finished unit
    uint64_t tmem_empty[2];           // rank 0: both CTAs' epilogues have drained set b
    uint64_t xbar[4];                 // exchange between the two warps of a lane pair
    uint32_t tmem_base;
    int abort;
    int32_t col[EPI_WARPS][PAIR_TILE];  // per epilogue warp: one index per column of a unit
};

template <class P>
__host__ __device__ constexpr int pair_smem() {
    return P::STAGES * P::STAGE_BYTES + 1024 + (int)sizeof(PairSmem) + P::XCH_BYTES;
}

// One unit as one CTA of the pair loads and multiplies it: the policy's coordinates and
// the MMA's shape.
struct PairGeom {
    int32_t ax, ay, ay2;  // A half (per policy)
    int32_t bx, by;       // B half (per policy)
    int nbox;
    int n_mma;            // N of each pair MMA (multiple of 16; of 128 for MN-major B)
    int k_steps;          // 16-element K steps; 0 leaves the accumulators unwritten
};

// What an epilogue warp gets besides its accumulator: a scratch of one index per column,
// the CTA's exchange buffers and barriers (policies whose SwiGLU pairs lanes of two warps),
// this warp's exchange phase, and the status / abort words of its bounded waits.
struct PairEpi {
    int32_t *col;
    float *xch;
    uint64_t *xbar;
    uint32_t *xph;
    int *status;
    volatile int *abort;
};

// 32 accumulator columns from TMEM address c (this warp's lane quadrant), one round trip
MOK_DEV void tmem_ld32(uint32_t c, float (&v)[32]) {
    float a[16], b[16];
    tc::tmem_ld16(c, a);
    tc::tmem_ld16(c + 16, b);
    tc::tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        v[j] = a[j];
        v[16 + j] = b[j];
    }
}

// Policy interface: STAGES x STAGE_BYTES of operand ring, the A region (A_BYTES) first in
// each stage; A_MN / B_MN operand majors; TWO: two MMAs per K step, on A rows 0-127 and
// 128-255 of the A region into accumulator columns 0 and 128 of a set (N <= 128), else one
// on A rows 0-127 into columns 0 (N <= 256); XCH_BYTES: shared memory for the epilogue's
// lane exchange; tx(g): bytes one CTA loads per stage; load(..): its copies of one stage;
// epilogue(..): TMEM -> outputs, false when a bounded wait gave up.

// weight gradient: out[e][n][m] = sum over the expert's padded rows p of A[p][m] B[p][n];
// a unit is (expert, 256-column block nb, 256-row block mb)
struct WgradPair {
    static constexpr bool A_MN = true, B_MN = true, TWO = false;
    static constexpr int A_BYTES = 2 * PAIR_BOX, STAGE_BYTES = 4 * PAIR_BOX, STAGES = 6;
    static constexpr int XCH_BYTES = 0;
    const int32_t *counts, *poff;
    void *out;     // [E][N][M], fp32 if out_f32, else bf16
    bool out_f32;
    int E, M, N;
    int nmb, nnb;  // ceil(M / 256), ceil(N / 256) (N is a multiple of 128)
    int *status;

    MOK_DEV int64_t n_units() const { return (int64_t)E * nmb * nnb; }
    MOK_DEV void get(int64_t u, int *e, int *mb, int *nb) const {
        *e = (int)(u / ((int64_t)nmb * nnb));
        const int rest = (int)(u % ((int64_t)nmb * nnb));
        *nb = rest / nmb;
        *mb = rest % nmb;
    }
    MOK_DEV int cols(int nb) const { return N - nb * 256 < 256 ? N - nb * 256 : 256; }
    MOK_DEV PairGeom geom(int64_t u, uint32_t rank) const {
        int e, mb, nb;
        get(u, &e, &mb, &nb);
        PairGeom g;
        g.n_mma = cols(nb);
        const int half = g.n_mma / 2;  // 64 or 128 columns of B per CTA
        g.ax = mb * 256 + (int)rank * 128;
        g.ay = poff[e];
        g.ay2 = 0;
        g.bx = nb * 256 + (int)rank * half;
        g.by = poff[e];
        g.nbox = half / 64;
        g.k_steps = ((counts[e] + 15) & ~15) / 16;
        return g;
    }
    MOK_DEV uint32_t tx(const PairGeom &g) const { return A_BYTES + g.nbox * PAIR_BOX; }
    // A: two 64-wide MN-major boxes of the CTA's 128 M rows; B: its columns, 64 per box
    MOK_DEV void load(uint8_t *st, uint32_t fb, const PairGeom &g, int k0,
                      const CUtensorMap *tmA, const CUtensorMap *tmB) const {
        tc::tma_load_2d_pair(st, tmA, fb, g.ax, g.ay + k0);
        tc::tma_load_2d_pair(st + PAIR_BOX, tmA, fb, g.ax + 64, g.ay + k0);
        for (int j = 0; j < g.nbox; ++j)
            tc::tma_load_2d_pair(st + A_BYTES + j * PAIR_BOX, tmB, fb, g.bx + 64 * j,
                                 g.by + k0);
    }
    MOK_DEV bool epilogue(int64_t u, uint32_t rank, uint32_t c, const PairEpi &, int q, int hw,
                          int lane) const {
        int e, mb, nb;
        get(u, &e, &mb, &nb);
        const int nn = cols(nb);
        const bool any = counts[e] > 0;
        const int m = mb * 256 + (int)rank * 128 + q * 32 + lane;
        const bool mok = m < M;
        const int64_t row0 = (int64_t)e * N + (int64_t)nb * 256;
        // 32 columns per TMEM round trip (nn is a multiple of 128)
        for (int n0 = 32 * hw; n0 < nn; n0 += 64) {
            float v[32];
            tmem_ld32(c + n0, v);
            if (mok) {
                const int64_t o = (row0 + n0) * M + m;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    st_val(out, o + (int64_t)j * M, any ? v[j] : 0.f, out_f32);
            }
        }
        return true;
    }
};

// Scatter of 32 accumulator columns n0.. of a token tile to output rows fcol[n] (< nr),
// column c; accumulate: add into the stored values (every load of the chunk before any
// store: a store to one row may alias the next row's load, which would otherwise
// serialise the round trips)
MOK_DEV void scatter32(void *outp, bool out_f32, bool accumulate, const int32_t *fcol, int n0,
                       int nr, int64_t ld_out, int c, float (&v)[32]) {
    if (accumulate) {
        float a[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const bool ok = n0 + j < nr;
            const int64_t o = (int64_t)fcol[ok ? n0 + j : 0] * ld_out + c;
            a[j] = !ok ? 0.f
                   : out_f32 ? static_cast<const float *>(outp)[o]
                             : bf16_to_f32(static_cast<const uint16_t *>(outp)[o]);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += a[j];
    }
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (n0 + j < nr) st_val(outp, (int64_t)fcol[n0 + j] * ld_out + c, v[j], out_f32);
}

// reverse dispatch: dx_slots[perm[r]][c] (+)= sum_j dA[r][j] W13[e][j][c] over the rows r
// of a token tile (e, r0, r1) of <= 256 rows; a unit is (tile, 256-feature block mb)
struct DgradPair {
    static constexpr bool A_MN = true, B_MN = false, TWO = false;
    static constexpr int A_BYTES = 2 * PAIR_BOX, STAGE_BYTES = 4 * PAIR_BOX, STAGES = 6;
    static constexpr int XCH_BYTES = 0;
    TileUnits tu;
    int H, I;
    const int32_t *offsets, *poff, *perm;
    void *dx_slots;   // [rows][H], fp32 if out_f32, else bf16
    bool out_f32;
    bool accumulate;  // add into the output rows (the shared expert adds into dx)
    int *status;

    MOK_DEV int64_t n_units() const { return tu.count(); }
    MOK_DEV PairGeom geom(int64_t u, uint32_t rank) const {
        int e, mb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &mb);
        PairGeom g;
        g.n_mma = (int)((r1 - r0 + 15) & ~15);
        g.ax = mb * 256 + (int)rank * 128;
        g.ay = e * 2 * I;
        g.ay2 = 0;
        g.bx = 0;
        g.by = (int32_t)(poff[e] + (r0 - offsets[e])) + (int)rank * (g.n_mma / 2);
        g.nbox = 1;
        g.k_steps = 2 * I / 16;
        return g;
    }
    MOK_DEV uint32_t tx(const PairGeom &) const { return A_BYTES + 2 * PAIR_BOX; }
    // A: two 64-wide MN-major boxes of W13^T; B: one 128-row K-major box of dA, of which
    // the MMA reads n_mma / 2 rows
    MOK_DEV void load(uint8_t *st, uint32_t fb, const PairGeom &g, int k0,
                      const CUtensorMap *tmA, const CUtensorMap *tmB) const {
        tc::tma_load_2d_pair(st, tmA, fb, g.ax, g.ay + k0);
        tc::tma_load_2d_pair(st + PAIR_BOX, tmA, fb, g.ax + 64, g.ay + k0);
        tc::tma_load_2d_pair(st + A_BYTES, tmB, fb, k0, g.by);
    }
    MOK_DEV bool epilogue(int64_t u, uint32_t rank, uint32_t c, const PairEpi &pe, int q, int hw,
                          int lane) const {
        int32_t *fcol = pe.col;
        int e, mb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &mb);
        const int nr = (int)(r1 - r0);
        const int n_mma = (nr + 15) & ~15;
        const int f = mb * 256 + (int)rank * 128 + q * 32 + lane;
        for (int n = lane; n < nr; n += 32) fcol[n] = perm[r0 + n];
        __syncwarp();
        for (int n0 = 32 * hw; n0 < n_mma; n0 += 64) {
            float v[32];
            tmem_ld32(c + n0, v);
            if (f < H) scatter32(dx_slots, out_f32, accumulate, fcol, n0, nr, H, f, v);
        }
        __syncwarp();
        return true;
    }
};

// both warps of a lane pair arrive (all 64 threads), then wait for the other (bounded)
MOK_DEV bool xsync(const PairEpi &pe, int pair) {
    tc::mbar_arrive(&pe.xbar[pair]);
    const bool ok = tc::wait_bounded(&pe.xbar[pair], *pe.xph, pe.status, pe.abort,
                                     tc::WAIT_LIMIT_NS);
    *pe.xph ^= 1u;
    return ok;
}

// forward gate/up with SwiGLU (BF16) on token tiles of <= 256 rows: a unit is (tile,
// 128-feature block fb), rank r taking features [fb*128 + 64r, +64) with their gate rows as
// A rows 0-63 and their up rows as A rows 64-127: one MMA per K step, N up to 256. A
// feature's gate value then sits on TMEM lane l of quadrant q < 2 and its up value on lane
// l of quadrant q + 2, in two warps: per 32-column chunk each of the two hands the other
// half of its columns through shared memory, and each computes SwiGLU for 16 columns.
struct UpPair {
    static constexpr bool A_MN = false, B_MN = false, TWO = false;
    static constexpr int A_BYTES = 2 * PAIR_BOX, STAGE_BYTES = 4 * PAIR_BOX, STAGES = 6;
    static constexpr int XCH_BYTES = 4 * 2 * 16 * 32 * 4;  // per lane pair: 2 x 16 x 32 fp32
    TileUnits tu;   // n_mblocks = I / 128
    int H, I;
    Ring ring;
    void *hring;    // [rows][I] bf16
    void *preact;   // [R][I] (gate, up) pairs, fp32 if preact_f32, else bf16; or nullptr
    bool preact_f32;
    int *status;

    MOK_DEV int64_t n_units() const { return tu.count(); }
    MOK_DEV PairGeom geom(int64_t u, uint32_t rank) const {
        int e, fb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &fb);
        PairGeom g;
        g.n_mma = (int)((r1 - r0 + 15) & ~15);
        g.ax = 0;
        g.ay = e * 2 * I + fb * 128 + (int)rank * 64;  // gate rows of the CTA's features
        g.ay2 = g.ay + I;                              // their up rows
        g.bx = 0;
        // a tile never straddles a lap of the ring: its rows are consecutive ring rows
        g.by = (int32_t)RingMap{ring.R, ring.MB, ring.n_slots}(r0) + (int)rank * (g.n_mma / 2);
        g.nbox = 1;
        g.k_steps = H / 16;
        return g;
    }
    MOK_DEV uint32_t tx(const PairGeom &) const { return A_BYTES + 2 * PAIR_BOX; }
    // A: two 64-row K-major boxes of W13 (gate, up); B: one 128-row K-major box of the x
    // ring, of which the MMA reads n_mma / 2 rows
    MOK_DEV void load(uint8_t *st, uint32_t fb, const PairGeom &g, int k0,
                      const CUtensorMap *tmA, const CUtensorMap *tmB) const {
        tc::tma_load_2d_pair(st, tmA, fb, k0, g.ay);
        tc::tma_load_2d_pair(st + PAIR_BOX, tmA, fb, k0, g.ay2);
        tc::tma_load_2d_pair(st + A_BYTES, tmB, fb, k0, g.by);
    }
    MOK_DEV bool epilogue(int64_t u, uint32_t rank, uint32_t c, const PairEpi &pe, int q, int hw,
                          int lane) const {
        int e, fb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &fb);
        const int nr = (int)(r1 - r0);
        const int n_mma = (nr + 15) & ~15;
        const int64_t hrow0 = RingMap{ring.R, ring.MB, ring.n_slots}(r0);
        const int i = fb * 128 + (int)rank * 64 + (q & 1) * 32 + lane;  // this lane's feature
        const int pair = (q & 1) + 2 * hw;  // the two warps of a lane pair share hw
        const bool gate_side = q < 2;
        float *xg = pe.xch + pair * 1024;   // written by the gate side: its columns 16-31
        float *xu = xg + 512;               // written by the up side: its columns 0-15
        for (int n0 = 32 * hw; n0 < n_mma; n0 += 64) {
            float v[32];
            tmem_ld32(c + n0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (gate_side)
                    xg[j * 32 + lane] = v[16 + j];
                else
                    xu[j * 32 + lane] = v[j];
            }
            if (!xsync(pe, pair)) return false;
            // the gate side finishes columns n0..n0+15, the up side n0+16..n0+31
            float g[16], up[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                g[j] = gate_side ? v[j] : xg[j * 32 + lane];
                up[j] = gate_side ? xu[j * 32 + lane] : v[16 + j];
            }
            if (!xsync(pe, pair)) return false;  // the buffers are free again
            const int nb = gate_side ? n0 : n0 + 16;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int n = nb + j;
                if (n < nr) {
                    const int64_t r = r0 + n;
                    if (preact != nullptr) {
                        if (preact_f32)
                            static_cast<float2 *>(preact)[r * I + i] = make_float2(g[j], up[j]);
                        else
                            static_cast<uint32_t *>(preact)[r * I + i] = pack_bf16x2(g[j], up[j]);
                    }
                    ((uint16_t *)hring)[(hrow0 + n) * I + i] = f32_to_bf16(silu_f(g[j]) * up[j]);
                }
            }
        }
        return true;
    }
};

// forward down with the push scatter (BF16): slots[perm[r]][c] (+)= sum_i W2[e][c][i]
// hring[r][i]; a unit is (tile of <= 128 rows, 512-feature block pb), rank r taking
// features [pb*512 + 128r, +128) and [pb*512 + 256 + 128r, +128) as A rows 0-127 and
// 128-255: two MMAs per K step
struct DownPair {
    static constexpr bool A_MN = false, B_MN = false, TWO = true;
    static constexpr int A_BYTES = 4 * PAIR_BOX, STAGE_BYTES = 5 * PAIR_BOX, STAGES = 5;
    static constexpr int XCH_BYTES = 0;
    TileUnits tu;  // n_mblocks = ceil(H / 512)
    int H, I;
    Ring ring;
    const int32_t *perm;  // output row of each sorted row (nullptr: the row itself)
    void *slots;          // [rows][H], fp32 if out_f32, else bf16
    bool out_f32;
    bool accumulate;      // add into the output (the shared expert adds into y)
    int *status;

    MOK_DEV int64_t n_units() const { return tu.count(); }
    MOK_DEV PairGeom geom(int64_t u, uint32_t rank) const {
        int e, pb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &pb);
        PairGeom g;
        g.n_mma = (int)((r1 - r0 + 15) & ~15);
        g.ax = 0;
        // rows past this expert's H (a partial last block) read the next expert's rows or
        // the zero fill; their results are discarded
        g.ay = e * H + pb * 512 + (int)rank * 128;
        g.ay2 = g.ay + 256;
        g.bx = 0;
        g.by = (int32_t)RingMap{ring.R, ring.MB, ring.n_slots}(r0) + (int)rank * (g.n_mma / 2);
        g.nbox = 1;
        g.k_steps = I / 16;
        return g;
    }
    MOK_DEV uint32_t tx(const PairGeom &) const { return A_BYTES + PAIR_BOX; }
    // A: two 128-row K-major boxes of W2; B: 64 K-major rows of the h ring
    MOK_DEV void load(uint8_t *st, uint32_t fb, const PairGeom &g, int k0,
                      const CUtensorMap *tmA, const CUtensorMap *tmB) const {
        tc::tma_load_2d_pair(st, tmA, fb, k0, g.ay);
        tc::tma_load_2d_pair(st + 2 * PAIR_BOX, tmA, fb, k0, g.ay2);
        tc::tma_load_2d_pair(st + A_BYTES, tmB, fb, k0, g.by);
    }
    MOK_DEV bool epilogue(int64_t u, uint32_t rank, uint32_t c, const PairEpi &pe, int q, int hw,
                          int lane) const {
        int32_t *fcol = pe.col;
        int e, pb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &pb);
        const int nr = (int)(r1 - r0);
        const int n_mma = (nr + 15) & ~15;
        const int f0 = pb * 512 + (int)rank * 128 + q * 32 + lane, f1 = f0 + 256;
        for (int n = lane; n < nr; n += 32)
            fcol[n] = perm != nullptr ? perm[r0 + n] : (int)(r0 + n);
        __syncwarp();
        // warps of hw 0 drain accumulator 0 (features f0), of hw 1 accumulator 1 (f1), 32
        // columns per TMEM round trip
        const int f = hw ? f1 : f0;
        const uint32_t ca = c + (hw ? 128u : 0u);
        for (int n0 = 0; n0 < n_mma; n0 += 32) {
            float v[32];
            tmem_ld32(ca + n0, v);
            if (f < H) scatter32(slots, out_f32, accumulate, fcol, n0, nr, H, f, v);
        }
        __syncwarp();
        return true;
    }
};

MOK_DEV bool pair_wait(uint64_t *bar, uint32_t parity, int *status, volatile int *abort) {
    return tc::wait_bounded_cluster(bar, parity, status, abort, tc::WAIT_LIMIT_NS);
}

// bounded drain of a barrier phase on the way out (no status: the loops already ended)
MOK_DEV void pair_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait_cluster(bar, parity) && tc::globaltimer() - t0 < 100000000ull) {
    }
}

template <class P>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const P p) {
    constexpr int NS = P::STAGES, SB = P::STAGE_BYTES;
    static_assert(NS <= PAIR_MAX_STAGES && pair_smem<P>() <= 232448, "pair kernel smem");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the same offset in both CTAs: the MMA finds the peer's tiles where this CTA has its own
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    PairSmem *sm = (PairSmem *)(base + NS * SB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_rank();
    const int64_t cid = tc::cluster_id_x(), ncl = tc::cluster_count_x();
    const int64_t n_units = p.n_units();

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(&sm->full[s], 1);
            tc::mbar_init(&sm->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sm->tmem_full[b], 1);
            tc::mbar_init(&sm->tmem_empty[b], 2 * EPI_WARPS);
        }
        for (int j = 0; j < 4; ++j) tc::mbar_init(&sm->xbar[j], 64);
        sm->abort = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tmA);
        tc::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tc::tmem_alloc_pair(&sm->tmem_base, TMEM_COLS);
        tc::tmem_relinquish_pair();
    }
    // both CTAs' barriers exist and TMEM is allocated before either CTA touches the other
    tc::tc_fence_before();
    tc::cluster_sync();
    tc::tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    volatile int *abort = &sm->abort;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (tc::elect_one()) {
            const uint32_t full0 = tc::cluster_addr(&sm->full[0], 0);  // rank 0's full[0]
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t u = cid; u < n_units && ok; u += ncl) {
                const PairGeom g = p.geom(u, rank);
                const uint32_t tx = p.tx(g);
                const int kblocks = (g.k_steps + 3) / 4;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!pair_wait(&sm->empty[s], ph ^ 1u, p.status, abort)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0) tc::mbar_arrive_expect_tx(&sm->full[s], 2 * tx);
                    p.load(base + s * SB, full0 + (uint32_t)s * 8u, g, kb * BK, &tmA, &tmB);
                    ++issued;
                    if (++s == NS) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // do not leave while copies may still be landing: the MMAs that read the last
            // stages have finished (bounded)
            for (int q = 0; q < NS && q < issued; ++q) {
                if (--s < 0) {
                    s = NS - 1;
                    ph ^= 1u;
                }
                pair_drain(&sm->empty[s], ph);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (rank 0)
        if (rank == 0 && tc::elect_one()) {
            int s = 0;
            uint32_t ph = 0;
            int64_t a = 0;  // units so far: unit a uses accumulator set a % 2
            bool ok = true;
            for (int64_t u = cid; u < n_units && ok; u += ncl, ++a) {
                const PairGeom g = p.geom(u, 0);
                const uint32_t idesc = tc::idesc_bf16(256, g.n_mma, P::A_MN, P::B_MN);
                const int ab = (int)(a & 1);
                const uint32_t use = (uint32_t)((a >> 1) & 1);
                if (!pair_wait(&sm->tmem_empty[ab], use ^ 1u, p.status, abort)) break;
                tc::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)ab * PAIR_SET_COLS;
                const int kblocks = (g.k_steps + 3) / 4;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!pair_wait(&sm->full[s], ph, p.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t sa = tc::smem_u32(base + s * SB);
                    const uint32_t sb = sa + P::A_BYTES;
                    const int steps = g.k_steps - kb * 4 < 4 ? g.k_steps - kb * 4 : 4;
                    for (int kk = 0; kk < steps; ++kk) {
                        // MN-major: 16 K rows = 2 groups of eight 128-byte rows, the two
                        // 64-wide blocks of 128 M rows PAIR_BOX apart; K-major: 16 elements
                        // = 32 bytes along the swizzled row, 128 rows = 16 KB
                        const uint64_t db =
                            P::B_MN ? tc::sdesc_sw128(sb + kk * 2048, PAIR_BOX, 1024)
                                    : tc::sdesc_sw128(sb + kk * 32, 16, 1024);
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
                        for (int h = 0; h < (P::TWO ? 2 : 1); ++h) {
                            const uint32_t sah = sa + (uint32_t)h * 2 * PAIR_BOX;
                            const uint64_t da =
                                P::A_MN ? tc::sdesc_sw128(sah + kk * 2048, PAIR_BOX, 1024)
                                        : tc::sdesc_sw128(sah + kk * 32, 16, 1024);
                            tc::mma_f16_pair(d + (uint32_t)h * 128, da, db, idesc, acc);
                        }
                    }
                    tc::mma_commit_pair(&sm->empty[s], 3);  // frees the stage in both CTAs
                    if (++s == NS) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                tc::mma_commit_pair(&sm->tmem_full[ab], 3);
            }
            // do not free TMEM under MMAs still in flight (bounded)
            if (a > 0) {
                const int lb = (int)((a - 1) & 1);
                pair_drain(&sm->tmem_full[lb], (uint32_t)(((a - 1) >> 1) & 1));
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;            // TMEM lane quadrant this warp may access
        const int hw = (warp - 2) >> 2;    // which alternate 32-column chunks it takes
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const uint32_t empty0 = tc::cluster_addr(&sm->tmem_empty[0], 0);
        uint32_t xph = 0;
        const PairEpi pe{sm->col[warp - 2], (float *)((uint8_t *)sm + sizeof(PairSmem)), sm->xbar,
                         &xph, p.status, abort};
        int64_t a = 0;
        for (int64_t u = cid; u < n_units; u += ncl, ++a) {
            const int ab = (int)(a & 1);
            if (!pair_wait(&sm->tmem_full[ab], (uint32_t)((a >> 1) & 1), p.status, abort))
                break;
            tc::tc_fence_after();
            // this quadrant's lanes of the unit's accumulator set
            if (!p.epilogue(u, rank, tmem + lane_base + (uint32_t)ab * PAIR_SET_COLS, pe, q, hw,
                            lane))
                break;
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster(empty0 + (uint32_t)ab * 8u);
        }
    }

    // no MMA, copy or arrival of either CTA targets the other past this point
    tc::tc_fence_before();
    tc::cluster_sync();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

// clusters of two that fit on a device at once, per device and kernel; queried once per
// device outside stream capture (a launch under capture before then uses one cluster per
// two SMs)
template <class P>
cudaError_t pair_clusters(int *out, cudaStream_t s) {
    static std::atomic<int> cache[MAX_DEV];
    static std::atomic<uint64_t> attr_set[2] = {{0}, {0}};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEV) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << (dev & 63);
    if ((attr_set[dev >> 6].load(std::memory_order_acquire) & bit) == 0) {
        e = cudaFuncSetAttribute(tc_pair_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 pair_smem<P>());
        if (e != cudaSuccess) return e;
        attr_set[dev >> 6].fetch_or(bit, std::memory_order_acq_rel);
    }
    int nc = cache[dev].load(std::memory_order_acquire);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (nc == 0 && cudaStreamIsCapturing(s, &cs) == cudaSuccess &&
        cs != cudaStreamCaptureStatusNone) {
        *out = device_sm_count() / 2 > 0 ? device_sm_count() / 2 : 1;
        return cudaSuccess;
    }
    if (nc == 0) {
        cudaLaunchConfig_t q = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        q.gridDim = dim3((unsigned)(2 * device_sm_count()), 1, 1);
        q.blockDim = dim3(NTHREADS, 1, 1);
        q.dynamicSmemBytes = pair_smem<P>();
        q.attrs = at;
        q.numAttrs = 1;
        // where the query fails, one cluster per two SMs: clusters that do not fit wait for
        // a free pair and take their units then (the static stride still covers them all)
        if (cudaOccupancyMaxActiveClusters(&nc, tc_pair_kernel<P>, &q) != cudaSuccess ||
            nc < 1) {
            (void)cudaGetLastError();
            nc = device_sm_count() / 2 > 0 ? device_sm_count() / 2 : 1;
        }
        cache[dev].store(nc, std::memory_order_release);
    }
    *out = nc;
    return cudaSuccess;
}

// units_cap: a host-side bound on the device-side unit count
template <class P>
cudaError_t launch_pair(const CUtensorMap &ma, const CUtensorMap &mb, const P &p,
                        int64_t units_cap, cudaStream_t s) {
    if (units_cap < 1) return cudaSuccess;
    if (units_cap > 0x7FFFFFFF) return cudaErrorInvalidValue;
    int nc = 0;
    cudaError_t e = pair_clusters<P>(&nc, s);
    if (e != cudaSuccess) return e;
    const int64_t clusters = units_cap < nc ? units_cap : nc;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = pair_smem<P>();
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, tc_pair_kernel<P>, ma, mb, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool wgrad_pair_supported(int M, int N) { return M > 0 && N > 0 && N % 128 == 0; }

// out [E][N][M] = per expert sum over padded rows of A[p][m] B[p][n]; N % 128 == 0
cudaError_t launch_wgrad_pair_tc(const int32_t *counts, const int32_t *poff, const uint16_t *A,
                                 const uint16_t *Bm, void *out, bool out_f32, int E, int M,
                                 int N, int64_t rows_a, int64_t rows_b, int *status,
                                 cudaStream_t s) {
    if (!wgrad_pair_supported(M, N)) return cudaErrorInvalidValue;
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // rows past an operand's own rows read the copy engine's zero fill
    if ((e = make_map_bf16(&ma, A, rows_a, M, 64)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, Bm, rows_b, N, 64)) != cudaSuccess) return e;
    const int nmb = (M + 255) / 256, nnb = (N + 255) / 256;
    WgradPair p{counts, poff, out, out_f32, E, M, N, nmb, nnb, status};
    return launch_pair(ma, mb, p, (int64_t)E * nmb * nnb, s);
}

// BF16 forward gate/up over tiles of <= PAIR_TILE_ROWS rows
cudaError_t launch_gemm_up_pair_tc(const GemmUpArgs &a, int64_t ring_rows, cudaStream_t s) {
    if (a.mxfp8) return cudaErrorInvalidValue;
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W13 as [E*2I][H], 64-row boxes; B: the x ring, 128-row boxes
    if ((e = make_map_bf16(&ma, a.w13, (int64_t)a.E * 2 * a.I, a.H, 64)) != cudaSuccess)
        return e;
    if ((e = make_map_bf16(&mb, a.xring, ring_rows, a.H, KBOX_ROWS)) != cudaSuccess) return e;
    UpPair p{TileUnits{a.tiles, a.tiles_cap, a.I / 128}, a.H, a.I, a.ring, a.hring, a.preact,
              a.preact_f32, a.status};
    return launch_pair(ma, mb, p, a.tiles_cap * (a.I / 128), s);
}

// BF16 forward down with the push scatter over tiles of <= 128 rows
cudaError_t launch_gemm_down_pair_tc(const GemmDownArgs &a, int64_t ring_rows, cudaStream_t s) {
    if (a.mxfp8) return cudaErrorInvalidValue;
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W2 as [E*H][I], 128-row boxes; B: the h ring, 64-row boxes
    if ((e = make_map_bf16(&ma, a.w2, (int64_t)a.E * a.H, a.I, 128)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, a.hring, ring_rows, a.I, 64)) != cudaSuccess) return e;
    const int npb = (a.H + 511) / 512;
    DownPair p{TileUnits{a.tiles, a.tiles_cap, npb}, a.H, a.I, a.ring, a.perm, a.slots,
               a.out_f32, a.accumulate, a.status};
    return launch_pair(ma, mb, p, a.tiles_cap * npb, s);
}

// BF16 dgrad over tiles of <= PAIR_TILE_ROWS rows
cudaError_t launch_gemm_dgrad_pair_tc(const GemmDgradArgs &a, int E, int64_t rpad_cap,
                                      cudaStream_t s) {
    if (a.mxfp8) return cudaErrorInvalidValue;
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb;  // A: W13 as [E*2I][H] (MN-major over H); B: dA [rpad][2I]
    if ((e = make_map_bf16(&ma, a.w13, (int64_t)E * 2 * a.I, a.H, 64)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, a.dA, rpad_cap, 2 * a.I, KBOX_ROWS)) != cudaSuccess) return e;
    const int nmb = (a.H + 255) / 256;
    DgradPair p{TileUnits{a.tiles, a.tiles_cap, nmb}, a.H, a.I, a.offsets, a.poff, a.perm,
                a.dx_slots, a.out_f32, a.accumulate, a.status};
    return launch_pair(ma, mb, p, a.tiles_cap * nmb, s);
}

}  // namespace mok
