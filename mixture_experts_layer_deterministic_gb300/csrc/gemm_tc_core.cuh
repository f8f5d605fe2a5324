// gemm_tc_core.cuh -- the tensor-core GEMM engine shared by its translation units: tile
// constants and shared-memory layout, the forward problem policies, the persistent kernel
// template and the host-side tensor-map helpers. The engine itself is described in
// gemm_tc.cu; the forward through a partial ring instantiates the same kernel in
// ring_fwd.cu.
#pragma once

#include <cudaTypedefs.h>

#include <atomic>
#include <cstddef>

#include "common.cuh"
#include "mok_internal.h"
#include "tc.cuh"

namespace mok {
namespace {

constexpr int BK = 64;            // bf16 K elements per stage (128 bytes per row)
constexpr int BK_MX = 128;        // E4M3 K elements per stage (128 bytes per row)
constexpr int STAGES = 4;
constexpr int TILE_ROWS = 128;    // max N per unit (bf16)
constexpr int TILE_ROWS_MX = 112; // max N per unit (MXFP8: TMEM also holds the scales)
constexpr int KBOX_ROWS = 128;    // rows of the TMA box of a K-major B operand: a tile's rows
                                  // and whatever follows them (unused) or zero fill past the end
constexpr int A_BYTES = 128 * 128;                // 128 rows x 128 bytes
constexpr int B_BYTES = TILE_ROWS * 128;          // 128 rows x 128 bytes
constexpr int SF_BYTES = 2048;    // MXFP8 scale atoms per stage: A0, A1, B (512 B each), pad
constexpr int EPI_WARPS = 8;
constexpr int QD = 8;             // depth of the shared-memory queue of unit indices
constexpr int NTHREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL = 480;  // MXFP8: TMEM columns of the stage's scale atoms
// TMEM column of accumulator a (0: A0, 1: A1) of accumulator set b
template <bool MX>
__host__ __device__ constexpr uint32_t acc_col(int b, int a) {
    return (uint32_t)((2 * b + a) * (MX ? TILE_ROWS_MX : TILE_ROWS));
}
template <bool MX>
__host__ __device__ constexpr int stage_bytes() { return 2 * A_BYTES + B_BYTES + (MX ? SF_BYTES : 0); }


// per epilogue warp: one value per token column of the unit (a routing weight or a slot
// index), a transpose buffer for fixed-order reductions over the warp's 32 lanes, and a
// staging area that turns per-lane byte results into 16-byte stores
struct alignas(16) EpiScratch {
    float col[TILE_ROWS];
    float red[16][33];
    alignas(16) uint8_t stage[512];
};

struct Smem {
    uint4 clc_resp;          // Cluster Launch Control response (16-byte aligned)
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t qfull[QD];      // unit queue: the producer published slot j
    uint64_t qempty[QD];     // the MMA thread and every epilogue warp read slot j
    uint64_t clc_bar;        // a cancel response has landed
    int32_t q[QD];           // unit indices, -1 = no more work
    uint64_t tmem_full[2];   // accumulator set b holds a finished unit
    uint64_t tmem_empty[2];  // the epilogue has drained accumulator set b
    uint32_t tmem_base;
    int abort;
    EpiScratch epi[EPI_WARPS];
};

// the MXFP8 epilogues stage codes in EpiScratch with 16-byte accesses
static_assert(sizeof(EpiScratch) % 16 == 0 && offsetof(Smem, epi) % 16 == 0,
              "epilogue scratch alignment");
static_assert(STAGES * stage_bytes<true>() + 1024 + (int)sizeof(Smem) <= 232448,
              "MXFP8 kernels exceed the shared memory of a CTA");

template <bool MX>
__host__ __device__ constexpr int smem_bytes() {
    return STAGES * stage_bytes<MX>() + 1024 /*align*/ + (int)sizeof(Smem);
}

// How the producer fetches A0 and A1 (128 rows each) for one stage:
enum AMode {
    A_ROWS256 = 0,  // K-major, A1 directly below A0: one 256-row box at (k, ay0)
    A_PAIR5D = 1,   // K-major W13 gate/up blocks: one 5D box at (k, 0, ay0 = block, 0, ay1 = e)
    A_MN4 = 2,      // MN-major: four 64x64 boxes at (ax0, ay0 + k), (ax0 + 64, ..), (ax1, ..)
};

// One work unit as the producer and the MMA issuer see it.
struct Geom {
    int32_t ax0, ay0, ax1, ay1;  // A0 and A1 coordinates (x innermost), per the policy's AMode
    int32_t bx, by;              // first box of B
    int n_mma;                   // N of each MMA (multiple of 16, <= 256)
    int nbox;                    // B boxes per stage (MN-major B only)
    int k_steps;                 // K steps of one MMA (16 bf16 or 32 E4M3 elements); 0 leaves
                                 // the accumulators unwritten
    int64_t sfa0, sfa1, sfb;     // MXFP8: byte offsets of the first stage's scale atoms
};

MOK_DEV float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Saved pre-activations of a row: [I] pairs (gate, up) of one feature each, so that the lane
// holding feature i stores and loads both halves with one access (a bf16 pair is one 32-bit
// word, an fp32 pair one 64-bit word) and a warp's 32 consecutive features are one run.

// element i of a stored-value array held as fp32 (f32) or bf16
MOK_DEV void st_val(void *p, int64_t i, float v, bool f32) {
    if (f32)
        static_cast<float *>(p)[i] = v;
    else
        static_cast<uint16_t *>(p)[i] = f32_to_bf16(v);
}
// the values an accumulating epilogue adds to: rows fcol[n0 + j] (j < 16, rows past nr read
// as 0), columns c and c + 128 (the latter when has1), all loads issued before any is used
template <bool F32>
MOK_DEV void load_rows16(const void *p, const int *fcol, int n0, int nr, int H, int c,
                         bool has1, float (&a0)[16], float (&a1)[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const bool ok = n0 + j < nr;
        const int64_t o = (int64_t)fcol[ok ? n0 + j : 0] * H + c;
        if (F32) {
            const float *pf = static_cast<const float *>(p);
            a0[j] = ok ? pf[o] : 0.f;
            a1[j] = ok && has1 ? pf[o + 128] : 0.f;
        } else {
            const uint16_t *pb = static_cast<const uint16_t *>(p);
            a0[j] = ok ? bf16_to_f32(pb[o]) : 0.f;
            a1[j] = ok && has1 ? bf16_to_f32(pb[o + 128]) : 0.f;
        }
    }
}

// bounded wait; gives up when another role has aborted or after the wall-time limit
MOK_DEV bool wait_or_abort(uint64_t *bar, uint32_t parity, int *status, volatile int *abort) {
    return tc::wait_bounded(bar, parity, status, abort, tc::WAIT_LIMIT_NS);
}

// ---------------------------------------------------------------- problem policies

// tile-based problems: units = tiles x weight blocks, tile = (e, r0, r1)
struct TileUnits {
    const int32_t *tiles;
    int64_t cap;
    int n_mblocks;
    MOK_DEV int64_t count() const {
        const int64_t n = tiles[-4] < cap ? tiles[-4] : cap;
        return n * n_mblocks;
    }
    MOK_DEV void get(int64_t u, int *e, int64_t *r0, int64_t *r1, int *mb) const {
        const int64_t t = u / n_mblocks;
        *mb = (int)(u % n_mblocks);
        *e = tiles[4 * t + 0];
        *r0 = tiles[4 * t + 1];
        *r1 = tiles[4 * t + 2];
    }
};

// MXFP8 scale atoms: 128 rows x 4 blocks of 32 K elements as 32 rows of 16 bytes, row i
// holding rows i, i+32, i+64, i+96 (4 bytes each, one per block). Weights: atom
// (row/128, k/128) at ((row/128) * K/128 + k/128) * 512; token tiles: one atom per
// 128-wide K block at (tile * K/128 + k/128) * 512.
// ATOMS: MXFP8 h's scales are also written as the down GEMM's scale atoms (hs_atoms)
template <bool MXv, bool ATOMS = false>
struct FwdUpT {
    static constexpr bool A_MN = false, B_MN = false, MX = MXv;
    static constexpr int A_MODE = A_PAIR5D;
    static constexpr bool CLC = true;
    static constexpr bool FUSED = false;  // the engine's own producer
    TileUnits tu;
    int H, I;
    Ring ring;
    void *hring;
    uint8_t *hring_s;
    void *preact;        // [R][2I] pre-activations (fp32 if preact_f32, else bf16), or nullptr
    bool preact_f32;
    bool mxfp8;
    int *status;
    const uint8_t *sf_a, *sf_b;
    // backward recompute: B rows in the padded expert layout, no h output (else nullptr)
    const int32_t *offsets_b, *poff_b;
    // ATOMS: h's scales also as the down GEMM's scale atoms, one per tile of the list and
    // 128-feature block
    uint8_t *hs_atoms = nullptr;

    MOK_DEV int64_t n_units() const { return tu.count(); }
    MOK_DEV Geom geom(int64_t u) const {
        int e, mb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &mb);
        return geom_of(u / tu.n_mblocks, e, r0, r1, mb);
    }
    // the unit of tile t = (e, r0, r1) and weight block mb
    MOK_DEV Geom geom_of(int64_t t, int e, int64_t r0, int64_t r1, int mb) const {
        const RingMap rm{ring.R, ring.MB, ring.n_slots};
        Geom g;
        g.ax0 = 0;
        g.ay0 = mb;
        g.ax1 = 0;
        g.ay1 = e;
        g.bx = 0;
        g.by = poff_b != nullptr ? (int32_t)(poff_b[e] + (r0 - offsets_b[e])) : (int32_t)rm(r0);
        g.n_mma = (int)((r1 - r0 + 15) & ~15);
        g.nbox = 1;
        g.k_steps = MX ? H / 32 : H / 16;
        const int64_t kg = H / 128;
        const int64_t gate_row = (int64_t)e * 2 * I + mb * 128;
        g.sfa0 = (gate_row / 128) * kg * 512;
        g.sfa1 = ((gate_row + I) / 128) * kg * 512;
        g.sfb = t * kg * 512;
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
        // a tile never straddles a lap of the ring: its rows are consecutive ring rows
        const int64_t hrow0 = RingMap{ring.R, ring.MB, ring.n_slots}(r0);
        const int i = mb * 128 + q * 32 + lane;  // gate feature; its up feature is I + i
        for (int n0 = 16 * half; n0 < n_mma; n0 += 32) {
            float d0[16], d1[16];
            ld(n0, d0, d1);
            float h[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int n = n0 + j;
                const int64_t r = r0 + n;
                h[j] = silu_f(d0[j]) * d1[j];
                if (n < nr && preact != nullptr) {
                    if (preact_f32)
                        static_cast<float2 *>(preact)[r * I + i] = make_float2(d0[j], d1[j]);
                    else
                        static_cast<uint32_t *>(preact)[r * I + i] = pack_bf16x2(d0[j], d1[j]);
                }
                if (hring != nullptr && !mxfp8 && n < nr)
                    ((uint16_t *)hring)[(hrow0 + n) * I + i] = f32_to_bf16(h[j]);
            }
            if (hring == nullptr || !mxfp8) continue;
            // MXFP8: the warp's 32 lanes hold one 32-feature block of each of the chunk's 16
            // rows. A block's maximum magnitude comes from one integer reduction (the bit
            // patterns of non-negative floats order like the floats); two rows share one
            // conversion. The codes are staged in the warp's scratch as 16 rows x 32 bytes
            // and written back one 16-byte piece per lane, the scales by lanes 0-15.
            uint8_t *stage = reinterpret_cast<uint8_t *>(es.col);
            uint32_t my_sb = 0;
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const float a0 = __uint_as_float(
                    __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(h[j]))));
                const float a1 = __uint_as_float(
                    __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(h[j + 1]))));
                const uint32_t sb0 = mx_scale_byte(a0), sb1 = mx_scale_byte(a1);
                const uint32_t c2 = e4m3x2(h[j] * mx_inv_scale(sb0), h[j + 1] * mx_inv_scale(sb1));
                stage[j * 32 + lane] = (uint8_t)(c2 & 0xFFu);
                stage[(j + 1) * 32 + lane] = (uint8_t)(c2 >> 8);
                if (lane == j) my_sb = sb0;
                if (lane == j + 1) my_sb = sb1;
            }
            __syncwarp();
            if (lane < 16 && n0 + lane < nr) {
                hring_s[(hrow0 + n0 + lane) * (I / 32) + (mb * 128 + q * 32) / 32] =
                    (uint8_t)my_sb;
                if (ATOMS) {
                    const int n = n0 + lane;
                    hs_atoms[((u / tu.n_mblocks) * (I / 128) + mb) * 512 + (n & 31) * 16 +
                             (n >> 5) * 4 + q] = (uint8_t)my_sb;
                }
            }
            const int jr = lane >> 1, hb = lane & 1;
            if (n0 + jr < nr) {
                const uint4 v = *reinterpret_cast<const uint4 *>(stage + jr * 32 + hb * 16);
                *reinterpret_cast<uint4 *>((uint8_t *)hring + (hrow0 + n0 + jr) * I +
                                           mb * 128 + q * 32 + hb * 16) = v;
            }
            __syncwarp();
        }
    }
};

template <bool MXv>
struct FwdDownT {
    static constexpr bool A_MN = false, B_MN = false, MX = MXv;
    static constexpr int A_MODE = A_ROWS256;
    static constexpr bool CLC = true;
    static constexpr bool FUSED = false;  // the engine's own producer
    TileUnits tu;
    int H, I;
    Ring ring;
    const int32_t *perm;  // output row of each sorted row (nullptr: the row itself)
    void *slots;          // [rows][H], fp32 if out_f32, else bf16
    bool out_f32;
    int *status;
    const uint8_t *sf_a, *sf_b;
    bool accumulate;      // add into the output (the shared expert adds into y)

    MOK_DEV int64_t n_units() const { return tu.count(); }
    MOK_DEV Geom geom(int64_t u) const {
        int e, mb;
        int64_t r0, r1;
        tu.get(u, &e, &r0, &r1, &mb);
        return geom_of(u / tu.n_mblocks, e, r0, r1, mb);
    }
    // the unit of tile t = (e, r0, r1) and weight block mb
    MOK_DEV Geom geom_of(int64_t t, int e, int64_t r0, int64_t r1, int mb) const {
        const RingMap rm{ring.R, ring.MB, ring.n_slots};
        Geom g;
        g.ax0 = 0;
        g.ay0 = e * H + mb * 256;
        g.ax1 = 0;
        g.ay1 = g.ay0 + 128;
        g.bx = 0;
        g.by = (int32_t)rm(r0);
        g.n_mma = (int)((r1 - r0 + 15) & ~15);
        g.nbox = 1;
        g.k_steps = MX ? I / 32 : I / 16;
        const int64_t kg = I / 128;
        g.sfa0 = (int64_t)(g.ay0 / 128) * kg * 512;
        // when H is not a multiple of 256 the last block's A1 lies past this expert (its
        // results are discarded); keep its scale reads inside the expert
        g.sfa1 = mb * 256 + 128 < H ? (int64_t)(g.ay1 / 128) * kg * 512 : g.sfa0;
        g.sfb = t * kg * 512;
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
        for (int n = lane; n < nr; n += 32)
            fcol[n] = perm != nullptr ? perm[r0 + n] : (int)(r0 + n);
        __syncwarp();
        const bool has1 = c + 128 < H;
        for (int n0 = 16 * half; n0 < n_mma; n0 += 32) {
            float d0[16], d1[16];
            ld(n0, d0, d1);
            if (accumulate) {
                // every load of the chunk before any store: a store to one row may alias
                // the next row's load, which would otherwise serialise the round trips
                float a0[16], a1[16];
                if (out_f32)
                    load_rows16<true>(slots, fcol, n0, nr, H, c, has1, a0, a1);
                else
                    load_rows16<false>(slots, fcol, n0, nr, H, c, has1, a0, a1);
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
                    const int64_t o = (int64_t)fcol[n] * H + c;
                    st_val(slots, o, d0[j], out_f32);
                    if (has1) st_val(slots, o + 128, d1[j], out_f32);
                }
            }
        }
        __syncwarp();
    }
};

// ---------------------------------------------------------------- the kernel
// The kernel body. tmA / tmB: the A and B operand maps of the policy's own producer; a
// policy with its own producer (P::FUSED) gets all four maps.
template <class P>
MOK_DEV void gemm_body(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                       const CUtensorMap &tmD, const P &p, const int use_clc) {
    constexpr bool MX = P::MX;
    constexpr int SB = stage_bytes<MX>();
    constexpr int BKE = MX ? BK_MX : BK;             // K elements per stage
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Smem *sm = (Smem *)(base + STAGES * SB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_units = p.n_units();
    const bool clc = P::CLC && use_clc != 0;  // else static striding, one CTA per SM
    if ((int64_t)blockIdx.x >= n_units) return;  // uniform across the CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&sm->full[s], 1);
            tc::mbar_init(&sm->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sm->tmem_full[b], 1);
            tc::mbar_init(&sm->tmem_empty[b], 32 * EPI_WARPS);
        }
        for (int j = 0; j < QD; ++j) {
            tc::mbar_init(&sm->qfull[j], 1);
            tc::mbar_init(&sm->qempty[j], 1 + EPI_WARPS);
        }
        tc::mbar_init(&sm->clc_bar, 1);
        sm->abort = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tmA);
        tc::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tc::tmem_alloc(&sm->tmem_base, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    volatile int *abort = &sm->abort;
    constexpr int A_HALF = A_BYTES / 2;                        // one 64-wide MN-major box
    constexpr int B_BOX = P::B_MN ? 64 * 128 : KBOX_ROWS * 128;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if constexpr (P::FUSED) {
            // a policy with its own producer (the whole warp; see ring_fwd.cu)
            p.produce(sm, base, lane, &tmA, &tmB, &tmC, &tmD);
        } else if (tc::elect_one()) {
            int s = 0;
            uint32_t ph = 0, clc_ph = 0;
            int64_t issued = 0, j = 0;
            bool clc_live = true, clc_pending = false;
            int64_t u = blockIdx.x;
            for (;;) {
                // publish the unit (or the end marker) to the MMA thread and the epilogue
                const int slot = (int)(j % QD);
                if (!wait_or_abort(&sm->qempty[slot], (uint32_t)(((j / QD) & 1) ^ 1), p.status,
                                   abort))
                    break;
                *(volatile int32_t *)&sm->q[slot] = (int32_t)u;
                tc::mbar_arrive(&sm->qfull[slot]);
                ++j;
                if (u < 0) break;
                const Geom g = p.geom(u);
                const int kblocks = (g.k_steps + 3) / 4;
                // ask for the next unit while the last two stages of this one are issued:
                // asking later keeps units that share operand tiles (consecutive indices)
                // starting together on whichever CTAs free up, so L2 serves their re-reads
                const int ask_at = kblocks > 2 ? kblocks - 2 : 0;
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (clc && kb == ask_at && clc_live) {
                        tc::mbar_arrive_expect_tx(&sm->clc_bar, 16);
                        tc::clc_try_cancel(&sm->clc_resp, &sm->clc_bar);
                        clc_pending = true;
                    }
                    if (!wait_or_abort(&sm->empty[s], ph ^ 1u, p.status, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = base + s * SB;
                    uint64_t *fb = &sm->full[s];
                    tc::mbar_arrive_expect_tx(fb, 2 * A_BYTES +
                                                      (P::B_MN ? g.nbox * B_BOX : B_BYTES) +
                                                      (MX ? 1536 : 0));
                    const int k0 = kb * BKE;
                    if (MX) {
                        uint8_t *sf = st + 2 * A_BYTES + B_BYTES;
                        tc::bulk_load(sf, p.sf_a + g.sfa0 + kb * 512, 512, fb);
                        tc::bulk_load(sf + 512, p.sf_a + g.sfa1 + kb * 512, 512, fb);
                        tc::bulk_load(sf + 1024, p.sf_b + g.sfb + kb * 512, 512, fb);
                    }
                    if (P::A_MODE == A_MN4) {
                        tc::tma_load_2d(st, &tmA, fb, g.ax0, g.ay0 + k0);
                        tc::tma_load_2d(st + A_HALF, &tmA, fb, g.ax0 + 64, g.ay0 + k0);
                        tc::tma_load_2d(st + A_BYTES, &tmA, fb, g.ax1, g.ay1 + k0);
                        tc::tma_load_2d(st + A_BYTES + A_HALF, &tmA, fb, g.ax1 + 64, g.ay1 + k0);
                    } else if (P::A_MODE == A_PAIR5D) {
                        tc::tma_load_5d(st, &tmA, fb, k0, 0, g.ay0, 0, g.ay1);
                    } else {
                        tc::tma_load_2d(st, &tmA, fb, k0, g.ay0);
                    }
                    uint8_t *bt = st + 2 * A_BYTES;
                    if (P::B_MN) {
                        for (int j = 0; j < g.nbox; ++j)
                            tc::tma_load_2d(bt + j * B_BOX, &tmB, fb, g.bx + 64 * j, g.by + k0);
                    } else {
                        tc::tma_load_2d(bt, &tmB, fb, k0, g.by);
                    }
                    ++issued;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                int64_t next = -1;
                if (!clc) {
                    next = u + (int64_t)gridDim.x < n_units ? u + (int64_t)gridDim.x : -1;
                } else if (clc_pending) {
                    if (!wait_or_abort(&sm->clc_bar, clc_ph, p.status, abort)) break;
                    clc_ph ^= 1u;
                    clc_pending = false;
                    uint32_t x;
                    // after a failed or out-of-range answer no further request is made
                    if (tc::clc_query(&sm->clc_resp, &x) && (int64_t)x < n_units)
                        next = x;
                    else
                        clc_live = false;
                }
                u = next;
            }
            // do not leave while a cancel response may still be landing
            if (clc_pending) {
                const uint64_t t0 = tc::globaltimer();
                while (!tc::mbar_try_wait(&sm->clc_bar, clc_ph) &&
                       tc::globaltimer() - t0 < 100000000ull) {
                }
            }
            // do not leave while copies this CTA issued may still be landing
            for (int q = 0; q < STAGES && q < issued; ++q) {
                if (--s < 0) {
                    s = STAGES - 1;
                    ph ^= 1u;
                }
                const uint64_t t0 = tc::globaltimer();
                while (!tc::mbar_try_wait(&sm->full[s], ph) &&
                       tc::globaltimer() - t0 < 100000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (tc::elect_one()) {
            int s = 0;
            uint32_t ph = 0;
            int64_t i = 0;  // units of this CTA so far (queue entries)
            int64_t a = 0;  // of them, units with accumulators: unit a uses set a % 2
            for (;; ++i) {
                const int slot = (int)(i % QD);
                if (!wait_or_abort(&sm->qfull[slot], (uint32_t)((i / QD) & 1), p.status, abort))
                    break;
                const int64_t u = *(volatile int32_t *)&sm->q[slot];
                tc::mbar_arrive(&sm->qempty[slot]);
                if (u < 0) break;
                if constexpr (P::FUSED) {
                    // a unit that only copies through the stages: the policy drains them
                    if (p.is_copy(u)) {
                        if (!p.copy_out(u, base, sm->full, sm->empty, s, ph, abort)) break;
                        continue;
                    }
                }
                const Geom g = p.geom(u);
                const uint32_t idesc = tc::idesc_bf16(128, g.n_mma, P::A_MN, P::B_MN);
                const uint32_t idesc_mx = tc::idesc_mxf8(128, g.n_mma, 0);
                const int ab = (int)(a & 1);
                const uint32_t use = (uint32_t)((a >> 1) & 1);
                if (!wait_or_abort(&sm->tmem_empty[ab], use ^ 1u, p.status, abort)) break;
                tc::tc_fence_after();
                const uint32_t d0 = tmem + acc_col<MX>(ab, 0), d1 = tmem + acc_col<MX>(ab, 1);
                const int kblocks = (g.k_steps + 3) / 4;
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_or_abort(&sm->full[s], ph, p.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(base + s * SB);
                    const uint32_t a1 = a0 + A_BYTES;
                    const uint32_t b = a0 + 2 * A_BYTES;
                    const int steps = g.k_steps - kb * 4 < 4 ? g.k_steps - kb * 4 : 4;
                    if (MX) {
                        // this stage's scale atoms into TMEM: A0, A1, B
                        const uint32_t sf = b + B_BYTES;
                        tc::tmem_cp_32x128b_x4(tmem + SF_COL + 0, tc::sdesc_plain_rows16(sf));
                        tc::tmem_cp_32x128b_x4(tmem + SF_COL + 4, tc::sdesc_plain_rows16(sf + 512));
                        tc::tmem_cp_32x128b_x4(tmem + SF_COL + 8, tc::sdesc_plain_rows16(sf + 1024));
                    }
                    for (int kk = 0; kk < steps; ++kk) {
                        // K-major: 16 elements = 32 bytes along the swizzled row;
                        // MN-major: 16 K rows = 2 groups of eight 128-byte rows
                        const uint32_t ao = P::A_MN ? kk * 2048 : kk * 32;
                        const uint32_t bo = P::B_MN ? kk * 2048 : kk * 32;
                        const uint32_t albo = P::A_MN ? A_HALF : 16;
                        const uint32_t blbo = P::B_MN ? B_BOX : 16;
                        const uint64_t da0 = tc::sdesc_sw128(a0 + ao, albo, 1024);
                        const uint64_t da1 = tc::sdesc_sw128(a1 + ao, albo, 1024);
                        const uint64_t db = tc::sdesc_sw128(b + bo, blbo, 1024);
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        if (MX) {
                            // byte kk of each 32-bit scale word is this K=32 block's scale
                            const uint32_t id = idesc_mx | ((uint32_t)kk << 4) |
                                                ((uint32_t)kk << 29);
                            tc::mma_mxf8(d0, da0, db, id, tmem + SF_COL + 0, tmem + SF_COL + 8,
                                         acc);
                            tc::mma_mxf8(d1, da1, db, id, tmem + SF_COL + 4, tmem + SF_COL + 8,
                                         acc);
                        } else {
                            tc::mma_f16(d0, da0, db, idesc, acc);
                            tc::mma_f16(d1, da1, db, idesc, acc);
                        }
                    }
                    tc::mma_commit(&sm->empty[s]);  // frees the stage once these MMAs finish
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                tc::mma_commit(&sm->tmem_full[ab]);
                ++a;
            }
            // on an abort, do not free TMEM under MMAs still in flight: the last commit
            // completes once every earlier MMA of this thread has (bounded wait)
            if (a > 0) {
                const int lb = (int)((a - 1) & 1);
                const uint32_t lu = (uint32_t)(((a - 1) >> 1) & 1);
                const uint64_t t0 = tc::globaltimer();
                while (!tc::mbar_try_wait(&sm->tmem_full[lb], lu) &&
                       tc::globaltimer() - t0 < 100000000ull) {
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int half = (warp - 2) >> 2;  // which alternate 16-column chunks it takes
        EpiScratch &es = sm->epi[warp - 2];
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        uint32_t c0 = 0, c1 = 0;  // accumulator columns of the current unit
        auto ld = [&](int n0, float (&d0)[16], float (&d1)[16]) {
            tc::tmem_ld16(tmem + lane_base + c0 + n0, d0);
            tc::tmem_ld16(tmem + lane_base + c1 + n0, d1);
            tc::tmem_ld_wait();
        };
        int64_t a = 0;  // units with accumulators so far
        for (int64_t i = 0;; ++i) {
            const int slot = (int)(i % QD);
            if (!wait_or_abort(&sm->qfull[slot], (uint32_t)((i / QD) & 1), p.status, abort))
                break;
            const int64_t u = *(volatile int32_t *)&sm->q[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sm->qempty[slot]);
            if (u < 0) break;
            if constexpr (P::FUSED) {
                if (p.is_copy(u)) continue;
            }
            const int ab = (int)(a & 1);
            if (!wait_or_abort(&sm->tmem_full[ab], (uint32_t)((a >> 1) & 1), p.status, abort))
                break;
            tc::tc_fence_after();
            c0 = acc_col<MX>(ab, 0);
            c1 = acc_col<MX>(ab, 1);
            p.epilogue(u, ld, es, q, half, lane);
            tc::tc_fence_before();
            tc::mbar_arrive(&sm->tmem_empty[ab]);
            ++a;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <class P>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const P p, const int use_clc) {
    gemm_body<P>(tmA, tmB, tmA, tmB, p, use_clc);
}

// ---------------------------------------------------------------- host side
// the driver's tensor-map encoder: one process-wide entry point, looked up once
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};

cudaError_t init_host() {
    if (g_encode.load(std::memory_order_acquire) == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return cudaErrorNotSupported;
        g_encode.store((PFN_cuTensorMapEncodeTiled_v12000)fn, std::memory_order_release);
    }
    return cudaSuccess;
}

CUresult encode(CUtensorMap *m, CUtensorMapDataType t, cuuint32_t rank, void *ptr,
                const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                const cuuint32_t *estr) {
    return g_encode.load(std::memory_order_acquire)(
        m, t, rank, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// row-major bf16 matrix [rows][cols] -> 2D map of 64-column x box_rows boxes with
// 128-byte swizzle
cudaError_t make_map_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols,
                          int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                        strides, box, estr);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// row-major byte matrix [rows][cols] (E4M3) -> 2D map of 128-byte x box_rows boxes with
// 128-byte swizzle
cudaError_t make_map_u8(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols,
                        int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {(cuuint32_t)BK_MX, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims,
                        strides, box, estr);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// W13 [E][2I][H] (bf16, or E4M3 bytes when mx) viewed as 5D [E][2][I/128][128][H] (gate
// rows, then up rows): one box of {one 128-byte K block, 128 rows, 1 block, 2 halves, 1
// expert} puts the gate block and its up block one after the other in shared memory.
cudaError_t make_map_w13_pairs(CUtensorMap *m, const void *ptr, int64_t E, int64_t I,
                               int64_t H, bool mx) {
    const int64_t es = mx ? 1 : 2;
    cuuint64_t dims[5] = {(cuuint64_t)H, 128, (cuuint64_t)(I / 128), 2, (cuuint64_t)E};
    cuuint64_t strides[4] = {(cuuint64_t)(H * es), (cuuint64_t)(128 * H * es),
                             (cuuint64_t)(I * H * es), (cuuint64_t)(2 * I * H * es)};
    cuuint32_t box[5] = {(cuuint32_t)(mx ? BK_MX : BK), 128, 1, 2, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = encode(m, mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        5, const_cast<void *>(ptr), dims, strides, box, estr);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// units_cap: the host-side bound on the units (the grid under Cluster Launch Control);
// units_min: a lower bound on the units there will be. CTAs past the device-side count
// return at once, but each still costs a launch; when the bound is loose (more than twice
// the minimum, e.g. a ring pass that touches few experts) the launch strides statically
// over one CTA per SM instead.
template <class P>
cudaError_t launch(const CUtensorMap &ma, const CUtensorMap &mb, const P &p, int64_t units_cap,
                   int64_t units_min, cudaStream_t s) {
    constexpr int SMEM = smem_bytes<P::MX>();
    // the shared-memory opt-in is a per-device function attribute: set once per device
    static std::atomic<uint64_t> attr_set[2] = {{0}, {0}};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << (dev & 63);
    if ((attr_set[dev >> 6].load(std::memory_order_acquire) & bit) == 0) {
        e = cudaFuncSetAttribute(tc_gemm_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev >> 6].fetch_or(bit, std::memory_order_acq_rel);
    }
    // Cluster Launch Control: one CTA per unit, running CTAs take over the units of CTAs
    // not yet launched; static striding: one CTA per SM
    if (units_cap < 1) return cudaSuccess;
    if (units_cap > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const bool clc = P::CLC && units_cap <= 2 * units_min;
    const int n_sms = device_sm_count();
    const int grid = clc || units_cap < n_sms ? (int)units_cap : n_sms;
    tc_gemm_kernel<P><<<grid, NTHREADS, SMEM, s>>>(ma, mb, p, clc ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace
}  // namespace mok
