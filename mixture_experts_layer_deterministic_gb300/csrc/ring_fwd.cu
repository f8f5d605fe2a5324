// ring_fwd.cu -- the forward through a partial ring (capacity C below the routed rows R) as
// one persistent launch of the tensor-core GEMM engine.
//
// [arex] "Cursor 放出 MoK" (arex-research.com), section "pull 代替 push", point 2: tokens
// cycle through a fixed ring buffer that is refilled as work completes, never drops a token
// and needs no CPU synchronisation. [alphalab] "Mixture-of-Kittens" (alphalab.site),
// sections 一 and 二: one deterministic megakernel runs the pull dispatch, the expert FFN
// and the push back.
//
// Work. The sorted rows are cut into tiles (expert e, rows [r0, r1)) at expert boundaries,
// at multiples of C (so that a tile's ring rows r mod C are contiguous) and at `chunk` rows.
// Each tile has three groups of units:
//   one gather unit: the x rows of the tile's tokens (bf16, or MXFP8 codes of x quantized
//     once per token) into x ring rows r mod C, whole rows through the shared-memory stages
//     by bulk copies (the pull dispatch);
//   gate/up units, one per 128 features of I: A = the W13 gate/up block pair, B = the tile's
//     x ring rows; epilogue SwiGLU, h into h ring rows r mod C (MXFP8: quantized, its
//     scales also written as the down GEMM's scale atoms);
//   down units, one per 256 features of H: A = W2 rows, B = the tile's h ring rows;
//     epilogue push to the (token, k) slots.
// Order. Units are claimed one at a time from a device counter, in an order built on the
// device: groups keyed in half rows, gather 2 r0 - g, gate/up 2 r0, down 2 r0 + d, merged
// with gather before gate/up before down on equal keys. Gate/up units read the x rows of
// their own tile's gather (an earlier key for g >= 1); down units read the h rows of their
// own tile's gate/up units (an earlier key for d >= 1). A gather overwrites x ring rows last
// read by the gate/up units of the tiles one lap back (rows r - C), and gate/up units
// overwrite h ring rows last read by the down units one lap back: those keys are at most
// 2 (r1 - C - 1) + d (resp. 2 (r1 - C - 1)), below the overwriting unit's key when g, d <=
// 2 (C - chunk) + 1. So a unit only ever waits on units claimed before it, every claimed
// unit belongs to a running CTA, and the launch cannot deadlock.
// Waits. Only the producer warp waits, before it loads a unit's operands, on per-tile
// counters raised after the stores they cover: by the epilogue warps (a release per warp,
// with a proxy fence for the TMA reads of h) and, for a gather, by the MMA thread once its
// bulk stores are complete. The spin is bounded at 2 s; on a timeout it records
// MOK_ERR_TIMEOUT in the status word, and every CTA gives up at its next wait once the
// status word shows a problem.
// Every output element is the same fixed-order dot product as in the forward through a ring
// that holds every row, so y is bitwise equal to that forward's.
#include "gemm_tc_core.cuh"

namespace mok {
namespace {

constexpr int KIND_UP = 0, KIND_DOWN = 1, KIND_GATHER = 2;
constexpr int REC_AHEAD = 64;  // unit records a producer asks L2 for ahead of its claim

// One claimable unit, all the producer needs to start it with one 32-byte read: its tile,
// kind and weight block (code = kind << 16 | block), the tile's expert and rows, and the
// tiles one lap back over the tile's ring rows (dep_lo > dep_hi: none).
struct alignas(16) UnitRec {
    int32_t t, code, e, r0;
    int32_t r1, dep_lo, dep_hi, pad;
};

template <bool MXv>
struct RingFwdT {
    static constexpr bool A_MN = false, B_MN = false, MX = MXv;
    static constexpr bool CLC = false;
    static constexpr bool FUSED = true;
    FwdUpT<MXv, true> up;     // over the flat tile list; hring = the ring, RingMap{R, C, 1}
    FwdDownT<MXv> dn;
    const UnitRec *units;  // the unit of each claim index
    int32_t *hdr;       // [0] units, [1] next claim index
    int32_t *done_up;   // per tile: epilogue warps that finished one of its gate/up units
    int32_t *done_dn;   // likewise for its down units
    int32_t *done_g;    // per tile: its gather's bulk stores are complete
    const int32_t *perm;  // flat id t*K + k of each sorted row
    int K;
    int *status;
    const uint8_t *x;   // x rows (bf16, or MXFP8 codes), row_bytes each
    uint8_t *xring;     // [C] rows of row_bytes
    int64_t C;
    int row_bytes;
    int rows_per_stage; // x rows a stage holds in a gather (<= 32)
    int gather_pieces;  // gather units per tile, of gather_rows rows each (the last ones of
    int gather_rows;    // a short tile may be empty)

    MOK_DEV int64_t n_units() const { return hdr[0]; }
    MOK_DEV bool is_copy(int64_t u) const { return (units[u].code >> 16) == KIND_GATHER; }
    MOK_DEV Geom geom(int64_t u) const { return geom_rec(units[u]); }
    MOK_DEV Geom geom_rec(const UnitRec &r) const {
        const int mb = r.code & 0xFFFF;
        if ((r.code >> 16) == KIND_DOWN) return dn.geom_of(r.t, r.e, r.r0, r.r1, mb);
        return up.geom_of(r.t, r.e, r.r0, r.r1, mb);
    }
    template <class LD>
    MOK_DEV void epilogue(int64_t u, const LD &ld, EpiScratch &es, int q, int half,
                          int lane) const {
        const int4 a = *reinterpret_cast<const int4 *>(&units[u]);  // t, code
        const int mb = a.y & 0xFFFF;
        const bool down = (a.y >> 16) == KIND_DOWN;
        if (down)
            dn.epilogue((int64_t)a.x * dn.tu.n_mblocks + mb, ld, es, q, half, lane);
        else
            up.epilogue((int64_t)a.x * up.tu.n_mblocks + mb, ld, es, q, half, lane);
        // publish this warp's stores to the units that wait on them
        tc::fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            atomicAdd(down ? &done_dn[a.x] : &done_up[a.x], 1);
        }
    }

    // the next claim index, or -1 once every unit is taken
    MOK_DEV int32_t claim() const {
        const int32_t v = atomicAdd(&hdr[1], 1);
        return v < hdr[0] ? v : -1;
    }
    // bounded spin on a per-tile counter (gives up after 2 s, or once any CTA has)
    MOK_DEV bool wait_count(const int32_t *ctr, int32_t target, volatile int *abort) const {
        return tc::wait_count_bounded(ctr, target, status, abort, tc::WAIT_LIMIT_NS);
    }
    MOK_DEV UnitRec load_rec(int32_t u) const {
        const int4 *p = reinterpret_cast<const int4 *>(&units[u]);
        const int4 a = p[0], b = p[1];
        return UnitRec{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    }
    // the units a claimed unit depends on have finished (see the order above)
    MOK_DEV bool wait_inputs(const UnitRec &r, volatile int *abort) const {
        const int kind = r.code >> 16;
        bool ok = true;
        if (kind == KIND_DOWN) {
            ok = wait_count(&done_up[r.t], up.tu.n_mblocks * EPI_WARPS, abort);
        } else {
            // both rings: the same rows one lap back
            if (kind == KIND_UP) ok = wait_count(&done_g[r.t], gather_pieces, abort);
            const int32_t *ctr = kind == KIND_UP ? done_dn : done_up;
            const int32_t target =
                (kind == KIND_UP ? dn.tu.n_mblocks : up.tu.n_mblocks) * EPI_WARPS;
            for (int t = r.dep_lo; ok && t <= r.dep_hi; ++t)
                ok = wait_count(&ctr[t], target, abort);
        }
        tc::fence_proxy_async_global();  // the TMA reads that follow see those stores
        return ok;
    }

    // the sorted rows [*q0, *q1) a gather unit copies: piece `block` of its tile's rows
    MOK_DEV void gather_span(const UnitRec &r, int64_t *q0, int64_t *q1) const {
        const int64_t a = r.r0 + (int64_t)(r.code & 0xFFFF) * gather_rows;
        *q0 = a < r.r1 ? a : r.r1;
        *q1 = a + gather_rows < r.r1 ? a + gather_rows : r.r1;
        if (*q1 < *q0) *q1 = *q0;
    }
    // The MMA thread's side of a gather: per stage, the rows that landed go back out to
    // their x ring rows. A stage is freed once its stores have read it, one stage behind (the
    // stores of two stages in flight), and the tile's counter raised once every store is
    // complete.
    MOK_DEV bool copy_out(int64_t u, uint8_t *base, uint64_t *full, uint64_t *empty, int &s,
                          uint32_t &ph, volatile int *abort) const {
        constexpr int SB = stage_bytes<MX>();
        const UnitRec r = load_rec((int32_t)u);
        const int64_t t = r.t;
        int64_t r0, r1;
        gather_span(r, &r0, &r1);
        int prev = -1;  // the stage of the newest committed stores but one
        for (int64_t q0 = r0; q0 < r1; q0 += rows_per_stage) {
            if (!wait_or_abort(&full[s], ph, status, abort)) {
                tc::bulk_wait<0>();
                return false;
            }
            const int m = (int)(r1 - q0 < rows_per_stage ? r1 - q0 : rows_per_stage);
            const uint8_t *st = base + s * SB;
            const int64_t x0 = q0 % C;  // a tile stays within a lap: consecutive ring rows
            for (int i = 0; i < m; ++i)
                tc::bulk_store(xring + (x0 + i) * row_bytes, st + i * row_bytes,
                               (uint32_t)row_bytes);
            tc::bulk_commit();
            if (prev >= 0) {
                tc::bulk_wait_read<1>();
                tc::mbar_arrive(&empty[prev]);
            }
            prev = s;
            if (++s == STAGES) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (prev >= 0) {
            tc::bulk_wait_read<0>();
            tc::mbar_arrive(&empty[prev]);
        }
        tc::bulk_wait<0>();
        tc::fence_proxy_async_global();
        __threadfence();
        atomicAdd(&done_g[t], 1);
        return true;
    }

    MOK_DEV static UnitRec shfl_rec(const UnitRec &r) {
        constexpr uint32_t FULL = 0xFFFFFFFFu;
        return UnitRec{__shfl_sync(FULL, r.t, 0),      __shfl_sync(FULL, r.code, 0),
                       __shfl_sync(FULL, r.e, 0),      __shfl_sync(FULL, r.r0, 0),
                       __shfl_sync(FULL, r.r1, 0),     __shfl_sync(FULL, r.dep_lo, 0),
                       __shfl_sync(FULL, r.dep_hi, 0), 0};
    }

    // The producer, run by the whole warp: lane 0 claims, waits and issues the boxes of a
    // GEMM unit; for a gather, lane i copies row i of each stage's rows. Lane 0 claims the
    // next unit six stages before the end of the current one and reads its record three
    // stages before, so that both reads are in flight while the stages are issued.
    MOK_DEV void produce(Smem *sm, uint8_t *base, int lane, const CUtensorMap *tm_w13,
                         const CUtensorMap *tm_w2, const CUtensorMap *tm_x,
                         const CUtensorMap *tm_h) const {
        constexpr int SB = stage_bytes<MX>();
        constexpr int BKE = MX ? BK_MX : BK;
        constexpr uint32_t FULL = 0xFFFFFFFFu;
        volatile int *abort = &sm->abort;
        if (lane == 0) {
            tc::prefetch_tmap(tm_x);
            tc::prefetch_tmap(tm_h);
        }
        int s = 0;
        uint32_t ph = 0;
        int64_t issued = 0, j = 0;
        int32_t u = -1;
        UnitRec rec{};
        if (lane == 0) {
            u = claim();
            if (u >= 0) rec = load_rec(u);
        }
        u = __shfl_sync(FULL, u, 0);
        rec = shfl_rec(rec);
        for (;;) {
            // wait for the unit's inputs, then publish it (or the end marker) to the MMA
            // thread and the epilogue warps
            int ok = 1;
            if (lane == 0) {
                if (u >= 0) ok = wait_inputs(rec, abort);
                const int slot = (int)(j % QD);
                if (ok)
                    ok = wait_or_abort(&sm->qempty[slot], (uint32_t)(((j / QD) & 1) ^ 1),
                                       status, abort);
                if (ok) {
                    *(volatile int32_t *)&sm->q[slot] = u;
                    tc::mbar_arrive(&sm->qfull[slot]);
                }
            }
            if (!__shfl_sync(FULL, ok, 0)) break;
            ++j;
            if (u < 0) break;
            const int kind = rec.code >> 16;
            // lane 0: the next unit, claimed at step claim_at of this unit's n_steps and its
            // record read at step rec_at (or after the last step)
            int32_t next = -1;
            UnitRec nrec{};
            bool claimed = false, have = false;
            auto prefetch = [&](int64_t k, int64_t n_steps) {
                const int64_t claim_at = n_steps > 6 ? n_steps - 6 : 0;
                const int64_t rec_at = n_steps > 3 ? n_steps - 3 : n_steps;
                if (k == claim_at) {
                    next = claim();
                    claimed = true;
                }
                if (k == rec_at && next >= 0) {
                    nrec = load_rec(next);
                    have = true;
                    // records are claimed in order by every SM in turn: warm L2 with the
                    // one 64 claims ahead
                    if (next + REC_AHEAD < hdr[0])
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(units + next + REC_AHEAD));
                }
            };
            if (kind == KIND_GATHER) {
                int64_t r0, r1;
                gather_span(rec, &r0, &r1);
                const int64_t n_st = (r1 - r0 + rows_per_stage - 1) / rows_per_stage;
                for (int64_t si = 0; si < n_st; ++si) {
                    if (lane == 0) {
                        prefetch(si, n_st);
                        ok = wait_or_abort(&sm->empty[s], ph ^ 1u, status, abort);
                    }
                    if (!__shfl_sync(FULL, ok, 0)) break;
                    const int64_t q0 = r0 + si * rows_per_stage;
                    const int m = (int)(r1 - q0 < rows_per_stage ? r1 - q0 : rows_per_stage);
                    uint8_t *st = base + s * SB;
                    uint64_t *fb = &sm->full[s];
                    if (lane == 0) tc::mbar_arrive_expect_tx(fb, (uint32_t)(m * row_bytes));
                    __syncwarp();  // the expected bytes are set before any copy can land
                    if (lane < m)
                        tc::bulk_load(st + lane * row_bytes,
                                      x + (int64_t)(perm[q0 + lane] / K) * row_bytes,
                                      (uint32_t)row_bytes, fb);
                    ++issued;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            } else if (lane == 0) {
                const bool down = kind == KIND_DOWN;
                const Geom g = geom_rec(rec);
                const int kblocks = (g.k_steps + 3) / 4;
                const uint32_t tx = 2 * A_BYTES + B_BYTES + (MX ? 1536 : 0);
                const uint8_t *sfa = down ? dn.sf_a : up.sf_a;
                const uint8_t *sfb = down ? dn.sf_b : up.sf_b;
                for (int kb = 0; kb < kblocks; ++kb) {
                    prefetch(kb, kblocks);
                    if (!wait_or_abort(&sm->empty[s], ph ^ 1u, status, abort)) {
                        ok = 0;
                        break;
                    }
                    uint8_t *st = base + s * SB;
                    uint64_t *fb = &sm->full[s];
                    const int k0 = kb * BKE;
                    tc::mbar_arrive_expect_tx(fb, tx);
                    if (MX) {
                        uint8_t *sf = st + 2 * A_BYTES + B_BYTES;
                        tc::bulk_load(sf, sfa + g.sfa0 + kb * 512, 512, fb);
                        tc::bulk_load(sf + 512, sfa + g.sfa1 + kb * 512, 512, fb);
                        tc::bulk_load(sf + 1024, sfb + g.sfb + kb * 512, 512, fb);
                    }
                    if (down) {
                        tc::tma_load_2d(st, tm_w2, fb, k0, g.ay0);
                        tc::tma_load_2d(st + 2 * A_BYTES, tm_h, fb, k0, g.by);
                    } else {
                        tc::tma_load_5d(st, tm_w13, fb, k0, 0, g.ay0, 0, g.ay1);
                        tc::tma_load_2d(st + 2 * A_BYTES, tm_x, fb, k0, g.by);
                    }
                    ++issued;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // a unit without steps (an empty gather piece) claims its successor here
            if (lane == 0 && ok && !claimed) next = claim();
            if (lane == 0 && next >= 0 && !have) nrec = load_rec(next);
            // lane 0 holds the loop state of a GEMM unit and the next unit: broadcast them
            if (!__shfl_sync(FULL, ok, 0)) break;
            s = __shfl_sync(FULL, s, 0);
            ph = __shfl_sync(FULL, ph, 0);
            issued = __shfl_sync(FULL, issued, 0);
            u = __shfl_sync(FULL, next, 0);
            rec = shfl_rec(nrec);
        }
        // do not leave while copies this CTA issued may still be landing
        if (lane == 0) {
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
        __syncwarp();
    }
};

template <class P>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_ring_kernel(const __grid_constant__ CUtensorMap tm_w13,
                   const __grid_constant__ CUtensorMap tm_w2,
                   const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_h, const P p) {
    gemm_body<P>(tm_w13, tm_w2, tm_x, tm_h, p, 0);
}

// ---------------------------------------------------------------- the unit order
constexpr int BUILD_THREADS = 1024;

// tiles of rows [b, end) of one expert: cut at multiples of C, then each piece into tiles of
// at most `chunk` rows, of balanced heights rounded up to 16 (the last may be shorter)
struct PieceCut {
    int64_t C;
    int chunk;
    MOK_DEV int64_t size_of(int64_t len) const {
        const int64_t n0 = (len + chunk - 1) / chunk;
        int64_t size = (((len + n0 - 1) / n0) + 15) & ~(int64_t)15;
        return size > chunk ? chunk : size;
    }
    MOK_DEV int64_t count(int64_t b, int64_t end) const {
        int64_t n = 0;
        for (int64_t p = b; p < end;) {
            const int64_t lap_end = (p / C + 1) * C;
            const int64_t q = lap_end < end ? lap_end : end;
            const int64_t size = size_of(q - p);
            n += (q - p + size - 1) / size;
            p = q;
        }
        return n;
    }
};

// first index j in [0, n) with key(j) > v, for keys 2 * r0(j) + add (non-decreasing in j)
MOK_DEV int64_t upper_bound_key(const int32_t *tiles, int64_t n, int64_t add, int64_t v) {
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        const int64_t m = (lo + hi) >> 1;
        if (2 * (int64_t)tiles[4 * m + 1] + add <= v)
            lo = m + 1;
        else
            hi = m;
    }
    return lo;
}

// One block: the flat tile list (count at tiles[-4]), the unit records in claim order,
// zeroed counters and the unit count. Group keys in half rows:
// gather 2 r0 - g, gate/up 2 r0, down 2 r0 + d; on equal keys gather, then gate/up, then
// down.
__global__ void __launch_bounds__(BUILD_THREADS)
    build_ring_units(const int32_t *__restrict__ offsets, int E, int64_t C, int chunk,
                     int64_t g, int64_t d, int n_g, int n_up, int n_dn,
                     int32_t *__restrict__ tiles,
                     int64_t cap, UnitRec *__restrict__ units,
                     int32_t *__restrict__ hdr, int32_t *__restrict__ done_up,
                     int32_t *__restrict__ done_dn, int32_t *__restrict__ done_g,
                     int *status) {
    __shared__ int64_t sc[BUILD_THREADS];
    const int e = threadIdx.x;
    const PieceCut cut{C, chunk};
    int64_t b = 0, end = 0, n = 0;
    if (e < E) {
        b = offsets[e];
        end = offsets[e + 1];
        n = cut.count(b, end);
    }
    sc[e] = n;
    __syncthreads();
    for (int o = 1; o < BUILD_THREADS; o <<= 1) {
        const int64_t v = e >= o ? sc[e - o] : 0;
        __syncthreads();
        sc[e] += v;
        __syncthreads();
    }
    const int64_t total = sc[BUILD_THREADS - 1];
    if (total > cap) {
        // cannot happen for a valid schedule (cap bounds the tiles of any cut)
        if (e == 0) {
            raise_status(status, MOK_ERR_DEVICE_INVARIANT);
            tiles[-4] = 0;
            hdr[0] = 0;
            hdr[1] = 0;
        }
        return;
    }
    int64_t s = sc[e] - n;
    for (int64_t p = b; p < end;) {
        const int64_t lap_end = (p / C + 1) * C;
        const int64_t q = lap_end < end ? lap_end : end;
        const int64_t size = cut.size_of(q - p);
        for (int64_t r0 = p; r0 < q; r0 += size, ++s) {
            tiles[4 * s + 0] = e;
            tiles[4 * s + 1] = (int32_t)r0;
            tiles[4 * s + 2] = (int32_t)(r0 + size < q ? r0 + size : q);
            tiles[4 * s + 3] = 0;
        }
        p = q;
    }
    __syncthreads();
    const int64_t nt = total;
    // groups of each kind keyed at or below (or strictly below) a key
    auto at_most = [&](int64_t add, int64_t v) { return upper_bound_key(tiles, nt, add, v); };
    for (int64_t t = threadIdx.x; t < nt; t += BUILD_THREADS) {
        const int64_t r0 = tiles[4 * t + 1], r1 = tiles[4 * t + 2];
        // tiles one lap back over ring rows [r0, r1): rows [r0 - C, r1 - C)
        int2 dp = make_int2(0, -1);
        if (r1 - 1 - C >= 0) {
            const int64_t lo = r0 - C > 0 ? r0 - C : 0;
            dp.x = (int)(upper_bound_key(tiles, t, 0, 2 * lo) - 1);
            dp.y = (int)(upper_bound_key(tiles, t, 0, 2 * (r1 - 1 - C)) - 1);
        }
        const int e = tiles[4 * t];
        const UnitRec base{(int)t, 0, e, (int)r0, (int)r1, dp.x, dp.y, 0};
        auto put = [&](int64_t o, int kind, int m) {
            UnitRec r = base;
            r.code = (kind << 16) | m;
            units[o] = r;
        };
        // gather group (key 2 r0 - g): gate/up and down groups with smaller keys before it
        const int64_t kg = 2 * r0 - g, ku = 2 * r0, kd = 2 * r0 + d;
        int64_t o = t * n_g + at_most(0, kg - 1) * n_up + at_most(d, kg - 1) * n_dn;
        for (int m = 0; m < n_g; ++m) put(o + m, KIND_GATHER, m);
        // gate/up group: gathers at or below its key, down groups below it
        o = at_most(-g, ku) * n_g + t * n_up + at_most(d, ku - 1) * n_dn;
        for (int m = 0; m < n_up; ++m) put(o + m, KIND_UP, m);
        // down group: gathers and gate/up groups at or below its key
        o = at_most(-g, kd) * n_g + at_most(0, kd) * n_up + t * n_dn;
        for (int m = 0; m < n_dn; ++m) put(o + m, KIND_DOWN, m);
        done_up[t] = 0;
        done_dn[t] = 0;
        done_g[t] = 0;
    }
    if (threadIdx.x == 0) {
        tiles[-4] = (int32_t)nt;
        hdr[0] = (int32_t)(nt * (n_g + n_up + n_dn));
        hdr[1] = 0;
    }
}

// MXFP8: the scale atoms of the x rows of every tile (the gate/up GEMM's B scales), from x's
// token-major scales: atom (tile t, K block kb) row n holds the 4 scale bytes of block kb of
// row r0 + n (the last row of the tile for n past it).
__global__ void __launch_bounds__(128)
    ring_x_atoms(const int32_t *__restrict__ tiles, int64_t cap, const int32_t *__restrict__ perm,
                 int K, const uint8_t *__restrict__ xs, int H, uint8_t *__restrict__ atoms) {
    const int kg = H / 128;
    const int64_t nt = tiles[-4] < cap ? tiles[-4] : cap;
    const int n = threadIdx.x;
    for (int64_t bi = blockIdx.x; bi < nt * kg; bi += gridDim.x) {
        const int64_t t = bi / kg;
        const int kb = (int)(bi % kg);
        const int64_t r0 = tiles[4 * t + 1], r1 = tiles[4 * t + 2];
        const int64_t r = r0 + n < r1 ? r0 + n : r1 - 1;
        const int64_t tok = perm[r] / K;
        const uint32_t v = *reinterpret_cast<const uint32_t *>(xs + tok * (H / 32) + kb * 4);
        *reinterpret_cast<uint32_t *>(atoms + bi * 512 + (n & 31) * 16 + (n >> 5) * 4) = v;
    }
}

template <bool MX>
cudaError_t launch_ring(const RingFwdArgs &a, cudaStream_t s) {
    using P = RingFwdT<MX>;
    constexpr int SMEM = smem_bytes<MX>();
    static std::atomic<uint64_t> attr_set[2] = {{0}, {0}};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << (dev & 63);
    if ((attr_set[dev >> 6].load(std::memory_order_acquire) & bit) == 0) {
        e = cudaFuncSetAttribute(tc_ring_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev >> 6].fetch_or(bit, std::memory_order_acq_rel);
    }
    CUtensorMap m_w13, m_w2, m_x, m_h;
    if ((e = make_map_w13_pairs(&m_w13, a.w13, a.E, a.I, a.H, MX)) != cudaSuccess) return e;
    if (MX) {
        if ((e = make_map_u8(&m_w2, a.w2, (int64_t)a.E * a.H, a.I, 256)) != cudaSuccess) return e;
        if ((e = make_map_u8(&m_h, a.hring, a.C, a.I, KBOX_ROWS)) != cudaSuccess) return e;
    } else {
        if ((e = make_map_bf16(&m_w2, a.w2, (int64_t)a.E * a.H, a.I, 256)) != cudaSuccess)
            return e;
        if ((e = make_map_bf16(&m_h, a.hring, a.C, a.I, KBOX_ROWS)) != cudaSuccess) return e;
    }
    if (MX) {
        if ((e = make_map_u8(&m_x, a.xring, a.C, a.H, KBOX_ROWS)) != cudaSuccess) return e;
    } else if ((e = make_map_bf16(&m_x, a.xring, a.C, a.H, KBOX_ROWS)) != cudaSuccess) {
        return e;
    }
    const Ring ring{a.R, (int32_t)a.C, 1};
    const int nmb_dn = (a.H + 255) / 256;
    P p{};
    p.up = FwdUpT<MX, true>{TileUnits{a.tiles, a.tiles_cap, a.I / 128}, a.H, a.I, ring, a.hring,
                      a.hring_s, a.preact, a.preact_f32, MX, a.status,
                      MX ? a.sf_w13 : nullptr, MX ? a.sf_x : nullptr, nullptr, nullptr,
                      MX ? a.sf_h : nullptr};
    p.dn = FwdDownT<MX>{TileUnits{a.tiles, a.tiles_cap, nmb_dn}, a.H, a.I, ring, a.perm,
                        a.slots, a.out_f32, a.status, MX ? a.sf_w2 : nullptr,
                        MX ? a.sf_h : nullptr, false};
    p.units = static_cast<const UnitRec *>(a.units);
    p.hdr = a.hdr;
    p.done_up = a.done_up;
    p.done_dn = a.done_dn;
    p.done_g = a.done_g;
    p.perm = a.perm;
    p.K = a.K;
    p.status = a.status;
    p.x = static_cast<const uint8_t *>(a.x);
    p.xring = static_cast<uint8_t *>(a.xring);
    p.C = a.C;
    p.row_bytes = a.H * (MX ? 1 : 2);
    p.rows_per_stage = ring_stage_rows(MX, a.H);
    p.gather_pieces = a.gather_pieces;
    p.gather_rows = (a.chunk + a.gather_pieces - 1) / a.gather_pieces;
    tc_ring_kernel<P><<<device_sm_count(), NTHREADS, SMEM, s>>>(m_w13, m_w2, m_x, m_h, p);
    return cudaGetLastError();
}

}  // namespace

int ring_tile_rows(bool mxfp8, int64_t C) {
    const int chunk = gemm_tc_tile_rows(mxfp8);
    if (C >= 2 * (int64_t)chunk) return chunk;
    return C / 2 > 1 ? (int)(C / 2) : 1;
}

// The lags, in half rows, of a tile's gather before its gate/up units (g) and of its down
// units after them (d): g = C and d = 3C/2, both capped at 2 (C - chunk) + 1. On the
// 65536-token imbalanced workload (2960-row ring) a sweep of g, d over C/4 .. 1.9 C found
// this pair fastest; d = g = C was 2.4% slower, d = C/4 nearly twice as slow.
void ring_lags(bool mxfp8, int64_t C, int64_t *g, int64_t *d) {
    const int64_t most = 2 * (C - ring_tile_rows(mxfp8, C)) + 1;
    *g = C < most ? C : most;
    *d = C + C / 2 < most ? C + C / 2 : most;
}

// x rows of one stage in a gather: a stage's operand bytes (48 KB) over a row's, at most
// one per lane
int ring_stage_rows(bool mxfp8, int H) {
    const int n = (2 * A_BYTES + B_BYTES) / (H * (mxfp8 ? 1 : 2));
    return n < 32 ? n : 32;
}

// gather units per tile: pieces of at most four stages (one fill of the stage ring), so a
// tile's rows are gathered by several CTAs at once. A tile's gate/up units wait for all of
// its pieces; on the 65536-token imbalanced workload a whole-tile gather took 28 us and
// gated 61% of the gate/up units' waits.
int ring_gather_pieces(bool mxfp8, int64_t C, int H) {
    const int per = 4 * ring_stage_rows(mxfp8, H);
    const int chunk = ring_tile_rows(mxfp8, C);
    return (chunk + per - 1) / per;
}

int64_t ring_tiles_cap(int64_t R, int E, int64_t C, int chunk) {
    return (R + chunk - 1) / chunk + E + (R + C - 1) / C;
}

cudaError_t launch_ring_forward(const RingFwdArgs &a, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    if (a.R < 1 || a.C < 1 || a.E > BUILD_THREADS) return cudaErrorInvalidValue;
    const int nmb_up = a.I / 128, nmb_dn = (a.H + 255) / 256;
    build_ring_units<<<1, BUILD_THREADS, 0, s>>>(a.offsets, a.E, a.C, a.chunk, a.lag_gather,
                                                 a.lag, a.gather_pieces, nmb_up, nmb_dn,
                                                 a.tiles, a.tiles_cap,
                                                 static_cast<UnitRec *>(a.units), a.hdr,
                                                 a.done_up, a.done_dn,
                                                 a.done_g, a.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.mx) {
        const int64_t blocks = a.tiles_cap * (a.H / 128);
        const int64_t cap_blocks = (int64_t)device_sm_count() * 16;
        ring_x_atoms<<<(unsigned)(blocks < cap_blocks ? blocks : cap_blocks), 128, 0, s>>>(
            a.tiles, a.tiles_cap, a.perm, a.K, a.xs, a.H, a.sf_x);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return launch_ring<true>(a, s);
    }
    return launch_ring<false>(a, s);
}

}  // namespace mok
