// wgrad_pair.cu -- the expert weight gradients on pairs of SMs that share their operand tiles.
//
// [alphalab] "Mixture-of-Kittens" (alphalab.site), section 一: the backward computes the
// expert gradients dW13 = dA^T x and dW2 = (w*h)^T dy per expert over its routed rows;
// section 五: warp specialization and PTX.
//
// out[e][n][m] = sum over the expert's padded rows p of A[p][m] B[p][n], the same fixed-order
// fp32 dot products as the one-SM weight-gradient GEMM (K in 16-row steps from the expert's
// first row), so the results are the same bit for bit.
//
// A cluster of two CTAs on two SMs computes one 256 x 256 output tile with the two-SM MMA
// (tcgen05 cta_group::2, M = 256): rank r holds output rows m in [mb*256 + 128r, +128) as
// its A half and loads columns [nb*256 + 128r, +128) of B; the MMA gives each CTA its 128
// rows against all 256 columns. Per 64-row K block a SM loads 32 KB for 128 x 256 outputs,
// where the one-SM kernel loads 48 KB (two A tiles and one B tile) for 256 x 128: the
// operand feed per FLOP falls by a third.
//
// Per CTA, 320 threads:
//   warp 0     TMA producer (both ranks): its own A half (two 64 x 64 MN-major boxes) and
//              B half into a 6-stage ring; the copies of both ranks complete on rank 0's
//              full barrier of the stage, whose expected bytes rank 0 sets
//   warp 1     TMEM owner (both ranks: the pair allocates together); on rank 0 the MMA
//              issuer, whose commits arrive on the stage-free and accumulator-full
//              barriers of both CTAs
//   warps 2-9  epilogue (both ranks): TMEM -> bf16/fp32 dW; each warp then arrives on rank
//              0's accumulator-free barrier
// Two accumulator sets of 256 columns alternate between consecutive units. Units are
// (expert, N block, M block) in that order, taken by the clusters in a static stride, so
// the clusters running at one time share an expert's operand tiles in L2.
//
// Every wait is bounded (2 s); a CTA that gives up records MOK_ERR_TIMEOUT and leaves its
// loops, and both CTAs meet at a cluster barrier before TMEM is freed.
#include "gemm_tc_core.cuh"

namespace mok {
namespace {

constexpr int PAIR_STAGES = 6;
constexpr int PAIR_BOX = 64 * 128;                // one 64 x 64 bf16 MN-major box
constexpr int PAIR_STAGE = 4 * PAIR_BOX;          // A half (2 boxes) + B half (<= 2 boxes)
constexpr uint32_t PAIR_SET_COLS = 256;           // TMEM columns of one accumulator set

struct PairSmem {
    uint64_t full[PAIR_STAGES];   // rank 0: both CTAs' copies of the stage have landed
    uint64_t empty[PAIR_STAGES];  // each CTA: the MMAs that read the stage are done
    uint64_t tmem_full[2];        // each CTA: accumulator set b holds a finished unit
    uint64_t tmem_empty[2];       // rank 0: both CTAs' epilogues have drained set b
    uint32_t tmem_base;
    int abort;
};

constexpr int PAIR_SMEM = PAIR_STAGES * PAIR_STAGE + 1024 + (int)sizeof(PairSmem);
static_assert(PAIR_SMEM <= 232448, "pair kernel exceeds the shared memory of a CTA");

struct PairArgs {
    const int32_t *counts, *poff;
    void *out;     // [E][N][M], fp32 if out_f32, else bf16
    bool out_f32;
    int E, M, N;
    int nmb, nnb;  // ceil(M / 256), N / 256 rounded up (N is a multiple of 128)
    int *status;
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

__global__ void __launch_bounds__(NTHREADS, 1)
    tc_wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, const PairArgs p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the same offset in both CTAs: the MMA finds the peer's tiles where this CTA has its own
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    PairSmem *sm = (PairSmem *)(base + PAIR_STAGES * PAIR_STAGE);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_rank();
    const int64_t cid = tc::cluster_id_x(), ncl = tc::cluster_count_x();
    const int64_t n_units = (int64_t)p.E * p.nmb * p.nnb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PAIR_STAGES; ++s) {
            tc::mbar_init(&sm->full[s], 1);
            tc::mbar_init(&sm->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sm->tmem_full[b], 1);
            tc::mbar_init(&sm->tmem_empty[b], 2 * EPI_WARPS);
        }
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

    auto unit = [&](int64_t u, int *e, int *mb, int *nb) {
        *e = (int)(u / ((int64_t)p.nmb * p.nnb));
        const int rest = (int)(u % ((int64_t)p.nmb * p.nnb));
        *nb = rest / p.nmb;
        *mb = rest % p.nmb;
    };
    auto cols = [&](int nb) { return p.N - nb * 256 < 256 ? p.N - nb * 256 : 256; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (tc::elect_one()) {
            const uint32_t full0 = tc::cluster_addr(&sm->full[0], 0);  // rank 0's full[0]
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t u = cid; u < n_units && ok; u += ncl) {
                int e, mb, nb;
                unit(u, &e, &mb, &nb);
                const int half = cols(nb) / 2;  // 64 or 128 columns of B per CTA
                const int nbox = half / 64;
                const int ax = mb * 256 + (int)rank * 128;
                const int bx = nb * 256 + (int)rank * half;
                const int y0 = p.poff[e];
                const int kblocks = (((p.counts[e] + 15) & ~15) / 16 + 3) / 4;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!pair_wait(&sm->empty[s], ph ^ 1u, p.status, abort)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0)
                        tc::mbar_arrive_expect_tx(&sm->full[s], 2 * (2 + nbox) * PAIR_BOX);
                    const uint32_t fb = full0 + (uint32_t)s * 8u;
                    uint8_t *st = base + s * PAIR_STAGE;
                    const int y = y0 + kb * BK;
                    tc::tma_load_2d_pair(st, &tmA, fb, ax, y);
                    tc::tma_load_2d_pair(st + PAIR_BOX, &tmA, fb, ax + 64, y);
                    for (int j = 0; j < nbox; ++j)
                        tc::tma_load_2d_pair(st + (2 + j) * PAIR_BOX, &tmB, fb, bx + 64 * j, y);
                    ++issued;
                    if (++s == PAIR_STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // do not leave while copies may still be landing: the MMAs that read the last
            // stages have finished (bounded)
            for (int q = 0; q < PAIR_STAGES && q < issued; ++q) {
                if (--s < 0) {
                    s = PAIR_STAGES - 1;
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
                int e, mb, nb;
                unit(u, &e, &mb, &nb);
                const int nn = cols(nb);
                const uint32_t idesc = tc::idesc_bf16(256, nn, true, true);
                const int k_steps = ((p.counts[e] + 15) & ~15) / 16;
                const int ab = (int)(a & 1);
                const uint32_t use = (uint32_t)((a >> 1) & 1);
                if (!pair_wait(&sm->tmem_empty[ab], use ^ 1u, p.status, abort)) break;
                tc::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)ab * PAIR_SET_COLS;
                const int kblocks = (k_steps + 3) / 4;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!pair_wait(&sm->full[s], ph, p.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t sa = tc::smem_u32(base + s * PAIR_STAGE);
                    const uint32_t sb = sa + 2 * PAIR_BOX;
                    const int steps = k_steps - kb * 4 < 4 ? k_steps - kb * 4 : 4;
                    for (int kk = 0; kk < steps; ++kk) {
                        // MN-major: 16 K rows = 2 groups of eight 128-byte rows; the two
                        // 64-wide blocks of each half are PAIR_BOX apart
                        const uint64_t da = tc::sdesc_sw128(sa + kk * 2048, PAIR_BOX, 1024);
                        const uint64_t db = tc::sdesc_sw128(sb + kk * 2048, PAIR_BOX, 1024);
                        tc::mma_f16_pair(d, da, db, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit_pair(&sm->empty[s], 3);  // frees the stage in both CTAs
                    if (++s == PAIR_STAGES) {
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
        int64_t a = 0;
        for (int64_t u = cid; u < n_units; u += ncl, ++a) {
            int e, mb, nb;
            unit(u, &e, &mb, &nb);
            const int nn = cols(nb);
            const int ab = (int)(a & 1);
            if (!pair_wait(&sm->tmem_full[ab], (uint32_t)((a >> 1) & 1), p.status, abort))
                break;
            tc::tc_fence_after();
            const bool any = p.counts[e] > 0;
            const int m = mb * 256 + (int)rank * 128 + q * 32 + lane;
            const bool mok = m < p.M;
            const uint32_t c = tmem + lane_base + (uint32_t)ab * PAIR_SET_COLS;
            const int64_t row0 = (int64_t)e * p.N + (int64_t)nb * 256;
            // 32 columns per TMEM round trip (nn is a multiple of 128)
            for (int n0 = 32 * hw; n0 < nn; n0 += 64) {
                float v0[16], v1[16];
                tc::tmem_ld16(c + n0, v0);
                tc::tmem_ld16(c + n0 + 16, v1);
                tc::tmem_ld_wait();
                if (mok) {
                    const int64_t o = (row0 + n0) * p.M + m;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        st_val(p.out, o + (int64_t)j * p.M, any ? v0[j] : 0.f, p.out_f32);
                        st_val(p.out, o + (int64_t)(16 + j) * p.M, any ? v1[j] : 0.f,
                               p.out_f32);
                    }
                }
            }
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

// clusters of two that fit on the device at once, per device
std::atomic<int> g_pair_clusters[MAX_DEV];

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
    const int64_t units = (int64_t)E * nmb * nnb;
    if (units < 1) return cudaSuccess;
    if (units > 0x7FFFFFFF) return cudaErrorInvalidValue;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEV) return cudaErrorInvalidDevice;
    int nc = g_pair_clusters[dev].load(std::memory_order_acquire);
    if (nc == 0) {
        e = cudaFuncSetAttribute(tc_wgrad_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PAIR_SMEM);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t q = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        q.gridDim = dim3((unsigned)(2 * device_sm_count()), 1, 1);
        q.blockDim = dim3(NTHREADS, 1, 1);
        q.dynamicSmemBytes = PAIR_SMEM;
        q.attrs = at;
        q.numAttrs = 1;
        // where the query fails, one cluster per two SMs: clusters that do not fit wait for
        // a free pair and take their units then (the static stride still covers them all)
        if (cudaOccupancyMaxActiveClusters(&nc, tc_wgrad_pair_kernel, &q) != cudaSuccess ||
            nc < 1) {
            (void)cudaGetLastError();
            nc = device_sm_count() / 2 > 0 ? device_sm_count() / 2 : 1;
        }
        g_pair_clusters[dev].store(nc, std::memory_order_release);
    }
    const int64_t clusters = units < nc ? units : nc;
    PairArgs p{counts, poff, out, out_f32, E, M, N, nmb, nnb, status};
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = PAIR_SMEM;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, tc_wgrad_pair_kernel, ma, mb, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mok
