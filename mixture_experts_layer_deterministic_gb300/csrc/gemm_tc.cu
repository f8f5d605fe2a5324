// gemm_tc.cu -- expert-grouped GEMMs of the forward on the 5th-generation tensor cores.
//
// [alphalab] "Mixture-of-Kittens" (alphalab.site), section 一: routed experts run a SwiGLU
// FFN (gate/up GEMM, SwiGLU, down GEMM); section 五: warp specialization and PTX.
// [arex] "Cursor 放出 MoK" (arex-research.com), section "pull 代替 push": expert-grouped
// GEMMs fed by a pull dispatch, results pushed back to their (token, k) slots.
//
// One persistent kernel per GEMM, 192 threads per CTA, one CTA per SM:
//   warp 0     TMA producer: weight tiles A0, A1 (128 rows each) and the token tile B
//              (up to 256 rows) of each 64-wide K block into a 3-stage ring
//   warp 1     TMEM owner and MMA issuer: D0 += A0 B^T, D1 += A1 B^T (M=128, N<=256, K=16
//              per instruction), fp32 accumulators at TMEM columns 0 and 256
//   warps 2-5  epilogue: TMEM -> registers -> fused SwiGLU / scatter -> global memory
// Work unit = (token tile, weight block). Swapping the GEMM so that the weights are M and
// the expert's routed rows are N keeps the ragged dimension at a 16-row granularity.
// Every output element is one fixed-order fp32 dot product, so results do not depend on
// which CTA computes a unit.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "mok_internal.h"
#include "tc.cuh"

namespace mok {
namespace {

constexpr int BK = 64;            // K elements per stage (128 bytes of bf16)
constexpr int STAGES = 3;
constexpr int TILE_ROWS = 256;    // max token rows per unit (N)
constexpr int BOX_ROWS = 32;      // token rows per TMA box
constexpr int A_BYTES = 128 * BK * 2;
constexpr int B_BYTES = TILE_ROWS * BK * 2;
constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;
constexpr int NTHREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;

struct PairArgs {
    const int32_t *tiles;   // (e, r0, r1, _) list, count at tiles[-4]
    int64_t tiles_cap;
    int n_mblocks;          // weight blocks per tile
    int k_blocks;           // K / BK
    int a_rows_per_expert;  // rows of A per expert in the 2D A map
    int a_off1;             // row offset of A1 relative to A0 inside the expert
    int a_mb_stride;        // row step per weight block
    Ring ring;
    int *status;
};

struct EpiUpArgs {
    void *hring;
    uint8_t *hring_s;
    float *preact;
    int I;
    bool mxfp8;
};

struct EpiDownArgs {
    const int32_t *perm;
    float *slots;
    int H;
};

struct Smem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint32_t tmem_base;
    int abort;
};

MOK_DEV float silu_f(float g) { return g / (1.0f + expf(-g)); }

// bounded wait; gives up when another role has aborted or after the wall-time limit
MOK_DEV bool wait_or_abort(uint64_t *bar, uint32_t parity, int *status, volatile int *abort) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer();
    uint32_t n = 0;
    while (!tc::mbar_try_wait(bar, parity)) {
        if ((++n & 255u) == 0) {
            if (*abort) return false;
            if (tc::globaltimer() - t0 > tc::WAIT_LIMIT_NS) {
                raise_status(status, MOK_ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
    return true;
}

template <int KIND>  // 0: gate/up + SwiGLU, 1: down + push scatter
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, PairArgs p, EpiUpArgs up,
                     EpiDownArgs down) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Smem *sm = (Smem *)(base + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int64_t n_tiles = p.tiles[-4] < p.tiles_cap ? p.tiles[-4] : p.tiles_cap;
    const int64_t n_units = n_tiles * p.n_mblocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&sm->full[s], 1);
            tc::mbar_init(&sm->empty[s], 1);
        }
        tc::mbar_init(&sm->tmem_full, 1);
        tc::mbar_init(&sm->tmem_empty, 128);
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

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (tc::elect_one()) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            for (int64_t u = blockIdx.x; u < n_units && !*abort; u += gridDim.x) {
                const int64_t t = u / p.n_mblocks;
                const int mb = (int)(u % p.n_mblocks);
                const int e = p.tiles[4 * t + 0];
                const int64_t r0 = p.tiles[4 * t + 1], r1 = p.tiles[4 * t + 2];
                const int nbox = (int)((r1 - r0 + BOX_ROWS - 1) / BOX_ROWS);
                const RingMap rm{p.ring.R, p.ring.MB, p.ring.n_slots};
                const int32_t brow = (int32_t)rm(r0);
                const int32_t arow0 = e * p.a_rows_per_expert + mb * p.a_mb_stride;
                const int32_t arow1 = arow0 + p.a_off1;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!wait_or_abort(&sm->empty[s], ph ^ 1u, p.status, abort)) break;
                    uint8_t *st = base + s * STAGE_BYTES;
                    tc::mbar_arrive_expect_tx(&sm->full[s],
                                              2 * A_BYTES + nbox * BOX_ROWS * BK * 2);
                    tc::tma_load_2d(st, &tmA, &sm->full[s], kb * BK, arow0);
                    tc::tma_load_2d(st + A_BYTES, &tmA, &sm->full[s], kb * BK, arow1);
                    for (int j = 0; j < nbox; ++j)
                        tc::tma_load_2d(st + 2 * A_BYTES + j * BOX_ROWS * BK * 2, &tmB,
                                        &sm->full[s], kb * BK, brow + j * BOX_ROWS);
                    ++issued;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
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
            uint32_t ph = 0, acc_ph = 0;
            for (int64_t u = blockIdx.x; u < n_units && !*abort; u += gridDim.x) {
                const int64_t t = u / p.n_mblocks;
                const int64_t r0 = p.tiles[4 * t + 1], r1 = p.tiles[4 * t + 2];
                const int n_mma = (int)((r1 - r0 + 15) & ~15);
                const uint32_t idesc = tc::idesc_bf16(128, n_mma, false, false);
                if (!wait_or_abort(&sm->tmem_empty, acc_ph ^ 1u, p.status, abort)) break;
                tc::tc_fence_after();
                bool ok = true;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!wait_or_abort(&sm->full[s], ph, p.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(base + s * STAGE_BYTES);
                    const uint32_t a1 = a0 + A_BYTES;
                    const uint32_t b = a0 + 2 * A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t da0 = tc::sdesc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t da1 = tc::sdesc_sw128(a1 + kk * 32, 16, 1024);
                        const uint64_t db = tc::sdesc_sw128(b + kk * 32, 16, 1024);
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        tc::mma_f16(tmem + 0, da0, db, idesc, acc);
                        tc::mma_f16(tmem + 256, da1, db, idesc, acc);
                    }
                    tc::mma_commit(&sm->empty[s]);  // frees the stage once these MMAs finish
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                tc::mma_commit(&sm->tmem_full);
                acc_ph ^= 1u;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int fl = q * 32 + lane;
        uint32_t acc_ph = 0;
        for (int64_t u = blockIdx.x; u < n_units && !*abort; u += gridDim.x) {
            const int64_t t = u / p.n_mblocks;
            const int mb = (int)(u % p.n_mblocks);
            const int64_t r0 = p.tiles[4 * t + 1], r1 = p.tiles[4 * t + 2];
            const int nr = (int)(r1 - r0);
            const int n_mma = (nr + 15) & ~15;
            if (!wait_or_abort(&sm->tmem_full, acc_ph, p.status, abort)) break;
            tc::tc_fence_after();
            const uint32_t lane_base = (uint32_t)(q * 32) << 16;
            const RingMap rm{p.ring.R, p.ring.MB, p.ring.n_slots};
            for (int n0 = 0; n0 < n_mma; n0 += 16) {
                float d0[16], d1[16];
                tc::tmem_ld16(tmem + lane_base + 0 + n0, d0);
                tc::tmem_ld16(tmem + lane_base + 256 + n0, d1);
                tc::tmem_ld_wait();
                if (KIND == 0) {
                    const int I = up.I;
                    const int i = mb * 128 + fl;  // gate feature; up feature is I + i
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = n0 + j;
                        const bool live = n < nr;
                        const int64_t r = r0 + n;
                        const float h = silu_f(d0[j]) * d1[j];
                        if (live && up.preact != nullptr) {
                            up.preact[r * 2 * I + i] = d0[j];
                            up.preact[r * 2 * I + I + i] = d1[j];
                        }
                        if (!up.mxfp8) {
                            if (live)
                                ((uint16_t *)up.hring)[rm(r) * I + i] = f32_to_bf16(h);
                        } else {
                            // the warp's 32 lanes hold one 32-feature MXFP8 block of row r
                            float amax = fabsf(h);
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1)
                                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                            const uint32_t sb = mx_scale_byte(amax);
                            const uint32_t code = e4m3x2(h * mx_inv_scale(sb), 0.f) & 0xFFu;
                            if (live) {
                                const int64_t slot = rm(r);
                                ((uint8_t *)up.hring)[slot * I + i] = (uint8_t)code;
                                if (lane == 0) up.hring_s[slot * (I / 32) + i / 32] = (uint8_t)sb;
                            }
                        }
                    }
                } else {
                    const int H = down.H;
                    const int c = mb * 256 + fl;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = n0 + j;
                        if (n < nr) {
                            const int64_t f = down.perm[r0 + n];
                            down.slots[f * H + c] = d0[j];
                            if (c + 128 < H) down.slots[f * H + c + 128] = d1[j];
                        }
                    }
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&sm->tmem_empty);
            acc_ph ^= 1u;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_num_sms = 0;
bool g_attr_set[2] = {false, false};

cudaError_t init_host() {
    if (g_encode == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return cudaErrorNotSupported;
        g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaError_t e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// row-major bf16 matrix [rows][cols] -> 2D map with 64 x box_rows boxes, 128-byte swizzle
cudaError_t make_map_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols,
                          int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int KIND>
cudaError_t launch_pair(const CUtensorMap &ma, const CUtensorMap &mb, const PairArgs &p,
                        const EpiUpArgs &up, const EpiDownArgs &dn, cudaStream_t s) {
    if (!g_attr_set[KIND]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<KIND>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        g_attr_set[KIND] = true;
    }
    const int64_t units = p.tiles_cap * p.n_mblocks;
    const int grid = (int)(units < g_num_sms ? units : g_num_sms);
    if (grid < 1) return cudaSuccess;
    gemm_pair_kernel<KIND><<<grid, NTHREADS, SMEM_BYTES, s>>>(ma, mb, p, up, dn);
    return cudaGetLastError();
}

}  // namespace

int gemm_tc_tile_rows() { return TILE_ROWS; }

cudaError_t launch_gemm_up_tc(const GemmUpArgs &a, int64_t ring_rows, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    // A: W13 viewed as [E*2I][H]; B: the ring [ring_rows][H]
    CUtensorMap ma, mb;
    if ((e = make_map_bf16(&ma, a.w13, (int64_t)a.E * 2 * a.I, a.H, 128)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, a.xring, ring_rows, a.H, BOX_ROWS)) != cudaSuccess) return e;
    PairArgs p{a.tiles, a.tiles_cap, a.I / 128, a.H / BK, 2 * a.I, a.I, 128, a.ring, a.status};
    EpiUpArgs up{a.hring, a.hring_s, a.preact, a.I, a.mxfp8};
    EpiDownArgs dn{nullptr, nullptr, 0};
    return launch_pair<0>(ma, mb, p, up, dn, s);
}

cudaError_t launch_gemm_down_tc(const GemmDownArgs &a, int64_t ring_rows, cudaStream_t s) {
    cudaError_t e = init_host();
    if (e != cudaSuccess) return e;
    // A: W2 viewed as [E*H][I]; B: the h ring [ring_rows][I]
    CUtensorMap ma, mb;
    if ((e = make_map_bf16(&ma, a.w2, (int64_t)a.E * a.H, a.I, 128)) != cudaSuccess) return e;
    if ((e = make_map_bf16(&mb, a.hring, ring_rows, a.I, BOX_ROWS)) != cudaSuccess) return e;
    PairArgs p{a.tiles, a.tiles_cap, (a.H + 255) / 256, a.I / BK, a.H, 128, 256, a.ring,
               a.status};
    EpiUpArgs up{nullptr, nullptr, nullptr, 0, false};
    EpiDownArgs dn{a.perm, a.slots, a.H};
    return launch_pair<1>(ma, mb, p, up, dn, s);
}

}  // namespace mok
