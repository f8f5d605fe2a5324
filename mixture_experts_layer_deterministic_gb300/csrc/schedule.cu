// schedule.cu -- the deterministic expert schedule and the device-built tile lists.
//
// [arex] "Cursor 放出 MoK：NVL72 训练提速 2.37 倍" (arex-research.com), section "pull 代替
// push，ring buffer 踢掉 CPU": one schedule table drives dispatch, combine and their
// backward twins, and costs a few percent of the layer. Here it is a stable counting sort
// of the routed ids f = t*K + k by expert, built from integer counts only, so every
// output is bit-exact and independent of thread scheduling.
//
// Passes (R routed ids cut into chunks of CHUNK ids, one warp per chunk):
//   1. hist:     per-chunk expert counts (warp match + shared-memory counters)
//   2. colscan:  per expert, the exclusive prefix of the chunk counts (in place) and counts[e]
//   3. offsets:  exclusive scan of counts over experts; minibatch segments
//   4. rank:     each id's row = offsets[e] + prefix of its chunk + its rank among equal
//                experts earlier in the chunk -> perm and inv
#include "common.cuh"
#include "mok_internal.h"

namespace mok {
namespace {

constexpr int CHUNK = 1024;        // routed ids per warp in passes 1 and 4
constexpr int SCHED_WARPS = 8;     // warps per block in passes 1 and 4
constexpr int MAX_E = 1024;

__global__ void __launch_bounds__(SCHED_WARPS * 32)
    sched_hist(const int32_t *__restrict__ idx, int64_t R, int E, int64_t n_chunks,
               int32_t *__restrict__ hist, int *status) {
    extern __shared__ int32_t cnt_all[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *cnt = cnt_all + warp * E;
    const int64_t chunk = (int64_t)blockIdx.x * SCHED_WARPS + warp;
    if (chunk >= n_chunks) return;
    for (int e = lane; e < E; e += 32) cnt[e] = 0;
    __syncwarp();
    const int64_t f0 = chunk * CHUNK;
    for (int base = 0; base < CHUNK; base += 32) {
        const int64_t f = f0 + base + lane;
        int e = -1;
        if (f < R) {
            e = idx[f];
            if (e < 0 || e >= E) {
                raise_status(status, MOK_ERR_DEVICE_INVARIANT);
                e = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
        __syncwarp();
    }
    for (int e = lane; e < E; e += 32) hist[chunk * E + e] = cnt[e];
}

// grid: ceil(E/32) blocks of 32x32 threads; lane = expert within the block's 32, warp j
// owns a contiguous range of chunks. Exclusive prefix over chunks, in place.
__global__ void __launch_bounds__(1024)
    sched_colscan(int32_t *__restrict__ hist, int E, int64_t n_chunks,
                  int32_t *__restrict__ counts) {
    __shared__ int32_t part[32][33];
    const int lane = threadIdx.x & 31, j = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    const int64_t per = (n_chunks + 31) / 32;
    const int64_t c0 = j * per;
    const int64_t c1 = (c0 + per < n_chunks) ? c0 + per : n_chunks;
    int32_t sum = 0;
    if (e < E)
        for (int64_t c = c0; c < c1; ++c) sum += hist[c * E + e];
    part[j][lane] = sum;
    __syncthreads();
    if (j == 0) {
        int32_t run = 0;
        for (int q = 0; q < 32; ++q) {
            const int32_t v = part[q][lane];
            part[q][lane] = run;
            run += v;
        }
        if (e < E) counts[e] = run;
    }
    __syncthreads();
    int32_t run = part[j][lane];
    if (e < E)
        for (int64_t c = c0; c < c1; ++c) {
            const int32_t v = hist[c * E + e];
            hist[c * E + e] = run;
            run += v;
        }
}

// one block of MAX_E threads: offsets = exclusive scan of counts; segments.
__global__ void __launch_bounds__(MAX_E)
    sched_offsets(const int32_t *__restrict__ counts, int E, int64_t MB, int64_t seg_cap,
                  int32_t *__restrict__ offsets, int32_t *__restrict__ segs,
                  int32_t *__restrict__ n_segs, int *status) {
    __shared__ int32_t sc[MAX_E];
    __shared__ int32_t ss[MAX_E];
    const int e = threadIdx.x;
    const int32_t c = (e < E) ? counts[e] : 0;
    sc[e] = c;
    __syncthreads();
    // Hillis-Steele inclusive scan of counts (integers: order does not matter)
    for (int o = 1; o < MAX_E; o <<= 1) {
        const int32_t v = (e >= o) ? sc[e - o] : 0;
        __syncthreads();
        sc[e] += v;
        __syncthreads();
    }
    const int32_t off = sc[e] - c;  // exclusive
    if (e < E) offsets[e] = off;
    if (e == E - 1) offsets[E] = sc[e];
    // segments of expert e: its row range cut at multiples of MB
    int32_t nseg = 0;
    if (e < E && c > 0) nseg = (int32_t)((off + c - 1) / MB - off / MB + 1);
    ss[e] = nseg;
    __syncthreads();
    for (int o = 1; o < MAX_E; o <<= 1) {
        const int32_t v = (e >= o) ? ss[e - o] : 0;
        __syncthreads();
        ss[e] += v;
        __syncthreads();
    }
    int64_t s = ss[e] - nseg;
    if (e == MAX_E - 1) n_segs[0] = ss[e] <= seg_cap ? ss[e] : (int32_t)seg_cap;
    int64_t b = off;
    const int64_t end = (int64_t)off + c;
    for (int32_t q = 0; q < nseg; ++q, ++s) {
        int64_t mb_end = (b / MB + 1) * MB;
        const int64_t se = end < mb_end ? end : mb_end;
        if (s < seg_cap) {
            segs[3 * s + 0] = e;
            segs[3 * s + 1] = (int32_t)b;
            segs[3 * s + 2] = (int32_t)se;
        } else {
            raise_status(status, MOK_ERR_DEVICE_INVARIANT);
        }
        b = se;
    }
}

__global__ void __launch_bounds__(SCHED_WARPS * 32)
    sched_rank(const int32_t *__restrict__ idx, int64_t R, int E, int64_t n_chunks,
               const int32_t *__restrict__ hist, const int32_t *__restrict__ offsets,
               int32_t *__restrict__ perm, int32_t *__restrict__ inv) {
    extern __shared__ int32_t cnt_all[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *cnt = cnt_all + warp * E;
    const int64_t chunk = (int64_t)blockIdx.x * SCHED_WARPS + warp;
    if (chunk >= n_chunks) return;
    for (int e = lane; e < E; e += 32) cnt[e] = offsets[e] + hist[chunk * E + e];
    __syncwarp();
    const unsigned lt = (1u << lane) - 1u;
    const int64_t f0 = chunk * CHUNK;
    for (int base = 0; base < CHUNK; base += 32) {
        const int64_t f = f0 + base + lane;
        int e = -1;
        if (f < R) {
            e = idx[f];
            if (e < 0 || e >= E) e = -1;
        }
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0) {
            const int32_t row = cnt[e] + __popc(peers & lt);
            perm[row] = (int32_t)f;
            inv[f] = row;
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
        __syncwarp();
    }
}

// ---------------------------------------------------------------- tile lists
// One block per row window m: for each expert, the part of its rows inside [p0, p1) with
// p0 = first + m * span and p1 = min(p0 + span, last), cut into tiles of at most `chunk`
// rows (balanced heights, multiples of 16 but for the last), written in expert order to the
// window's list at list0 + m * stride. count at list[-4].
__global__ void __launch_bounds__(MAX_E)
    build_tiles(const int32_t *__restrict__ offsets, int E, int64_t first, int64_t span,
                int64_t last, int chunk, int32_t *__restrict__ list0, int64_t stride,
                int64_t cap, int *status) {
    __shared__ int32_t sc[MAX_E];
    const int e = threadIdx.x;
    const int64_t p0 = first + (int64_t)blockIdx.x * span;
    const int64_t p1 = p0 + span < last ? p0 + span : last;
    int32_t *__restrict__ list = list0 + (int64_t)blockIdx.x * stride;
    int64_t b = 0, end = 0, size = chunk;
    int32_t n = 0;
    if (e < E) {
        b = offsets[e];
        end = offsets[e + 1];
        if (b < p0) b = p0;
        if (end > p1) end = p1;
        if (end > b) {
            // balanced cut: as many tiles as chunk-sized tiles would need, of equal height
            // rounded up to 16 rows (the last one may be shorter)
            const int64_t len = end - b;
            const int64_t n0 = (len + chunk - 1) / chunk;
            size = (((len + n0 - 1) / n0) + 15) & ~(int64_t)15;
            if (size > chunk) size = chunk;
            n = (int32_t)((len + size - 1) / size);
        }
    }
    sc[e] = n;
    __syncthreads();
    for (int o = 1; o < MAX_E; o <<= 1) {
        const int32_t v = (e >= o) ? sc[e - o] : 0;
        __syncthreads();
        sc[e] += v;
        __syncthreads();
    }
    int64_t s = sc[e] - n;
    if (e == MAX_E - 1) {
        list[-4] = (int32_t)(sc[e] <= cap ? sc[e] : cap);
        if (sc[e] > cap) raise_status(status, MOK_ERR_DEVICE_INVARIANT);
    }
    for (int32_t q = 0; q < n; ++q, ++s) {
        const int64_t r0 = b + (int64_t)q * size;
        const int64_t r1 = (r0 + size < end) ? r0 + size : end;
        if (s < cap) {
            list[4 * s + 0] = e;
            list[4 * s + 1] = (int32_t)r0;
            list[4 * s + 2] = (int32_t)r1;
            list[4 * s + 3] = 0;
        }
    }
}

// poff[e] = sum over e' < e of roundup16(counts[e']); poff[E] = padded total
__global__ void __launch_bounds__(MAX_E)
    pad_offsets(const int32_t *__restrict__ counts, int E, int32_t *__restrict__ poff) {
    __shared__ int32_t sc[MAX_E];
    const int e = threadIdx.x;
    const int32_t c = (e < E) ? ((counts[e] + 15) & ~15) : 0;
    sc[e] = c;
    __syncthreads();
    for (int o = 1; o < MAX_E; o <<= 1) {
        const int32_t v = (e >= o) ? sc[e - o] : 0;
        __syncthreads();
        sc[e] += v;
        __syncthreads();
    }
    if (e < E) poff[e] = sc[e] - c;
    if (e == E - 1) poff[E] = sc[e];
}

}  // namespace

static int64_t n_chunks_of(int64_t R) { return (R + CHUNK - 1) / CHUNK; }

size_t schedule_ws_bytes(int64_t R, int E) {
    return (size_t)(n_chunks_of(R) > 0 ? n_chunks_of(R) : 1) * (size_t)E * sizeof(int32_t);
}

ScheduleWs schedule_ws_carve(void *ws, int64_t R, int E) {
    (void)E;
    ScheduleWs w;
    w.hist = (int32_t *)ws;
    w.n_chunks = n_chunks_of(R);
    return w;
}

cudaError_t launch_build_schedule(const int32_t *idx, int64_t R, int E, int MB,
                                  const mok_schedule &sch, const ScheduleWs &ws, int *status,
                                  cudaStream_t s) {
    const int64_t nc = ws.n_chunks;
    const size_t smem = (size_t)SCHED_WARPS * E * sizeof(int32_t);
    const unsigned blocks = (unsigned)((nc + SCHED_WARPS - 1) / SCHED_WARPS);
    const int64_t seg_cap = (int64_t)E + (R + MB - 1) / MB - 1 > 0
                                ? (int64_t)E + (R + MB - 1) / MB - 1
                                : 1;
    if (nc > 0) {
        sched_hist<<<blocks, SCHED_WARPS * 32, smem, s>>>(idx, R, E, nc, ws.hist, status);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        sched_colscan<<<(E + 31) / 32, 1024, 0, s>>>(ws.hist, E, nc, sch.counts);
    } else {
        cudaError_t err = cudaMemsetAsync(sch.counts, 0, sizeof(int32_t) * E, s);
        if (err != cudaSuccess) return err;
    }
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    sched_offsets<<<1, MAX_E, 0, s>>>(sch.counts, E, MB, seg_cap, sch.offsets, sch.segs,
                                      sch.n_segs, status);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (nc > 0) {
        sched_rank<<<blocks, SCHED_WARPS * 32, smem, s>>>(idx, R, E, nc, ws.hist, sch.offsets,
                                                         sch.perm, sch.inv);
        err = cudaGetLastError();
    }
    return err;
}

int64_t tile_list_cap(int64_t rows, int E, int chunk) {
    return (int64_t)E + (rows + chunk - 1) / chunk;
}

cudaError_t launch_build_tiles(const int32_t *offsets, int E, int64_t p0, int64_t p1, int chunk,
                               int32_t *list, int64_t cap, int *status, cudaStream_t s) {
    build_tiles<<<1, MAX_E, 0, s>>>(offsets, E, p0, p1 - p0, p1, chunk, list, 0, cap, status);
    return cudaGetLastError();
}

cudaError_t launch_pad_offsets(const int32_t *counts, int E, int32_t *poff, cudaStream_t s) {
    pad_offsets<<<1, MAX_E, 0, s>>>(counts, E, poff);
    return cudaGetLastError();
}

}  // namespace mok
