// route.cu -- top-k routing over router logits.
//
// [alphalab] "Mixture-of-Kittens" analysis (alphalab.site), section 四: the benchmark routes
// by top-k over Gaussian router logits. Weights are a softmax over the chosen K logits.
//
// One warp per token; lane l holds the logits of experts 32j + l. Each logit becomes an
// unsigned order-preserving image of its fp32 value (-0 folded onto +0; every finite
// value maps above 0, which marks a retired or absent expert). Each lane keeps its largest
// remaining value, the lowest j among equal ones. A round takes the warp-wide maximum
// value with one integer reduction, then the lowest expert id among the lanes holding it
// with a second, so the experts come out by descending logit with ties to the lower id;
// only the winning lane retires that logit and rescans its own. The chosen logit is read
// back from its image (-0 comes back as +0, which has the same exponential).
// HBM-bound: T*E*4 bytes read, T*K*8 bytes written.
#include "common.cuh"
#include "mok_internal.h"

namespace mok {
namespace {

MOK_DEV uint32_t logit_order(float v) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0u;  // -0 ties with +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

MOK_DEV float order_logit(uint32_t ord) {
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

// PER = logits per lane (E <= 32 * PER)
template <int PER>
__global__ void __launch_bounds__(256) route_topk_kernel(const float *__restrict__ logits,
                                                         int64_t T, int E, int K,
                                                         int32_t *__restrict__ idx,
                                                         float *__restrict__ wout) {
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
         t += warps_total) {
        const float *row = logits + t * E;
        uint32_t v[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = j * 32 + lane;  // coalesced: lanes read consecutive experts
            v[j] = (e < E) ? logit_order(__ldg(row + e)) : 0u;
        }
        // this lane's largest remaining value and its slot (the lowest j among equals)
        uint32_t best = 0u;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if (v[j] > best) {
                best = v[j];
                bj = j;
            }
        float sel_logit = 0.f;  // lane k keeps the k-th chosen logit
        int sel_e = 0;
        float first = 0.f;
        for (int k = 0; k < K; ++k) {
            const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
            const uint32_t cand = best == top ? (uint32_t)(bj * 32 + lane) : 0xFFFFFFFFu;
            const uint32_t e = __reduce_min_sync(0xFFFFFFFFu, cand);
            if (cand == e) {  // the lane that held the winner retires it and rescans
#pragma unroll
                for (int j = 0; j < PER; ++j)
                    if (j == bj) v[j] = 0u;
                best = 0u;
                bj = 0;
#pragma unroll
                for (int j = 0; j < PER; ++j)
                    if (v[j] > best) {
                        best = v[j];
                        bj = j;
                    }
            }
            const float lv = order_logit(top);
            if (k == 0) first = lv;
            if (lane == k) {
                sel_logit = lv;
                sel_e = (int)e;
            }
        }
        // softmax over the chosen logits, shifted by the largest, summed in k order
        float den = 0.f;
        for (int k = 0; k < K; ++k) {
            const float lk = __shfl_sync(0xFFFFFFFFu, sel_logit, k);
            den += expf(lk - first);
        }
        if (lane < K) {
            idx[t * K + lane] = sel_e;
            wout[t * K + lane] = expf(sel_logit - first) / den;
        }
    }
}

template <int PER>
cudaError_t launch_per(const float *logits, int64_t T, int E, int K, int32_t *idx, float *w,
                       cudaStream_t s) {
    const int threads = 256;
    int64_t blocks = (T + 7) / 8;
    const int64_t cap = (int64_t)device_sm_count() * 64;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    route_topk_kernel<PER><<<(unsigned)blocks, threads, 0, s>>>(logits, T, E, K, idx, w);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route_topk(const float *logits, int64_t T, int E, int K, int32_t *idx,
                              float *w, int *status, cudaStream_t s) {
    (void)status;
    if (T == 0) return cudaSuccess;
    const int per = (E + 31) / 32;
    if (per <= 1) return launch_per<1>(logits, T, E, K, idx, w, s);
    if (per <= 2) return launch_per<2>(logits, T, E, K, idx, w, s);
    if (per <= 4) return launch_per<4>(logits, T, E, K, idx, w, s);
    if (per <= 8) return launch_per<8>(logits, T, E, K, idx, w, s);
    if (per <= 16) return launch_per<16>(logits, T, E, K, idx, w, s);
    return launch_per<32>(logits, T, E, K, idx, w, s);
}

}  // namespace mok
