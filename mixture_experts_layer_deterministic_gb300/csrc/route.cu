// route.cu -- top-k routing over router logits.
//
// [alphalab] "Mixture-of-Kittens" analysis (alphalab.site), section 四: the benchmark routes
// by top-k over Gaussian router logits. Weights are a softmax over the chosen K logits.
//
// One warp per token. Each logit becomes a 64-bit key: an order-preserving image of the
// fp32 value (with -0 folded onto +0) in the high half and (2^32-1 - expert) in the low
// half, so the unsigned maximum is the largest logit and, among equal logits, the lowest
// expert id. Each lane keeps the maximum of its own keys; K rounds of a warp-wide maximum
// over those pick the experts in descending order, and only the lane that owned the
// winner retires it and rescans its keys. The chosen logit is read back from the key
// (the image inverts; -0 comes back as +0, which has the same exponential).
// HBM-bound: T*E*4 bytes read, T*K*8 bytes written.
#include "common.cuh"
#include "mok_internal.h"

namespace mok {
namespace {

MOK_DEV uint64_t logit_key(float v, uint32_t e) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0u;  // -0 ties with +0
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)ord << 32) | (uint64_t)(0xFFFFFFFFu - e);
}

MOK_DEV float key_logit(uint64_t key) {
    const uint32_t ord = (uint32_t)(key >> 32);
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

MOK_DEV uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = w > v ? w : v;
    }
    return v;
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
        uint64_t key[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = j * 32 + lane;  // coalesced: lanes read consecutive experts
            key[j] = (e < E) ? logit_key(__ldg(row + e), (uint32_t)e) : 0ull;
        }
        float sel_logit = 0.f;  // lane k keeps the k-th chosen logit
        int sel_e = 0;
        float first = 0.f;
        uint64_t mine = 0ull;  // this lane's largest remaining key
#pragma unroll
        for (int j = 0; j < PER; ++j) mine = key[j] > mine ? key[j] : mine;
        for (int k = 0; k < K; ++k) {
            const uint64_t best = warp_max_u64(mine);
            const uint32_t e = 0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull);
            // keys are unique: exactly one lane owns the winner; it retires it and rescans
            if (mine == best) {
                mine = 0ull;
#pragma unroll
                for (int j = 0; j < PER; ++j) {
                    if (key[j] == best) key[j] = 0ull;
                    mine = key[j] > mine ? key[j] : mine;
                }
            }
            const float lv = key_logit(best);
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
    if (blocks > 152 * 64) blocks = 152 * 64;
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
