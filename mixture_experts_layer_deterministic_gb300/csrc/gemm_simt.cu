// gemm_simt.cu -- grouped GEMMs of the layer on CUDA cores (fp32 FMA), with the fused
// epilogues of the forward and backward.
//
// [alphalab] "Mixture-of-Kittens" (alphalab.site), section 一: expert FFN with SwiGLU in the
// forward; reverse-combine, expert gradients and reverse-dispatch in the backward.
// [arex] "Cursor 放出 MoK" (arex-research.com), section "pull 代替 push": router-weight
// gradient computed inside the SwiGLU backward.
//
// Orientation: the weight dimension is M (tile 128) and the expert's routed rows are N
// (tile 64), so a tile never mixes experts and a ragged expert wastes at most 63 rows.
#include "common.cuh"
#include "mok_internal.h"

namespace mok {
namespace {

constexpr int BM = 128, BN = 64, BK = 16, NT = 256;

MOK_DEV float silu_f(float g) { return g / (1.0f + expf(-g)); }

struct Acc {
    float v[8][4];
};

// C[m][n] += sum_k A(m, k) * B(n, k) over k < klen; thread (tx = tid & 15, ty = tid >> 4)
// owns m = ty*8 + i, n = tx*4 + j.
template <class LA, class LB>
MOK_DEV void mainloop(Acc &acc, int klen, const LA &la, const LB &lb, float (*As)[BM],
                      float (*Bs)[BN]) {
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc.v[i][j] = 0.f;
    for (int k0 = 0; k0 < klen; k0 += BK) {
#pragma unroll
        for (int q = 0; q < (BM * BK) / NT; ++q) {
            const int id = tid + q * NT, m = id >> 4, kk = id & 15;
            As[kk][m] = (k0 + kk < klen) ? la(m, k0 + kk) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < (BN * BK) / NT; ++q) {
            const int id = tid + q * NT, n = id >> 4, kk = id & 15;
            Bs[kk][n] = (k0 + kk < klen) ? lb(n, k0 + kk) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[8], b[4];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = As[kk][ty * 8 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc.v[i][j] = fmaf(a[i], b[j], acc.v[i][j]);
        }
        __syncthreads();
    }
}

MOK_DEV void stage(const Acc &acc, float (*C)[BN + 1]) {
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) C[ty * 8 + i][tx * 4 + j] = acc.v[i][j];
    __syncthreads();
}

struct Smem {
    float As[BK][BM];
    float Bs[BK][BN];
    float C[BM][BN + 1];
};

MOK_DEV bool read_tile(const int32_t *tiles, int64_t cap, int *e, int64_t *r0, int64_t *r1) {
    const int64_t n = tiles[-4];
    if ((int64_t)blockIdx.x >= n || (int64_t)blockIdx.x >= cap) return false;
    *e = tiles[4 * blockIdx.x + 0];
    *r0 = tiles[4 * blockIdx.x + 1];
    *r1 = tiles[4 * blockIdx.x + 2];
    return true;
}

// operand element loaders ----------------------------------------------------------------
MOK_DEV float ld_bf16(const uint16_t *p) { return bf16_to_f32(*p); }
MOK_DEV float ld_mx(const uint8_t *q, const uint8_t *s, int64_t row, int ld, int64_t k) {
    return e4m3_to_f32(q[row * ld + k]) * mx_scale(s[row * (ld / 32) + k / 32]);
}

// ---------------------------------------------------------------- forward gate/up
// grid (tiles_cap, I/64); M tile = 64 gate rows + the matching 64 up rows.
__global__ void __launch_bounds__(NT) gemm_up_kernel(GemmUpArgs a) {
    __shared__ Smem sm;
    int e;
    int64_t r0, r1;
    if (!read_tile(a.tiles, a.tiles_cap, &e, &r0, &r1)) return;
    const int H = a.H, I = a.I, i0 = blockIdx.y * 64;
    const int nr = (int)(r1 - r0);
    RingMap rm{a.ring.R, a.ring.MB, a.ring.n_slots};
    auto jrow = [&](int m) { return m < 64 ? i0 + m : I + i0 + m - 64; };
    Acc acc;
    if (!a.mxfp8) {
        const uint16_t *W = (const uint16_t *)a.w13 + (int64_t)e * 2 * I * H;
        const uint16_t *X = (const uint16_t *)a.xring;
        mainloop(
            acc, H, [&](int m, int k) { return ld_bf16(W + (int64_t)jrow(m) * H + k); },
            [&](int n, int k) { return n < nr ? ld_bf16(X + rm(r0 + n) * H + k) : 0.f; },
            sm.As, sm.Bs);
    } else {
        const uint8_t *Wq = (const uint8_t *)a.w13 + (int64_t)e * 2 * I * H;
        const uint8_t *Ws = a.w13_s + (int64_t)e * 2 * I * (H / 32);
        const uint8_t *Xq = (const uint8_t *)a.xring;
        mainloop(
            acc, H, [&](int m, int k) { return ld_mx(Wq, Ws, jrow(m), H, k); },
            [&](int n, int k) { return n < nr ? ld_mx(Xq, a.xring_s, rm(r0 + n), H, k) : 0.f; },
            sm.As, sm.Bs);
    }
    stage(acc, sm.C);
    const int tid = threadIdx.x;
    if (a.preact != nullptr) {
        for (int id = tid; id < BM * nr; id += NT) {
            const int n = id / BM, m = id % BM;
            a.preact[(r0 + n) * 2 * I + jrow(m)] = sm.C[m][n];
        }
    }
    if (!a.mxfp8) {
        uint16_t *Hb = (uint16_t *)a.hring;
        for (int id = tid; id < 64 * nr; id += NT) {
            const int n = id / 64, il = id % 64;
            const float h = silu_f(sm.C[il][n]) * sm.C[64 + il][n];
            Hb[rm(r0 + n) * I + i0 + il] = f32_to_bf16(h);
        }
    } else {
        // each (row, 32-block) pair: 32 h values -> E4M3 codes + E8M0 scale
        uint8_t *Hq = (uint8_t *)a.hring;
        for (int id = tid; id < 2 * nr; id += NT) {
            const int n = id >> 1, b = id & 1;
            float hv[32];
            float amax = 0.f;
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int il = b * 32 + q;
                hv[q] = silu_f(sm.C[il][n]) * sm.C[64 + il][n];
                amax = fmaxf(amax, fabsf(hv[q]));
            }
            const uint32_t sb = mx_scale_byte(amax);
            const float inv = mx_inv_scale(sb);
            const int64_t slot = rm(r0 + n);
            uint8_t *dst = Hq + slot * I + i0 + b * 32;
#pragma unroll
            for (int q = 0; q < 32; q += 2) {
                const uint32_t c = e4m3x2(hv[q] * inv, hv[q + 1] * inv);
                dst[q] = (uint8_t)(c & 0xFF);
                dst[q + 1] = (uint8_t)(c >> 8);
            }
            a.hring_s[slot * (I / 32) + (i0 / 32) + b] = (uint8_t)sb;
        }
    }
}

// ---------------------------------------------------------------- forward down + push
// grid (tiles_cap, H/128)
__global__ void __launch_bounds__(NT) gemm_down_kernel(GemmDownArgs a) {
    __shared__ Smem sm;
    int e;
    int64_t r0, r1;
    if (!read_tile(a.tiles, a.tiles_cap, &e, &r0, &r1)) return;
    const int H = a.H, I = a.I, c0 = blockIdx.y * BM;
    const int nr = (int)(r1 - r0);
    RingMap rm{a.ring.R, a.ring.MB, a.ring.n_slots};
    Acc acc;
    if (!a.mxfp8) {
        const uint16_t *W = (const uint16_t *)a.w2 + (int64_t)e * H * I;
        const uint16_t *Hb = (const uint16_t *)a.hring;
        mainloop(
            acc, I, [&](int m, int k) { return ld_bf16(W + (int64_t)(c0 + m) * I + k); },
            [&](int n, int k) { return n < nr ? ld_bf16(Hb + rm(r0 + n) * I + k) : 0.f; },
            sm.As, sm.Bs);
    } else {
        const uint8_t *Wq = (const uint8_t *)a.w2 + (int64_t)e * H * I;
        const uint8_t *Ws = a.w2_s + (int64_t)e * H * (I / 32);
        const uint8_t *Hq = (const uint8_t *)a.hring;
        mainloop(
            acc, I, [&](int m, int k) { return ld_mx(Wq, Ws, c0 + m, I, k); },
            [&](int n, int k) { return n < nr ? ld_mx(Hq, a.hring_s, rm(r0 + n), I, k) : 0.f; },
            sm.As, sm.Bs);
    }
    stage(acc, sm.C);
    for (int id = threadIdx.x; id < BM * nr; id += NT) {
        const int n = id / BM, m = id % BM;
        const int64_t f = a.perm[r0 + n];
        a.slots[f * H + c0 + m] = sm.C[m][n];
    }
}

// ---------------------------------------------------------------- backward G + SwiGLU bwd
// grid (tiles_cap, I/128)
__global__ void __launch_bounds__(NT) gemm_g_kernel(GemmGArgs a) {
    __shared__ Smem sm;
    int e;
    int64_t r0, r1;
    if (!read_tile(a.tiles, a.tiles_cap, &e, &r0, &r1)) return;
    const int H = a.H, I = a.I, i0 = blockIdx.y * BM;
    const int nr = (int)(r1 - r0);
    const int64_t oe = a.offsets[e], pe = a.poff[e];
    const int64_t pbase = pe + (r0 - oe);
    const uint16_t *W = a.w2 + (int64_t)e * H * I;
    const uint16_t *D = a.dy_perm;
    Acc acc;
    mainloop(
        acc, H, [&](int m, int k) { return ld_bf16(W + (int64_t)k * I + i0 + m); },
        [&](int n, int k) { return n < nr ? ld_bf16(D + (pbase + n) * H + k) : 0.f; }, sm.As,
        sm.Bs);
    stage(acc, sm.C);
    const int tid = threadIdx.x;
    for (int id = tid; id < BM * nr; id += NT) {
        const int n = id / BM, m = id % BM;
        const int64_t r = r0 + n, p = pbase + n;
        const int i = i0 + m;
        const float ag = a.preact[r * 2 * I + i];
        const float au = a.preact[r * 2 * I + I + i];
        const float s = a.topk_w[a.perm[r]];
        const float g = sm.C[m][n];
        const float sig = 1.0f / (1.0f + expf(-ag));
        const float sl = ag * sig;
        const float h = sl * au;
        const float dh = s * g;
        a.dA[p * 2 * I + i] = f32_to_bf16(dh * au * sig * (1.0f + ag * (1.0f - sig)));
        a.dA[p * 2 * I + I + i] = f32_to_bf16(dh * sl);
        a.sh[p * I + i] = f32_to_bf16(s * h);
        sm.C[m][n] = g * h;
    }
    // pad rows after the expert's last row, up to the next multiple of 16
    if (r1 == a.offsets[e + 1]) {
        const int npad = ((nr + 15) & ~15) - nr;
        for (int id = tid; id < BM * npad; id += NT) {
            const int n = nr + id / BM, m = id % BM;
            const int64_t p = pbase + n;
            a.dA[p * 2 * I + i0 + m] = 0;
            a.dA[p * 2 * I + I + i0 + m] = 0;
            a.sh[p * I + i0 + m] = 0;
        }
    }
    __syncthreads();
    const int n_parts = I / BM;
    for (int n = tid; n < nr; n += NT) {
        float d = 0.f;
        for (int m = 0; m < BM; ++m) d += sm.C[m][n];
        a.dS_part[(r0 + n) * n_parts + blockIdx.y] = d;
    }
}

// ---------------------------------------------------------------- backward dgrad + push
// grid (tiles_cap, H/128)
__global__ void __launch_bounds__(NT) gemm_dgrad_kernel(GemmDgradArgs a) {
    __shared__ Smem sm;
    int e;
    int64_t r0, r1;
    if (!read_tile(a.tiles, a.tiles_cap, &e, &r0, &r1)) return;
    const int H = a.H, I = a.I, c0 = blockIdx.y * BM;
    const int nr = (int)(r1 - r0);
    const int64_t pbase = a.poff[e] + (r0 - a.offsets[e]);
    const uint16_t *W = a.w13 + (int64_t)e * 2 * I * H;
    Acc acc;
    mainloop(
        acc, 2 * I, [&](int m, int k) { return ld_bf16(W + (int64_t)k * H + c0 + m); },
        [&](int n, int k) { return n < nr ? ld_bf16(a.dA + (pbase + n) * 2 * I + k) : 0.f; },
        sm.As, sm.Bs);
    stage(acc, sm.C);
    for (int id = threadIdx.x; id < BM * nr; id += NT) {
        const int n = id / BM, m = id % BM;
        const int64_t f = a.perm[r0 + n];
        a.dx_slots[f * H + c0 + m] = sm.C[m][n];
    }
}

// ---------------------------------------------------------------- weight gradients
// grid (E, M/128, N/64)
__global__ void __launch_bounds__(NT) gemm_wgrad_kernel(GemmWgradArgs a) {
    __shared__ Smem sm;
    const int e = blockIdx.x, m0 = blockIdx.y * BM, n0 = blockIdx.z * BN;
    const int M = a.M, N = a.N;
    const int klen = (a.counts[e] + 15) & ~15;
    const int64_t pb = a.poff[e];
    Acc acc;
    mainloop(
        acc, klen, [&](int m, int k) { return ld_bf16(a.A + (pb + k) * M + m0 + m); },
        [&](int n, int k) { return ld_bf16(a.B + (pb + k) * N + n0 + n); }, sm.As, sm.Bs);
    stage(acc, sm.C);
    float *out = a.out + (int64_t)e * M * N;
    for (int id = threadIdx.x; id < BM * BN; id += NT) {
        const int m = id / BN, n = id % BN;
        out[(int64_t)(m0 + m) * N + n0 + n] = sm.C[m][n];
    }
}

}  // namespace

// tiles for these kernels are cut at BN rows
int gemm_tile_rows() { return BN; }

cudaError_t launch_gemm_up(const GemmUpArgs &a, cudaStream_t s) {
    if (a.tiles_cap == 0) return cudaSuccess;
    gemm_up_kernel<<<dim3((unsigned)a.tiles_cap, a.I / 64), NT, 0, s>>>(a);
    return cudaGetLastError();
}
cudaError_t launch_gemm_down(const GemmDownArgs &a, cudaStream_t s) {
    if (a.tiles_cap == 0) return cudaSuccess;
    gemm_down_kernel<<<dim3((unsigned)a.tiles_cap, a.H / BM), NT, 0, s>>>(a);
    return cudaGetLastError();
}
cudaError_t launch_gemm_g(const GemmGArgs &a, cudaStream_t s) {
    if (a.tiles_cap == 0) return cudaSuccess;
    gemm_g_kernel<<<dim3((unsigned)a.tiles_cap, a.I / BM), NT, 0, s>>>(a);
    return cudaGetLastError();
}
cudaError_t launch_gemm_dgrad(const GemmDgradArgs &a, cudaStream_t s) {
    if (a.tiles_cap == 0) return cudaSuccess;
    gemm_dgrad_kernel<<<dim3((unsigned)a.tiles_cap, a.H / BM), NT, 0, s>>>(a);
    return cudaGetLastError();
}
cudaError_t launch_gemm_wgrad(const GemmWgradArgs &a, cudaStream_t s) {
    if (a.E == 0) return cudaSuccess;
    gemm_wgrad_kernel<<<dim3(a.E, a.M / BM, a.N / BN), NT, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace mok
