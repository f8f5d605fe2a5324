// dispatch.cu -- HBM-bound steps: pull dispatch, push-combine reduction, their backward
// twins, MXFP8 quantization and the router gradient.
//
// [arex] "Cursor 放出 MoK：NVL72 训练提速 2.37 倍" (arex-research.com), section "pull 代替
// push": the receiver pulls token rows into expert order (dispatch), results go back to
// their source (combine), and the backward uses the same schedule in reverse; MXFP8
// activation quantization is fused into dispatch. [alphalab] "Mixture-of-Kittens"
// (alphalab.site), section 二: a final router-weighted reduction follows combine; section
// 六: a fixed accumulation order makes results bitwise reproducible.
#include "common.cuh"
#include "mok_internal.h"

namespace mok {
namespace {

constexpr int TPB = 256;

// blocks for `items` work items at `per_block` items per block (grid-stride loops), capped
// at `per_sm` blocks per streaming multiprocessor of the device
inline unsigned grid_for(int64_t items, int per_block, int per_sm = 32) {
    const int64_t cap = (int64_t)device_sm_count() * per_sm;
    int64_t b = (items + per_block - 1) / per_block;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return (unsigned)b;
}

// ---------------------------------------------------------------- BF16 gather
// Token-major, into a ring that holds every row (slot r = r): one warp per token t reads
// x[t] once and writes it to the ring rows inv[t*K + k] of its K routed copies. Reading
// each token row once keeps the gather at the bytes it must write, where the sorted-order
// form re-reads every row K times from scattered positions.
__global__ void __launch_bounds__(TPB)
    gather_tok_bf16_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ inv,
                           int64_t T, int K, int H, uint16_t *__restrict__ ring) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (TPB / 32);
    const int nv = H / 8;
    for (int64_t t = (int64_t)blockIdx.x * (TPB / 32) + (threadIdx.x >> 5); t < T; t += nw) {
        const int32_t rk = lane < K ? inv[t * K + lane] : 0;  // K <= 32
        const uint4 *src = reinterpret_cast<const uint4 *>(x + t * H);
        for (int v0 = 0; v0 < nv; v0 += 32 * 16) {
            uint4 b[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int v = v0 + j * 32 + lane;
                if (v < nv) b[j] = ldg_nc_v4(src + v);
            }
            for (int k = 0; k < K; ++k) {
                const int64_t r = __shfl_sync(0xFFFFFFFFu, rk, k);
                uint4 *dst = reinterpret_cast<uint4 *>(ring + r * H);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int v = v0 + j * 32 + lane;
                    if (v < nv) dst[v] = b[j];
                }
            }
        }
    }
}

// ---------------------------------------------------------------- MXFP8 quantizer
// One 32-element bf16 block -> 32 E4M3 bytes (out[8]) and its E8M0 byte.
MOK_DEV uint32_t quant_block32_regs(const uint16_t *__restrict__ src, uint32_t (&out)[8]) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = ldg_nc_v4(src + 8 * j);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(v);
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    const uint32_t sb = mx_scale_byte(amax);
    const float inv = mx_inv_scale(sb);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t a = e4m3x2(bf16_lo(w[2 * j]) * inv, bf16_hi(w[2 * j]) * inv);
        const uint32_t b = e4m3x2(bf16_lo(w[2 * j + 1]) * inv, bf16_hi(w[2 * j + 1]) * inv);
        out[j] = a | (b << 16);
    }
    return sb;
}

MOK_DEV void quant_block32(const uint16_t *__restrict__ src, uint8_t *__restrict__ q,
                           uint8_t *__restrict__ sbyte) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = ldg_nc_v4(src + 8 * j);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(v);
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    const uint32_t sb = mx_scale_byte(amax);
    const float inv = mx_inv_scale(sb);
    uint32_t out[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t a = e4m3x2(bf16_lo(w[2 * j]) * inv, bf16_hi(w[2 * j]) * inv);
        const uint32_t b = e4m3x2(bf16_lo(w[2 * j + 1]) * inv, bf16_hi(w[2 * j + 1]) * inv);
        out[j] = a | (b << 16);
    }
    uint4 *qd = reinterpret_cast<uint4 *>(q);
    qd[0] = make_uint4(out[0], out[1], out[2], out[3]);
    qd[1] = make_uint4(out[4], out[5], out[6], out[7]);
    *sbyte = (uint8_t)sb;
}

// Along rows, stored transposed: one thread per (matrix b, column c, 32-row block j); the
// block src[b][32j..32j+31][c] (neighbouring threads read neighbouring columns) becomes
// q[b][c][32j..32j+31] and scale[b][c][j].
__global__ void __launch_bounds__(TPB)
    quantize_transposed_kernel(const uint16_t *__restrict__ src, int64_t batch, int rows,
                               int cols, uint8_t *__restrict__ q, uint8_t *__restrict__ sc) {
    const int nb = rows / 32;
    const int64_t total = batch * nb * cols;
    const int64_t stride = (int64_t)gridDim.x * TPB;
    for (int64_t i = (int64_t)blockIdx.x * TPB + threadIdx.x; i < total; i += stride) {
        const int c = (int)(i % cols);
        const int j = (int)((i / cols) % nb);
        const int64_t b = i / ((int64_t)cols * nb);
        const uint16_t *s0 = src + (b * rows + (int64_t)j * 32) * cols + c;
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
            w[k] = (uint32_t)__ldg(s0 + (int64_t)(2 * k) * cols) |
                   ((uint32_t)__ldg(s0 + (int64_t)(2 * k + 1) * cols) << 16);
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
        const uint32_t sb = mx_scale_byte(amax);
        const float inv = mx_inv_scale(sb);
        uint32_t out[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t a = e4m3x2(bf16_lo(w[2 * k]) * inv, bf16_hi(w[2 * k]) * inv);
            const uint32_t bb = e4m3x2(bf16_lo(w[2 * k + 1]) * inv, bf16_hi(w[2 * k + 1]) * inv);
            out[k] = a | (bb << 16);
        }
        uint4 *qd = reinterpret_cast<uint4 *>(q + (b * cols + c) * (int64_t)rows + j * 32);
        qd[0] = make_uint4(out[0], out[1], out[2], out[3]);
        qd[1] = make_uint4(out[4], out[5], out[6], out[7]);
        sc[(b * cols + c) * (int64_t)nb + j] = (uint8_t)sb;
    }
}

// Token-major form (ring holds every row): one thread per 32-element block of token t,
// quantized once and written to the ring rows of its K routed copies.
__global__ void __launch_bounds__(TPB)
    gather_tok_mxfp8_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ inv,
                            int64_t T, int K, int H, uint8_t *__restrict__ rq,
                            uint8_t *__restrict__ rs) {
    const int nb = H / 32;
    const int64_t total = T * nb;
    const int64_t stride = (int64_t)gridDim.x * TPB;
    for (int64_t i = (int64_t)blockIdx.x * TPB + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / nb;
        const int b = (int)(i % nb);
        uint32_t out[8];
        const uint32_t sb = quant_block32_regs(x + t * H + b * 32, out);
        for (int k = 0; k < K; ++k) {
            const int64_t r = __ldg(inv + t * K + k);
            uint4 *qd = reinterpret_cast<uint4 *>(rq + r * H + b * 32);
            qd[0] = make_uint4(out[0], out[1], out[2], out[3]);
            qd[1] = make_uint4(out[4], out[5], out[6], out[7]);
            rs[r * nb + b] = (uint8_t)sb;
        }
    }
}

__global__ void __launch_bounds__(TPB)
    quantize_kernel(const uint16_t *__restrict__ src, int64_t rows, int cols,
                    uint8_t *__restrict__ q, uint8_t *__restrict__ sc) {
    const int nb = cols / 32;
    const int64_t total = rows * nb;
    const int64_t stride = (int64_t)gridDim.x * TPB;
    for (int64_t i = (int64_t)blockIdx.x * TPB + threadIdx.x; i < total; i += stride) {
        const int64_t r = i / nb;
        const int b = (int)(i % nb);
        quant_block32(src + r * cols + b * 32, q + r * cols + b * 32, sc + r * nb + b);
    }
}

// ---------------------------------------------------------------- combine
// y[t][c..c+3] = sum over k = 0..K-1 of w[t,k] * slots[t*K+k][c..c+3] in fp32, k ascending
// (fmaf from zero); w == nullptr sums with weight one.
// y[t] = sum over k ascending of w[t,k] * slots[t*K + k], fp32 fused multiply-adds; each
// thread owns 4 (fp32) or 8 (bf16) consecutive columns and reads every slot with one
// 16-byte load. bf16 storage rounds y once, after the sum.
template <bool F32>
__global__ void __launch_bounds__(TPB)
    combine_kernel(const void *__restrict__ slots, const float *__restrict__ w, int64_t T,
                   int K, int H, void *__restrict__ y) {
    constexpr int PER = F32 ? 4 : 8;  // columns per thread
    const int nv = H / PER;
    const int64_t total = T * nv;
    const int64_t stride = (int64_t)gridDim.x * TPB;
    for (int64_t i = (int64_t)blockIdx.x * TPB + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / nv;
        const int v = (int)(i % nv);
        float acc[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) acc[q] = 0.f;
        for (int k = 0; k < K; ++k) {
            const int64_t f = t * K + k;
            const float s = (w != nullptr) ? __ldg(w + f) : 1.0f;
            const uint4 o = ldg_nc_v4(static_cast<const uint8_t *>(slots) +
                                      (f * H + (int64_t)v * PER) * (F32 ? 4 : 2));
            const uint32_t u[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (F32) {
                    acc[q] = fmaf(s, __uint_as_float(u[q]), acc[q]);
                } else {
                    acc[2 * q] = fmaf(s, bf16_lo(u[q]), acc[2 * q]);
                    acc[2 * q + 1] = fmaf(s, bf16_hi(u[q]), acc[2 * q + 1]);
                }
            }
        }
        uint4 r;
        if (F32) {
            r = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                           __float_as_uint(acc[2]), __float_as_uint(acc[3]));
        } else {
            r = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                           pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
        }
        *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(y) +
                                   (t * H + (int64_t)v * PER) * (F32 ? 4 : 2)) = r;
    }
}

// ---------------------------------------------------------------- backward gather
// Padded row space: expert e owns rows [poff[e], poff[e+1]) with its counts[e] real rows
// first and zero rows after; sorted row r of expert e sits at poff[e] + r - offsets[e].
// One warp per token t reads dy[t] and x[t] once and writes them to the padded rows of its
// K routed copies (the row of copy k found from inv[t*K + k] by binary search over the
// expert offsets: the last e with offsets[e] <= r, which skips empty experts).
__global__ void __launch_bounds__(TPB)
    gather_bwd_kernel(const uint16_t *__restrict__ dy, const uint16_t *__restrict__ x,
                      const int32_t *__restrict__ inv, const int32_t *__restrict__ offsets,
                      const int32_t *__restrict__ poff, int E, int64_t T, int K, int H,
                      uint16_t *__restrict__ dyp, uint16_t *__restrict__ xp,
                      int32_t *__restrict__ prow) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (TPB / 32);
    const int nv = H / 8;
    for (int64_t t = (int64_t)blockIdx.x * (TPB / 32) + (threadIdx.x >> 5); t < T; t += nw) {
        int64_t pk = 0;
        if (lane < K) {
            const int32_t r = inv[t * K + lane];
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
            }
            pk = poff[lo] + (int64_t)(r - offsets[lo]);
            if (prow != nullptr) prow[t * K + lane] = (int32_t)pk;
        }
        for (int which = 0; which < 2; ++which) {
            const uint4 *src = reinterpret_cast<const uint4 *>((which ? x : dy) + t * H);
            uint16_t *dbase = which ? xp : dyp;
            for (int v0 = 0; v0 < nv; v0 += 32 * 16) {
                uint4 b[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int v = v0 + j * 32 + lane;
                    if (v < nv) b[j] = ldg_nc_v4(src + v);
                }
                for (int k = 0; k < K; ++k) {
                    const int64_t p = __shfl_sync(0xFFFFFFFFu, pk, k);
                    uint4 *dst = reinterpret_cast<uint4 *>(dbase + p * H);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int v = v0 + j * 32 + lane;
                        if (v < nv) dst[v] = b[j];
                    }
                }
            }
        }
    }
}

// MXFP8 backward: dy quantized along H into the padded layout, one thread per 32-element
// block of token t, quantized once and written to the padded rows prow[t*K + k] of its K
// routed copies.
__global__ void __launch_bounds__(TPB)
    quantize_dy_padded_kernel(const uint16_t *__restrict__ dy, const int32_t *__restrict__ prow,
                              int64_t T, int K, int H, uint8_t *__restrict__ q,
                              uint8_t *__restrict__ sc) {
    const int nb = H / 32;
    const int64_t total = T * nb;
    const int64_t stride = (int64_t)gridDim.x * TPB;
    for (int64_t i = (int64_t)blockIdx.x * TPB + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / nb;
        const int b = (int)(i % nb);
        uint32_t out[8];
        const uint32_t sb = quant_block32_regs(dy + t * H + b * 32, out);
        for (int k = 0; k < K; ++k) {
            const int64_t p = __ldg(prow + t * K + k);
            uint4 *qd = reinterpret_cast<uint4 *>(q + p * H + b * 32);
            qd[0] = make_uint4(out[0], out[1], out[2], out[3]);
            qd[1] = make_uint4(out[4], out[5], out[6], out[7]);
            sc[p * nb + b] = (uint8_t)sb;
        }
    }
}

// The pad rows of every expert (at most 15) are zero in both padded arrays: one warp per
// (expert, pad row).
__global__ void __launch_bounds__(TPB)
    zero_pad_rows_kernel(const int32_t *__restrict__ counts, const int32_t *__restrict__ poff,
                         int E, int H, uint16_t *__restrict__ dyp, uint16_t *__restrict__ xp,
                         uint8_t *__restrict__ dyq, uint8_t *__restrict__ dys) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (TPB / 32);
    const int nv = H / 8;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t w = (int64_t)blockIdx.x * (TPB / 32) + (threadIdx.x >> 5); w < (int64_t)E * 16;
         w += nw) {
        const int e = (int)(w / 16), j = (int)(w % 16);
        const int64_t p = poff[e] + counts[e] + j;
        if (p >= poff[e + 1]) continue;
        uint4 *d0 = reinterpret_cast<uint4 *>(dyp + p * H);
        uint4 *d1 = reinterpret_cast<uint4 *>(xp + p * H);
        for (int v = lane; v < nv; v += 32) {
            d0[v] = z;
            d1[v] = z;
        }
        if (dyq != nullptr) {  // MXFP8 copy of dy: E4M3 bytes and scale bytes
            uint4 *d2 = reinterpret_cast<uint4 *>(dyq + p * H);
            for (int v = lane; v < H / 16; v += 32) d2[v] = z;
            for (int v = lane; v < H / 32; v += 32) dys[p * (H / 32) + v] = 0;
        }
    }
}

// ---------------------------------------------------------------- router gradient
// One warp per token. dS of routed id f is the fixed-order sum of its per-feature-block
// partials; d_topk = dS; d_logits through the top-k softmax (zero for unchosen logits).
__global__ void __launch_bounds__(TPB)
    router_grad_kernel(const float *__restrict__ part, int n_parts, const int32_t *__restrict__ inv,
                       const int32_t *__restrict__ offsets, const float *__restrict__ w,
                       int64_t T, int K, int E, float *__restrict__ d_topk,
                       float *__restrict__ d_logits) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (TPB / 32);
    for (int64_t t = (int64_t)blockIdx.x * (TPB / 32) + (threadIdx.x >> 5); t < T; t += nw) {
        float dS = 0.f, wk = 0.f;
        int ek = 0;
        if (lane < K) {
            const int64_t f = t * K + lane;
            const int64_t r = inv[f];
            for (int j = 0; j < n_parts; ++j) dS += part[r * n_parts + j];
            d_topk[f] = dS;
            wk = w[f];
            // expert of sorted row r: last e with offsets[e] <= r
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
            }
            ek = lo;
        }
        if (d_logits == nullptr) continue;
        float sw = 0.f;
        for (int k = 0; k < K; ++k) sw += __shfl_sync(0xFFFFFFFFu, wk * dS, k);
        float *dl = d_logits + t * E;
        for (int e = lane; e < E; e += 32) dl[e] = 0.f;
        __syncwarp();
        if (lane < K) dl[ek] = wk * (dS - sw);
        __syncwarp();
    }
}

// ---------------------------------------------------------------- MXFP8 scale atoms
// The tensor cores read an operand's E8M0 scales as atoms of 128 rows x 4 K-blocks (512
// bytes: 32 rows of 16 bytes, row i holding the 4 scales of rows i, i+32, i+64, i+96).
// Weights: plain [rows][K/32] -> atom (row/128, kg) at ((row/128) * K/128 + kg) * 512.
// Token tiles: the rows n < 128 of tile t = (e, r0, r1) (rows past the tile get byte 0) ->
// one atom per 128-wide K block at (t * K/128 + kg) * 512; sorted row r sits at ring slot
// rm(r), or, with poff (the backward's padded layout), at poff[e] + r - offsets[e].
//
// Both go through shared memory: one block iteration loads the scales of 128 rows x 8 K
// groups (32 bytes per row, 16-byte loads) and writes the 8 atoms with 16-byte stores, so
// neither side is a scatter of 4-byte accesses.
constexpr int ATOM_KG = 8;  // K groups (atoms) per block iteration

struct AtomRows {  // where row n of atom row-block b starts in the source (-1: absent)
    const int32_t *tiles;   // nullptr: plain rows
    int64_t rows;
    RingMap rm;
    const int32_t *offsets, *poff;
    MOK_DEV int64_t operator()(int64_t b, int n, int rowbytes) const {
        if (tiles == nullptr) {
            const int64_t r = b * 128 + n;
            return r < rows ? r * rowbytes : -1;
        }
        const int64_t r0 = tiles[4 * b + 1], r1 = tiles[4 * b + 2];
        if (n >= r1 - r0) return -1;
        const int e = tiles[4 * b];
        const int64_t row = poff != nullptr ? poff[e] + (r0 - offsets[e]) + n : rm(r0 + n);
        return row * rowbytes;
    }
};

__global__ void __launch_bounds__(256)
    scale_atoms_kernel(const uint8_t *__restrict__ src, int64_t n_blocks, int64_t cap, int K,
                       AtomRows where, uint8_t *__restrict__ dst) {
    __shared__ __align__(16) uint8_t tile[128][ATOM_KG * 4];
    const int kgn = K / 128, rowbytes = K / 32;
    const int nkc = (kgn + ATOM_KG - 1) / ATOM_KG;
    int64_t nb = n_blocks;
    if (where.tiles != nullptr) nb = where.tiles[-4] < cap ? where.tiles[-4] : cap;
    for (int64_t it = blockIdx.x; it < nb * nkc; it += gridDim.x) {
        const int64_t b = it / nkc;
        const int kc = (int)(it % nkc);
        const int nkg = kgn - kc * ATOM_KG < ATOM_KG ? kgn - kc * ATOM_KG : ATOM_KG;
        {  // 128 rows x (4 * nkg) bytes: two threads per row, 16 bytes each
            const int n = threadIdx.x >> 1, half = threadIdx.x & 1;
            const int64_t at = where(b, n, rowbytes);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (at >= 0 && half * 16 < nkg * 4) {
                const uint8_t *sp = src + at + kc * ATOM_KG * 4 + half * 16;
                const int left = nkg * 4 - half * 16;  // bytes of this row in the patch
                // 16-byte loads only where every row starts on a 16-byte boundary (a row
                // is K/32 bytes, a multiple of 4); else 4-byte loads
                if (left >= 16 && rowbytes % 16 == 0) {
                    v = *reinterpret_cast<const uint4 *>(sp);
                } else {
                    uint32_t w[4] = {0, 0, 0, 0};
                    const int nw = left < 16 ? left / 4 : 4;
                    for (int q = 0; q < nw; ++q)
                        w[q] = *reinterpret_cast<const uint32_t *>(sp + 4 * q);
                    v = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            *reinterpret_cast<uint4 *>(&tile[n][half * 16]) = v;
        }
        __syncthreads();
        {  // atom a (K group kc*8 + a), its 16-byte row r16: scales of rows r16 + 32j
            const int a = threadIdx.x >> 5, r16 = threadIdx.x & 31;
            if (a < nkg) {
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    w[j] = *reinterpret_cast<const uint32_t *>(&tile[r16 + 32 * j][a * 4]);
                uint8_t *o = dst + (b * kgn + kc * ATOM_KG + a) * 512 + r16 * 16;
                *reinterpret_cast<uint4 *>(o) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        __syncthreads();
    }
}

}  // namespace

__global__ void single_expert_offsets_kernel(int32_t *off, int64_t rows) {
    off[0] = 0;
    off[1] = (int32_t)rows;
}

cudaError_t launch_single_expert_offsets(int32_t *off, int64_t rows, cudaStream_t s) {
    single_expert_offsets_kernel<<<1, 1, 0, s>>>(off, rows);
    return cudaGetLastError();
}

__global__ void __launch_bounds__(TPB)
    single_expert_bwd_setup_kernel(int32_t *offsets, int32_t *poff, int32_t *counts,
                                   float *ones, int32_t *perm, int64_t T) {
    const int64_t i = (int64_t)blockIdx.x * TPB + threadIdx.x;
    if (i < T) {
        ones[i] = 1.0f;
        perm[i] = (int32_t)i;
    }
    if (i == 0) {
        offsets[0] = 0;
        offsets[1] = (int32_t)T;
        poff[0] = 0;
        poff[1] = (int32_t)((T + 15) & ~(int64_t)15);
        counts[0] = (int32_t)T;
    }
}

cudaError_t launch_single_expert_bwd_setup(int32_t *offsets, int32_t *poff, int32_t *counts,
                                           float *ones, int32_t *perm, int64_t T,
                                           cudaStream_t s) {
    single_expert_bwd_setup_kernel<<<(unsigned)((T + TPB - 1) / TPB > 0 ? (T + TPB - 1) / TPB
                                                                          : 1),
                                     TPB, 0, s>>>(offsets, poff, counts, ones, perm, T);
    return cudaGetLastError();
}

cudaError_t launch_gather_tok_bf16(const uint16_t *x, const int32_t *inv, int64_t T, int K,
                                   int H, uint16_t *ring, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    gather_tok_bf16_kernel<<<grid_for(T, TPB / 32, 16), TPB, 0, s>>>(x, inv, T, K, H,
                                                                           ring);
    return cudaGetLastError();
}

cudaError_t launch_gather_tok_mxfp8(const uint16_t *x, const int32_t *inv, int64_t T, int K,
                                    int H, uint8_t *ring_q, uint8_t *ring_s, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    gather_tok_mxfp8_kernel<<<grid_for(T * (H / 32), TPB, 16), TPB, 0, s>>>(
        x, inv, T, K, H, ring_q, ring_s);
    return cudaGetLastError();
}

cudaError_t launch_quantize_mxfp8(const uint16_t *src, int64_t rows, int cols, uint8_t *q,
                                  uint8_t *scale, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    quantize_kernel<<<grid_for(rows * (cols / 32), TPB, 16), TPB, 0, s>>>(src, rows, cols,
                                                                                q, scale);
    return cudaGetLastError();
}

cudaError_t launch_quantize_mxfp8_transposed(const uint16_t *src, int64_t batch, int rows,
                                             int cols, uint8_t *q, uint8_t *scale,
                                             cudaStream_t s) {
    if (batch == 0 || rows == 0 || cols == 0) return cudaSuccess;
    quantize_transposed_kernel<<<grid_for(batch * (rows / 32) * cols, TPB, 16), TPB, 0,
                                 s>>>(src, batch, rows, cols, q, scale);
    return cudaGetLastError();
}

cudaError_t launch_combine(const void *slots, const float *w, int64_t T, int K, int H,
                           void *y, bool f32, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (f32)
        combine_kernel<true><<<grid_for(T * (H / 4), TPB, 16), TPB, 0, s>>>(slots, w, T, K, H, y);
    else
        combine_kernel<false><<<grid_for(T * (H / 8), TPB, 16), TPB, 0, s>>>(slots, w, T, K, H, y);
    return cudaGetLastError();
}

cudaError_t launch_gather_bwd(const uint16_t *dy, const uint16_t *x, const int32_t *inv,
                              const int32_t *counts, const int32_t *offsets,
                              const int32_t *poff, int E, int64_t T, int K, int H,
                              uint16_t *dy_perm, uint16_t *x_perm, int32_t *prow, uint8_t *dy_q,
                              uint8_t *dy_s, cudaStream_t s) {
    if (E == 0) return cudaSuccess;
    if (T > 0)
        gather_bwd_kernel<<<grid_for(T, TPB / 32, 16), TPB, 0, s>>>(
            dy, x, inv, offsets, poff, E, T, K, H, dy_perm, x_perm, prow);
    if (T > 0 && dy_q != nullptr)
        quantize_dy_padded_kernel<<<grid_for(T * (H / 32), TPB, 16), TPB, 0, s>>>(
            dy, prow, T, K, H, dy_q, dy_s);
    zero_pad_rows_kernel<<<grid_for((int64_t)E * 16, TPB / 32, 16), TPB, 0, s>>>(
        counts, poff, E, H, dy_perm, x_perm, dy_q, dy_s);
    return cudaGetLastError();
}

cudaError_t launch_router_grad(const float *dS_part, int n_parts, const int32_t *inv,
                               const int32_t *offsets, const float *w, int64_t T, int K, int E,
                               float *d_topk, float *d_logits, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    router_grad_kernel<<<grid_for(T, TPB / 32, 16), TPB, 0, s>>>(
        dS_part, n_parts, inv, offsets, w, T, K, E, d_topk, d_logits);
    return cudaGetLastError();
}

}  // namespace mok

namespace mok {

cudaError_t launch_scale_atoms_rows(const uint8_t *src, int64_t rows, int K, uint8_t *dst,
                                    cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t nb = (rows + 127) / 128;
    const int nkc = (K / 128 + ATOM_KG - 1) / ATOM_KG;
    scale_atoms_kernel<<<grid_for(nb * nkc, 1, 8), 256, 0, s>>>(
        src, nb, 0, K, AtomRows{nullptr, rows, RingMap{1, 1, 0}, nullptr, nullptr}, dst);
    return cudaGetLastError();
}

cudaError_t launch_scale_atoms_tiles(const int32_t *tiles, int64_t cap, const uint8_t *src,
                                     int64_t R, int MB, int n_slots, int K, uint8_t *dst,
                                     cudaStream_t s) {
    if (cap == 0) return cudaSuccess;
    const int nkc = (K / 128 + ATOM_KG - 1) / ATOM_KG;
    scale_atoms_kernel<<<grid_for(cap * nkc, 1, 8), 256, 0, s>>>(
        src, 0, cap, K, AtomRows{tiles, 0, RingMap{R, MB, n_slots}, nullptr, nullptr}, dst);
    return cudaGetLastError();
}

cudaError_t launch_scale_atoms_tiles_padded(const int32_t *tiles, int64_t cap,
                                            const uint8_t *src, const int32_t *offsets,
                                            const int32_t *poff, int K, uint8_t *dst,
                                            cudaStream_t s) {
    if (cap == 0) return cudaSuccess;
    const int nkc = (K / 128 + ATOM_KG - 1) / ATOM_KG;
    scale_atoms_kernel<<<grid_for(cap * nkc, 1, 8), 256, 0, s>>>(
        src, 0, cap, K, AtomRows{tiles, 0, RingMap{1, 1, 0}, offsets, poff}, dst);
    return cudaGetLastError();
}

}  // namespace mok
