// common.cuh -- device helpers shared by the layer's kernels.
//
// Pages cited (by title and section):
//   [arex]     "Cursor 放出 MoK：NVL72 训练提速 2.37 倍" (arex-research.com)
//   [alphalab] "Mixture-of-Kittens" analysis (alphalab.site)
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mok.h"

#define MOK_DEV __device__ __forceinline__

namespace mok {

// ---------------------------------------------------------------- device status word
// Kernels record the first problem they find here and skip the offending access; the
// host reads it with mok_read_device_status.
MOK_DEV void raise_status(int *status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- bf16 helpers
MOK_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOK_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
MOK_DEV float bf16_to_f32(uint16_t v) { return __uint_as_float(((uint32_t)v) << 16); }
// round to nearest even (finite inputs)
MOK_DEV uint16_t f32_to_bf16(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
MOK_DEV uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
}

// ---------------------------------------------------------------- MXFP8 (OCP MX, E4M3 + E8M0)
// Shared scale of a 32-element block ([arex] section "pull 代替 push": MXFP8 activations
// quantized on the fly): 2^(floor(log2 amax) - 8), 8 being the largest E4M3 exponent,
// clamped at 2^-127. For amax >= 0 with fp32 exponent field ef, floor(log2 amax) = ef - 127
// for normal amax, so the E8M0 byte is ef - 8, and 0 when that is negative (subnormal or
// zero amax, or amax below 2^-119).
MOK_DEV uint32_t mx_scale_byte(float amax) {
    const int ef = (int)(__float_as_uint(amax) >> 23);
    return (uint32_t)(ef > 8 ? ef - 8 : 0);
}
// 2^-(byte-127) as an fp32 power of two (byte <= 246 keeps it a normal number)
MOK_DEV float mx_inv_scale(uint32_t byte) { return __uint_as_float((254u - byte) << 23); }
MOK_DEV float mx_scale(uint32_t byte) {
    // 2^(byte-127); byte 0 is 2^-127, a subnormal fp32
    return byte == 0 ? 5.877471754111438e-39f : __uint_as_float(byte << 23);
}
// two fp32 values to E4M3 (round to nearest even, finite overflow saturates), lo in byte 0
MOK_DEV uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}
// E4M3 byte to fp32, from the format's definition (bias 7, subnormal step 2^-9)
MOK_DEV float e4m3_to_f32(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    float v = (e == 0) ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (c & 0x80u) ? -v : v;
}

// ---------------------------------------------------------------- ring mapping
// Ring row of sorted row r ([arex] section "pull 代替 push", point 2: a fixed ring that
// rows cycle through): identity when the ring holds every row, otherwise row
// ((r / MB) mod n_slots) * MB + r mod MB; the forward through a ring of C rows uses MB = C,
// n_slots = 1, i.e. row r mod C.
struct RingMap {
    int64_t R;
    int32_t MB;
    int32_t n_slots;  // 0: ring holds every row
    MOK_DEV int64_t operator()(int64_t r) const {
        if (n_slots == 0) return r;
        return (int64_t)((r / MB) % n_slots) * MB + (r % MB);
    }
};

// ---------------------------------------------------------------- loads
MOK_DEV uint4 ldg_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

}  // namespace mok
