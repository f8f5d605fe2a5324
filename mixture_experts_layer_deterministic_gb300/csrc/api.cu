// api.cu -- the C ABI entry points (include/mok.h): argument validation, workspace layout
// and the stream-ordered sequence of kernels for each call.
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "mok_internal.h"

using namespace mok;

// ---------------------------------------------------------------- device status word
static __device__ int g_status;

namespace {

int g_cc_ok[MAX_DEV];        // 0 unknown, 1 ok, 2 unsupported
int *g_status_ptr[MAX_DEV];  // device address of g_status, per device

mok_status check_device(int **status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return MOK_ERR_CUDA;
    if (g_cc_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return MOK_ERR_CUDA;
        g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
        if (g_cc_ok[dev] == 1) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return MOK_ERR_CUDA;
            g_status_ptr[dev] = (int *)p;
        }
    }
    if (g_cc_ok[dev] != 1) return MOK_ERR_UNSUPPORTED;
    *status = g_status_ptr[dev];
    return MOK_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// values that are only stored are fp32 under MOK_FLAG_FP32_STORAGE, else bf16
bool f32_storage(const mok_config *c) { return (c->flags & MOK_FLAG_FP32_STORAGE) != 0; }
size_t stored_bytes(const mok_config *c) { return f32_storage(c) ? 4 : 2; }

// Which GEMMs run on SM pairs (the results are the same bit for bit). Unless the caller
// forces one form, the BF16 gate/up, down and dx GEMMs of the routed experts always do, the
// shared expert's gate/up too, and the weight gradients when an expert averages at least
// PAIR_ROWS rows. Measured on 4096 x 1024 experts, pairs against one SM: gate/up 6-16%, dx
// 6-16% and down 2-9% faster from 160 rows per expert up (down once 4% slower at 1280);
// weight gradients 18-23% faster from 640 rows, but 2-16% slower at 320 rows and below.
// There the dW writes bound the kernel, and the pair's two pipelines must both finish a
// unit before it moves on, which costs more than the operand bytes it saves. The same
// holds for GEMMs that add into their output (the shared expert's down and dx: 19% slower
// on pairs), whose epilogues wait on the loads of the values they add to. The MXFP8 GEMMs
// run on one SM: their scale atoms are cut per one-SM tile.
constexpr int64_t PAIR_ROWS = 512;
bool gemm_pairs(const mok_config *c, bool mx, bool by_default) {
    if (mx || (c->flags & MOK_FLAG_ONE_SM_GEMMS) != 0) return false;
    return (c->flags & MOK_FLAG_SM_PAIR_GEMMS) != 0 || by_default;
}

// the weight gradients; avg_rows: an expert's average rows
cudaError_t launch_wgrad(const mok_config *c, int64_t avg_rows, const int32_t *counts,
                         const int32_t *poff, const uint16_t *A, const uint16_t *Bm, void *out,
                         int E, int M, int N, int64_t rows_a, int64_t rows_b, int *status,
                         cudaStream_t s) {
    if (gemm_pairs(c, false, avg_rows >= PAIR_ROWS) && wgrad_pair_supported(M, N))
        return launch_wgrad_pair_tc(counts, poff, A, Bm, out, f32_storage(c), E, M, N, rows_a,
                                    rows_b, status, s);
    return launch_wgrad_tc(counts, poff, A, Bm, out, f32_storage(c), E, M, N, rows_a, rows_b,
                           status, s);
}

int64_t rows_R(const mok_config *c) { return (int64_t)c->T * c->K; }

// The forward runs in one of two ways:
//   a ring that holds every routed row (capacity 0 or >= R): gather every row, then the
//   gate/up and down GEMMs over all tiles (three launches);
//   a partial ring (capacity C < R): one persistent launch over rows cycling through a ring of
//   C rows, row r in ring row r mod C (ring_fwd.cu).
// Both give the same results bit for bit.
bool partial_ring(const mok_config *c) {
    return c->ring_capacity != 0 && (int64_t)c->ring_capacity < rows_R(c);
}
// rows of the h ring (and, for the full ring, of the x ring)
int64_t ring_rows(const mok_config *c) { return partial_ring(c) ? c->ring_capacity : rows_R(c); }

// ---------------------------------------------------------------- workspace layouts
struct Carver {
    char *base;
    size_t off = 0;
    template <class T>
    T *take(size_t bytes) {
        off = (off + 255) & ~(size_t)255;
        T *p = base ? (T *)((uintptr_t)base + off) : nullptr;
        off += bytes;
        return p;
    }
};

// A stand-in workspace address for locating pieces without a workspace: carving against it
// gives each piece's offset (never dereferenced).
char *const kVirtualWs = (char *)(uintptr_t)(1u << 20);
size_t ws_offset(const void *p) { return (size_t)((uintptr_t)p - (uintptr_t)kVirtualWs); }

struct FwdWs {
    int32_t *tiles;  // points past a 16-byte header holding the count
    int64_t tiles_cap;
    void *xring;              // gathered x [ring rows][H]
    uint8_t *xring_s;         // MXFP8, full ring: its scales [R][H/32]
    void *xq;                 // MXFP8, partial ring: x quantized token-major [T][H] and
    uint8_t *xq_s;            // its scales [T][H/32]
    void *hring;              // [ring rows][I]
    uint8_t *hring_s;         // MXFP8: [ring rows][I/32]
    void *slots;              // [R][H], the storage type of cfg->flags
    uint8_t *sf_w13, *sf_w2;  // MXFP8 weight scales as tensor-core atoms
    uint8_t *sf_x, *sf_h;     // MXFP8 token-tile scales as atoms, per tile of the list
    // partial ring: the unit records in claim order, the unit count and claim counter,
    // per-tile completion counters
    void *units;
    int32_t *hdr, *done_up, *done_dn, *done_g;
    int chunk;
    int gather_pieces;
};

size_t carve_fwd(const mok_config *c, void *ws, FwdWs *o) {
    Carver cv{(char *)ws};
    const int64_t R = rows_R(c);
    const bool mx = c->prec == MOK_MXFP8;
    const bool part = partial_ring(c);
    const int64_t rr = ring_rows(c);
    const int esz = mx ? 1 : 2;
    FwdWs w;
    w.chunk = part ? ring_tile_rows(mx, c->ring_capacity) : gemm_tc_tile_rows(mx);
    w.gather_pieces = part ? ring_gather_pieces(mx, c->ring_capacity, c->H) : 0;
    w.tiles_cap = part ? ring_tiles_cap(R, c->E, c->ring_capacity, w.chunk)
                       : tile_list_cap(R, c->E, w.chunk);
    int32_t *t = cv.take<int32_t>(16 + (size_t)w.tiles_cap * 16);
    w.tiles = t ? t + 4 : nullptr;
    w.xring = cv.take<void>((size_t)rr * c->H * esz);
    w.xring_s = mx && !part ? cv.take<uint8_t>((size_t)R * (c->H / 32)) : nullptr;
    w.xq = nullptr;
    w.xq_s = nullptr;
    if (part && mx) {
        w.xq = cv.take<void>((size_t)c->T * c->H);
        w.xq_s = cv.take<uint8_t>((size_t)c->T * (c->H / 32));
    }
    w.hring = cv.take<void>((size_t)rr * c->I * esz);
    w.hring_s = mx ? cv.take<uint8_t>((size_t)rr * (c->I / 32)) : nullptr;
    w.slots = cv.take<void>((size_t)R * c->H * stored_bytes(c));
    w.sf_w13 = w.sf_w2 = w.sf_x = w.sf_h = nullptr;
    if (mx) {
        w.sf_w13 = cv.take<uint8_t>((size_t)c->E * 2 * c->I * (c->H / 32));
        w.sf_w2 = cv.take<uint8_t>((size_t)c->E * c->H * (c->I / 32));
        w.sf_x = cv.take<uint8_t>((size_t)w.tiles_cap * (c->H / 128) * 512);
        w.sf_h = cv.take<uint8_t>((size_t)w.tiles_cap * (c->I / 128) * 512);
    }
    w.units = nullptr;
    w.hdr = w.done_up = w.done_dn = w.done_g = nullptr;
    if (part) {
        const int64_t units =
            w.tiles_cap * (w.gather_pieces + c->I / 128 + (c->H + 255) / 256);
        w.units = cv.take<void>((size_t)units * 32);
        w.hdr = cv.take<int32_t>(16);
        w.done_up = cv.take<int32_t>((size_t)w.tiles_cap * 4);
        w.done_dn = cv.take<int32_t>((size_t)w.tiles_cap * 4);
        w.done_g = cv.take<int32_t>((size_t)w.tiles_cap * 4);
    }
    if (o) *o = w;
    return cv.off;
}

struct BwdWs {
    int32_t *poff;
    int32_t *tiles;
    int64_t tiles_cap;
    int64_t rpad_cap;
    uint16_t *dy_perm, *x_perm, *dA, *sh;
    void *dx_slots;  // [R][H], the storage type of cfg->flags
    float *dS_part;
    void *preact;    // recomputed pre-activations [R][2I] (recompute workspace only)
    // MXFP8: padded row of every flat id; dy and dA quantized along H / 2I; scale atoms of
    // the transposed weights and of the dy and dA tiles
    int32_t *prow;
    uint8_t *dy_q, *dy_s, *dA_q, *dA_s, *sf_w2t, *sf_w13t, *sf_dy, *sf_dA;
};

size_t carve_bwd(const mok_config *c, void *ws, BwdWs *o, bool recompute = false) {
    Carver cv{(char *)ws};
    const int64_t R = rows_R(c);
    const bool mx = c->prec == MOK_MXFP8;
    BwdWs w;
    w.rpad_cap = R + 15 * (int64_t)c->E;
    w.poff = cv.take<int32_t>((size_t)(c->E + 1) * 4);
    w.tiles_cap = tile_list_cap(R, c->E, gemm_tc_tile_rows(mx));
    int32_t *t = cv.take<int32_t>(16 + (size_t)w.tiles_cap * 16);
    w.tiles = t ? t + 4 : nullptr;
    w.dy_perm = cv.take<uint16_t>((size_t)w.rpad_cap * c->H * 2);
    w.x_perm = cv.take<uint16_t>((size_t)w.rpad_cap * c->H * 2);
    w.dA = cv.take<uint16_t>((size_t)w.rpad_cap * 2 * c->I * 2);
    w.sh = cv.take<uint16_t>((size_t)w.rpad_cap * c->I * 2);
    w.dS_part = cv.take<float>((size_t)R * gemm_tc_dS_parts(c->I) * 4);
    w.dx_slots = cv.take<void>((size_t)R * c->H * stored_bytes(c));
    w.preact = recompute ? cv.take<void>((size_t)R * 2 * c->I * stored_bytes(c)) : nullptr;
    w.prow = nullptr;
    w.dy_q = w.dy_s = w.dA_q = w.dA_s = w.sf_w2t = w.sf_w13t = w.sf_dy = w.sf_dA = nullptr;
    if (mx) {
        const int64_t H = c->H, I2 = 2 * (int64_t)c->I, E = c->E;
        w.prow = cv.take<int32_t>((size_t)R * 4);
        w.dy_q = cv.take<uint8_t>((size_t)(w.rpad_cap * H));
        w.dy_s = cv.take<uint8_t>((size_t)(w.rpad_cap * (H / 32)));
        w.dA_q = cv.take<uint8_t>((size_t)(w.rpad_cap * I2));
        w.dA_s = cv.take<uint8_t>((size_t)(w.rpad_cap * (I2 / 32)));
        w.sf_w2t = cv.take<uint8_t>((size_t)(E * c->I * H / 32));
        w.sf_w13t = cv.take<uint8_t>((size_t)(E * H * I2 / 32));
        w.sf_dy = cv.take<uint8_t>((size_t)(w.tiles_cap * (H / 128) * 512));
        w.sf_dA = cv.take<uint8_t>((size_t)(w.tiles_cap * (I2 / 128) * 512));
    }
    if (o) *o = w;
    return cv.off;
}

// shared-expert forward: the expert's offsets, its tile list and h [T][I] bf16; MXFP8:
// x and h quantized (with scales) and the scale atoms of the weights and of the tiles
struct SharedWs {
    int32_t *offsets;
    int32_t *tiles;
    int64_t tiles_cap;
    uint16_t *h;
    uint8_t *x_q, *x_s, *h_q, *h_s, *sf_w13, *sf_w2, *sf_x, *sf_h;
};

size_t carve_shared(const mok_config *c, void *ws, SharedWs *o) {
    Carver cv{(char *)ws};
    const bool mx = c->prec == MOK_MXFP8;
    const int64_t T = c->T, H = c->H, I = c->I;
    SharedWs w;
    w.offsets = cv.take<int32_t>(2 * 4);
    w.tiles_cap = tile_list_cap(T, 1, gemm_tc_tile_rows(mx));
    int32_t *t = cv.take<int32_t>(16 + (size_t)w.tiles_cap * 16);
    w.tiles = t ? t + 4 : nullptr;
    w.h = mx ? nullptr : cv.take<uint16_t>((size_t)(T * I * 2));
    w.x_q = w.x_s = w.h_q = w.h_s = w.sf_w13 = w.sf_w2 = w.sf_x = w.sf_h = nullptr;
    if (mx) {
        w.x_q = cv.take<uint8_t>((size_t)(T * H));
        w.x_s = cv.take<uint8_t>((size_t)(T * (H / 32)));
        w.h_q = cv.take<uint8_t>((size_t)(T * I));
        w.h_s = cv.take<uint8_t>((size_t)(T * (I / 32)));
        w.sf_w13 = cv.take<uint8_t>((size_t)(2 * I * H / 32));
        w.sf_w2 = cv.take<uint8_t>((size_t)(H * I / 32));
        w.sf_x = cv.take<uint8_t>((size_t)(w.tiles_cap * (H / 128) * 512));
        w.sf_h = cv.take<uint8_t>((size_t)(w.tiles_cap * (I / 128) * 512));
    }
    if (o) *o = w;
    return cv.off;
}

// shared-expert backward: the single expert's offsets, padded offsets, count, weights of
// one and identity row map; its tile list; dA [Tpad][2I], h [Tpad][I] (bf16, rows past T
// zero) and the G epilogue's (unused) router-gradient partials. MXFP8: dy quantized along
// H [T][H], dA quantized along 2I [Tpad][2I] (with scales), and the scale atoms of the
// transposed weights and of the dy and dA tiles.
struct SharedBwdWs {
    int32_t *offsets, *poff, *counts, *perm;
    float *ones;
    int32_t *tiles;
    int64_t tiles_cap, tpad;
    uint16_t *dA, *sh;
    float *dS_part;
    uint8_t *dy_q, *dy_s, *dA_q, *dA_s, *sf_w2t, *sf_w13t, *sf_dy, *sf_dA;
};

size_t carve_shared_bwd(const mok_config *c, void *ws, SharedBwdWs *o) {
    Carver cv{(char *)ws};
    SharedBwdWs w;
    w.tpad = ((int64_t)c->T + 15) & ~(int64_t)15;
    w.offsets = cv.take<int32_t>(2 * 4);
    w.poff = cv.take<int32_t>(2 * 4);
    w.counts = cv.take<int32_t>(4);
    w.perm = cv.take<int32_t>((size_t)c->T * 4 + 4);
    w.ones = cv.take<float>((size_t)c->T * 4 + 4);
    const bool mx = c->prec == MOK_MXFP8;
    w.tiles_cap = tile_list_cap(c->T, 1, gemm_tc_tile_rows(mx));
    int32_t *t = cv.take<int32_t>(16 + (size_t)w.tiles_cap * 16);
    w.tiles = t ? t + 4 : nullptr;
    w.dA = cv.take<uint16_t>((size_t)(w.tpad * 2 * c->I * 2));
    w.sh = cv.take<uint16_t>((size_t)(w.tpad * c->I * 2));
    w.dS_part = cv.take<float>((size_t)c->T * gemm_tc_dS_parts(c->I) * 4 + 4);
    w.dy_q = w.dy_s = w.dA_q = w.dA_s = w.sf_w2t = w.sf_w13t = w.sf_dy = w.sf_dA = nullptr;
    if (mx) {
        const int64_t T = c->T, H = c->H, I2 = 2 * (int64_t)c->I;
        w.dy_q = cv.take<uint8_t>((size_t)(T * H));
        w.dy_s = cv.take<uint8_t>((size_t)(T * (H / 32)));
        w.dA_q = cv.take<uint8_t>((size_t)(w.tpad * I2));
        w.dA_s = cv.take<uint8_t>((size_t)(w.tpad * (I2 / 32)));
        w.sf_w2t = cv.take<uint8_t>((size_t)(c->I * H / 32));
        w.sf_w13t = cv.take<uint8_t>((size_t)(H * I2 / 32));
        w.sf_dy = cv.take<uint8_t>((size_t)(w.tiles_cap * (H / 128) * 512));
        w.sf_dA = cv.take<uint8_t>((size_t)(w.tiles_cap * (I2 / 128) * 512));
    }
    if (o) *o = w;
    return cv.off;
}

cudaError_t first_error(cudaError_t a, cudaError_t b) { return a != cudaSuccess ? a : b; }

mok_status check_ws(void *ws, size_t ws_bytes, size_t need) {
    if (need == 0) return MOK_OK;
    if (ws == nullptr || ws_bytes < need) return MOK_ERR_WORKSPACE;
    if (((uintptr_t)ws & 255u) != 0) return MOK_ERR_WORKSPACE;
    return MOK_OK;
}

mok_status check_sched(const mok_config *c, const mok_schedule *s) {
    if (s == nullptr) return MOK_ERR_INVALID_ARG;
    const void *ps[] = {s->counts, s->offsets, s->perm, s->inv, s->segs, s->n_segs};
    for (const void *p : ps)
        if (p == nullptr) return MOK_ERR_INVALID_ARG;
    (void)c;
    return MOK_OK;
}

}  // namespace

namespace mok {
mok_status current_device_status_word(int **status) { return check_device(status); }

int device_sm_count() {
    static std::atomic<int> cache[MAX_DEV];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return 1;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n < 1)
            n = 1;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}
}  // namespace mok

// a launch of `nk` kernels of one kind, bracketed by events while profiling is on
#define MOK_LAUNCH(kind, nk, expr)                         \
    do {                                                   \
        prof_begin(kind, stream);                          \
        cudaError_t _e = (expr);                           \
        prof_end(kind, stream, nk);                        \
        if (_e != cudaSuccess) return MOK_ERR_CUDA;        \
    } while (0)

extern "C" {

uint32_t mok_abi_version(void) { return MOK_ABI_VERSION; }

const char *mok_status_string(mok_status s) {
    switch (s) {
        case MOK_OK: return "ok";
        case MOK_ERR_INVALID_ARG: return "invalid argument";
        case MOK_ERR_UNSUPPORTED: return "unsupported device (compute capability 10.3 required)";
        case MOK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOK_ERR_CUDA: return "CUDA runtime error";
        case MOK_ERR_TIMEOUT: return "device wait timed out";
        case MOK_ERR_DEVICE_INVARIANT: return "device-side invariant violated";
        case MOK_ERR_ABI: return "ABI version mismatch";
    }
    return "unknown status";
}

mok_status mok_check_config(const mok_config *c) {
    if (c == nullptr) return MOK_ERR_INVALID_ARG;
    if (c->abi_version != MOK_ABI_VERSION) return MOK_ERR_ABI;
    if (c->T < 0 || c->E < 1 || c->E > 1024 || c->K < 1 || c->K > 32 || c->K > c->E)
        return MOK_ERR_INVALID_ARG;
    if (c->H < 128 || c->H > 16384 || c->H % 128 != 0) return MOK_ERR_INVALID_ARG;
    if (c->I < 128 || c->I > 8192 || c->I % 128 != 0) return MOK_ERR_INVALID_ARG;
    if (c->minibatch < 1) return MOK_ERR_INVALID_ARG;
    if ((int64_t)c->T * c->K >= ((int64_t)1 << 31) - 16 * 1024) return MOK_ERR_INVALID_ARG;
    if (c->ring_capacity < 0) return MOK_ERR_INVALID_ARG;
    if (c->ring_capacity != 0 && (int64_t)c->ring_capacity < rows_R(c) &&
        c->ring_capacity < c->minibatch)
        return MOK_ERR_INVALID_ARG;
    if (c->prec != MOK_BF16 && c->prec != MOK_MXFP8) return MOK_ERR_INVALID_ARG;
    const uint32_t known =
        MOK_FLAG_FP32_STORAGE | MOK_FLAG_ONE_SM_GEMMS | MOK_FLAG_SM_PAIR_GEMMS;
    if ((c->flags & ~known) != 0) return MOK_ERR_INVALID_ARG;
    if ((c->flags & MOK_FLAG_ONE_SM_GEMMS) && (c->flags & MOK_FLAG_SM_PAIR_GEMMS))
        return MOK_ERR_INVALID_ARG;
    return MOK_OK;
}

int64_t mok_segment_capacity(const mok_config *c) {
    if (mok_check_config(c) != MOK_OK) return 0;
    const int64_t R = rows_R(c);
    const int64_t cap = (int64_t)c->E + (R + c->minibatch - 1) / c->minibatch - 1;
    return cap > 0 ? cap : 1;
}

mok_status mok_workspace_item(const mok_config *c, int which, int item, size_t *offset,
                              size_t *bytes) {
    if (offset == nullptr || bytes == nullptr) return MOK_ERR_INVALID_ARG;
    if (mok_check_config(c) != MOK_OK) return MOK_ERR_INVALID_ARG;
    const bool mx = c->prec == MOK_MXFP8;
    const size_t H = (size_t)c->H, I = (size_t)c->I, R = (size_t)rows_R(c), T = (size_t)c->T;
    const void *p = nullptr;
    size_t n = 0;
    if (which == MOK_WS_FORWARD) {
        FwdWs w;
        carve_fwd(c, kVirtualWs, &w);
        const size_t rr = (size_t)ring_rows(c);
        const bool part = partial_ring(c);
        const size_t esz = mx ? 1 : 2;
        switch (item) {
            case MOK_ITEM_X_RING: p = w.xring; n = rr * H * esz; break;
            case MOK_ITEM_X_RING_SCALE:  // a partial ring: the scales of x's token rows
                p = part ? (const void *)w.xq_s : (const void *)w.xring_s;
                n = (part ? T : R) * (H / 32);
                break;
            case MOK_ITEM_H_RING: p = w.hring; n = (size_t)rr * I * esz; break;
            case MOK_ITEM_H_RING_SCALE: p = w.hring_s; n = (size_t)rr * (I / 32); break;
            case MOK_ITEM_SLOTS: p = w.slots; n = R * H * stored_bytes(c); break;
            case MOK_ITEM_RING_TILES:
                p = w.units ? (const void *)(w.tiles - 4) : nullptr;
                n = 16 + (size_t)w.tiles_cap * 16;
                break;
            case MOK_ITEM_RING_ORDER:
                p = w.units;
                n = (size_t)w.tiles_cap * (w.gather_pieces + I / 128 + (H + 255) / 256) * 32;
                break;
            default: break;
        }
    } else if (which == MOK_WS_BACKWARD || which == MOK_WS_BACKWARD_RECOMPUTE) {
        BwdWs w;
        carve_bwd(c, kVirtualWs, &w, which == MOK_WS_BACKWARD_RECOMPUTE);
        const size_t rp = (size_t)w.rpad_cap;
        switch (item) {
            case MOK_ITEM_PAD_OFFSETS: p = w.poff; n = ((size_t)c->E + 1) * 4; break;
            case MOK_ITEM_DA: p = w.dA; n = rp * 2 * I * 2; break;
            case MOK_ITEM_WH: p = w.sh; n = rp * I * 2; break;
            case MOK_ITEM_SLOTS: p = w.dx_slots; n = R * H * stored_bytes(c); break;
            case MOK_ITEM_DA_Q: p = w.dA_q; n = rp * 2 * I; break;
            case MOK_ITEM_DA_SCALE: p = w.dA_s; n = rp * (2 * I / 32); break;
            case MOK_ITEM_DY_Q: p = w.dy_q; n = rp * H; break;
            case MOK_ITEM_DY_SCALE: p = w.dy_s; n = rp * (H / 32); break;
            default: break;
        }
    } else if (which == MOK_WS_SHARED) {
        SharedWs w;
        carve_shared(c, kVirtualWs, &w);
        switch (item) {
            case MOK_ITEM_H_RING:
                p = mx ? (const void *)w.h_q : (const void *)w.h;
                n = T * I * (mx ? 1 : 2);
                break;
            case MOK_ITEM_H_RING_SCALE: p = w.h_s; n = T * (I / 32); break;
            case MOK_ITEM_X_RING: p = w.x_q; n = T * H; break;
            case MOK_ITEM_X_RING_SCALE: p = w.x_s; n = T * (H / 32); break;
            default: break;
        }
    } else if (which == MOK_WS_SHARED_BACKWARD) {
        SharedBwdWs w;
        carve_shared_bwd(c, kVirtualWs, &w);
        const size_t tp = (size_t)w.tpad;
        switch (item) {
            case MOK_ITEM_DA: p = w.dA; n = tp * 2 * I * 2; break;
            case MOK_ITEM_WH: p = w.sh; n = tp * I * 2; break;
            case MOK_ITEM_DA_Q: p = w.dA_q; n = tp * 2 * I; break;
            case MOK_ITEM_DA_SCALE: p = w.dA_s; n = tp * (2 * I / 32); break;
            case MOK_ITEM_DY_Q: p = w.dy_q; n = T * H; break;
            case MOK_ITEM_DY_SCALE: p = w.dy_s; n = T * (H / 32); break;
            default: break;
        }
    }
    if (p == nullptr) return MOK_ERR_INVALID_ARG;
    *offset = ws_offset(p);
    *bytes = n;
    return MOK_OK;
}

size_t mok_workspace_size(const mok_config *c, int which) {
    if (mok_check_config(c) != MOK_OK) return 0;
    switch (which) {
        case MOK_WS_SCHEDULE: return schedule_ws_bytes(rows_R(c), c->E);
        case MOK_WS_FORWARD: return carve_fwd(c, nullptr, nullptr);
        case MOK_WS_BACKWARD_RECOMPUTE: return carve_bwd(c, nullptr, nullptr, true);
        case MOK_WS_SHARED: return carve_shared(c, nullptr, nullptr);
        case MOK_WS_SHARED_BACKWARD: return carve_shared_bwd(c, nullptr, nullptr);
        case MOK_WS_BACKWARD: return carve_bwd(c, nullptr, nullptr);
    }
    return 0;
}

mok_status mok_route_topk(const mok_config *c, const float *logits, int32_t *topk_idx,
                          float *topk_w, cudaStream_t stream) {
    mok_status st = mok_check_config(c);
    if (st != MOK_OK) return st;
    int *status;
    if ((st = check_device(&status)) != MOK_OK) return st;
    if (c->T == 0) return MOK_OK;
    if (!logits || !topk_idx || !topk_w) return MOK_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(topk_w))
        return MOK_ERR_INVALID_ARG;
    MOK_LAUNCH(KK_ROUTE, 1,
               launch_route_topk(logits, c->T, c->E, c->K, topk_idx, topk_w, status, stream));
    return MOK_OK;
}

mok_status mok_build_schedule(const mok_config *c, const int32_t *topk_idx,
                              const mok_schedule *sch, void *ws, size_t ws_bytes,
                              cudaStream_t stream) {
    mok_status st = mok_check_config(c);
    if (st != MOK_OK) return st;
    int *status;
    if ((st = check_device(&status)) != MOK_OK) return st;
    if ((st = check_sched(c, sch)) != MOK_OK) return st;
    const int64_t R = rows_R(c);
    if (R > 0 && (topk_idx == nullptr || !aligned16(topk_idx))) return MOK_ERR_INVALID_ARG;
    if ((st = check_ws(ws, ws_bytes, schedule_ws_bytes(R, c->E))) != MOK_OK) return st;
    ScheduleWs w = schedule_ws_carve(ws, R, c->E);
    MOK_LAUNCH(KK_SCHEDULE, R > 0 ? 4 : 1,
               launch_build_schedule(topk_idx, R, c->E, c->minibatch, *sch, w, status, stream));
    return MOK_OK;
}

mok_status mok_forward(const mok_config *c, const void *x, const mok_schedule *sch,
                       const float *topk_w, const void *w13, const uint8_t *w13_scale,
                       const void *w2, const uint8_t *w2_scale, void *y, void *saved_preact,
                       void *ws, size_t ws_bytes, cudaStream_t stream) {
    mok_status st = mok_check_config(c);
    if (st != MOK_OK) return st;
    int *status;
    if ((st = check_device(&status)) != MOK_OK) return st;
    if ((st = check_sched(c, sch)) != MOK_OK) return st;
    const bool mx = c->prec == MOK_MXFP8;
    if (!x || !topk_w || !w13 || !w2 || !y) return MOK_ERR_INVALID_ARG;
    if (mx && (!w13_scale || !w2_scale)) return MOK_ERR_INVALID_ARG;
    if (!mx && (w13_scale || w2_scale)) return MOK_ERR_INVALID_ARG;
    const void *ps[] = {x, topk_w, w13, w2, y, w13_scale, w2_scale, saved_preact};
    for (const void *p : ps)
        if (p && !aligned16(p)) return MOK_ERR_INVALID_ARG;
    const size_t need = carve_fwd(c, nullptr, nullptr);
    if ((st = check_ws(ws, ws_bytes, need)) != MOK_OK) return st;
    const int64_t R = rows_R(c);
    if (R == 0) return MOK_OK;
    FwdWs w;
    carve_fwd(c, ws, &w);
    const int chunk = w.chunk;
    const int64_t cap = w.tiles_cap;
    if (mx) {
        // the weights' scales in the tensor cores' atom layout, once per call
        MOK_LAUNCH(KK_SCALE_ATOMS, 2,
                   first_error(launch_scale_atoms_rows(w13_scale, (int64_t)c->E * 2 * c->I,
                                                       c->H, w.sf_w13, stream),
                               launch_scale_atoms_rows(w2_scale, (int64_t)c->E * c->H, c->I,
                                                       w.sf_w2, stream)));
    }
    if (partial_ring(c)) {
        // one persistent launch through the ring; MXFP8 quantizes x once, token-major
        if (mx)
            MOK_LAUNCH(KK_QUANTIZE, 1,
                       launch_quantize_mxfp8((const uint16_t *)x, c->T, c->H,
                                             (uint8_t *)w.xq, w.xq_s, stream));
        RingFwdArgs ra{};
        ra.offsets = sch->offsets;
        ra.perm = sch->perm;
        ra.tiles = w.tiles;
        ra.tiles_cap = cap;
        ra.units = w.units;
        ra.hdr = w.hdr;
        ra.done_up = w.done_up;
        ra.done_dn = w.done_dn;
        ra.done_g = w.done_g;
        ra.x = mx ? (const void *)w.xq : x;
        ra.xs = w.xq_s;
        ra.xring = w.xring;
        ra.w13 = w13;
        ra.w2 = w2;
        ra.sf_w13 = w.sf_w13;
        ra.sf_w2 = w.sf_w2;
        ra.sf_x = w.sf_x;
        ra.sf_h = w.sf_h;
        ra.hring = w.hring;
        ra.hring_s = w.hring_s;
        ra.preact = saved_preact;
        ra.preact_f32 = f32_storage(c);
        ra.slots = w.slots;
        ra.out_f32 = f32_storage(c);
        ra.T = c->T;
        ra.R = R;
        ra.C = c->ring_capacity;
        ra.chunk = chunk;
        ra.gather_pieces = w.gather_pieces;
        ring_lags(mx, c->ring_capacity, &ra.lag_gather, &ra.lag);
        ra.H = c->H;
        ra.I = c->I;
        ra.E = c->E;
        ra.K = c->K;
        ra.mx = mx;
        ra.status = status;
        MOK_LAUNCH(KK_RING_FWD, mx ? 3 : 2, launch_ring_forward(ra, stream));
    } else {
        // a ring that holds every row: filled token by token (each x row read once), then
        // the two GEMMs over every tile
        const Ring ring{R, c->minibatch, 0};
        // the gate/up GEMM on SM pairs takes tiles of up to 256 rows, the down GEMM (either
        // form) tiles of up to 128: the list is rebuilt in place between the two
        const bool up_pairs = gemm_pairs(c, mx, true);
        MOK_LAUNCH(KK_TILES, 1,
                   launch_build_tiles(sch->offsets, c->E, 0, R, up_pairs ? PAIR_TILE_ROWS : chunk,
                                      w.tiles, cap, status, stream));
        if (!mx)
            MOK_LAUNCH(KK_GATHER, 1,
                       launch_gather_tok_bf16((const uint16_t *)x, sch->inv, c->T, c->K, c->H,
                                              (uint16_t *)w.xring, stream));
        else
            MOK_LAUNCH(KK_GATHER, 1,
                       launch_gather_tok_mxfp8((const uint16_t *)x, sch->inv, c->T, c->K, c->H,
                                               (uint8_t *)w.xring, w.xring_s, stream));
        GemmUpArgs ua{w.tiles, cap, w.xring, w.xring_s, w13, w13_scale, w.hring,
                      w.hring_s, saved_preact, c->H, c->I, c->E, mx, ring, status};
        ua.preact_f32 = f32_storage(c);
        GemmDownArgs da{w.tiles, cap, w.hring, w.hring_s, w2, w2_scale, sch->perm,
                        w.slots, c->H, c->I, c->E, mx, ring, status, false};
        da.out_f32 = f32_storage(c);
        if (mx) {
            MOK_LAUNCH(KK_SCALE_ATOMS, 1,
                       launch_scale_atoms_tiles(w.tiles, cap, w.xring_s, R, c->minibatch, 0,
                                                c->H, w.sf_x, stream));
            MOK_LAUNCH(KK_GEMM_UP, 1, launch_gemm_up_tc_mx(ua, R, w.sf_w13, w.sf_x, stream));
            MOK_LAUNCH(KK_SCALE_ATOMS, 1,
                       launch_scale_atoms_tiles(w.tiles, cap, w.hring_s, R, c->minibatch, 0,
                                                c->I, w.sf_h, stream));
            MOK_LAUNCH(KK_GEMM_DOWN, 1,
                       launch_gemm_down_tc_mx(da, R, w.sf_w2, w.sf_h, stream));
        } else {
            if (up_pairs) {
                MOK_LAUNCH(KK_GEMM_UP, 1, launch_gemm_up_pair_tc(ua, R, stream));
                MOK_LAUNCH(KK_TILES, 1,
                           launch_build_tiles(sch->offsets, c->E, 0, R, chunk, w.tiles, cap,
                                              status, stream));
            } else {
                MOK_LAUNCH(KK_GEMM_UP, 1, launch_gemm_up_tc(ua, R, stream));
            }
            MOK_LAUNCH(KK_GEMM_DOWN, 1,
                       gemm_pairs(c, mx, true) ? launch_gemm_down_pair_tc(da, R, stream)
                                               : launch_gemm_down_tc(da, R, stream));
        }
    }
    MOK_LAUNCH(KK_COMBINE, 1,
               launch_combine(w.slots, topk_w, c->T, c->K, c->H, y, f32_storage(c), stream));
    return MOK_OK;
}

}  // extern "C"

namespace mok {
// the transposed, MXFP8-quantized weights of the MXFP8 backward
struct MxBwdWeights {
    const uint8_t *w13t_q, *w13t_s, *w2t_q, *w2t_s;
};

mok_status backward_impl(const mok_config *c, const void *x, const mok_schedule *sch,
                         const float *topk_w, const void *saved_preact, const void *w13,
                         const void *w2, const MxBwdWeights *mxw, const void *dy, void *dx,
                         void *dw13, void *dw2, float *d_topk_w, float *d_logits, void *ws,
                         size_t ws_bytes, cudaStream_t stream) {
    mok_status st = mok_check_config(c);
    if (st != MOK_OK) return st;
    int *status;
    if ((st = check_device(&status)) != MOK_OK) return st;
    if ((st = check_sched(c, sch)) != MOK_OK) return st;
    const bool mx = mxw != nullptr;
    if (c->prec != (mx ? MOK_MXFP8 : MOK_BF16)) return MOK_ERR_INVALID_ARG;
    if (!x || !topk_w || !dy || !dx || !dw13 || !dw2 || !d_topk_w) return MOK_ERR_INVALID_ARG;
    if (!mx && (!w13 || !w2)) return MOK_ERR_INVALID_ARG;
    if (mx && (!saved_preact || !mxw->w13t_q || !mxw->w13t_s || !mxw->w2t_q || !mxw->w2t_s))
        return MOK_ERR_INVALID_ARG;
    const bool recompute = saved_preact == nullptr;
    const void *ps[] = {x, topk_w, saved_preact, w13, w2, dy, dx, dw13, dw2, d_topk_w, d_logits,
                        mx ? mxw->w13t_q : nullptr, mx ? mxw->w2t_q : nullptr};
    for (const void *p : ps)
        if (p && !aligned16(p)) return MOK_ERR_INVALID_ARG;
    const size_t need = carve_bwd(c, nullptr, nullptr, recompute);
    if ((st = check_ws(ws, ws_bytes, need)) != MOK_OK) return st;
    const int64_t R = rows_R(c);
    BwdWs w;
    carve_bwd(c, ws, &w, recompute);
    const int E = c->E, H = c->H, I = c->I, K = c->K;
    MOK_LAUNCH(KK_PAD, 1, launch_pad_offsets(sch->counts, E, w.poff, stream));
    MOK_LAUNCH(KK_TILES, 1,
               launch_build_tiles(sch->offsets, E, 0, R, gemm_tc_tile_rows(mx), w.tiles,
                                  w.tiles_cap, status, stream));
    MOK_LAUNCH(KK_GATHER_BWD, 1,
               launch_gather_bwd((const uint16_t *)dy, (const uint16_t *)x, sch->inv,
                                 sch->counts, sch->offsets, w.poff, E, c->T, K, H, w.dy_perm,
                                 w.x_perm, w.prow, w.dy_q, w.dy_s, stream));
    if (recompute)
        MOK_LAUNCH(KK_GEMM_UP, 1,
                   launch_gemm_up_recompute_tc(w.tiles, w.tiles_cap, w.x_perm, w.rpad_cap, w13,
                                               sch->offsets, w.poff, w.preact, f32_storage(c),
                                               H, I, E, status, stream));
    if (mx)  // the tensor cores' scale atoms of W2t, W13t and of the dy tiles
        MOK_LAUNCH(KK_SCALE_ATOMS, 3,
                   first_error(first_error(launch_scale_atoms_rows(mxw->w2t_s, (int64_t)E * I,
                                                                   H, w.sf_w2t, stream),
                                           launch_scale_atoms_rows(mxw->w13t_s, (int64_t)E * H,
                                                                   2 * I, w.sf_w13t, stream)),
                               launch_scale_atoms_tiles_padded(w.tiles, w.tiles_cap, w.dy_s,
                                                               sch->offsets, w.poff, H,
                                                               w.sf_dy, stream)));
    const void *pre = recompute ? w.preact : saved_preact;
    GemmGArgs ga{w.tiles, w.tiles_cap, sch->offsets, w.poff, (const uint16_t *)w2, w.dy_perm,
                 pre, sch->perm, topk_w, w.dA, w.sh, w.dS_part, H, I, status};
    ga.preact_f32 = f32_storage(c);
    if (mx) {
        ga.mxfp8 = true;
        ga.w2t_q = mxw->w2t_q;
        ga.sf_w2t = w.sf_w2t;
        ga.dy_q = w.dy_q;
        ga.sf_dy = w.sf_dy;
        ga.dA_q = w.dA_q;
        ga.dA_s = w.dA_s;
    }
    MOK_LAUNCH(KK_GEMM_G, 1, launch_gemm_g_tc(ga, E, w.rpad_cap, stream));
    MOK_LAUNCH(KK_ROUTER_GRAD, 1,
               launch_router_grad(w.dS_part, gemm_tc_dS_parts(I), sch->inv, sch->offsets,
                                  topk_w, c->T, K, E, d_topk_w, d_logits, stream));
    GemmDgradArgs dg{w.tiles, w.tiles_cap, sch->offsets, w.poff, (const uint16_t *)w13, w.dA,
                     sch->perm, w.dx_slots, H, I, status};
    dg.out_f32 = f32_storage(c);
    if (mx) {
        MOK_LAUNCH(KK_SCALE_ATOMS, 1,
                   launch_scale_atoms_tiles_padded(w.tiles, w.tiles_cap, w.dA_s, sch->offsets,
                                                   w.poff, 2 * I, w.sf_dA, stream));
        dg.mxfp8 = true;
        dg.w13t_q = mxw->w13t_q;
        dg.sf_w13t = w.sf_w13t;
        dg.dA_q = w.dA_q;
        dg.sf_dA = w.sf_dA;
    }
    if (gemm_pairs(c, mx, true)) {
        // the pair form's tiles hold up to 256 rows; the list is rebuilt in place (nothing
        // after this GEMM reads it)
        MOK_LAUNCH(KK_TILES, 1,
                   launch_build_tiles(sch->offsets, E, 0, R, PAIR_TILE_ROWS, w.tiles,
                                      w.tiles_cap, status, stream));
        MOK_LAUNCH(KK_GEMM_DGRAD, 1, launch_gemm_dgrad_pair_tc(dg, E, w.rpad_cap, stream));
    } else {
        MOK_LAUNCH(KK_GEMM_DGRAD, 1, launch_gemm_dgrad_tc(dg, E, w.rpad_cap, stream));
    }
    MOK_LAUNCH(KK_DX_REDUCE, 1,
               launch_combine(w.dx_slots, nullptr, c->T, K, H, dx, f32_storage(c), stream));
    // dW13[e] is [2I][H]: rows j (N) x contiguous c (M)
    const int64_t avg_rows = E > 0 ? (int64_t)c->T * K / E : 0;
    MOK_LAUNCH(KK_WGRAD13, 1,
               launch_wgrad(c, avg_rows, sch->counts, w.poff, w.x_perm, w.dA, dw13, E, H,
                            2 * I, w.rpad_cap, w.rpad_cap, status, stream));
    // dW2[e] is [H][I]: rows c (N) x contiguous i (M)
    MOK_LAUNCH(KK_WGRAD2, 1,
               launch_wgrad(c, avg_rows, sch->counts, w.poff, w.sh, w.dy_perm, dw2, E, I, H,
                            w.rpad_cap, w.rpad_cap, status, stream));
    return MOK_OK;
}
}  // namespace mok

extern "C" {

mok_status mok_backward(const mok_config *c, const void *x, const mok_schedule *sch,
                        const float *topk_w, const void *saved_preact, const void *w13,
                        const void *w2, const void *dy, void *dx, void *dw13, void *dw2,
                        float *d_topk_w, float *d_logits, void *ws, size_t ws_bytes,
                        cudaStream_t stream) {
    return backward_impl(c, x, sch, topk_w, saved_preact, w13, w2, nullptr, dy, dx, dw13, dw2,
                         d_topk_w, d_logits, ws, ws_bytes, stream);
}

mok_status mok_backward_mxfp8(const mok_config *c, const void *x, const mok_schedule *sch,
                              const float *topk_w, const void *saved_preact,
                              const uint8_t *w13t_q, const uint8_t *w13t_s,
                              const uint8_t *w2t_q, const uint8_t *w2t_s, const void *dy,
                              void *dx, void *dw13, void *dw2, float *d_topk_w,
                              float *d_logits, void *ws, size_t ws_bytes, cudaStream_t stream) {
    const MxBwdWeights mxw{w13t_q, w13t_s, w2t_q, w2t_s};
    return backward_impl(c, x, sch, topk_w, saved_preact, nullptr, nullptr, &mxw, dy, dx, dw13,
                         dw2, d_topk_w, d_logits, ws, ws_bytes, stream);
}

mok_status mok_shared_expert_forward(const mok_config *c, const void *x, const void *w13_s,
                                     const void *w2_s, void *y, void *saved_preact_s, void *ws,
                                     size_t ws_bytes, cudaStream_t stream) {
    mok_status st = mok_check_config(c);
    if (st != MOK_OK) return st;
    int *status;
    if ((st = check_device(&status)) != MOK_OK) return st;
    if (c->prec != MOK_BF16) return MOK_ERR_UNSUPPORTED;
    if (!x || !w13_s || !w2_s || !y) return MOK_ERR_INVALID_ARG;
    const void *ps[] = {x, w13_s, w2_s, y, saved_preact_s};
    for (const void *p : ps)
        if (p && !aligned16(p)) return MOK_ERR_INVALID_ARG;
    const size_t need = carve_shared(c, nullptr, nullptr);
    if ((st = check_ws(ws, ws_bytes, need)) != MOK_OK) return st;
    if (c->T == 0) return MOK_OK;
    SharedWs w;
    carve_shared(c, ws, &w);
    // one expert owning every token, in token order: x itself is the ring (slot t = t)
    const Ring ring{c->T, c->minibatch, 0};
    // gate/up on SM pairs over tiles of up to 256 rows, then the down GEMM over tiles of up
    // to 128 (the list rebuilt in place)
    const bool up_pairs = gemm_pairs(c, false, true);
    MOK_LAUNCH(KK_TILES, 2,
               first_error(launch_single_expert_offsets(w.offsets, c->T, stream),
                           launch_build_tiles(w.offsets, 1, 0, c->T,
                                              up_pairs ? PAIR_TILE_ROWS : gemm_tc_tile_rows(false),
                                              w.tiles, w.tiles_cap, status, stream)));
    GemmUpArgs ua{w.tiles, w.tiles_cap, x, nullptr, w13_s, nullptr, w.h, nullptr,
                  saved_preact_s, c->H, c->I, 1, false, ring, status};
    ua.preact_f32 = f32_storage(c);
    MOK_LAUNCH(KK_SHARED_UP, 1,
               up_pairs ? launch_gemm_up_pair_tc(ua, c->T, stream)
                        : launch_gemm_up_tc(ua, c->T, stream));
    if (up_pairs)
        MOK_LAUNCH(KK_TILES, 1,
                   launch_build_tiles(w.offsets, 1, 0, c->T, gemm_tc_tile_rows(false), w.tiles,
                                      w.tiles_cap, status, stream));
    GemmDownArgs da{w.tiles, w.tiles_cap, w.h, nullptr, w2_s, nullptr, nullptr, y,
                    c->H, c->I, 1, false, ring, status, true};
    da.out_f32 = f32_storage(c);
    MOK_LAUNCH(KK_SHARED_DOWN, 1,
               gemm_pairs(c, false, false) ? launch_gemm_down_pair_tc(da, c->T, stream)
                                           : launch_gemm_down_tc(da, c->T, stream));
    return MOK_OK;
}

mok_status mok_shared_expert_forward_mxfp8(const mok_config *c, const void *x,
                                           const uint8_t *w13s_q, const uint8_t *w13s_scale,
                                           const uint8_t *w2s_q, const uint8_t *w2s_scale,
                                           void *y, void *saved_preact_s, void *ws,
                                           size_t ws_bytes, cudaStream_t stream) {
    mok_status st = mok_check_config(c);
    if (st != MOK_OK) return st;
    int *status;
    if ((st = check_device(&status)) != MOK_OK) return st;
    if (c->prec != MOK_MXFP8) return MOK_ERR_INVALID_ARG;
    if (!x || !w13s_q || !w13s_scale || !w2s_q || !w2s_scale || !y) return MOK_ERR_INVALID_ARG;
    const void *ps[] = {x, w13s_q, w2s_q, y, saved_preact_s};
    for (const void *p : ps)
        if (p && !aligned16(p)) return MOK_ERR_INVALID_ARG;
    const size_t need = carve_shared(c, nullptr, nullptr);
    if ((st = check_ws(ws, ws_bytes, need)) != MOK_OK) return st;
    if (c->T == 0) return MOK_OK;
    SharedWs w;
    carve_shared(c, ws, &w);
    const int64_t T = c->T;
    const int H = c->H, I = c->I;
    const Ring ring{T, c->minibatch, 0};  // token order: row t is x[t]
    MOK_LAUNCH(KK_TILES, 2,
               first_error(launch_single_expert_offsets(w.offsets, T, stream),
                           launch_build_tiles(w.offsets, 1, 0, T, gemm_tc_tile_rows(true),
                                              w.tiles, w.tiles_cap, status, stream)));
    MOK_LAUNCH(KK_QUANTIZE, 1,
               launch_quantize_mxfp8((const uint16_t *)x, T, H, w.x_q, w.x_s, stream));
    MOK_LAUNCH(KK_SCALE_ATOMS, 3,
               first_error(first_error(launch_scale_atoms_rows(w13s_scale, 2 * (int64_t)I, H,
                                                               w.sf_w13, stream),
                                       launch_scale_atoms_rows(w2s_scale, H, I, w.sf_w2,
                                                               stream)),
                           launch_scale_atoms_tiles(w.tiles, w.tiles_cap, w.x_s, T,
                                                    c->minibatch, 0, H, w.sf_x, stream)));
    GemmUpArgs ua{w.tiles, w.tiles_cap, w.x_q, w.x_s, w13s_q, w13s_scale, w.h_q, w.h_s,
                  saved_preact_s, H, I, 1, true, ring, status};
    ua.preact_f32 = f32_storage(c);
    MOK_LAUNCH(KK_SHARED_UP, 1, launch_gemm_up_tc_mx(ua, T, w.sf_w13, w.sf_x, stream));
    MOK_LAUNCH(KK_SCALE_ATOMS, 1,
               launch_scale_atoms_tiles(w.tiles, w.tiles_cap, w.h_s, T, c->minibatch, 0, I,
                                        w.sf_h, stream));
    GemmDownArgs da{w.tiles, w.tiles_cap, w.h_q, w.h_s, w2s_q, w2s_scale, nullptr, y,
                    H, I, 1, true, ring, status, true};
    da.out_f32 = f32_storage(c);
    MOK_LAUNCH(KK_SHARED_DOWN, 1, launch_gemm_down_tc_mx(da, T, w.sf_w2, w.sf_h, stream));
    return MOK_OK;
}

}  // extern "C"

namespace {
// the shared expert's transposed, MXFP8-quantized weights (its MXFP8 backward)
struct MxSharedWeights {
    const uint8_t *w13t_q, *w13t_s, *w2t_q, *w2t_s;
};

mok_status shared_backward_impl(const mok_config *c, const void *x, const void *w13_s,
                                const void *w2_s, const MxSharedWeights *mxw,
                                const void *saved_preact_s, const void *dy, void *dx,
                                void *dw13_s, void *dw2_s, void *ws, size_t ws_bytes,
                                cudaStream_t stream) {
    mok_status st = mok_check_config(c);
    if (st != MOK_OK) return st;
    int *status;
    if ((st = check_device(&status)) != MOK_OK) return st;
    const bool mx = mxw != nullptr;
    if (!mx && c->prec != MOK_BF16) return MOK_ERR_UNSUPPORTED;
    if (mx && c->prec != MOK_MXFP8) return MOK_ERR_INVALID_ARG;
    if (!x || !saved_preact_s || !dy || !dx || !dw13_s || !dw2_s) return MOK_ERR_INVALID_ARG;
    if (!mx && (!w13_s || !w2_s)) return MOK_ERR_INVALID_ARG;
    if (mx && (!mxw->w13t_q || !mxw->w13t_s || !mxw->w2t_q || !mxw->w2t_s))
        return MOK_ERR_INVALID_ARG;
    const void *ps[] = {x, w13_s, w2_s, saved_preact_s, dy, dx, dw13_s, dw2_s,
                        mx ? mxw->w13t_q : nullptr, mx ? mxw->w2t_q : nullptr};
    for (const void *p : ps)
        if (p && !aligned16(p)) return MOK_ERR_INVALID_ARG;
    const size_t need = carve_shared_bwd(c, nullptr, nullptr);
    if ((st = check_ws(ws, ws_bytes, need)) != MOK_OK) return st;
    SharedBwdWs w;
    carve_shared_bwd(c, ws, &w);
    const int64_t T = c->T;
    const int H = c->H, I = c->I;
    // one expert owning every token in token order, weight one: x and dy are read directly
    MOK_LAUNCH(KK_SHARED_BWD, 2,
               first_error(launch_single_expert_bwd_setup(w.offsets, w.poff, w.counts, w.ones,
                                                          w.perm, T, stream),
                           launch_build_tiles(w.offsets, 1, 0, T, gemm_tc_tile_rows(mx),
                                              w.tiles, w.tiles_cap, status, stream)));
    if (T > 0) {
        GemmGArgs ga{w.tiles, w.tiles_cap, w.offsets, w.poff, (const uint16_t *)w2_s,
                     (const uint16_t *)dy, saved_preact_s, w.perm, w.ones, w.dA,
                     w.sh, w.dS_part, H, I, status};
        ga.preact_f32 = f32_storage(c);
        GemmDgradArgs dg{w.tiles, w.tiles_cap, w.offsets, w.poff, (const uint16_t *)w13_s,
                         w.dA, w.perm, dx, H, I, status};
        dg.accumulate = true;
        dg.out_f32 = f32_storage(c);
        if (mx) {
            // dy quantized along H in token order (the padded layout of a single expert is
            // the token order; rows past T are outside the TMA map and read zero)
            MOK_LAUNCH(KK_QUANTIZE, 1,
                       launch_quantize_mxfp8((const uint16_t *)dy, T, H, w.dy_q, w.dy_s,
                                             stream));
            MOK_LAUNCH(KK_SCALE_ATOMS, 3,
                       first_error(first_error(launch_scale_atoms_rows(mxw->w2t_s, I, H,
                                                                       w.sf_w2t, stream),
                                               launch_scale_atoms_rows(mxw->w13t_s, H, 2 * I,
                                                                       w.sf_w13t, stream)),
                                   launch_scale_atoms_tiles_padded(w.tiles, w.tiles_cap,
                                                                   w.dy_s, w.offsets, w.poff,
                                                                   H, w.sf_dy, stream)));
            ga.mxfp8 = true;
            ga.w2t_q = mxw->w2t_q;
            ga.sf_w2t = w.sf_w2t;
            ga.dy_q = w.dy_q;
            ga.sf_dy = w.sf_dy;
            ga.dA_q = w.dA_q;
            ga.dA_s = w.dA_s;
            dg.mxfp8 = true;
            dg.w13t_q = mxw->w13t_q;
            dg.sf_w13t = w.sf_w13t;
            dg.dA_q = w.dA_q;
            dg.sf_dA = w.sf_dA;
        }
        MOK_LAUNCH(KK_SHARED_BWD, 1, launch_gemm_g_tc(ga, 1, T, stream));  // dy: T rows
        if (mx)
            MOK_LAUNCH(KK_SCALE_ATOMS, 1,
                       launch_scale_atoms_tiles_padded(w.tiles, w.tiles_cap, w.dA_s, w.offsets,
                                                       w.poff, 2 * I, w.sf_dA, stream));
        if (gemm_pairs(c, mx, false)) {  // dx adds into the routed part
            MOK_LAUNCH(KK_TILES, 1,
                       launch_build_tiles(w.offsets, 1, 0, T, PAIR_TILE_ROWS, w.tiles,
                                          w.tiles_cap, status, stream));
            MOK_LAUNCH(KK_SHARED_BWD, 1, launch_gemm_dgrad_pair_tc(dg, 1, w.tpad, stream));
        } else {
            MOK_LAUNCH(KK_SHARED_BWD, 1, launch_gemm_dgrad_tc(dg, 1, w.tpad, stream));
        }
    }
    // the weight gradients' K runs over the padded rows: x and dy rows past T read zeros
    MOK_LAUNCH(KK_SHARED_BWD, 2,
               first_error(launch_wgrad(c, T, w.counts, w.poff, (const uint16_t *)x, w.dA,
                                        dw13_s, 1, H, 2 * I, T > 0 ? T : 1,
                                        w.tpad > 0 ? w.tpad : 1, status, stream),
                           launch_wgrad(c, T, w.counts, w.poff, w.sh, (const uint16_t *)dy,
                                        dw2_s, 1, I, H, w.tpad > 0 ? w.tpad : 1,
                                        T > 0 ? T : 1, status, stream)));
    return MOK_OK;
}
}  // namespace

extern "C" {

mok_status mok_shared_expert_backward(const mok_config *c, const void *x, const void *w13_s,
                                      const void *w2_s, const void *saved_preact_s,
                                      const void *dy, void *dx, void *dw13_s, void *dw2_s,
                                      void *ws, size_t ws_bytes, cudaStream_t stream) {
    return shared_backward_impl(c, x, w13_s, w2_s, nullptr, saved_preact_s, dy, dx, dw13_s,
                                dw2_s, ws, ws_bytes, stream);
}

mok_status mok_shared_expert_backward_mxfp8(const mok_config *c, const void *x,
                                            const uint8_t *w13st_q, const uint8_t *w13st_scale,
                                            const uint8_t *w2st_q, const uint8_t *w2st_scale,
                                            const void *saved_preact_s, const void *dy,
                                            void *dx, void *dw13_s, void *dw2_s, void *ws,
                                            size_t ws_bytes, cudaStream_t stream) {
    const MxSharedWeights mxw{w13st_q, w13st_scale, w2st_q, w2st_scale};
    return shared_backward_impl(c, x, nullptr, nullptr, &mxw, saved_preact_s, dy, dx, dw13_s,
                                dw2_s, ws, ws_bytes, stream);
}

mok_status mok_quantize_mxfp8(const void *src_bf16, int64_t rows, int32_t cols, uint8_t *q,
                              uint8_t *scale, cudaStream_t stream) {
    int *status;
    mok_status st = check_device(&status);
    if (st != MOK_OK) return st;
    if (rows < 0 || cols <= 0 || cols % 32 != 0) return MOK_ERR_INVALID_ARG;
    if (rows == 0) return MOK_OK;
    if (!src_bf16 || !q || !scale) return MOK_ERR_INVALID_ARG;
    if (!aligned16(src_bf16) || !aligned16(q)) return MOK_ERR_INVALID_ARG;
    MOK_LAUNCH(KK_QUANTIZE, 1,
               launch_quantize_mxfp8((const uint16_t *)src_bf16, rows, cols, q, scale, stream));
    return MOK_OK;
}

mok_status mok_quantize_mxfp8_transposed(const void *src_bf16, int64_t batch, int32_t rows,
                                         int32_t cols, uint8_t *q, uint8_t *scale,
                                         cudaStream_t stream) {
    int *status;
    mok_status st = check_device(&status);
    if (st != MOK_OK) return st;
    if (batch < 0 || rows <= 0 || cols <= 0 || rows % 32 != 0) return MOK_ERR_INVALID_ARG;
    if (batch == 0) return MOK_OK;
    if (!src_bf16 || !q || !scale) return MOK_ERR_INVALID_ARG;
    // each 32-byte block of q is written with two 16-byte stores
    if (!aligned16(src_bf16) || !aligned16(q)) return MOK_ERR_INVALID_ARG;
    MOK_LAUNCH(KK_QUANTIZE, 1,
               launch_quantize_mxfp8_transposed((const uint16_t *)src_bf16, batch, rows, cols,
                                                q, scale, stream));
    return MOK_OK;
}

mok_status mok_selftest_bounded_wait(uint32_t limit_us, cudaStream_t stream) {
    int *status;
    mok_status st = check_device(&status);
    if (st != MOK_OK) return st;
    if (limit_us == 0 || limit_us > 1000000u) return MOK_ERR_INVALID_ARG;
    if (launch_bounded_wait_probe(status, (uint64_t)limit_us * 1000ull, stream) != cudaSuccess)
        return MOK_ERR_CUDA;
    return MOK_OK;
}

mok_status mok_selftest_bounded_count_wait(uint32_t limit_us, cudaStream_t stream) {
    int *status;
    mok_status st = check_device(&status);
    if (st != MOK_OK) return st;
    if (limit_us == 0 || limit_us > 1000000u) return MOK_ERR_INVALID_ARG;
    if (launch_bounded_count_probe(status, (uint64_t)limit_us * 1000ull, stream) != cudaSuccess)
        return MOK_ERR_CUDA;
    return MOK_OK;
}

mok_status mok_read_device_status(mok_status *out) {
    if (out == nullptr) return MOK_ERR_INVALID_ARG;
    int *status;
    mok_status st = check_device(&status);
    if (st != MOK_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOK_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return MOK_ERR_CUDA;
    *out = (mok_status)v;
    return MOK_OK;
}

mok_status mok_clear_device_status(void) {
    int *status;
    mok_status st = check_device(&status);
    if (st != MOK_OK) return st;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return MOK_ERR_CUDA;
    return MOK_OK;
}

}  // extern "C"
