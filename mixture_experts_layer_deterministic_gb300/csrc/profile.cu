// profile.cu -- opt-in per-kernel timing with CUDA events (host code only).
#include <vector>

#include "common.cuh"
#include "mok_internal.h"

namespace mok {
namespace {

const char *const kNames[KK_COUNT] = {
    "route_topk", "schedule", "build_tiles", "gather", "gemm_up_swiglu", "gemm_down_push",
    "combine", "quantize_mxfp8", "pad_offsets", "gather_bwd", "gemm_g_swiglu_bwd",
    "router_grad", "gemm_dgrad_push", "dx_reduce", "wgrad_w13", "wgrad_w2", "scale_atoms",
    "shared_up_swiglu", "shared_down_add", "shared_backward", "ring_forward"};

struct Rec {
    int kind;
    int n;
    size_t ev;  // index of the start event; ev + 1 is the end event
};

bool g_on = false;
std::vector<cudaEvent_t> g_events;
std::vector<Rec> g_recs;
size_t g_next = 0;
int g_open_kind = -1;

cudaEvent_t next_event() {
    if (g_next == g_events.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_events.push_back(e);
    }
    return g_events[g_next++];
}

}  // namespace

bool prof_on() { return g_on; }

void prof_begin(int kind, cudaStream_t s) {
    if (!g_on) return;
    cudaEvent_t a = next_event();
    if (a) cudaEventRecord(a, s);
    g_open_kind = kind;
}

void prof_end(int kind, cudaStream_t s, int n_kernels) {
    if (!g_on || g_open_kind != kind) return;
    cudaEvent_t b = next_event();
    if (b) cudaEventRecord(b, s);
    g_recs.push_back(Rec{kind, n_kernels, g_next - 2});
    g_open_kind = -1;
}

}  // namespace mok

extern "C" mok_status mok_profile_enable(int on) {
    mok::g_on = on != 0;
    if (mok::g_on) {
        mok::g_recs.clear();
        mok::g_next = 0;
    }
    return MOK_OK;
}

extern "C" mok_status mok_profile_read(int32_t max, int32_t *n_kinds, const char **names,
                                       int64_t *launches, double *ms) {
    using namespace mok;
    if (n_kinds == nullptr) return MOK_ERR_INVALID_ARG;
    double tot[KK_COUNT] = {0};
    int64_t cnt[KK_COUNT] = {0};
    for (const Rec &r : g_recs) {
        if (cudaEventSynchronize(g_events[r.ev + 1]) != cudaSuccess) return MOK_ERR_CUDA;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, g_events[r.ev], g_events[r.ev + 1]) != cudaSuccess)
            return MOK_ERR_CUDA;
        tot[r.kind] += t;
        cnt[r.kind] += r.n;
    }
    int32_t n = 0;
    for (int k = 0; k < KK_COUNT; ++k) {
        if (cnt[k] == 0) continue;
        if (n < max) {
            if (names) names[n] = kNames[k];
            if (launches) launches[n] = cnt[k];
            if (ms) ms[n] = tot[k];
        }
        ++n;
    }
    *n_kinds = n;
    return MOK_OK;
}
