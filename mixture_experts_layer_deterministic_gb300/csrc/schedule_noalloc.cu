// schedule_noalloc.cu -- mok_build_schedule_noalloc, the schedule builder for callers that
// cannot allocate device memory.
//
// mok_build_schedule needs a caller-allocated workspace for its per-chunk expert
// histograms. Some callers cannot make one: code that runs under a device-memory budget
// owned by someone else (a host framework or server that hands out all GPU memory from its
// own pool and forbids raw cudaMalloc), or a time-critical loop that cannot afford
// cudaMalloc's latency and implicit device synchronisation. This variant keeps that scratch
// in a fixed array in the library's own device memory instead. The array is a file-scope
// __device__ variable of MOK_NOALLOC_SCHEDULE_SCRATCH_BYTES (4 MiB): every GPU that loads
// the library holds it until the process exits, and the entry point allocates nothing.
#include <atomic>

#include "common.cuh"
#include "mok_internal.h"

namespace {

static __device__ __align__(256) int32_t
    g_noalloc_sched_scratch[MOK_NOALLOC_SCHEDULE_SCRATCH_BYTES / sizeof(int32_t)];

// Device address of the scratch array, per device. In host code the array's name is only
// a host-side stand-in, never a device address, so the address is looked up once per
// device (with that device current) and cached here. Host threads may make their first
// call on a device at the same time: the cache is atomic, and both store the same address.
std::atomic<int32_t *> g_scratch_dev[mok::MAX_DEV];

}  // namespace

extern "C" mok_status mok_build_schedule_noalloc(const mok_config *cfg,
                                                 const int32_t *topk_idx,
                                                 const mok_schedule *sched,
                                                 cudaStream_t stream) {
    mok_status st = mok_check_config(cfg);
    if (st != MOK_OK) return st;
    int *status = nullptr;
    if ((st = mok::current_device_status_word(&status)) != MOK_OK) return st;
    if (sched == nullptr || !sched->counts || !sched->offsets || !sched->perm || !sched->inv ||
        !sched->segs || !sched->n_segs)
        return MOK_ERR_INVALID_ARG;
    const int64_t R = (int64_t)cfg->T * cfg->K;
    if (R > 0 && (topk_idx == nullptr || ((uintptr_t)topk_idx & 15u) != 0))
        return MOK_ERR_INVALID_ARG;
    // the scratch holds the per-chunk histograms; refuse sizes that would not fit
    if (mok::schedule_ws_bytes(R, cfg->E) > MOK_NOALLOC_SCHEDULE_SCRATCH_BYTES)
        return MOK_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= mok::MAX_DEV) return MOK_ERR_CUDA;
    int32_t *scratch = g_scratch_dev[dev].load(std::memory_order_acquire);
    if (scratch == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_sched_scratch) != cudaSuccess || p == nullptr)
            return MOK_ERR_CUDA;
        scratch = (int32_t *)p;
        g_scratch_dev[dev].store(scratch, std::memory_order_release);
    }
    // Nothing in the scratch has to start at zero: the first kernel writes every
    // histogram entry that the later kernels read.
    mok::ScheduleWs w = mok::schedule_ws_carve(scratch, R, cfg->E);
    // timed under the same kind as mok_build_schedule while profiling is on
    mok::prof_begin(mok::KK_SCHEDULE, stream);
    const cudaError_t e =
        mok::launch_build_schedule(topk_idx, R, cfg->E, cfg->minibatch, *sched, w, status, stream);
    mok::prof_end(mok::KK_SCHEDULE, stream, R > 0 ? 4 : 1);
    return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}
