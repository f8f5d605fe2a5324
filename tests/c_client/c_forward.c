/* A plain C client of libmok: routes, schedules and runs the BF16 layer forward on inputs
 * read from files, then writes y and the top-k indices. It uses nothing but the C ABI of
 * include/mok.h and the CUDA runtime.
 *
 * usage: c_forward T H I E K minibatch ring_capacity dir
 *   dir/x.bin      bf16 [T][H]       dir/logits.bin  fp32 [T][E]
 *   dir/w13.bin    bf16 [E][2I][H]   dir/w2.bin      bf16 [E][H][I]
 * writes dir/y.bin (bf16 [T][H]) and dir/idx.bin (int32 [T][K]); exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "mok.h"

#define MOK_CHECK(x)                                                                 \
    do {                                                                             \
        mok_status s_ = (x);                                                         \
        if (s_ != MOK_OK) {                                                          \
            fprintf(stderr, "%s: %s\n", #x, mok_status_string(s_));                  \
            return 1;                                                                \
        }                                                                            \
    } while (0)
#define CUDA_CHECK(x)                                                                \
    do {                                                                             \
        cudaError_t e_ = (x);                                                        \
        if (e_ != cudaSuccess) {                                                     \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                 \
            return 1;                                                                \
        }                                                                            \
    } while (0)

static void *read_file(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (f == NULL) return NULL;
    void *p = malloc(bytes ? bytes : 1);
    if (p != NULL && fread(p, 1, bytes, f) != bytes) {
        free(p);
        p = NULL;
    }
    fclose(f);
    return p;
}

static int write_file(const char *dir, const char *name, const void *p, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (f == NULL) return 1;
    const int bad = fwrite(p, 1, bytes, f) != bytes;
    return fclose(f) != 0 || bad;
}

int main(int argc, char **argv) {
    if (argc != 9) {
        fprintf(stderr, "usage: %s T H I E K minibatch ring_capacity dir\n", argv[0]);
        return 2;
    }
    mok_config cfg;
    cfg.abi_version = MOK_ABI_VERSION;
    cfg.T = atoi(argv[1]);
    cfg.H = atoi(argv[2]);
    cfg.I = atoi(argv[3]);
    cfg.E = atoi(argv[4]);
    cfg.K = atoi(argv[5]);
    cfg.minibatch = atoi(argv[6]);
    cfg.ring_capacity = atoi(argv[7]);
    cfg.prec = MOK_BF16;
    cfg.flags = 0; /* bf16 storage: y is bf16 */
    const char *dir = argv[8];
    MOK_CHECK(mok_check_config(&cfg));

    const size_t T = (size_t)cfg.T, H = (size_t)cfg.H, I = (size_t)cfg.I, E = (size_t)cfg.E,
                 K = (size_t)cfg.K, R = T * K;
    const size_t nx = T * H * 2, nl = T * E * 4, n13 = E * 2 * I * H * 2, n2 = E * H * I * 2;
    void *hx = read_file(dir, "x.bin", nx), *hl = read_file(dir, "logits.bin", nl);
    void *h13 = read_file(dir, "w13.bin", n13), *h2 = read_file(dir, "w2.bin", n2);
    if (!hx || !hl || !h13 || !h2) {
        fprintf(stderr, "missing or short input file in %s\n", dir);
        return 1;
    }

    /* caller-owned device buffers: inputs, routing, schedule, output, workspaces */
    void *x, *logits, *w13, *w2, *y, *ws_s, *ws_f;
    int32_t *idx, *counts, *offsets, *perm, *inv, *segs, *n_segs;
    float *topk_w;
    const size_t cap = (size_t)mok_segment_capacity(&cfg);
    const size_t nws_s = mok_workspace_size(&cfg, MOK_WS_SCHEDULE);
    const size_t nws_f = mok_workspace_size(&cfg, MOK_WS_FORWARD);
    CUDA_CHECK(cudaMalloc(&x, nx));
    CUDA_CHECK(cudaMalloc(&logits, nl));
    CUDA_CHECK(cudaMalloc(&w13, n13));
    CUDA_CHECK(cudaMalloc(&w2, n2));
    CUDA_CHECK(cudaMalloc(&y, T * H * 2));
    CUDA_CHECK(cudaMalloc((void **)&idx, R * 4));
    CUDA_CHECK(cudaMalloc((void **)&topk_w, R * 4));
    CUDA_CHECK(cudaMalloc((void **)&counts, E * 4));
    CUDA_CHECK(cudaMalloc((void **)&offsets, (E + 1) * 4));
    CUDA_CHECK(cudaMalloc((void **)&perm, R * 4));
    CUDA_CHECK(cudaMalloc((void **)&inv, R * 4));
    CUDA_CHECK(cudaMalloc((void **)&segs, cap * 3 * 4));
    CUDA_CHECK(cudaMalloc((void **)&n_segs, 4));
    CUDA_CHECK(cudaMalloc(&ws_s, nws_s ? nws_s : 1));
    CUDA_CHECK(cudaMalloc(&ws_f, nws_f ? nws_f : 1));
    CUDA_CHECK(cudaMemcpy(x, hx, nx, cudaMemcpyHostToDevice));
    CUDA_CHECK(cudaMemcpy(logits, hl, nl, cudaMemcpyHostToDevice));
    CUDA_CHECK(cudaMemcpy(w13, h13, n13, cudaMemcpyHostToDevice));
    CUDA_CHECK(cudaMemcpy(w2, h2, n2, cudaMemcpyHostToDevice));
    mok_schedule sched = {counts, offsets, perm, inv, segs, n_segs};

    cudaStream_t stream;
    CUDA_CHECK(cudaStreamCreate(&stream));
    MOK_CHECK(mok_clear_device_status());
    MOK_CHECK(mok_route_topk(&cfg, (const float *)logits, idx, topk_w, stream));
    MOK_CHECK(mok_build_schedule(&cfg, idx, &sched, ws_s, nws_s, stream));
    MOK_CHECK(mok_forward(&cfg, x, &sched, topk_w, w13, NULL, w2, NULL, y, NULL, ws_f, nws_f,
                          stream));
    CUDA_CHECK(cudaStreamSynchronize(stream));
    mok_status dev = MOK_OK;
    MOK_CHECK(mok_read_device_status(&dev));
    if (dev != MOK_OK) {
        fprintf(stderr, "device status: %s\n", mok_status_string(dev));
        return 1;
    }

    uint16_t *hy = (uint16_t *)malloc(T * H * 2);
    int32_t *hidx = (int32_t *)malloc(R * 4);
    if (!hy || !hidx) return 1;
    CUDA_CHECK(cudaMemcpy(hy, y, T * H * 2, cudaMemcpyDeviceToHost));
    CUDA_CHECK(cudaMemcpy(hidx, idx, R * 4, cudaMemcpyDeviceToHost));
    if (write_file(dir, "y.bin", hy, T * H * 2) || write_file(dir, "idx.bin", hidx, R * 4)) {
        fprintf(stderr, "cannot write outputs to %s\n", dir);
        return 1;
    }

    void *dev_ptrs[] = {x, logits, w13, w2, y, idx, topk_w, counts, offsets, perm, inv, segs,
                        n_segs, ws_s, ws_f};
    for (size_t i = 0; i < sizeof dev_ptrs / sizeof dev_ptrs[0]; ++i) cudaFree(dev_ptrs[i]);
    cudaStreamDestroy(stream);
    free(hx);
    free(hl);
    free(h13);
    free(h2);
    free(hy);
    free(hidx);
    return 0;
}
