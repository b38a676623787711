/* A plain C client of the C ABI (include/slide.h): no Python, no torch.
 *
 *   abi_client cpu   host-only calls (accounting, argument checks)
 *   abi_client gpu   a layer step on the GPU with gradients allocated by the
 *                    client: zero gradients from zero moments make the update
 *                    pure decay, theta_1 = fl(theta_0 * (1 - lr*wd)), and the
 *                    BF16 copy is the RNE rounding of that master.
 * Exit status 0 on success; prints what failed otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "slide.h"

#define CHECK(cond, ...)                                                                  \
    do {                                                                                  \
        if (!(cond)) {                                                                    \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__);                          \
            fprintf(stderr, __VA_ARGS__);                                                 \
            fprintf(stderr, " (last error: %s)\n", slide_last_error());                  \
            return 1;                                                                     \
        }                                                                                 \
    } while (0)

static uint16_t to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    uint32_t keep = u >> 16, rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep++;
    return (uint16_t)keep;
}

static int cpu_checks(void)
{
    int64_t numel[3] = {1000, 7, 0};
    slide_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.n_layers = 3;
    cfg.layer_numel = numel;
    cfg.n_replicas = 2;
    cfg.residency = SLIDE_RESIDENCY_HOST_STREAMED;
    int64_t dev = -1, host = -1;
    CHECK(slide_state_bytes(&cfg, &dev, &host) == SLIDE_OK, "slide_state_bytes");
    CHECK(host >= 14 * 1007 && host <= 14 * 1007 + 4 * 256 * 3, "host bytes %lld", (long long)host);
    CHECK(dev > 0, "window bytes");
    cfg.n_replicas = 9;
    CHECK(slide_state_bytes(&cfg, &dev, &host) == SLIDE_ERR_INVALID_ARG, "R = 9 accepted");
    CHECK(strstr(slide_last_error(), "n_replicas") != NULL, "message");
    CHECK(slide_abi_version() == SLIDE_ABI_VERSION, "abi version");
    slide_state_destroy(NULL);
    return 0;
}

static int gpu_checks(void)
{
    const int64_t n = 100003;
    const int R = 2;
    int64_t numel[1] = {n};
    slide_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.n_layers = 1;
    cfg.layer_numel = numel;
    cfg.n_replicas = R;
    cfg.residency = SLIDE_RESIDENCY_HBM;
    slide_state *st = NULL;
    CHECK(slide_state_create(&cfg, &st) == SLIDE_OK && st, "slide_state_create");

    float *th0 = malloc(n * sizeof(float)), *th = malloc(n * sizeof(float));
    float *m = malloc(n * sizeof(float)), *v = malloc(n * sizeof(float));
    uint16_t *w = malloc(n * sizeof(uint16_t));
    for (int64_t i = 0; i < n; ++i)
        th0[i] = (float)((i % 2001) - 1000) * 1e-5f;
    CHECK(slide_layer_set(st, 0, th0, NULL, NULL, 0) == SLIDE_OK, "slide_layer_set");

    void *grads[2] = {NULL, NULL};
    for (int r = 0; r < R; ++r) {
        CHECK(cudaMalloc(&grads[r], (size_t)n * 2) == cudaSuccess, "cudaMalloc");
        CHECK(cudaMemset(grads[r], 0, (size_t)n * 2) == cudaSuccess, "cudaMemset");
    }
    slide_adam_hparams hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.1f, 1.0f};
    const float decay = (float)(1.0 - (double)hp.lr * (double)hp.weight_decay);
    for (int t = 1; t <= 3; ++t)
        CHECK(slide_layer_step(st, 0, (const void *const *)grads, &hp, NULL, NULL) == SLIDE_OK, "step %d", t);
    int64_t t = 0;
    CHECK(slide_layer_get(st, 0, th, m, v, w, &t) == SLIDE_OK && t == 3, "slide_layer_get / t");
    for (int64_t i = 0; i < n; ++i) {
        float e = th0[i];
        for (int k = 0; k < 3; ++k)
            e = e * decay;
        CHECK(th[i] == e, "theta[%lld] = %.9g, want %.9g", (long long)i, th[i], e);
        CHECK(m[i] == 0.0f && v[i] == 0.0f, "moments not zero at %lld", (long long)i);
        CHECK(w[i] == to_bf16(th[i]), "bf16 copy at %lld", (long long)i);
    }
    /* a misaligned replica pointer is refused and nothing changes */
    void *bad[2] = {(char *)grads[0] + 2, grads[1]};
    CHECK(slide_layer_step(st, 0, (const void *const *)bad, &hp, NULL, NULL) == SLIDE_ERR_INVALID_ARG, "misaligned");
    CHECK(slide_layer_get(st, 0, NULL, NULL, NULL, NULL, &t) == SLIDE_OK && t == 3, "t after refused step");
    for (int r = 0; r < R; ++r)
        cudaFree(grads[r]);
    slide_state_destroy(st);

    /* the same closed form with the gradients in host memory and the BF16
     * copy delivered to host memory: slide_layer_step_host */
    cfg.flags = SLIDE_FLAG_HOST_INPUTS;
    CHECK(slide_state_create(&cfg, &st) == SLIDE_OK && st, "slide_state_create (host inputs)");
    CHECK(slide_layer_set(st, 0, th0, NULL, NULL, 0) == SLIDE_OK, "slide_layer_set (host inputs)");
    uint16_t *hg[2] = {calloc(n, 2), calloc(n, 2)};
    uint16_t *wout = malloc(n * sizeof(uint16_t));
    const void *hptr[2] = {hg[0], hg[1]};
    for (int k = 1; k <= 3; ++k)
        CHECK(slide_layer_step_host(st, 0, hptr, &hp, NULL, wout) == SLIDE_OK, "host step %d", k);
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "sync");
    CHECK(slide_layer_get(st, 0, th, m, v, w, &t) == SLIDE_OK && t == 3, "slide_layer_get / t (host inputs)");
    for (int64_t i = 0; i < n; ++i) {
        float e = th0[i];
        for (int k = 0; k < 3; ++k)
            e = e * decay;
        CHECK(th[i] == e, "host inputs: theta[%lld] = %.9g, want %.9g", (long long)i, th[i], e);
        CHECK(wout[i] == to_bf16(e), "host inputs: delivered bf16 copy at %lld", (long long)i);
    }
    slide_state_destroy(st);
    free(hg[0]), free(hg[1]), free(wout);
    free(th0), free(th), free(m), free(v), free(w);
    return 0;
}

int main(int argc, char **argv)
{
    if (argc < 2) {
        fprintf(stderr, "usage: abi_client cpu|gpu\n");
        return 2;
    }
    int rc = cpu_checks();
    if (rc == 0 && strcmp(argv[1], "gpu") == 0)
        rc = gpu_checks();
    if (rc == 0)
        printf("abi_client %s: ok\n", argv[1]);
    return rc;
}
