/* The C ABI used from plain C (no Python, no C++): one round of two clients over two keys,
 * client 1 sending only key 0, with values whose weighted means are exact in fp32 and bf16.
 *   key 0: (1*2.0 + 3*6.0) / (1 + 3) = 5.0
 *   key 1: only client 0 sends it: (1*-1.5) / 1 = -1.5
 * Exits 0 on success; prints what differs otherwise. */
#include <fedavg.h>

#include <cuda_runtime.h>

#include <stdio.h>
#include <stdlib.h>

#define CHECK(cond, ...)                      \
    do {                                      \
        if (!(cond)) {                        \
            fprintf(stderr, __VA_ARGS__);     \
            fprintf(stderr, "\n");            \
            return 1;                         \
        }                                     \
    } while (0)

int main(void) {
    enum { N0 = 4099, N1 = 17 };
    fa_key layout[2] = {{"weight", N0}, {"bias", N1}};
    fa_ctx* ctx = NULL;
    fa_status st = fa_open(layout, 2, FA_F32, FA_F32, 2, NULL, &ctx);
    CHECK(st == FA_OK, "fa_open: %s", fa_strerror(st));

    float* host = (float*)malloc(sizeof(float) * N0);
    float *c0k0, *c1k0, *c0k1, *out0, *out1;
    CHECK(cudaMalloc((void**)&c0k0, sizeof(float) * N0) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&c1k0, sizeof(float) * N0) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&c0k1, sizeof(float) * N1) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&out0, sizeof(float) * N0) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&out1, sizeof(float) * N1) == cudaSuccess, "cudaMalloc");
    for (int i = 0; i < N0; ++i) host[i] = 2.0f;
    cudaMemcpy(c0k0, host, sizeof(float) * N0, cudaMemcpyHostToDevice);
    for (int i = 0; i < N0; ++i) host[i] = 6.0f;
    cudaMemcpy(c1k0, host, sizeof(float) * N0, cudaMemcpyHostToDevice);
    for (int i = 0; i < N1; ++i) host[i] = -1.5f;
    cudaMemcpy(c0k1, host, sizeof(float) * N1, cudaMemcpyHostToDevice);

    /* client 0 sends key 0 in two chunks and key 1; client 1 sends key 0 */
    st = fa_accumulate(ctx, 0, 1.0, 0, 0, c0k0, 1000, NULL);
    CHECK(st == FA_OK, "accumulate: %s (%s)", fa_strerror(st), fa_last_error(ctx));
    st = fa_accumulate(ctx, 0, 1.0, 0, 1000, c0k0 + 1000, N0 - 1000, NULL);
    CHECK(st == FA_OK, "accumulate: %s", fa_strerror(st));
    st = fa_accumulate(ctx, 0, 1.0, 1, 0, c0k1, N1, NULL);
    CHECK(st == FA_OK, "accumulate: %s", fa_strerror(st));
    st = fa_accumulate(ctx, 1, 3.0, 0, 0, c1k0, N0, NULL);
    CHECK(st == FA_OK, "accumulate: %s", fa_strerror(st));
    /* a weight unlike client 1's earlier chunk is refused and changes nothing */
    st = fa_accumulate(ctx, 1, 4.0, 1, 0, c0k1, N1, NULL);
    CHECK(st == FA_ERR_WEIGHT, "expected FA_ERR_WEIGHT, got %d", (int)st);

    void* outs[2] = {out0, out1};
    st = fa_finalize(ctx, outs, NULL);
    CHECK(st == FA_OK, "finalize: %s (%s)", fa_strerror(st), fa_last_error(ctx));
    st = fa_sync(ctx);
    CHECK(st == FA_OK, "sync: %s", fa_strerror(st));

    double total = 0.0;
    uint32_t reporters = 0;
    CHECK(fa_key_total(ctx, 0, &total, &reporters) == FA_OK && total == 4.0 && reporters == 2,
          "key 0 totals %g / %u", total, reporters);
    CHECK(fa_key_total(ctx, 1, &total, &reporters) == FA_OK && total == 1.0 && reporters == 1,
          "key 1 totals %g / %u", total, reporters);

    cudaMemcpy(host, out0, sizeof(float) * N0, cudaMemcpyDeviceToHost);
    for (int i = 0; i < N0; ++i) CHECK(host[i] == 5.0f, "key 0 [%d] = %g, want 5", i, host[i]);
    cudaMemcpy(host, out1, sizeof(float) * N1, cudaMemcpyDeviceToHost);
    for (int i = 0; i < N1; ++i) CHECK(host[i] == -1.5f, "key 1 [%d] = %g, want -1.5", i, host[i]);

    fa_stats stats;
    CHECK(fa_get_stats(ctx, &stats) == FA_OK && stats.chunks == 4, "stats: %llu chunks",
          (unsigned long long)stats.chunks);
    CHECK(fa_close(ctx) == FA_OK, "fa_close");
    cudaFree(c0k0);
    cudaFree(c1k0);
    cudaFree(c0k1);
    cudaFree(out0);
    cudaFree(out1);
    free(host);
    printf("c abi example ok\n");
    return 0;
}
