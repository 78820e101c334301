/*
 * pa_c_client.c -- drives libpagedattn from plain C (no Python, no torch):
 * create a bf16 pool, take blocks from the free stack, append tokens with
 * pa_write_kv, decode with pa_decode_attention (split and unsplit), read the
 * status word, and compare against the CPU oracle linked into this test.
 * Exit code 0 on success.  Test infrastructure only.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "pagedattn.h"

/* from oracle/pa_oracle.c */
int oracle_decode_attention(double* out, const void* q, const void* pool, int dtype,
                            int num_blocks, int num_layers, int num_kv_heads, int block_size,
                            int head_dim, int layer, const int* block_tables,
                            int max_blocks_per_seq, const int* context_lens, int batch,
                            int num_heads, double scale, int num_threads);
int oracle_write_kv(void* pool, int dtype, int num_blocks, int num_layers, int num_kv_heads,
                    int block_size, int head_dim, int layer, const void* k, const void* v,
                    const int* block_tables, int max_blocks_per_seq, const int* positions,
                    int batch);

#define CHECK(x)                                                                   \
    do {                                                                           \
        int rc_ = (x);                                                             \
        if (rc_ != 0) {                                                            \
            fprintf(stderr, "%s:%d %s -> %d (%s)\n", __FILE__, __LINE__, #x, rc_,  \
                    pa_last_error_string());                                       \
            return 1;                                                              \
        }                                                                          \
    } while (0)

static uint16_t to_bf16(float f) { /* round to nearest even */
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static uint32_t lcg = 12345u;
static float frand(void) { /* uniform in [-1, 1) */
    lcg = lcg * 1664525u + 1013904223u;
    return (float)((lcg >> 8) & 0xffffff) / 8388608.0f - 1.0f;
}

int main(void) {
    enum { NB = 64, L = 2, HKV = 2, B = 16, D = 128, H = 8, BATCH = 3, MAXB = 8, STEPS = 40 };
    const size_t pool_elems = (size_t)NB * 2 * L * HKV * B * D;
    uint16_t* host_pool = calloc(pool_elems, 2);
    void* dpool = NULL;
    if (cudaMalloc(&dpool, pool_elems * 2) != cudaSuccess) return 2;
    if (cudaMemset(dpool, 0, pool_elems * 2) != cudaSuccess) return 2;
    pa_pool* pool = NULL;
    CHECK(pa_pool_create(&pool, dpool, NB, L, HKV, B, D, PA_DTYPE_BF16));

    int tables[BATCH * MAXB];
    int lens[BATCH] = {0, 0, 0};
    for (int i = 0; i < BATCH * MAXB; ++i) tables[i] = -1;
    int *dbt, *dpos, *dlens;
    void *dk, *dv, *dq;
    float* dout;
    cudaMalloc((void**)&dbt, sizeof tables);
    cudaMalloc((void**)&dpos, sizeof lens);
    cudaMalloc((void**)&dlens, sizeof lens);
    cudaMalloc(&dk, BATCH * HKV * D * 2);
    cudaMalloc(&dv, BATCH * HKV * D * 2);
    cudaMalloc(&dq, BATCH * H * D * 2);
    cudaMalloc((void**)&dout, BATCH * H * D * 4);
    uint16_t k[BATCH * HKV * D], v[BATCH * HKV * D], q[BATCH * H * D];
    for (int step = 0; step < STEPS; ++step) {
        for (int b = 0; b < BATCH; ++b) {
            if (b == 2 && step >= 25) continue; /* ragged: sequence 2 stops at 25 tokens */
            if (lens[b] % B == 0) CHECK(pa_alloc_block(pool, &tables[b * MAXB + lens[b] / B]));
        }
        for (int layer = 0; layer < L; ++layer) {
            for (int i = 0; i < BATCH * HKV * D; ++i) {
                k[i] = to_bf16(frand());
                v[i] = to_bf16(frand());
            }
            int pos[BATCH];
            int nb = 0;
            for (int b = 0; b < BATCH; ++b)
                if (!(b == 2 && step >= 25)) pos[nb++] = lens[b];
            /* sequences 0, 1 (and 2 while it grows) append at their length */
            cudaMemcpy(dbt, tables, sizeof tables, cudaMemcpyHostToDevice);
            cudaMemcpy(dpos, pos, sizeof pos, cudaMemcpyHostToDevice);
            cudaMemcpy(dk, k, sizeof k, cudaMemcpyHostToDevice);
            cudaMemcpy(dv, v, sizeof v, cudaMemcpyHostToDevice);
            CHECK(pa_write_kv(pool, layer, dk, dv, dbt, MAXB, dpos, nb, NULL));
            CHECK(oracle_write_kv(host_pool, 1, NB, L, HKV, B, D, layer, k, v, tables, MAXB, pos,
                                  nb));
        }
        for (int b = 0; b < BATCH; ++b)
            if (!(b == 2 && step >= 25)) lens[b] += 1;
    }
    for (int i = 0; i < BATCH * H * D; ++i) q[i] = to_bf16(frand());
    cudaMemcpy(dq, q, sizeof q, cudaMemcpyHostToDevice);
    cudaMemcpy(dlens, lens, sizeof lens, cudaMemcpyHostToDevice);
    const float scale = 1.0f / sqrtf((float)D);
    double* ref = malloc(sizeof(double) * BATCH * H * D);
    float* got = malloc(sizeof(float) * BATCH * H * D);
    for (int layer = 0; layer < L; ++layer) {
        CHECK(oracle_decode_attention(ref, q, host_pool, 1, NB, L, HKV, B, D, layer, tables, MAXB,
                                      lens, BATCH, H, scale, 1));
        for (int pb = 0; pb <= 2; pb += 2) { /* heuristic (here one partition), then 2 blocks */
            size_t ws_bytes = 0;
            CHECK(pa_decode_workspace_size(pool, BATCH, H, MAXB, pb, &ws_bytes));
            void* ws = NULL;
            if (ws_bytes) cudaMalloc(&ws, ws_bytes);
            CHECK(pa_decode_attention_partitioned(dout, dq, pool, layer, dbt, MAXB, dlens, BATCH,
                                                  B, H, HKV, D, scale, pb, ws, ws_bytes, NULL));
            cudaMemcpy(got, dout, sizeof(float) * BATCH * H * D, cudaMemcpyDeviceToHost);
            double err = 0.0;
            for (int i = 0; i < BATCH * H * D; ++i) err = fmax(err, fabs(got[i] - ref[i]));
            printf("layer %d partition_blocks %d: max abs err %.3e\n", layer, pb, err);
            if (!(err <= 2e-3)) return 3;
            if (ws) cudaFree(ws);
        }
    }
    /* the appended pool is bit-identical to the oracle's */
    uint16_t* back = malloc(pool_elems * 2);
    cudaMemcpy(back, dpool, pool_elems * 2, cudaMemcpyDeviceToHost);
    if (memcmp(back, host_pool, pool_elems * 2) != 0) {
        fprintf(stderr, "pool bytes differ\n");
        return 4;
    }
    unsigned status = 0;
    CHECK(pa_get_status(&status, NULL));
    if (status != 0) return 5;
    int nfree = 0;
    CHECK(pa_num_free(pool, &nfree));
    printf("free blocks left: %d\n", nfree);
    CHECK(pa_pool_destroy(pool));
    printf("c client ok\n");
    return 0;
}
