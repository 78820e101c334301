/*
 * pa_oracle.c -- plain, slow, CPU reference for paged KV-cache decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, constant or helper with
 * the CUDA library.
 *
 * What it follows:
 *  - Pool layout: one tensor [num_blocks, 2 (K/V), num_layers, num_kv_heads,
 *    block_size, head_dim] ("Paged KV-Cache Memory Management", mini-infer,
 *    section "Python Implementation: Physical Block Pool", BlockPool.__init__).
 *  - Slot resolution: logical token t of a sequence lives in physical block
 *    block_table[t / B] at offset t % B ("vllmini", section "PagedAttention
 *    Metaphor"; "kv-cache" skill, section 2 "Block Tables"; mini-infer,
 *    section "The Solution", Block Table).
 *  - Decode attention: for every sequence b and query head h, walk the block
 *    table, gather the n = context_lens[b] cached K and V rows contiguously,
 *    then out = softmax(scale * K q) V, entirely in fp64.  Query head h reads
 *    KV head h / (num_heads / num_kv_heads) (contiguous GQA groups).
 *  - KV append: the new token's K and V rows are copied into slot
 *    (block_table[p / B], p % B) of the given layer, p = positions[b]
 *    ("kv-cache" skill, section 2, Zero-Waste Allocation; mini-infer,
 *    Physical Blocks).
 *  - Batched gather: past K/V of every sequence copied into contiguous
 *    [batch, T, num_kv_heads, head_dim] plus a validity mask (mini-infer,
 *    section "Zero-Copy Batched Attention Gather").
 *
 * Element types: 0 = fp32, 1 = bf16.  bf16 values are widened exactly
 * (bits << 16) to fp32 and then to fp64.
 *
 * Every function returns 0 on success and a negative value when an argument
 * is out of range (a block id outside [0, num_blocks), a length above the
 * table's capacity, a layer outside [0, num_layers), ...).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1

static size_t elem_bytes(int dtype) { return dtype == ORC_F32 ? 4u : 2u; }

/* Exact widening of one stored element to fp64. */
static double load_elem(const void* base, int dtype, int64_t idx) {
    if (dtype == ORC_F32) return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Flat element index of pool[blk][kv][layer][kvh][slot][0]: the row-major
 * offset of the six-dimensional BlockPool tensor. */
static int64_t row_index(int64_t blk, int kv, int layer, int kvh, int slot,
                         int L, int Hkv, int B, int D) {
    int64_t i = blk;
    i = i * 2 + kv;
    i = i * L + layer;
    i = i * Hkv + kvh;
    i = i * B + slot;
    return i * D;
}

static int check_geometry(int num_blocks, int L, int Hkv, int B, int D, int layer, int dtype) {
    if (num_blocks <= 0 || L <= 0 || Hkv <= 0 || B <= 0 || D <= 0) return -1;
    if (layer < 0 || layer >= L) return -1;
    if (dtype != ORC_F32 && dtype != ORC_BF16) return -1;
    return 0;
}

/* Validate every table entry a sequence of length n reads. */
static int check_sequence(const int* bt_row, int maxb, int n, int B, int num_blocks) {
    if (n < 0) return -1;
    int64_t nblk = ((int64_t)n + B - 1) / B;
    if (nblk > maxb) return -1;
    for (int64_t j = 0; j < nblk; ++j)
        if (bt_row[j] < 0 || bt_row[j] >= num_blocks) return -1;
    return 0;
}

int oracle_decode_attention(double* out, const void* q, const void* pool, int dtype,
                            int num_blocks, int num_layers, int num_kv_heads,
                            int block_size, int head_dim, int layer,
                            const int* block_tables, int max_blocks_per_seq,
                            const int* context_lens, int batch, int num_heads,
                            double scale, int num_threads) {
    const int L = num_layers, Hkv = num_kv_heads, B = block_size, D = head_dim;
    if (check_geometry(num_blocks, L, Hkv, B, D, layer, dtype)) return -1;
    if (batch < 0 || num_heads <= 0 || num_heads % Hkv != 0 || max_blocks_per_seq <= 0) return -1;
    for (int b = 0; b < batch; ++b)
        if (check_sequence(block_tables + (int64_t)b * max_blocks_per_seq, max_blocks_per_seq,
                           context_lens[b], B, num_blocks))
            return -2;
    const int g = num_heads / Hkv;
    int bad_alloc = 0;
    if (num_threads <= 0) num_threads = 1;

#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(num_threads) reduction(| : bad_alloc)
    for (int b = 0; b < batch; ++b) {
        for (int h = 0; h < num_heads; ++h) {
            const int n = context_lens[b];
            const int kvh = h / g;
            double* o = out + ((int64_t)b * num_heads + h) * D;
            if (n == 0) {  /* no cached token: defined as a zero vector */
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                continue;
            }
            double* Kc = (double*)malloc(sizeof(double) * (size_t)n * D);
            double* Vc = (double*)malloc(sizeof(double) * (size_t)n * D);
            double* s = (double*)malloc(sizeof(double) * (size_t)n);
            double* qv = (double*)malloc(sizeof(double) * (size_t)D);
            if (!Kc || !Vc || !s || !qv) {
                free(Kc); free(Vc); free(s); free(qv);
                bad_alloc = 1;
                continue;
            }
            /* 1. walk the block table and gather K and V contiguously */
            const int* bt_row = block_tables + (int64_t)b * max_blocks_per_seq;
            for (int t = 0; t < n; ++t) {
                const int64_t blk = bt_row[t / B];
                const int slot = t % B;
                const int64_t ki = row_index(blk, 0, layer, kvh, slot, L, Hkv, B, D);
                const int64_t vi = row_index(blk, 1, layer, kvh, slot, L, Hkv, B, D);
                for (int d = 0; d < D; ++d) {
                    Kc[(int64_t)t * D + d] = load_elem(pool, dtype, ki + d);
                    Vc[(int64_t)t * D + d] = load_elem(pool, dtype, vi + d);
                }
            }
            for (int d = 0; d < D; ++d)
                qv[d] = load_elem(q, dtype, ((int64_t)b * num_heads + h) * D + d);
            /* 2. scores s = scale * K q */
            double m = -INFINITY;
            for (int t = 0; t < n; ++t) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += Kc[(int64_t)t * D + d] * qv[d];
                s[t] = scale * acc;
                if (s[t] > m) m = s[t];
            }
            /* 3. softmax weights and the weighted sum of V */
            double z = 0.0;
            for (int t = 0; t < n; ++t) {
                s[t] = exp(s[t] - m);
                z += s[t];
            }
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int t = 0; t < n; ++t) acc += s[t] * Vc[(int64_t)t * D + d];
                o[d] = acc / z;
            }
            free(Kc); free(Vc); free(s); free(qv);
        }
    }
    return bad_alloc ? -3 : 0;
}

int oracle_write_kv(void* pool, int dtype, int num_blocks, int num_layers, int num_kv_heads,
                    int block_size, int head_dim, int layer, const void* k, const void* v,
                    const int* block_tables, int max_blocks_per_seq, const int* positions,
                    int batch) {
    const int L = num_layers, Hkv = num_kv_heads, B = block_size, D = head_dim;
    if (check_geometry(num_blocks, L, Hkv, B, D, layer, dtype)) return -1;
    if (batch < 0 || max_blocks_per_seq <= 0) return -1;
    const size_t eb = elem_bytes(dtype);
    for (int b = 0; b < batch; ++b) {
        const int p = positions[b];
        if (p < 0 || p / B >= max_blocks_per_seq) return -2;
        const int blk = block_tables[(int64_t)b * max_blocks_per_seq + p / B];
        if (blk < 0 || blk >= num_blocks) return -2;
    }
    for (int b = 0; b < batch; ++b) {
        const int p = positions[b];
        const int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + p / B];
        for (int kvh = 0; kvh < Hkv; ++kvh) {
            const int64_t src = ((int64_t)b * Hkv + kvh) * D;
            const int64_t kd = row_index(blk, 0, layer, kvh, p % B, L, Hkv, B, D);
            const int64_t vd = row_index(blk, 1, layer, kvh, p % B, L, Hkv, B, D);
            memcpy((char*)pool + kd * eb, (const char*)k + src * eb, (size_t)D * eb);
            memcpy((char*)pool + vd * eb, (const char*)v + src * eb, (size_t)D * eb);
        }
    }
    return 0;
}

int oracle_gather_kv(void* k_out, void* v_out, unsigned char* mask, const void* pool, int dtype,
                     int num_blocks, int num_layers, int num_kv_heads, int block_size,
                     int head_dim, int layer, const int* block_tables, int max_blocks_per_seq,
                     const int* context_lens, int batch, int max_len) {
    const int L = num_layers, Hkv = num_kv_heads, B = block_size, D = head_dim;
    if (check_geometry(num_blocks, L, Hkv, B, D, layer, dtype)) return -1;
    if (batch < 0 || max_len < 0 || max_blocks_per_seq <= 0) return -1;
    for (int b = 0; b < batch; ++b) {
        if (context_lens[b] > max_len) return -2;
        if (check_sequence(block_tables + (int64_t)b * max_blocks_per_seq, max_blocks_per_seq,
                           context_lens[b], B, num_blocks))
            return -2;
    }
    const size_t eb = elem_bytes(dtype);
    const size_t row = (size_t)D * eb;
    for (int b = 0; b < batch; ++b) {
        const int n = context_lens[b];
        for (int t = 0; t < max_len; ++t) {
            mask[(int64_t)b * max_len + t] = (unsigned char)(t < n);
            for (int kvh = 0; kvh < Hkv; ++kvh) {
                const int64_t dst = (((int64_t)b * max_len + t) * Hkv + kvh) * D;
                if (t < n) {
                    const int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / B];
                    const int64_t ks = row_index(blk, 0, layer, kvh, t % B, L, Hkv, B, D);
                    const int64_t vs = row_index(blk, 1, layer, kvh, t % B, L, Hkv, B, D);
                    memcpy((char*)k_out + dst * eb, (const char*)pool + ks * eb, row);
                    memcpy((char*)v_out + dst * eb, (const char*)pool + vs * eb, row);
                } else {
                    memset((char*)k_out + dst * eb, 0, row);
                    memset((char*)v_out + dst * eb, 0, row);
                }
            }
        }
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
