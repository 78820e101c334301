// pa_internal.h -- launch interface between the C ABI layer and the kernels.
// Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Device status bits (mirror of the public PA_STATUS_* values).
constexpr unsigned kStatusBadBlock = 0x1u;
constexpr unsigned kStatusBadLength = 0x2u;
constexpr unsigned kStatusTimeout = 0x4u;
constexpr unsigned kStatusNoFreeBlocks = 0x8u;

// Where a pool's rows live.  The B x D tile of (block, layer, kv head) is
// contiguous and starts at element  blk*s_blk + layer*s_layer + head*s_head
// from k_base (K rows) or v_base (V rows).  The fused tensor
// [num_blocks, 2, L, Hkv, B, D] is the instance v_base = k_base + L*Hkv*B*D,
// s_blk = 2*L*Hkv*B*D, s_layer = Hkv*B*D, s_head = B*D.
struct PoolGeom {
    void* k_base;
    void* v_base;
    long long s_blk, s_layer, s_head;  // element strides
    long long num_blocks;
    int L, Hkv, B, D;
    int elt;    // bytes per element (4 = fp32, 2 = bf16)
    int dtype;  // 0 = fp32, 1 = bf16
};

struct DecodeParams {
    float* out;           // [batch, H, D] fp32
    const void* q;        // [batch, H, D] pool dtype
    const void* k_base;   // K rows (see PoolGeom)
    const void* v_base;   // V rows
    long long s_blk;      // element stride between physical blocks
    long long tile_off;   // layer * s_layer (elements)
    long long s_head;     // element stride between kv heads
    long long num_blocks;
    int Hkv, layer;
    const int* bt;        // [batch, maxb]
    int maxb;
    const int* lens;      // [batch]
    int batch, H;
    float qscale;         // softmax scale * log2(e): scores live in the base-2 domain
    float* part_o;        // [batch, H, Cmax, D] unnormalised partial outputs
    float* part_ml;       // [batch, H, Cmax, 2] (running max, sum of weights)
    int PB;               // blocks per partition
    int Cmax;             // partitions per (sequence, kv head) grid slot
    unsigned* status;     // device status word
    // fused append (all null unless pa_write_kv_and_decode): new K/V rows
    // [batch, Hkv, D] stored at slot positions[b] before the decode reads it
    const void* new_k;
    const void* new_v;
    const int* positions;
    // tensor-core kernel only: which of the tensor maps' outer dimensions
    // (2, 3, 4) index the physical block, the layer and the kv head
    int tma_slot_blk, tma_slot_layer, tma_slot_head;
    // tensor-core kernels only: the group (num_heads / Hkv) is served in
    // `nchunks` chunks of `chunk` heads (the kernel's compile-time G); the last
    // chunk holds the rest of a group that is no multiple of it, and the
    // tcgen05 kernel's partial slots are `chunk` heads wide
    int gsize, nchunks, chunk;
    // tcgen05 kernel only: its persistent grid, and (with tc_grid > 1) one
    // int4 per (sequence, head group) {first CTA, pieces, slot of the first
    // piece} that tells the combine where the pieces of a split context are;
    // the partials then sit in part_o / part_ml as [CTA][2 slots][chunk head]
    int tc_grid;
    int4* tc_desc;
    // tcgen05 kernel: per decode CTA, the (sequence, head group) pair whose
    // first piece it holds and which continues past its range, as {pair, first
    // CTA, pieces, slot of the first piece} (pair -1: none)
    int4* tc_cut;
};

struct WriteParams {
    void* k_base;
    void* v_base;
    long long s_blk, tile_off, s_head;  // elements; tile_off = layer * s_layer
    long long num_blocks;
    int Hkv, B, row_bytes, elt, layer;
    const void* k;
    const void* v;
    const int* bt;
    int maxb;
    const int* positions;
    int batch;
    unsigned* status;
};

struct GatherParams {
    void* k_out;
    void* v_out;
    uint8_t* mask;
    const void* k_base;
    const void* v_base;
    long long s_blk, tile_off, s_head;  // elements; tile_off = layer * s_layer
    long long num_blocks;
    int Hkv, B, row_bytes, elt, layer;
    const int* bt;
    int maxb;
    const int* lens;
    int batch, max_len;
    unsigned* status;
};

// Returns cudaErrorNotSupported (without launching) when no kernel is built
// for (dtype, D, B, G).
cudaError_t launch_decode_bf16(const DecodeParams& p, int D, int B, int G, cudaStream_t s);
cudaError_t launch_decode_f32(const DecodeParams& p, int D, int B, int G, cudaStream_t s);
bool decode_supported(int dtype, int D, int B, int G);
// The CUDA-core kernel's head chunk for group G: G itself for 1, 2, 4, 8;
// the next power of two below 8, 8 above (the last chunk masks the heads past
// the group); 0 for G < 1.
inline int decode_cc_chunk(int G) {
    if (G < 1) return 0;
    if (G > 8) return 8;
    int c = 1;
    while (c < G) c <<= 1;
    return c;
}

// Tensor-core kernel for bf16 pools; `tmaps` points to two CUtensorMap (K, V).
// Groups of up to 8 or exactly 16 heads run in one CTA per KV head; larger
// multiples of 8 in chunks (decode_mma_chunk gives the chunk size, 0 if none).
bool decode_mma_supported(int D, int B, int G);
int decode_mma_chunk(int G);
cudaError_t launch_decode_mma(const DecodeParams& p, const void* tmaps, int D, int B, int G,
                              cudaStream_t s);
// The same kernel in wide CTAs (many warps, one partition per context: p.Cmax
// must be 1).  decode_mma_wide_fits: whether a call with group G and `ctas`
// (sequence, KV head, chunk) CTAs over tables of maxb blocks suits it (a third
// to all of one wave, a few blocks per warp).
bool decode_mma_wide_fits(int D, int G, int maxb, long long ctas, int num_sms);
cudaError_t launch_decode_mma_wide(const DecodeParams& p, const void* tmaps, int D, int B, int G,
                                   cudaStream_t s);
// Encodes the K and V tensor maps of a bf16 pool (5-D, box 64 x 16, 128-byte
// swizzle) into tmaps[0..1]; slots receives the outer-dimension order.
cudaError_t encode_pool_tmaps(const PoolGeom& g, void* tmaps, int* slot_blk, int* slot_layer,
                              int* slot_head);
// Encodes a 2-D tensor map over `rows` contiguous rows of 128 bf16 (boxes of 64
// columns x box_rows rows, 128-byte swizzle) into one CUtensorMap at tmap.
cudaError_t encode_rows_tmap(void* tmap, const void* base, long long rows, int box_rows);

// tcgen05 kernel for bf16 pools, head_dim 128, groups that are multiples of
// 16 (chunks of 64, 32 or 16 heads; decode_umma_chunk gives the chunk, 0 if
// none); persistent, one CTA per SM.
bool decode_umma_supported(int D, int B, int G);
int decode_umma_chunk(int G);
cudaError_t launch_decode_umma(const DecodeParams& p, const void* tmaps, int B, int G,
                               cudaStream_t s);

cudaError_t launch_combine(const DecodeParams& p, int D, int B, cudaStream_t s);
// Merges the tcgen05 kernel's cut pairs: every pair (direct) or the pairs its
// CTAs recorded in tc_cut; pieces_hint estimates the pieces per cut pair.
cudaError_t launch_combine_tc(const DecodeParams& p, int D, bool direct, int pieces_hint,
                              cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned* status, cudaStream_t s);
cudaError_t launch_write_kv(const WriteParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_gather_kv(const GatherParams& p, int num_sms, cudaStream_t s);

cudaError_t launch_device_alloc(int* stack, int* bt, int maxb, const int* positions,
                                int* next_lens, int batch, int B, unsigned* status,
                                cudaStream_t s);
cudaError_t launch_device_free(int* stack, int* bt, int maxb, const int* lens,
                               const uint8_t* finished, int batch, int B, long long num_blocks,
                               unsigned* status, cudaStream_t s);

// Records `message` as the calling thread's last error; returns `code`.
int set_last_error(int code, const char* message);

// Device address of the status word of the current device (looked up once per device).
cudaError_t status_word(unsigned** ptr);
cudaError_t read_and_clear_status(unsigned* host_value, cudaStream_t s);

}  // namespace pa
