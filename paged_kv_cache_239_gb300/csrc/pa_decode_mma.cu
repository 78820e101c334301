// bf16 tensor-core decode: instantiations, launch, and the tensor maps.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "pa_decode_mma.cuh"

namespace pa {

namespace {

constexpr int kMmaWarps = 4;
// Stages per warp: a head_dim-64 stage is half the size, so four of them keep
// the CTA at the 64 KB (three CTAs per SM) of two head_dim-128 stages.  GB300,
// mini-infer shape (head_dim 64): 8.6 -> 7.7 us per decode call with four; four
// at head_dim 128 (one CTA per SM) halved the MHA batch-64 throughput.
template <int D>
constexpr int kMmaStages = D == 64 ? 4 : 2;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

}  // namespace

int decode_mma_chunk(int G) {
    if (G >= 1 && G <= 8) return G;
    if (G == 16) return 16;
    if (G > 16 && G % 16 == 0) return 16;
    if (G > 8) return 8;  // (the last chunk holds G % 8 heads when G is no multiple of 8)
    return 0;
}

bool decode_mma_supported(int D, int B, int G) {
    if (D != 64 && D != 128) return false;
    if (B != 16 && B != 32) return false;
    // heads past G in the 8-wide mma tiles are masked; larger groups in chunks
    // (a ragged last chunk masks the heads past the group the same way)
    return decode_mma_chunk(G) > 0;
}

cudaError_t launch_decode_mma(const DecodeParams& p_in, const void* tmaps, int D, int B, int Gtot,
                              cudaStream_t s) {
    const CUtensorMap* tm = static_cast<const CUtensorMap*>(tmaps);
    const int G = decode_mma_chunk(Gtot);
    if (G == 0) return cudaErrorNotSupported;
    DecodeParams p = p_in;
    p.gsize = Gtot;
    p.nchunks = (Gtot + G - 1) / G;
    p.chunk = G;
    if (D == 64) {
        if (B == 16) return launch_mma_g<64, 16, kMmaWarps, kMmaStages<64>>(p, tm, G, s);
        if (B == 32) return launch_mma_g<64, 32, kMmaWarps, kMmaStages<64>>(p, tm, G, s);
    } else if (D == 128) {
        if (B == 16) return launch_mma_g<128, 16, kMmaWarps, kMmaStages<128>>(p, tm, G, s);
        if (B == 32) return launch_mma_g<128, 32, kMmaWarps, kMmaStages<128>>(p, tm, G, s);
    }
    return cudaErrorNotSupported;
}

cudaError_t encode_pool_tmaps(const PoolGeom& g, void* tmaps, int* slot_blk, int* slot_layer,
                              int* slot_head) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    // Outer dimensions (block, layer, kv head) ordered by increasing stride; a
    // dimension of extent 1 gets the stride that follows the previous one.
    struct Outer {
        long long stride, count;
        int which;  // 0 block, 1 layer, 2 head
    } od[3] = {{g.s_blk, g.num_blocks, 0}, {g.s_layer, g.L, 1}, {g.s_head, g.Hkv, 2}};
    std::sort(od, od + 3, [](const Outer& a, const Outer& b) {
        const long long sa = a.count > 1 ? a.stride : (1LL << 62);
        const long long sb = b.count > 1 ? b.stride : (1LL << 62);
        return sa < sb;
    });
    const long long row = (long long)g.D * g.elt;  // bytes
    cuuint64_t dims[5] = {(cuuint64_t)g.D, (cuuint64_t)g.B, 0, 0, 0};
    cuuint64_t strides[4] = {(cuuint64_t)row, 0, 0, 0};
    long long prev_extent = row * g.B;  // bytes of one tile
    for (int i = 0; i < 3; ++i) {
        long long st = od[i].stride * g.elt;
        if (od[i].count <= 1) st = prev_extent;
        dims[2 + i] = (cuuint64_t)od[i].count;
        strides[1 + i] = (cuuint64_t)st;
        prev_extent = st * od[i].count;
        if (od[i].which == 0) *slot_blk = 2 + i;
        if (od[i].which == 1) *slot_layer = 2 + i;
        if (od[i].which == 2) *slot_head = 2 + i;
    }
    cuuint32_t box[5] = {64, 16, 1, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUtensorMap* tm = static_cast<CUtensorMap*>(tmaps);
    void* bases[2] = {g.k_base, g.v_base};
    for (int i = 0; i < 2; ++i) {
        CUresult r = fn(&tm[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, bases[i], dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

// A 2-D map over `rows` contiguous rows of 128 bf16 (256 bytes): boxes of
// 64 columns x box_rows rows with the 128-byte swizzle.
cudaError_t encode_rows_tmap(void* tmap, const void* base, long long rows, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if (rows <= 0 || box_rows <= 0 || box_rows > 256) return cudaErrorInvalidValue;
    cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(static_cast<CUtensorMap*>(tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace pa
