// bf16 decode for large GQA groups on tcgen05: instantiations and launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa_decode_umma.cuh"

namespace pa {

namespace {

template <int B, int G>
cudaError_t launch_inst(const DecodeParams& p, const CUtensorMap* tm, cudaStream_t stream) {
    // q of one piece is copied as two boxes of 64 columns x G heads
    CUtensorMap tq;
    cudaError_t eq = encode_rows_tmap(&tq, p.q, (long long)p.batch * p.H, G);
    if (eq != cudaSuccess) return eq;
    using Cfg = UmmaCfg<B, G>;
    auto kern = pa_decode_umma_kernel<B, G>;
    static std::mutex mu;
    static unsigned long long done_mask = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        const unsigned long long bit = 1ull << (dev & 63);
        if (!(done_mask & bit)) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cfg::SMEM_BYTES);
            if (e != cudaSuccess) return e;
            done_mask |= bit;
        }
    }
    if (p.tc_grid <= 0) return cudaErrorInvalidConfiguration;
    // persistent: one CTA per SM (the shared memory admits no second one),
    // each taking an equal share of the tiles
    return launch_pdl(kern, dim3((unsigned)p.tc_grid), dim3(Cfg::THREADS), Cfg::SMEM_BYTES,
                      stream, p, tm[0], tm[1], tq);
}

template <int B>
cudaError_t launch_g(const DecodeParams& p, const CUtensorMap* tm, int G, cudaStream_t s) {
    switch (G) {
        case 16: return launch_inst<B, 16>(p, tm, s);
        case 32: return launch_inst<B, 32>(p, tm, s);
        case 48: return launch_inst<B, 48>(p, tm, s);
        case 64: return launch_inst<B, 64>(p, tm, s);
        case 128: return launch_inst<B, 128>(p, tm, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

int decode_umma_chunk(int G) {
    if (G <= 0 || G % 16 != 0) return 0;
    if (G % 128 == 0) return 128;
    // 80, 96 and 112 heads: one 128-head chunk, the rows past the group
    // computed and dropped (one K/V pass at the 128-head rate, instead of five,
    // two or seven sibling chunks)
    if (G > 64 && G < 128) return 128;
    if (G % 64 == 0) return 64;
    if (G % 48 == 0) return 48;
    if (G % 32 == 0) return 32;
    return 16;
}

bool decode_umma_supported(int D, int B, int G) {
    return D == 128 && (B == 16 || B == 32) && decode_umma_chunk(G) > 0;
}

cudaError_t launch_decode_umma(const DecodeParams& p_in, const void* tmaps, int B, int Gtot,
                               cudaStream_t s) {
    const CUtensorMap* tm = static_cast<const CUtensorMap*>(tmaps);
    const int G = decode_umma_chunk(Gtot);
    if (G == 0) return cudaErrorNotSupported;
    DecodeParams p = p_in;
    p.gsize = Gtot;
    p.nchunks = (Gtot + G - 1) / G;
    p.chunk = G;
    if (B == 16) return launch_g<16>(p, tm, G, s);
    if (B == 32) return launch_g<32>(p, tm, G, s);
    return cudaErrorNotSupported;
}

}  // namespace pa
