// pa_decode_launch.cuh -- host-side launch of one decode kernel instantiation.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "pa_decode.cuh"

namespace pa {

constexpr int kDecodeWarps = 4;

// Pipeline depth per warp.  Two stages of >= 8 KiB keep a 4-warp CTA at about
// 66 KiB of shared memory, so three CTAs (12 warps) fit on an SM; measured on
// GB300 this beats three stages at two CTAs per SM by ~20% (the kernel is
// latency-bound at 8 warps per SM).  Small stages (4 KiB) take four.
template <typename T, int D, int B>
constexpr int decode_stages() {
    constexpr int R = B < 16 ? B : 16;
    constexpr int stage = 2 * R * D * (int)sizeof(T);
    return stage <= 4096 ? 4 : 2;
}

template <typename T, int D, int B, int G>
cudaError_t launch_decode_inst(const DecodeParams& p, cudaStream_t stream) {
    constexpr int S = decode_stages<T, D, B>();
    using C = DecodeCfg<T, D, B, G, kDecodeWarps, S>;
    auto kern = pa_decode_kernel<T, D, B, G, kDecodeWarps, S>;
    // The dynamic shared-memory opt-in is per device; set it once per device.
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
                                     C::SMEM_BYTES);
            if (e != cudaSuccess) return e;
            done_mask |= bit;
        }
    }
    const long long grid = (long long)p.batch * p.Hkv * p.nchunks * p.Cmax;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kDecodeWarps * 32), C::SMEM_BYTES, stream,
                      p);
}

template <typename T, int D, int B>
cudaError_t launch_decode_g(const DecodeParams& p, int G, cudaStream_t s) {
    switch (G) {
        case 1: return launch_decode_inst<T, D, B, 1>(p, s);
        case 2: return launch_decode_inst<T, D, B, 2>(p, s);
        case 4: return launch_decode_inst<T, D, B, 4>(p, s);
        case 8: return launch_decode_inst<T, D, B, 8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

template <typename T>
cudaError_t launch_decode_typed(const DecodeParams& p_in, int D, int B, int Gtot, cudaStream_t s) {
    const int G = decode_cc_chunk(Gtot);
    if (G == 0) return cudaErrorNotSupported;
    DecodeParams p = p_in;
    p.gsize = Gtot;
    p.nchunks = (Gtot + G - 1) / G;
    p.chunk = G;
    if (D == 64) {
        if (B == 16) return launch_decode_g<T, 64, 16>(p, G, s);
        if (B == 32) return launch_decode_g<T, 64, 32>(p, G, s);
    } else if (D == 128) {
        if (B == 16) return launch_decode_g<T, 128, 16>(p, G, s);
        if (B == 32) return launch_decode_g<T, 128, 32>(p, G, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace pa
