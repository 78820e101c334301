// pa_fused_append.cuh -- the KV append of pa_write_kv_and_decode, done inside
// the decode kernels by one warp.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// All 32 lanes of a warp store sequence b's new K and V rows of KV head kvh
// (ROW_BYTES each, in 16-byte chunks) at row pos % B of physical block blk,
// each lane fencing its stores against the bulk-copy (async) proxy; after the
// closing __syncwarp a copy that this warp issues reads the new row.
template <int ROW_BYTES, int ELT>
__device__ __forceinline__ void warp_store_new_row(const DecodeParams& p, int b, int kvh, int blk,
                                                   int pos, int B, int lane) {
    constexpr int CPR = ROW_BYTES / 16;  // chunks per row
    const long long row = (long long)blk * p.s_blk + p.tile_off + (long long)kvh * p.s_head +
                          (long long)(pos % B) * (ROW_BYTES / ELT);
    const long long src = ((long long)b * p.Hkv + kvh) * ROW_BYTES;
    for (int i = lane; i < 2 * CPR; i += 32) {
        const int kv = i / CPR;
        const int ci = i % CPR;
        const uint4 val = ld_dep(reinterpret_cast<const uint4*>(
            static_cast<const unsigned char*>(kv ? p.new_v : p.new_k) + src + ci * 16));
        unsigned char* dst = static_cast<unsigned char*>(const_cast<void*>(kv ? p.v_base : p.k_base)) +
                             row * ELT;
        reinterpret_cast<uint4*>(dst)[ci] = val;
        fence_proxy_async_global();
    }
    __syncwarp();
}

// The same store in two steps, so that the loads leave the critical path: a
// warp loads the new rows at its start (lane i < 2 * ROW_BYTES / 16 holds
// chunk i, K chunks first; the source depends only on the sequence and KV
// head), and stores them once the block and slot are known.
template <int ROW_BYTES>
__device__ __forceinline__ uint4 load_new_row(const DecodeParams& p, int b, int kvh, int lane) {
    constexpr int CPR = ROW_BYTES / 16;
    static_assert(2 * CPR <= 32, "one 16-byte chunk per lane");
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (lane < 2 * CPR) {
        const int kv = lane / CPR;
        const long long src = ((long long)b * p.Hkv + kvh) * ROW_BYTES + (lane % CPR) * 16;
        val = ld_dep(reinterpret_cast<const uint4*>(
            static_cast<const unsigned char*>(kv ? p.new_v : p.new_k) + src));
    }
    return val;
}

template <int ROW_BYTES, int ELT>
__device__ __forceinline__ void store_new_row(const DecodeParams& p, int kvh, int blk, int pos,
                                              int B, int lane, const uint4 val) {
    constexpr int CPR = ROW_BYTES / 16;
    if (lane < 2 * CPR) {
        const int kv = lane / CPR;
        const long long row = (long long)blk * p.s_blk + p.tile_off + (long long)kvh * p.s_head +
                              (long long)(pos % B) * (ROW_BYTES / ELT);
        unsigned char* dst = static_cast<unsigned char*>(const_cast<void*>(kv ? p.v_base : p.k_base)) +
                             row * ELT;
        reinterpret_cast<uint4*>(dst)[lane % CPR] = val;
        fence_proxy_async_global();
    }
    __syncwarp();
}

}  // namespace pa
