// pa_alloc.cu -- the free-block stack on the device: batch allocation of the
// next block for every sequence whose new token starts one, and batch freeing
// of finished sequences, without a host round trip.
//
// Semantics follow the host allocator (mini-infer BlockPool, "Python
// Implementation: Physical Block Pool": pop from the end, append on free) with
// the batch processed in increasing sequence order, so the ids handed out are
// exactly those of the same sequence of host calls.  The stack lives in a
// caller-owned int32 array: [0] = height, [1 + i] = i-th id from the bottom.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kScanThreads = 1024;

// Exclusive prefix sum of `v` over the CTA; `total` receives the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int& total) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        if (lane < nw) s_warp[lane] = w;  // inclusive totals per warp
    }
    __syncthreads();
    const int warp_prefix = warp > 0 ? s_warp[warp - 1] : 0;
    total = s_warp[(blockDim.x >> 5) - 1];
    __syncthreads();  // s_warp is reused by the next call
    return warp_prefix + incl - v;
}

__global__ void __launch_bounds__(kScanThreads)
pa_device_alloc_kernel(int* stack, int* bt, int maxb, const int* positions, int* next_lens,
                       int batch, int B, unsigned* status) {
    pdl_trigger();
    pdl_wait();
    __shared__ int s_warp[32];
    __shared__ int s_height;
    if (threadIdx.x == 0) s_height = stack[0];
    __syncthreads();
    const int height = s_height;
    int taken = 0;  // ids handed out by earlier chunks
    for (int chunk = 0; chunk < batch; chunk += blockDim.x) {
        const int b = chunk + threadIdx.x;
        int need = 0, pos = 0;
        if (b < batch) {
            pos = positions[b];
            if (next_lens != nullptr) next_lens[b] = pos + 1;
            if (pos < 0 || pos / B >= maxb) {
                atomicOr(status, kStatusBadLength);
            } else if (pos % B == 0) {
                need = 1;
            }
        }
        int total = 0;
        const int r = taken + block_exclusive_scan(need, s_warp, total);
        if (need) {
            int id = -1;
            if (r < height) {
                id = stack[1 + height - 1 - r];
            } else {
                atomicOr(status, kStatusNoFreeBlocks);
            }
            bt[(long long)b * maxb + pos / B] = id;
        }
        taken += total;
    }
    if (threadIdx.x == 0) stack[0] = taken < height ? height - taken : 0;
}

__global__ void __launch_bounds__(kScanThreads)
pa_device_free_kernel(int* stack, int* bt, int maxb, const int* lens, const uint8_t* finished,
                      int batch, int B, long long num_blocks, unsigned* status) {
    pdl_trigger();
    pdl_wait();
    __shared__ int s_warp[32];
    __shared__ int s_height;
    if (threadIdx.x == 0) s_height = stack[0];
    __syncthreads();
    const int height = s_height;
    int pushed = 0;
    for (int chunk = 0; chunk < batch; chunk += blockDim.x) {
        const int b = chunk + threadIdx.x;
        int cnt = 0, nblk = 0;
        int* row = bt + (long long)(b < batch ? b : 0) * maxb;
        if (b < batch && finished[b]) {
            const int n = lens[b];
            if (n < 0 || n > maxb * B) {
                atomicOr(status, kStatusBadLength);
            } else {
                nblk = (n + B - 1) / B;
                for (int j = 0; j < nblk; ++j) {
                    const int id = row[j];
                    if (id >= 0 && id < num_blocks) {
                        ++cnt;
                    } else {
                        atomicOr(status, kStatusBadBlock);
                    }
                }
            }
        }
        int total = 0;
        int slot = height + pushed + block_exclusive_scan(cnt, s_warp, total);
        for (int j = 0; j < nblk; ++j) {
            const int id = row[j];
            if (id >= 0 && id < num_blocks) {
                if (slot < num_blocks) {
                    stack[1 + slot] = id;
                } else {
                    atomicOr(status, kStatusBadBlock);  // more ids than the pool holds
                }
                ++slot;
            }
            row[j] = -1;
        }
        pushed += total;
    }
    if (threadIdx.x == 0) {
        const long long h = (long long)height + pushed;
        stack[0] = (int)(h < num_blocks ? h : num_blocks);
    }
}

}  // namespace

cudaError_t launch_device_alloc(int* stack, int* bt, int maxb, const int* positions,
                                int* next_lens, int batch, int B, unsigned* status,
                                cudaStream_t s) {
    if (batch <= 0) return cudaSuccess;
    return launch_pdl(pa_device_alloc_kernel, dim3(1), dim3(kScanThreads), 0, s, stack, bt, maxb,
                      positions, next_lens, batch, B, status);
}

cudaError_t launch_device_free(int* stack, int* bt, int maxb, const int* lens,
                               const uint8_t* finished, int batch, int B, long long num_blocks,
                               unsigned* status, cudaStream_t s) {
    if (batch <= 0) return cudaSuccess;
    return launch_pdl(pa_device_free_kernel, dim3(1), dim3(kScanThreads), 0, s, stack, bt, maxb,
                      lens, finished, batch, B, num_blocks, status);
}

}  // namespace pa
