// pa_aux.cu -- device status word, split-K combine launch, KV append and
// batched gather kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pa_decode.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// One status word per device per loaded library (file-scope device variable:
// no allocation).  Kernels OR PA_STATUS_* bits into it.
__device__ unsigned int g_status_word = 0;

cudaError_t status_word(unsigned** ptr) {
    static std::mutex mu;
    static unsigned* cached[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return e;
        cached[dev] = static_cast<unsigned*>(p);
    }
    *ptr = cached[dev];
    return cudaSuccess;
}

cudaError_t read_and_clear_status(unsigned* host_value, cudaStream_t s) {
    unsigned* dptr = nullptr;
    cudaError_t e = status_word(&dptr);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpy(host_value, dptr, sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    return cudaMemset(dptr, 0, sizeof(unsigned));
}

// Self-test of the bounded wait: one warp waits on an mbarrier phase that no
// thread or copy ever completes.  The wait gives up after 20 ms, the kernel
// records PA_STATUS_TIMEOUT and returns; the context stays usable.
constexpr unsigned long long kSelftestWaitNs = 20000000ull;

__global__ void pa_wait_selftest_kernel(unsigned* status) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t a = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(a, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded<kSelftestWaitNs>(a, 0);
    if (!__all_sync(kFullMask, ok) && threadIdx.x == 0) atomicOr(status, kStatusTimeout);
}

cudaError_t launch_wait_selftest(unsigned* status, cudaStream_t s) {
    pa_wait_selftest_kernel<<<1, 32, 0, s>>>(status);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_combine_d(const DecodeParams& p, int B, long long heads, cudaStream_t s) {
    // warps per (sequence, head): one warp for up to 4 partials (one round of
    // four loads), more as the partial count grows (ncu on GB300: with 4
    // partials a single warp is faster than two; with 64-128, eight warps)
    const int W = p.Cmax > 32 ? 8 : (p.Cmax > 8 ? 4 : (p.Cmax > 4 ? 2 : 1));
    const long long hpc = 8 / W;
    const long long grid = (heads + hpc - 1) / hpc;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaError_t e;
    switch (W) {
        case 8: e = launch_pdl(pa_combine_kernel<D, 8>, dim3((unsigned)grid), dim3(256), 0, s, p, B); break;
        case 4: e = launch_pdl(pa_combine_kernel<D, 4>, dim3((unsigned)grid), dim3(256), 0, s, p, B); break;
        case 2: e = launch_pdl(pa_combine_kernel<D, 2>, dim3((unsigned)grid), dim3(256), 0, s, p, B); break;
        default: e = launch_pdl(pa_combine_kernel<D, 1>, dim3((unsigned)grid), dim3(256), 0, s, p, B); break;
    }
    return e;
}

cudaError_t launch_combine(const DecodeParams& p, int D, int B, cudaStream_t s) {
    const long long heads = (long long)p.batch * p.H;
    if (heads <= 0) return cudaSuccess;
    if (D == 64) return launch_combine_d<64>(p, B, heads, s);
    if (D == 128) return launch_combine_d<128>(p, B, heads, s);
    return cudaErrorNotSupported;
}

// CTAs of pa_combine_tc_kernel<128, W> resident on the device at once (per
// device, looked up once).
template <int W>
static cudaError_t combine_tc_wave(long long* wave) {
    static std::mutex mu;
    static long long cached[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        int per_sm = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pa_combine_tc_kernel<128, W>,
                                                          256, 0);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cached[dev] = (long long)(per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
    }
    *wave = cached[dev];
    return cudaSuccess;
}

template <int W>
static cudaError_t launch_combine_tc_w(const DecodeParams& p, long long groups, int direct,
                                       cudaStream_t s) {
    constexpr int HPC = 8 / W;
    const int chunk = p.chunk;
    if (groups <= 0 || chunk <= 0) return cudaSuccess;
    // heads per warp: one, unless a CTA per 8 / W heads would take more than
    // one wave of CTAs (the second wave starts only as the first one ends)
    long long wave = 0;
    cudaError_t e = combine_tc_wave<W>(&wave);
    if (e != cudaSuccess) return e;
    const int max_rounds = (chunk + HPC - 1) / HPC;
    int rounds = 1;
    while (rounds < max_rounds && groups * ((chunk + HPC * rounds - 1) / (HPC * rounds)) > wave)
        ++rounds;
    const long long grid = groups * ((chunk + HPC * rounds - 1) / (HPC * rounds));
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_pdl(pa_combine_tc_kernel<128, W>, dim3((unsigned)grid), dim3(256), 0, s, p,
                      direct, rounds);
}

cudaError_t launch_combine_tc(const DecodeParams& p, int D, bool direct, int pieces_hint,
                              cudaStream_t s) {
    if (D != 128) return cudaErrorNotSupported;
    const long long groups = direct ? (long long)p.batch * p.Hkv * p.nchunks : p.tc_grid;
    // warps per head from the expected pieces per cut pair (as for partitions)
    const int W = pieces_hint > 32 ? 8 : (pieces_hint > 8 ? 4 : (pieces_hint > 4 ? 2 : 1));
    switch (W) {
        case 8: return launch_combine_tc_w<8>(p, groups, direct ? 1 : 0, s);
        case 4: return launch_combine_tc_w<4>(p, groups, direct ? 1 : 0, s);
        case 2: return launch_combine_tc_w<2>(p, groups, direct ? 1 : 0, s);
        default: return launch_combine_tc_w<1>(p, groups, direct ? 1 : 0, s);
    }
}

// ---------------------------------------------------------------------------
// KV append: one thread per 16-byte chunk of every (sequence, K/V, kv head) row.
// Consecutive threads cover consecutive chunks of one row, so both the read of
// k/v and the write into the pool row are coalesced.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pa_write_kv_kernel(const WriteParams p) {
    pdl_trigger();
    pdl_wait();
    const int cpr = p.row_bytes / 16;
    const long long total = (long long)p.batch * 2 * p.Hkv * cpr;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int ci = (int)(i % cpr);
        long long r = i / cpr;
        const int kvh = (int)(r % p.Hkv);
        r /= p.Hkv;
        const int kv = (int)(r % 2);
        const int b = (int)(r / 2);
        const int pos = ld_dep(p.positions + b);
        if (pos < 0 || pos / p.B >= p.maxb) {
            if (ci == 0 && kvh == 0 && kv == 0) atomicOr(p.status, kStatusBadLength);
            continue;
        }
        const int blk = ld_dep(p.bt + (long long)b * p.maxb + pos / p.B);
        if (blk < 0 || blk >= p.num_blocks) {
            if (ci == 0 && kvh == 0 && kv == 0) atomicOr(p.status, kStatusBadBlock);
            continue;
        }
        // element offset of the slot's row, then bytes
        const long long off = (long long)blk * p.s_blk + p.tile_off + (long long)kvh * p.s_head +
                              (long long)(pos % p.B) * (p.row_bytes / p.elt);
        const unsigned char* src = static_cast<const unsigned char*>(kv ? p.v : p.k) +
                                   ((long long)b * p.Hkv + kvh) * p.row_bytes + ci * 16;
        unsigned char* dst = static_cast<unsigned char*>(kv ? p.v_base : p.k_base) +
                             off * p.elt + ci * 16;
        *reinterpret_cast<uint4*>(dst) = ld_dep(reinterpret_cast<const uint4*>(src));
    }
}

cudaError_t launch_write_kv(const WriteParams& p, int num_sms, cudaStream_t s) {
    const long long total = (long long)p.batch * 2 * p.Hkv * (p.row_bytes / 16);
    if (total <= 0) return cudaSuccess;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(pa_write_kv_kernel, dim3((unsigned)blocks), dim3(256), 0, s, p);
}

// ---------------------------------------------------------------------------
// Batched gather: copies the first n rows of every sequence into contiguous
// [batch, max_len, Hkv, D] K and V, zero-fills the rest, writes the mask.
// One thread per 16-byte chunk of every output row (K and V).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pa_gather_kv_kernel(const GatherParams p) {
    pdl_trigger();
    pdl_wait();
    const int cpr = p.row_bytes / 16;
    const long long total = (long long)p.batch * p.max_len * p.Hkv * 2 * cpr;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int ci = (int)(i % cpr);
        long long r = i / cpr;
        const int kv = (int)(r % 2);
        r /= 2;
        const int kvh = (int)(r % p.Hkv);
        r /= p.Hkv;
        const int t = (int)(r % p.max_len);
        const int b = (int)(r / p.max_len);
        int n = ld_dep(p.lens + b);
        if (n < 0 || n > p.max_len || n > p.maxb * p.B) {
            if (t == 0 && kvh == 0 && kv == 0 && ci == 0) atomicOr(p.status, kStatusBadLength);
            n = 0;
        }
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        bool valid = t < n;
        if (valid) {
            const int blk = ld_dep(p.bt + (long long)b * p.maxb + t / p.B);
            if (blk < 0 || blk >= p.num_blocks) {
                if (kvh == 0 && kv == 0 && ci == 0) atomicOr(p.status, kStatusBadBlock);
            } else {
                const long long off = (long long)blk * p.s_blk + p.tile_off +
                                      (long long)kvh * p.s_head +
                                      (long long)(t % p.B) * (p.row_bytes / p.elt);
                val = ld_dep(reinterpret_cast<const uint4*>(
                    static_cast<const unsigned char*>(kv ? p.v_base : p.k_base) + off * p.elt +
                    ci * 16));
            }
        }
        const long long orow = ((long long)b * p.max_len + t) * p.Hkv + kvh;
        unsigned char* dst = static_cast<unsigned char*>(kv ? p.v_out : p.k_out) +
                             orow * p.row_bytes + ci * 16;
        *reinterpret_cast<uint4*>(dst) = val;
        if (kvh == 0 && kv == 0 && ci == 0) p.mask[(long long)b * p.max_len + t] = valid ? 1 : 0;
    }
}

// Tiled gather: one CTA per (logical block j, sequence b).  A thread owns one
// 16-byte chunk of a row (CPR chunks per row, 256 / CPR rows per pass) and
// walks the (K/V, kv head) pairs four at a time, so four independent loads are
// in flight before the stores.  Rows past the length (or behind a bad block id)
// are written as zeros; the mask rows of the block are written once.
template <int CPR>
__global__ void __launch_bounds__(256) pa_gather_kv_tiled(const GatherParams p) {
    pdl_trigger();
    pdl_wait();
    constexpr int RPP = 256 / CPR;  // rows per pass
    const int j = blockIdx.x;
    const int b = blockIdx.y;
    const int t0 = j * p.B;
    const int rows_here = min(p.B, p.max_len - t0);
    int n = ld_dep(p.lens + b);
    if (n < 0 || n > p.max_len || n > p.maxb * p.B) {
        if (j == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusBadLength);
        n = 0;
    }
    int valid = min(max(n - t0, 0), rows_here);
    int blk = -1;
    if (valid > 0) {
        blk = ld_dep(p.bt + (long long)b * p.maxb + j);
        if (blk < 0 || blk >= p.num_blocks) {
            if (threadIdx.x == 0) atomicOr(p.status, kStatusBadBlock);
            valid = 0;
        }
    }
    if (threadIdx.x < rows_here)
        p.mask[(long long)b * p.max_len + t0 + threadIdx.x] = threadIdx.x < valid ? 1 : 0;
    const int ci = threadIdx.x % CPR;
    const int elems_per_row = p.row_bytes / p.elt;
    const long long head_bytes = p.s_head * p.elt;
    for (int r = threadIdx.x / CPR; r < rows_here; r += RPP) {
        const bool live = r < valid;
        const long long src_row =
            live ? ((long long)blk * p.s_blk + p.tile_off + (long long)r * elems_per_row) * p.elt : 0;
        const long long dst_row = ((long long)b * p.max_len + t0 + r) * p.Hkv;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
            const unsigned char* sbase =
                static_cast<const unsigned char*>(kv ? p.v_base : p.k_base) + src_row + ci * 16;
            unsigned char* dbase = static_cast<unsigned char*>(kv ? p.v_out : p.k_out) +
                                   dst_row * p.row_bytes + ci * 16;
            for (int h0 = 0; h0 < p.Hkv; h0 += 4) {
                uint4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    v[u] = make_uint4(0u, 0u, 0u, 0u);
                    if (live && h0 + u < p.Hkv)
                        v[u] = ld_dep(reinterpret_cast<const uint4*>(sbase + (h0 + u) * head_bytes));
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (h0 + u < p.Hkv)
                        *reinterpret_cast<uint4*>(dbase + (long long)(h0 + u) * p.row_bytes) = v[u];
            }
        }
    }
}

cudaError_t launch_gather_kv(const GatherParams& p, int num_sms, cudaStream_t s) {
    const long long total = (long long)p.batch * p.max_len * p.Hkv * 2 * (p.row_bytes / 16);
    if (total <= 0) return cudaSuccess;
    const long long nj = ((long long)p.max_len + p.B - 1) / p.B;
    const int cpr = p.row_bytes / 16;
    if (p.batch <= 65535 && nj <= 0x7fffffffLL && p.B <= 256 && (cpr == 8 || cpr == 16 || cpr == 32)) {
        const dim3 grid((unsigned)nj, (unsigned)p.batch);
        if (cpr == 8) return launch_pdl(pa_gather_kv_tiled<8>, grid, dim3(256), 0, s, p);
        if (cpr == 16) return launch_pdl(pa_gather_kv_tiled<16>, grid, dim3(256), 0, s, p);
        return launch_pdl(pa_gather_kv_tiled<32>, grid, dim3(256), 0, s, p);
    }
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(pa_gather_kv_kernel, dim3((unsigned)blocks), dim3(256), 0, s, p);
}

}  // namespace pa
