// pa_decode_noalloc.cu -- decode attention whose split-K scratch lives in a
// fixed device array compiled into the library, for callers that must not
// allocate device memory while they run.
//
// Who needs this: code that runs inside a host framework which owns all device
// memory and forbids allocation during its execution step (a plugin or
// operator called from another engine's enqueue), or a latency-critical loop
// that cannot afford cudaMalloc, which can block on the device and can fail
// once the framework has reserved the memory.  Such a caller still passes its
// own inputs and outputs; only the partition partials need a home.
//
// The scratch array below is part of the loaded module, so every device on
// which this library's kernels are loaded holds PA_NOALLOC_SCRATCH_BYTES until
// the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "pa_internal.h"
#include "pagedattn.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

// Device address of g_decode_scratch on the current device.  The lookup runs
// once per device (on that device's first call) and is cached.
int scratch_address(void** out) {
    static std::mutex mu;
    static void* cached[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        char msg[256];
        std::snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
        return pa::set_last_error(PA_ERR_CUDA, msg);
    }
    if (dev < 0 || dev >= 64) return pa::set_last_error(PA_ERR_CUDA, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char msg[256];
            std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress(decode scratch): %s",
                          cudaGetErrorString(e));
            return pa::set_last_error(PA_ERR_CUDA, msg);
        }
        cached[dev] = p;
    }
    *out = cached[dev];
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_attention_noalloc(float* out, const void* q, const pa_pool* pool,
                                           int layer, const int* block_tables,
                                           int max_blocks_per_seq, const int* context_lens,
                                           int batch, int block_size, int num_heads,
                                           int num_kv_heads, int head_dim, float scale,
                                           int partition_blocks, pa_stream_t stream) {
    // Size (and validate) the scratch this call needs before touching the device array.
    size_t need = 0;
    int rc = pa_decode_workspace_size(pool, batch, num_heads, max_blocks_per_seq, partition_blocks,
                                      &need);
    if (rc != PA_OK) return rc;
    if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) {
        // The advice depends on the kernel the call would run: the tcgen05
        // kernel's scratch does not depend on partition_blocks.
        int kind = PA_DECODE_AUTO;
        rc = pa_decode_kernel_choice(pool, num_heads, &kind);
        if (rc != PA_OK) return rc;
        const char* advice =
            kind == PA_DECODE_TCGEN05
                ? "the tcgen05 kernel this call runs ignores partition_blocks (its scratch "
                  "follows the SM count and the (sequence, head group) pairs): use "
                  "pa_decode_attention with a caller-provided workspace"
                : "pass a larger partition_blocks or use pa_decode_attention with a "
                  "caller-provided workspace";
        char msg[512];
        std::snprintf(msg, sizeof msg,
                      "pa_decode_attention_noalloc: this call needs %zu bytes of split-K scratch "
                      "but the built-in scratch holds %zu; %s",
                      need, (size_t)PA_NOALLOC_SCRATCH_BYTES, advice);
        return pa::set_last_error(PA_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    if (need > 0) {
        rc = scratch_address(&scratch);
        if (rc != PA_OK) return rc;
    }
    // Same kernels as the workspace entry point; the partials go to the fixed array.
    return pa_decode_attention_partitioned(out, q, pool, layer, block_tables, max_blocks_per_seq,
                                           context_lens, batch, block_size, num_heads,
                                           num_kv_heads, head_dim, scale, partition_blocks,
                                           scratch, need > 0 ? (size_t)PA_NOALLOC_SCRATCH_BYTES : 0,
                                           stream);
}
