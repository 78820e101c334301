// pa_api.cpp -- the C ABI: pool handle, free-block stack allocator, argument
// validation and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "pa_internal.h"
#include "pagedattn.h"

struct pa_pool {
    pa::PoolGeom g;
    std::vector<int> free_stack;        // allocation pops from the back
    std::vector<unsigned char> in_use;  // 1 while a block is handed out
    bool on_device = false;             // the stack is held in a device copy
    int decode_kernel = PA_DECODE_AUTO;
    // tensor maps of the bf16 pool (K, V) for the tensor-core kernel, encoded
    // on first use
    mutable CUtensorMap tmaps[2];
    mutable bool tmaps_ready = false;
    mutable int tma_slots[3] = {2, 3, 4};
    mutable std::mutex mu;
};

namespace {

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(e == cudaErrorNotSupported ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA, "%s: %s (%s)",
                what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int num_sms_current(int* out) {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PA_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int v = 0;
        e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(multiProcessorCount)");
        cache[dev] = v;
    }
    *out = cache[dev];
    return PA_OK;
}

// Partition size heuristic.  The host does not see the lengths, so the batch's
// K+V is estimated from the table capacity (half full on average) and split so
// that about 12 partitions fall on each SM: enough CTAs of similar size that
// ragged lengths even out.  Bounds: at most 64 blocks and 1 MiB per CTA (more
// only adds partials and idle tail), at least 32 KiB (less is all ramp-up).
// The pick is rounded up to a multiple of 8 blocks (two per warp of a CTA), so
// that a context a little longer than the estimate does not leave a sliver of
// a second partition.  GB300 sweeps (graph-timed calls): large-batch 64 blocks
// (fastest; picks 64); long context 24-48 within 0.5 %, 40 fastest (picks
// 40); MHA batch 64 at lengths up to 1024: 16 / 20 / 24 / 28 blocks 72.8 /
// 71.3 / 71.1 / 75.2 us per call (picks 24; rounding down picked 16);
// mini-infer shape 4-8 (picks 8).
int auto_partition_blocks(const pa::PoolGeom& g, int batch, int maxb, int num_sms, int G) {
    const long long blk_bytes = 2LL * g.B * g.D * g.elt;
    const long long est_total = (long long)batch * g.Hkv * maxb * blk_bytes / 2;
    long long pb = est_total / ((long long)num_sms * 12 * blk_bytes);
    long long hi = 64;
    if (hi * blk_bytes > (1LL << 20)) hi = (1LL << 20) / blk_bytes;
    const long long lo = (32 * 1024 + blk_bytes - 1) / blk_bytes;
    // Groups of 16 and more carry G times the work per K/V byte: fewer, longer
    // partitions win (GB300, large-batch lengths: 64 blocks beat the estimate's
    // 16-32 by 10-54 % for G = 16, 32, 64).
    if (G >= 16) pb = hi;
    if (pb > hi) pb = hi;
    if (pb < lo) pb = lo;
    if (pb > 8) pb = (pb + 7) / 8 * 8;
    if (pb > maxb) pb = maxb;
    if (pb < 1) pb = 1;
    return (int)pb;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t workspace_bytes_for(int batch, int H, int Cmax, int D) {
    if (Cmax <= 1) return 0;
    const size_t slots = (size_t)batch * H * Cmax;
    return align256(slots * D * sizeof(float)) + slots * 2 * sizeof(float);
}

// tcgen05 kernel: two partial slots of `chunk` heads per CTA (its first and
// last piece), one int4 descriptor per (sequence, head group), then one int4
// per CTA naming the cut pair whose first piece it holds (with its
// descriptor).
size_t tc_partial_slots(int grid, int chunk) { return (size_t)grid * 2 * chunk; }
size_t tc_desc_offset(int grid, int chunk, int D) {
    const size_t S = tc_partial_slots(grid, chunk);
    return align256(S * D * sizeof(float)) + align256(S * 2 * sizeof(float));
}
size_t tc_cut_offset(int grid, int chunk, int D, long long pairs) {
    return tc_desc_offset(grid, chunk, D) + align256((size_t)pairs * sizeof(int4));
}
size_t tc_workspace_bytes(int grid, int chunk, int D, long long pairs) {
    if (grid <= 1) return 0;
    return tc_cut_offset(grid, chunk, D, pairs) + (size_t)grid * sizeof(int4);
}

int check_pool(const pa_pool* pool) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "pool handle is NULL");
    return PA_OK;
}

int check_layer(const pa_pool* pool, int layer) {
    if (layer < 0 || layer >= pool->g.L)
        return fail(PA_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, pool->g.L);
    return PA_OK;
}

// The kernels a decode call can run on.
enum class Kernel { CudaCores, MmaSync, Tcgen05 };

struct DecodeShape {
    int G, PB, Cmax;
    Kernel kernel;
    int chunk;    // heads per CTA chunk of the group
    int tc_grid;  // tcgen05 kernel: persistent grid
    size_t ws_bytes;
    bool combine;  // a second kernel merges split contexts
    bool wide;     // mma.sync kernel in wide CTAs, one per (sequence, KV head, chunk)
};

// The kernel the pool's choice selects for group G, or a PA_ERR_UNSUPPORTED
// failure.  Automatic: tcgen05 for groups that are multiples of 16 (head_dim
// 128), mma.sync for the other bf16 shapes, CUDA cores for fp32.  (GB300,
// large-batch lengths, GB/s tcgen05 / mma.sync: G = 64 3562 / 1593, G = 32
// 4854 / 2884, G = 16 5906 / 5152; long context G = 16 5159 / 5181.)
int pick_kernel(const pa_pool* pool, int G, Kernel* k) {
    const pa::PoolGeom& g = pool->g;
    const bool cuda_ok = pa::decode_supported(g.dtype, g.D, g.B, G);
    const bool mma_ok = g.dtype == 1 && pa::decode_mma_supported(g.D, g.B, G);
    const bool umma_ok = g.dtype == 1 && pa::decode_umma_supported(g.D, g.B, G);
    if (!cuda_ok && !mma_ok && !umma_ok)
        return fail(PA_ERR_UNSUPPORTED,
                    "no decode kernel for dtype=%d head_dim=%d block_size=%d group=%d "
                    "(built: head_dim 64/128, block_size 16/32, any group)",
                    g.dtype, g.D, g.B, G);
    switch (pool->decode_kernel) {
        case PA_DECODE_CUDA_CORES:
            if (!cuda_ok)
                return fail(PA_ERR_UNSUPPORTED, "no CUDA-core decode kernel for group size %d", G);
            *k = Kernel::CudaCores;
            return PA_OK;
        case PA_DECODE_TENSOR_CORES:
            if (!mma_ok)
                return fail(PA_ERR_UNSUPPORTED,
                            "no mma.sync tensor-core decode kernel for this pool / group size");
            *k = Kernel::MmaSync;
            return PA_OK;
        case PA_DECODE_TCGEN05:
            if (!umma_ok)
                return fail(PA_ERR_UNSUPPORTED,
                            "no tcgen05 decode kernel for this pool / group size (bf16, head_dim "
                            "128, group a multiple of 16)");
            *k = Kernel::Tcgen05;
            return PA_OK;
        default:
            *k = umma_ok ? Kernel::Tcgen05 : mma_ok ? Kernel::MmaSync : Kernel::CudaCores;
            return PA_OK;
    }
}

// Whether the mma.sync kernel's wide CTAs (one per sequence, KV head and head
// chunk, holding the whole context) suit a call: see decode_mma_wide_fits.
bool wide_fits(const pa_pool* pool, int G, int batch, int maxb, int sms) {
    const int chunk = pa::decode_mma_chunk(G);
    if (chunk == 0) return false;
    return pa::decode_mma_wide_fits(pool->g.D, G, maxb,
                                    (long long)batch * pool->g.Hkv * ((G + chunk - 1) / chunk), sms);
}

int resolve_decode_shape(const pa_pool* pool, int batch, int num_heads, int maxb,
                         int partition_blocks, DecodeShape* out) {
    if (batch < 0) return fail(PA_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (num_heads <= 0 || num_heads % pool->g.Hkv != 0)
        return fail(PA_ERR_INVALID_ARG, "num_heads %d is not a positive multiple of num_kv_heads %d",
                    num_heads, pool->g.Hkv);
    if (maxb <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq %d <= 0", maxb);
    if ((long long)maxb * pool->g.B > INT_MAX)
        return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq * block_size overflows int");
    if (partition_blocks < 0)
        return fail(PA_ERR_INVALID_ARG, "partition_blocks %d < 0", partition_blocks);
    const int G = num_heads / pool->g.Hkv;
    Kernel kernel = Kernel::CudaCores;
    if (int rc = pick_kernel(pool, G, &kernel)) return rc;
    if (kernel == Kernel::Tcgen05) {
        // The tcgen05 kernel splits the tiles evenly over its persistent grid
        // itself; partition_blocks does not apply to it.
        int sms = 0;
        if (int rc = num_sms_current(&sms)) return rc;
        const int chunk = pa::decode_umma_chunk(G);
        const long long pairs = (long long)batch * pool->g.Hkv * ((G + chunk - 1) / chunk);
        if (pairs > INT_MAX)
            return fail(PA_ERR_INVALID_ARG, "%lld (sequence, head group) pairs is too many", pairs);
        // groups served in nc chunks: nc groups of CTAs over the same work
        const long long nc = (G + chunk - 1) / chunk;
        const long long kv_pairs = (long long)batch * pool->g.Hkv;
        const long long tiles = ((long long)maxb * pool->g.B + 127) / 128;
        const long long units = kv_pairs * (tiles > 1 ? tiles : 1);  // upper bound per group
        const long long per_group = std::max(1LL, std::min(units, (long long)sms / nc));
        const int grid = (int)(per_group * nc);
        out->G = G;
        out->kernel = kernel;
        out->PB = maxb;
        // (Cmax only sizes the combine: pieces per pair when all contexts are
        // equally long -- fewer pairs than CTAs means long ones cut in many)
        out->Cmax = kv_pairs < per_group ? (int)((per_group + kv_pairs - 1) / kv_pairs) + 1 : 2;
        out->chunk = chunk;
        out->tc_grid = grid;
        out->ws_bytes = tc_workspace_bytes(grid, chunk, pool->g.D, pairs);
        out->combine = grid > 1;
        return PA_OK;
    }
    const int chunk =
        kernel == Kernel::MmaSync ? pa::decode_mma_chunk(G) : pa::decode_cc_chunk(G);
    const long long nchunks = (G + chunk - 1) / chunk;  // (mma.sync: a ragged last chunk)
    int pb = partition_blocks;
    bool wide = false;
    if (pb == 0) {
        int sms = 0;
        int rc = num_sms_current(&sms);
        if (rc != PA_OK) return rc;
        // Whole contexts in wide CTAs when those fit one wave and each warp
        // streams only a few blocks: no partials and no combine launch.
        wide = kernel == Kernel::MmaSync && wide_fits(pool, G, batch, maxb, sms);
        pb = wide ? maxb : auto_partition_blocks(pool->g, batch, maxb, sms, G);
    }
    if (pb > maxb) pb = maxb;
    const int Cmax = (maxb + pb - 1) / pb;
    if ((long long)batch * pool->g.Hkv * nchunks * Cmax > INT_MAX)
        return fail(PA_ERR_INVALID_ARG, "grid of %lld CTAs is too large",
                    (long long)batch * pool->g.Hkv * nchunks * Cmax);
    out->G = G;
    out->kernel = kernel;
    out->PB = pb;
    out->Cmax = Cmax;
    out->chunk = chunk;
    out->tc_grid = 0;
    out->ws_bytes = workspace_bytes_for(batch, num_heads, Cmax, pool->g.D);
    out->combine = Cmax > 1;
    out->wide = wide;
    return PA_OK;
}

}  // namespace

namespace pa {
int set_last_error(int code, const char* message) { return fail(code, "%s", message); }

bool decode_supported(int dtype, int D, int B, int G) {
    if (dtype != 0 && dtype != 1) return false;
    if (D != 64 && D != 128) return false;
    if (B != 16 && B != 32) return false;
    return decode_cc_chunk(G) > 0;  // (any group: chunks of a power of two)
}
}  // namespace pa

extern "C" {

const char* pa_last_error_string(void) { return t_last_error.c_str(); }

int pa_pool_create(pa_pool** out, void* pool_dev, int num_blocks, int num_layers,
                   int num_kv_heads, int block_size, int head_dim, pa_dtype dtype) {
    if (!out) return fail(PA_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!pool_dev) return fail(PA_ERR_INVALID_ARG, "pool_dev is NULL");
    if (num_blocks <= 0 || num_layers <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
        head_dim <= 0)
        return fail(PA_ERR_INVALID_ARG, "pool geometry must be positive (nb=%d L=%d Hkv=%d B=%d D=%d)",
                    num_blocks, num_layers, num_kv_heads, block_size, head_dim);
    if (dtype != PA_DTYPE_F32 && dtype != PA_DTYPE_BF16)
        return fail(PA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    // The fused mini-infer tensor [num_blocks, 2, L, Hkv, B, D] as strides.
    const long long tile = (long long)block_size * head_dim;
    const long long elt = dtype == PA_DTYPE_F32 ? 4 : 2;
    pa_pool_layout lay;
    lay.k_base = pool_dev;
    lay.v_base = static_cast<char*>(pool_dev) + (long long)num_layers * num_kv_heads * tile * elt;
    lay.block_stride = 2LL * num_layers * num_kv_heads * tile;
    lay.layer_stride = (long long)num_kv_heads * tile;
    lay.head_stride = tile;
    return pa_pool_create_strided(out, &lay, num_blocks, num_layers, num_kv_heads, block_size,
                                  head_dim, dtype);
}

int pa_pool_create_strided(pa_pool** out, const pa_pool_layout* layout, int num_blocks,
                           int num_layers, int num_kv_heads, int block_size, int head_dim,
                           pa_dtype dtype) {
    if (!out) return fail(PA_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!layout) return fail(PA_ERR_INVALID_ARG, "layout is NULL");
    if (!layout->k_base || !layout->v_base)
        return fail(PA_ERR_INVALID_ARG, "k_base and v_base must be non-NULL");
    if (!aligned(layout->k_base, 16) || !aligned(layout->v_base, 16))
        return fail(PA_ERR_INVALID_ARG, "k_base and v_base must be 16-byte aligned");
    if (num_blocks <= 0 || num_layers <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
        head_dim <= 0)
        return fail(PA_ERR_INVALID_ARG, "pool geometry must be positive (nb=%d L=%d Hkv=%d B=%d D=%d)",
                    num_blocks, num_layers, num_kv_heads, block_size, head_dim);
    if (dtype != PA_DTYPE_F32 && dtype != PA_DTYPE_BF16)
        return fail(PA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    const int elt = dtype == PA_DTYPE_F32 ? 4 : 2;
    if ((head_dim * elt) % 16 != 0)
        return fail(PA_ERR_INVALID_ARG, "head_dim * element size (%d) must be a multiple of 16",
                    head_dim * elt);
    // Strides: non-negative, 16-byte multiples, zero only for a dimension of
    // extent one, and tiles of one base must not overlap.
    struct Dim {
        long long stride, count;
        const char* name;
    } dims[3] = {{layout->block_stride, num_blocks, "block_stride"},
                 {layout->layer_stride, num_layers, "layer_stride"},
                 {layout->head_stride, num_kv_heads, "head_stride"}};
    for (const Dim& d : dims) {
        if (d.stride < 0) return fail(PA_ERR_INVALID_ARG, "%s is negative", d.name);
        if ((d.stride * elt) % 16 != 0)
            return fail(PA_ERR_INVALID_ARG, "%s * element size must be a multiple of 16 bytes",
                        d.name);
        if (d.stride == 0 && d.count > 1)
            return fail(PA_ERR_INVALID_ARG, "%s is 0 but that dimension has %lld entries", d.name,
                        d.count);
    }
    {
        Dim live[3];
        int n = 0;
        for (const Dim& d : dims)
            if (d.count > 1) live[n++] = d;
        for (int a = 0; a < n; ++a)
            for (int b = a + 1; b < n; ++b)
                if (live[b].stride < live[a].stride) {
                    Dim t = live[a];
                    live[a] = live[b];
                    live[b] = t;
                }
        long long extent = (long long)block_size * head_dim;  // one contiguous tile
        for (int a = 0; a < n; ++a) {
            if (live[a].stride < extent)
                return fail(PA_ERR_INVALID_ARG, "%s = %lld makes tiles overlap (needs >= %lld)",
                            live[a].name, live[a].stride, extent);
            const double ext = (double)live[a].stride * (double)live[a].count;
            if (ext > 4.0e18) return fail(PA_ERR_INVALID_ARG, "pool too large");
            extent = live[a].stride * live[a].count;
        }
    }
    try {
        pa_pool* p = new pa_pool();
        p->g.k_base = layout->k_base;
        p->g.v_base = layout->v_base;
        p->g.s_blk = layout->block_stride;
        p->g.s_layer = layout->layer_stride;
        p->g.s_head = layout->head_stride;
        p->g.num_blocks = num_blocks;
        p->g.L = num_layers;
        p->g.Hkv = num_kv_heads;
        p->g.B = block_size;
        p->g.D = head_dim;
        p->g.elt = elt;
        p->g.dtype = (int)dtype;
        p->free_stack.resize(num_blocks);
        for (int i = 0; i < num_blocks; ++i) p->free_stack[i] = i;
        p->in_use.assign(num_blocks, 0);
        *out = p;
    } catch (const std::bad_alloc&) {
        return fail(PA_ERR_INVALID_ARG, "host allocation failed for %d blocks", num_blocks);
    }
    return PA_OK;
}

int pa_pool_destroy(pa_pool* pool) {
    delete pool;
    return PA_OK;
}

int pa_pool_set_decode_kernel(pa_pool* pool, int kind) {
    if (int rc = check_pool(pool)) return rc;
    if (kind != PA_DECODE_AUTO && kind != PA_DECODE_CUDA_CORES && kind != PA_DECODE_TENSOR_CORES &&
        kind != PA_DECODE_TCGEN05)
        return fail(PA_ERR_INVALID_ARG, "unknown decode kernel kind %d", kind);
    std::lock_guard<std::mutex> lock(pool->mu);
    pool->decode_kernel = kind;
    return PA_OK;
}

int pa_decode_kernel_choice(const pa_pool* pool, int num_heads, int* kind) {
    if (int rc = check_pool(pool)) return rc;
    if (!kind) return fail(PA_ERR_INVALID_ARG, "kind is NULL");
    if (num_heads <= 0 || num_heads % pool->g.Hkv != 0)
        return fail(PA_ERR_INVALID_ARG, "num_heads %d is not a positive multiple of num_kv_heads %d",
                    num_heads, pool->g.Hkv);
    Kernel k = Kernel::CudaCores;
    if (int rc = pick_kernel(pool, num_heads / pool->g.Hkv, &k)) return rc;
    *kind = k == Kernel::Tcgen05   ? PA_DECODE_TCGEN05
            : k == Kernel::MmaSync ? PA_DECODE_TENSOR_CORES
                                   : PA_DECODE_CUDA_CORES;
    return PA_OK;
}

int pa_pool_block_bytes(const pa_pool* pool, size_t* bytes) {
    if (int rc = check_pool(pool)) return rc;
    if (!bytes) return fail(PA_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = (size_t)2 * pool->g.L * pool->g.Hkv * pool->g.B * pool->g.D * pool->g.elt;
    return PA_OK;
}

int pa_pool_seed_free_stack(pa_pool* pool, const int* order, int n) {
    if (int rc = check_pool(pool)) return rc;
    if (!order) return fail(PA_ERR_INVALID_ARG, "order is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    if (pool->on_device)
        return fail(PA_ERR_INVALID_ARG, "the free stack is held on the device; download it first");
    const long long nb = pool->g.num_blocks;
    if (n != nb) return fail(PA_ERR_INVALID_ARG, "order has %d entries, pool has %lld blocks", n, nb);
    if ((long long)pool->free_stack.size() != nb)
        return fail(PA_ERR_INVALID_ARG, "seeding requires every block to be free");
    std::vector<unsigned char> seen(nb, 0);
    for (int i = 0; i < n; ++i) {
        if (order[i] < 0 || order[i] >= nb || seen[order[i]])
            return fail(PA_ERR_INVALID_ARG, "order is not a permutation of 0..%lld (entry %d = %d)",
                        nb - 1, i, order[i]);
        seen[order[i]] = 1;
    }
    pool->free_stack.assign(order, order + n);
    return PA_OK;
}

int pa_alloc_block(pa_pool* pool, int* block_id) {
    if (int rc = check_pool(pool)) return rc;
    if (!block_id) return fail(PA_ERR_INVALID_ARG, "block_id is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    if (pool->on_device)
        return fail(PA_ERR_INVALID_ARG, "the free stack is held on the device; download it first");
    if (pool->free_stack.empty())
        return fail(PA_ERR_NO_FREE_BLOCKS, "Out of KV-Cache Physical Blocks");
    const int id = pool->free_stack.back();
    pool->free_stack.pop_back();
    pool->in_use[id] = 1;
    *block_id = id;
    return PA_OK;
}

int pa_free_block(pa_pool* pool, int block_id) {
    if (int rc = check_pool(pool)) return rc;
    std::lock_guard<std::mutex> lock(pool->mu);
    if (pool->on_device)
        return fail(PA_ERR_INVALID_ARG, "the free stack is held on the device; download it first");
    if (block_id < 0 || block_id >= pool->g.num_blocks)
        return fail(PA_ERR_INVALID_ARG, "block id %d outside [0, %lld)", block_id, pool->g.num_blocks);
    if (!pool->in_use[block_id])
        return fail(PA_ERR_DOUBLE_FREE, "block %d is not allocated", block_id);
    pool->in_use[block_id] = 0;
    pool->free_stack.push_back(block_id);
    return PA_OK;
}

int pa_num_free(const pa_pool* pool, int* n) {
    if (int rc = check_pool(pool)) return rc;
    if (!n) return fail(PA_ERR_INVALID_ARG, "n is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    *n = (int)pool->free_stack.size();
    return PA_OK;
}

int pa_device_stack_bytes(const pa_pool* pool, size_t* bytes) {
    if (int rc = check_pool(pool)) return rc;
    if (!bytes) return fail(PA_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = ((size_t)pool->g.num_blocks + 1) * sizeof(int);
    return PA_OK;
}

int pa_device_stack_upload(pa_pool* pool, void* dev_stack, pa_stream_t stream) {
    if (int rc = check_pool(pool)) return rc;
    if (!dev_stack || !aligned(dev_stack, 4))
        return fail(PA_ERR_INVALID_ARG, "dev_stack must be non-NULL and 4-byte aligned");
    std::lock_guard<std::mutex> lock(pool->mu);
    if (pool->on_device) return fail(PA_ERR_INVALID_ARG, "the free stack is already on the device");
    std::vector<int> img(pool->free_stack.size() + 1);
    img[0] = (int)pool->free_stack.size();
    std::copy(pool->free_stack.begin(), pool->free_stack.end(), img.begin() + 1);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(dev_stack, img.data(), img.size() * sizeof(int),
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "pa_device_stack_upload");
    pool->on_device = true;
    return PA_OK;
}

int pa_device_stack_download(pa_pool* pool, const void* dev_stack, pa_stream_t stream) {
    if (int rc = check_pool(pool)) return rc;
    if (!dev_stack || !aligned(dev_stack, 4))
        return fail(PA_ERR_INVALID_ARG, "dev_stack must be non-NULL and 4-byte aligned");
    std::lock_guard<std::mutex> lock(pool->mu);
    if (!pool->on_device) return fail(PA_ERR_INVALID_ARG, "the free stack is not on the device");
    const long long nb = pool->g.num_blocks;
    std::vector<int> img(nb + 1);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess)
        e = cudaMemcpy(img.data(), dev_stack, img.size() * sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "pa_device_stack_download");
    const int height = img[0];
    if (height < 0 || height > nb)
        return fail(PA_ERR_INVALID_ARG, "device stack height %d outside [0, %lld]", height, nb);
    std::vector<unsigned char> in_stack(nb, 0);
    for (int i = 0; i < height; ++i) {
        const int id = img[1 + i];
        if (id < 0 || id >= nb || in_stack[id])
            return fail(PA_ERR_INVALID_ARG, "device stack entry %d (= %d) is invalid or repeated",
                        i, id);
        in_stack[id] = 1;
    }
    pool->free_stack.assign(img.begin() + 1, img.begin() + 1 + height);
    for (long long i = 0; i < nb; ++i) pool->in_use[i] = in_stack[i] ? 0 : 1;
    pool->on_device = false;
    return PA_OK;
}

static int device_alloc(const char* who, pa_pool* pool, void* dev_stack, int* block_tables,
                        int max_blocks_per_seq, const int* positions, int* next_lens, int batch,
                        pa_stream_t stream) {
    if (int rc = check_pool(pool)) return rc;
    if (batch < 0 || max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "batch (%d) / max_blocks_per_seq (%d) out of range", batch,
                    max_blocks_per_seq);
    if (batch == 0) return PA_OK;
    if (!dev_stack || !block_tables || !positions || !aligned(dev_stack, 4) ||
        !aligned(block_tables, 4) || !aligned(positions, 4))
        return fail(PA_ERR_INVALID_ARG, "dev_stack, block_tables, positions: non-NULL, 4-byte aligned");
    if (next_lens) {
        if (!aligned(next_lens, 4))
            return fail(PA_ERR_INVALID_ARG, "next_lens: 4-byte aligned");
        const char* a = reinterpret_cast<const char*>(positions);
        const char* n = reinterpret_cast<const char*>(next_lens);
        const size_t bytes = (size_t)batch * sizeof(int);
        if (n < a + bytes && a < n + bytes)
            return fail(PA_ERR_INVALID_ARG, "next_lens overlaps positions");
    }
    unsigned* status = nullptr;
    cudaError_t e = pa::status_word(&status);
    if (e != cudaSuccess) return cuda_fail(e, "status word lookup");
    e = pa::launch_device_alloc(static_cast<int*>(dev_stack), block_tables, max_blocks_per_seq,
                                positions, next_lens, batch, pool->g.B, status,
                                reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return PA_OK;
}

int pa_device_alloc_blocks(pa_pool* pool, void* dev_stack, int* block_tables,
                           int max_blocks_per_seq, const int* positions, int batch,
                           pa_stream_t stream) {
    return device_alloc("pa_device_alloc_blocks launch", pool, dev_stack, block_tables,
                        max_blocks_per_seq, positions, nullptr, batch, stream);
}

int pa_device_alloc_blocks_step(pa_pool* pool, void* dev_stack, int* block_tables,
                                int max_blocks_per_seq, const int* positions, int* next_lens,
                                int batch, pa_stream_t stream) {
    if (!next_lens) return fail(PA_ERR_INVALID_ARG, "next_lens is NULL");
    return device_alloc("pa_device_alloc_blocks_step launch", pool, dev_stack, block_tables,
                        max_blocks_per_seq, positions, next_lens, batch, stream);
}

int pa_device_free_blocks(pa_pool* pool, void* dev_stack, int* block_tables,
                          int max_blocks_per_seq, const int* context_lens, const uint8_t* finished,
                          int batch, pa_stream_t stream) {
    if (int rc = check_pool(pool)) return rc;
    if (batch < 0 || max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "batch (%d) / max_blocks_per_seq (%d) out of range", batch,
                    max_blocks_per_seq);
    if (batch == 0) return PA_OK;
    if (!dev_stack || !block_tables || !context_lens || !finished || !aligned(dev_stack, 4) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return fail(PA_ERR_INVALID_ARG,
                    "dev_stack, block_tables, context_lens, finished: non-NULL, aligned");
    unsigned* status = nullptr;
    cudaError_t e = pa::status_word(&status);
    if (e != cudaSuccess) return cuda_fail(e, "status word lookup");
    e = pa::launch_device_free(static_cast<int*>(dev_stack), block_tables, max_blocks_per_seq,
                               context_lens, finished, batch, pool->g.B, pool->g.num_blocks,
                               status, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_device_free_blocks launch");
    return PA_OK;
}

int pa_write_kv(pa_pool* pool, int layer, const void* k, const void* v, const int* block_tables,
                int max_blocks_per_seq, const int* positions, int batch, pa_stream_t stream) {
    if (int rc = check_pool(pool)) return rc;
    if (int rc = check_layer(pool, layer)) return rc;
    if (batch < 0) return fail(PA_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq %d <= 0", max_blocks_per_seq);
    if (batch == 0) return PA_OK;
    if (!k || !v || !block_tables || !positions)
        return fail(PA_ERR_INVALID_ARG, "k, v, block_tables and positions must be non-NULL");
    if (!aligned(k, 16) || !aligned(v, 16))
        return fail(PA_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    if (!aligned(block_tables, 4) || !aligned(positions, 4))
        return fail(PA_ERR_INVALID_ARG, "block_tables and positions must be 4-byte aligned");
    int sms = 0;
    if (int rc = num_sms_current(&sms)) return rc;
    unsigned* status = nullptr;
    cudaError_t e = pa::status_word(&status);
    if (e != cudaSuccess) return cuda_fail(e, "status word lookup");
    const pa::PoolGeom& g = pool->g;
    pa::WriteParams p{g.k_base, g.v_base, g.s_blk, layer * g.s_layer, g.s_head, g.num_blocks,
                      g.Hkv, g.B, g.D * g.elt, g.elt, layer, k, v, block_tables,
                      max_blocks_per_seq, positions, batch, status};
    e = pa::launch_write_kv(p, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_write_kv launch");
    return PA_OK;
}

int pa_decode_partition_blocks(const pa_pool* pool, int batch, int num_heads,
                               int max_blocks_per_seq, int* partition_blocks) {
    if (int rc = check_pool(pool)) return rc;
    if (!partition_blocks) return fail(PA_ERR_INVALID_ARG, "partition_blocks is NULL");
    DecodeShape sh{};
    if (int rc = resolve_decode_shape(pool, batch, num_heads, max_blocks_per_seq, 0, &sh)) return rc;
    *partition_blocks = sh.PB;
    return PA_OK;
}

int pa_decode_workspace_size(const pa_pool* pool, int batch, int num_heads,
                             int max_blocks_per_seq, int partition_blocks, size_t* bytes) {
    if (int rc = check_pool(pool)) return rc;
    if (!bytes) return fail(PA_ERR_INVALID_ARG, "bytes is NULL");
    DecodeShape sh{};
    if (int rc = resolve_decode_shape(pool, batch, num_heads, max_blocks_per_seq, partition_blocks,
                                      &sh))
        return rc;
    *bytes = sh.ws_bytes;
    return PA_OK;
}

}  // extern "C"

namespace {

// Decode attention; with new_k/new_v/positions non-null the append of one
// token per sequence is fused into the decode kernel.
int decode_impl(float* out, const void* q, const pa_pool* pool, int layer,
                const int* block_tables, int max_blocks_per_seq, const int* context_lens,
                int batch, int block_size, int num_heads, int num_kv_heads, int head_dim,
                float scale, int partition_blocks, void* workspace, size_t workspace_bytes,
                pa_stream_t stream, const void* new_k, const void* new_v, const int* positions) {
    if (int rc = check_pool(pool)) return rc;
    if (int rc = check_layer(pool, layer)) return rc;
    const pa::PoolGeom& g = pool->g;
    if (block_size != g.B || num_kv_heads != g.Hkv || head_dim != g.D)
        return fail(PA_ERR_INVALID_ARG,
                    "block_size/num_kv_heads/head_dim (%d/%d/%d) do not match the pool (%d/%d/%d)",
                    block_size, num_kv_heads, head_dim, g.B, g.Hkv, g.D);
    if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale is not finite");
    DecodeShape sh{};
    if (int rc = resolve_decode_shape(pool, batch, num_heads, max_blocks_per_seq, partition_blocks,
                                      &sh))
        return rc;
    if (batch == 0) return PA_OK;
    if (!out || !q || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "out, q, block_tables and context_lens must be non-NULL");
    if (!aligned(out, 16) || !aligned(q, 16))
        return fail(PA_ERR_INVALID_ARG, "out and q must be 16-byte aligned");
    if (!aligned(block_tables, 4) || !aligned(context_lens, 4))
        return fail(PA_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");
    float* part_o = nullptr;
    float* part_ml = nullptr;
    int4* tc_desc = nullptr;
    int4* tc_cut = nullptr;
    if (sh.ws_bytes > 0) {
        if (!workspace || workspace_bytes < sh.ws_bytes || !aligned(workspace, 256))
            return fail(PA_ERR_WORKSPACE,
                        "workspace must be 256-byte aligned and hold %zu bytes (got %p, %zu)",
                        sh.ws_bytes, workspace, workspace_bytes);
        char* ws = static_cast<char*>(workspace);
        part_o = reinterpret_cast<float*>(ws);
        if (sh.kernel == Kernel::Tcgen05) {
            const size_t S = tc_partial_slots(sh.tc_grid, sh.chunk);
            const long long pairs = (long long)batch * g.Hkv * ((sh.G + sh.chunk - 1) / sh.chunk);
            part_ml = reinterpret_cast<float*>(ws + align256(S * g.D * sizeof(float)));
            tc_desc = reinterpret_cast<int4*>(ws + tc_desc_offset(sh.tc_grid, sh.chunk, g.D));
            tc_cut = reinterpret_cast<int4*>(ws + tc_cut_offset(sh.tc_grid, sh.chunk, g.D, pairs));
        } else {
            part_ml = reinterpret_cast<float*>(
                ws + align256((size_t)batch * num_heads * sh.Cmax * g.D * sizeof(float)));
        }
    }
    unsigned* status = nullptr;
    cudaError_t e = pa::status_word(&status);
    if (e != cudaSuccess) return cuda_fail(e, "status word lookup");
    pa::DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_base = g.k_base;
    p.v_base = g.v_base;
    p.s_blk = g.s_blk;
    p.tile_off = layer * g.s_layer;
    p.s_head = g.s_head;
    p.num_blocks = g.num_blocks;
    p.Hkv = g.Hkv;
    p.layer = layer;
    p.bt = block_tables;
    p.maxb = max_blocks_per_seq;
    p.lens = context_lens;
    p.batch = batch;
    p.H = num_heads;
    p.qscale = scale * 1.4426950408889634f;  // log2(e): softmax evaluated with exp2
    p.part_o = part_o;
    p.part_ml = part_ml;
    p.PB = sh.PB;
    p.Cmax = sh.Cmax;
    p.status = status;
    p.new_k = new_k;
    p.new_v = new_v;
    p.positions = positions;
    p.tc_grid = sh.tc_grid;
    p.tc_desc = tc_desc;
    p.tc_cut = tc_cut;
    p.gsize = sh.G;
    p.nchunks = (sh.G + sh.chunk - 1) / sh.chunk;
    p.chunk = sh.chunk;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!sh.wide && sh.kernel == Kernel::MmaSync && sh.Cmax == 1) {
        // an explicit partition that covers the table: wide CTAs where they fit
        int sms = 0;
        if (int rc = num_sms_current(&sms)) return rc;
        sh.wide = wide_fits(pool, sh.G, batch, max_blocks_per_seq, sms);
    }
    if (sh.kernel != Kernel::CudaCores) {
        {
            std::lock_guard<std::mutex> lock(pool->mu);
            if (!pool->tmaps_ready) {
                e = pa::encode_pool_tmaps(g, pool->tmaps, &pool->tma_slots[0],
                                          &pool->tma_slots[1], &pool->tma_slots[2]);
                if (e != cudaSuccess) return cuda_fail(e, "tensor map encoding");
                pool->tmaps_ready = true;
            }
        }
        p.tma_slot_blk = pool->tma_slots[0];
        p.tma_slot_layer = pool->tma_slots[1];
        p.tma_slot_head = pool->tma_slots[2];
        e = sh.kernel == Kernel::Tcgen05 ? pa::launch_decode_umma(p, pool->tmaps, g.B, sh.G, s)
            : sh.wide ? pa::launch_decode_mma_wide(p, pool->tmaps, g.D, g.B, sh.G, s)
                      : pa::launch_decode_mma(p, pool->tmaps, g.D, g.B, sh.G, s);
    } else {
        e = g.dtype == 1 ? pa::launch_decode_bf16(p, g.D, g.B, sh.G, s)
                         : pa::launch_decode_f32(p, g.D, g.B, sh.G, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    if (sh.combine && sh.kernel == Kernel::Tcgen05) {
        // (fewer pairs than CTAs: most are cut, so every pair gets a CTA group)
        const long long pairs = (long long)batch * g.Hkv * ((sh.G + sh.chunk - 1) / sh.chunk);
        e = pa::launch_combine_tc(p, g.D, pairs <= sh.tc_grid, sh.Cmax, s);
        if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    } else if (sh.combine) {
        e = pa::launch_combine(p, g.D, g.B, s);
        if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    }
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_decode_attention_partitioned(float* out, const void* q, const pa_pool* pool, int layer,
                                    const int* block_tables, int max_blocks_per_seq,
                                    const int* context_lens, int batch, int block_size,
                                    int num_heads, int num_kv_heads, int head_dim, float scale,
                                    int partition_blocks, void* workspace,
                                    size_t workspace_bytes, pa_stream_t stream) {
    return decode_impl(out, q, pool, layer, block_tables, max_blocks_per_seq, context_lens, batch,
                       block_size, num_heads, num_kv_heads, head_dim, scale, partition_blocks,
                       workspace, workspace_bytes, stream, nullptr, nullptr, nullptr);
}

int pa_write_kv_and_decode(float* out, const void* q, pa_pool* pool, int layer, const void* k,
                           const void* v, const int* positions, const int* block_tables,
                           int max_blocks_per_seq, const int* context_lens, int batch,
                           int block_size, int num_heads, int num_kv_heads, int head_dim,
                           float scale, int partition_blocks, void* workspace,
                           size_t workspace_bytes, pa_stream_t stream) {
    if (batch > 0) {
        if (!k || !v || !positions)
            return fail(PA_ERR_INVALID_ARG, "k, v and positions must be non-NULL");
        if (!aligned(k, 16) || !aligned(v, 16))
            return fail(PA_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
        if (!aligned(positions, 4))
            return fail(PA_ERR_INVALID_ARG, "positions must be 4-byte aligned");
    }
    return decode_impl(out, q, pool, layer, block_tables, max_blocks_per_seq, context_lens, batch,
                       block_size, num_heads, num_kv_heads, head_dim, scale, partition_blocks,
                       workspace, workspace_bytes, stream, k, v, positions);
}

int pa_decode_attention(float* out, const void* q, const pa_pool* pool, int layer,
                        const int* block_tables, int max_blocks_per_seq, const int* context_lens,
                        int batch, int block_size, int num_heads, int num_kv_heads, int head_dim,
                        float scale, void* workspace, size_t workspace_bytes,
                        pa_stream_t stream) {
    return pa_decode_attention_partitioned(out, q, pool, layer, block_tables, max_blocks_per_seq,
                                           context_lens, batch, block_size, num_heads,
                                           num_kv_heads, head_dim, scale, 0, workspace,
                                           workspace_bytes, stream);
}

int pa_gather_kv(void* k_out, void* v_out, uint8_t* mask, const pa_pool* pool, int layer,
                 const int* block_tables, int max_blocks_per_seq, const int* context_lens,
                 int batch, int max_len, pa_stream_t stream) {
    if (int rc = check_pool(pool)) return rc;
    if (int rc = check_layer(pool, layer)) return rc;
    if (batch < 0 || max_len < 0)
        return fail(PA_ERR_INVALID_ARG, "batch (%d) and max_len (%d) must be >= 0", batch, max_len);
    if (max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq %d <= 0", max_blocks_per_seq);
    if (batch == 0 || max_len == 0) return PA_OK;
    if (!k_out || !v_out || !mask || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "output and table pointers must be non-NULL");
    if (!aligned(k_out, 16) || !aligned(v_out, 16))
        return fail(PA_ERR_INVALID_ARG, "k_out and v_out must be 16-byte aligned");
    int sms = 0;
    if (int rc = num_sms_current(&sms)) return rc;
    unsigned* status = nullptr;
    cudaError_t e = pa::status_word(&status);
    if (e != cudaSuccess) return cuda_fail(e, "status word lookup");
    const pa::PoolGeom& g = pool->g;
    pa::GatherParams p{k_out,       v_out,   mask,       g.k_base,     g.v_base,
                       g.s_blk,     layer * g.s_layer, g.s_head, g.num_blocks, g.Hkv,
                       g.B,         g.D * g.elt, g.elt,   layer,      block_tables,
                       max_blocks_per_seq, context_lens, batch, max_len, status};
    e = pa::launch_gather_kv(p, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_gather_kv launch");
    return PA_OK;
}

int pa_selftest_wait_timeout(pa_stream_t stream) {
    unsigned* status = nullptr;
    cudaError_t e = pa::status_word(&status);
    if (e != cudaSuccess) return cuda_fail(e, "status word lookup");
    e = pa::launch_wait_selftest(status, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_selftest_wait_timeout launch");
    return PA_OK;
}

int pa_get_status(unsigned int* status, pa_stream_t stream) {
    if (!status) return fail(PA_ERR_INVALID_ARG, "status is NULL");
    cudaError_t e = pa::read_and_clear_status(status, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_get_status");
    return PA_OK;
}

}  // extern "C"
