/*
 * pagedattn.h -- C ABI of the GB300 paged KV-cache decode library.
 *
 * The library keeps a transformer's KV cache in ONE preallocated device tensor
 * of fixed-size physical blocks and runs decode attention directly on it,
 * resolving every token through a per-sequence block table.
 *
 * Sources of the semantics (page title, section):
 *  - "Paged KV-Cache Memory Management" (mini-infer), "The Solution" and
 *    "Python Implementation: Physical Block Pool": the pool tensor
 *    [num_blocks, 2 (K/V), num_layers, num_kv_heads, block_size, head_dim],
 *    zero-initialised once, and the free-block stack allocator
 *    (ids 0..n-1, allocation pops from the end, exhaustion is an error).
 *  - "vllmini", "PagedAttention Metaphor" and "The CUDA Block Kernel": logical
 *    block i of a sequence lives in physical block block_table[i]; the kernel
 *    resolves token t to (block_table[t / B], t % B) on the fly; the kernel's
 *    argument list (out, q, caches, block_tables, context_lens, block_size,
 *    num_heads, head_size).
 *  - "kv-cache" skill, section 2 "PagedAttention Architecture": blocks are
 *    taken one at a time as a sequence grows; only the last block is partly
 *    filled.
 *
 * Conventions for every call:
 *  - Return value: PA_OK (0) or a PA_ERR_* code; pa_last_error_string() then
 *    describes the failure (per calling thread).  Nothing throws across the ABI.
 *  - Device pointers are plain CUDA device addresses on the CURRENT device.
 *    The caller owns every device buffer (pool, q, k, v, out, tables, lengths,
 *    positions, workspace); the library owns only the pool handle and its
 *    host-side free stack.
 *  - Kernels are enqueued asynchronously on `stream` (NULL = legacy default
 *    stream).  Buffers must stay valid until the stream reaches the call.
 *  - Argument checks that need no device data happen on the host before any
 *    launch and return PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED.  Checks that
 *    need device data (block ids, lengths, positions) happen in the kernels:
 *    an offending row is skipped (never read or written out of bounds) and a
 *    bit is set in the device status word, read with pa_get_status().
 *  - The first launching call on a device looks up the device status word; do
 *    that call (or pa_get_status) once before capturing a stream into a graph.
 *  - Per device, for the life of the process, the library caches the status
 *    word's address, the SM count and the no-allocation scratch address
 *    (pa_decode_attention_noalloc).  These do not survive cudaDeviceReset():
 *    do not use the library on a device after resetting it in the same
 *    process.
 *  - Each declaration below names the passage of the source pages it restates
 *    ("Cites:"), or says that the pages have no counterpart.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Every entry point below is exported; the library hides all other symbols. */
#if defined(__GNUC__) || defined(__clang__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

/* Opaque pool handle: geometry + device pointer + host free-block stack. */
typedef struct pa_pool pa_pool;

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* pa_stream_t;

/* Element type of the pool, q, k and v. */
typedef enum pa_dtype { PA_DTYPE_F32 = 0, PA_DTYPE_BF16 = 1 } pa_dtype;

/* Return codes. */
enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, geometry mismatch */
    PA_ERR_NO_FREE_BLOCKS = 2, /* allocator exhausted ("Out of KV-Cache Physical Blocks") */
    PA_ERR_DOUBLE_FREE = 3,    /* freeing a block that is not allocated */
    PA_ERR_CUDA = 4,           /* a CUDA runtime call failed (message has the CUDA error) */
    PA_ERR_UNSUPPORTED = 5,    /* valid arguments, but no kernel is built for this shape */
    PA_ERR_WORKSPACE = 6       /* workspace missing, misaligned or smaller than required */
};

/* Bits of the device status word (pa_get_status). */
#define PA_STATUS_BAD_BLOCK_ID 0x1u /* a table entry read was outside [0, num_blocks) */
#define PA_STATUS_BAD_LENGTH 0x2u   /* a context length / position outside the table */
#define PA_STATUS_TIMEOUT 0x4u      /* a bounded wait for a shared-memory copy gave up */
#define PA_STATUS_NO_FREE_BLOCKS 0x8u /* the device free stack ran dry during an allocation */

/* Human-readable description of the calling thread's last error ("" if none).
 * Cites: no counterpart on the pages (this interface's error reporting); the one
 * error the pages name is the allocator's "Out of KV-Cache Physical Blocks"
 * (mini-infer, "Python Implementation: Physical Block Pool"). */
PA_API const char* pa_last_error_string(void);

/* ----------------------------------------------------------------------------
 * Pool and allocator (host only; none of these calls touches the GPU).
 * ------------------------------------------------------------------------- */

/*
 * Wrap an existing device tensor as a block pool (mini-infer BlockPool).
 *   pool_dev   device pointer to num_blocks * 2 * num_layers * num_kv_heads *
 *              block_size * head_dim elements of `dtype`, row-major in that
 *              order, 16-byte aligned.  Caller-owned; never freed here.
 *   geometry   all > 0; head_dim * sizeof(dtype) must be a multiple of 16.
 * The free stack starts as 0..num_blocks-1; pa_alloc_block pops the END, so
 * the first id handed out is num_blocks-1.
 * Cites: mini-infer, "Python Implementation: Physical Block Pool" (the pool
 * tensor's shape and order, one allocation at start-up, the free list
 * range(num_blocks)) and "The Solution" (fixed-size physical blocks).
 */
PA_API int pa_pool_create(pa_pool** out, void* pool_dev, int num_blocks, int num_layers,
                   int num_kv_heads, int block_size, int head_dim, pa_dtype dtype);

/*
 * Any other layout whose B x D tile of one (physical block, layer, KV head) is
 * a contiguous row-major [block_size, head_dim] array -- for instance vllmini's
 * separate k_cache / v_cache tensors ("vllmini", "The CUDA Block Kernel"), or
 * per-layer caches stacked layer-major.  K row t of the tile of (block, layer,
 * head) starts at element
 *     block*block_stride + layer*layer_stride + head*head_stride + t*head_dim
 * from k_base, V rows likewise from v_base (strides in elements).
 * Requirements: bases 16-byte aligned; strides >= 0 and multiples of 16 bytes;
 * a stride may be 0 only for a dimension of extent 1; the tiles reachable
 * from one base must not overlap (checked).  K and V tiles must not overlap
 * each other (not checked).  pa_pool_create is this call with the fused
 * layout's strides.
 * Cites: "vllmini", "The CUDA Block Kernel" (the kernel takes k_cache and
 * v_cache as separate arguments).
 */
typedef struct pa_pool_layout {
    void* k_base;
    void* v_base;
    int64_t block_stride;
    int64_t layer_stride;
    int64_t head_stride;
} pa_pool_layout;

PA_API int pa_pool_create_strided(pa_pool** out, const pa_pool_layout* layout, int num_blocks,
                                  int num_layers, int num_kv_heads, int block_size, int head_dim,
                                  pa_dtype dtype);

/* Release the handle (not the caller's device tensor).  NULL is accepted.
 * Cites: mini-infer, "Python Implementation: Physical Block Pool" (the pool
 * tensor is allocated once by its owner; the page shows no teardown, so this
 * call only drops what pa_pool_create made: the handle and its free stack). */
PA_API int pa_pool_destroy(pa_pool* pool);

/* Built shapes: head_dim 64 or 128, block_size 16 or 32; GQA group
 * (num_heads / num_kv_heads) of any size on the mma.sync tensor-core kernel
 * (bf16 pools; groups above 8 run as 16- or 8-head chunks whose CTAs share
 * each K/V tile through L2, the last chunk holding the rest of a group that
 * is no multiple of 8), any multiple of 16 on the
 * tcgen05 kernel (bf16 pools, head_dim 128; chunks of 128, 64, 48, 32 or 16
 * heads, groups of 80, 96 and 112 in one 128-head chunk), and of any size
 * on the CUDA-core kernel (every dtype; head chunks of a power of two up to 8,
 * the heads past the group masked).  Other shapes: PA_ERR_UNSUPPORTED.
 *
 * Which decode kernel a pool's decode calls use.  PA_DECODE_AUTO (default):
 * for bf16 pools with head_dim 128 the tcgen05 kernel for groups that are
 * multiples of 16 (S and O accumulate in tensor memory), else the mma.sync
 * kernel (K/V staged by tensor-map TMA); the CUDA-core kernel for fp32 pools.
 * PA_DECODE_CUDA_CORES forces the CUDA-core kernel (fp32 FMA on every dtype),
 * PA_DECODE_TENSOR_CORES the mma.sync kernel, PA_DECODE_TCGEN05 the tcgen05
 * kernel; a forced kernel that cannot serve a call makes it fail with
 * PA_ERR_UNSUPPORTED.  All compute the same result within the stated
 * tolerances.  The choice also fixes the automatic partition size (and so the
 * workspace size): query pa_decode_workspace_size after setting it.
 * The tcgen05 kernel does not use partitions: it runs one persistent CTA per
 * SM and gives each CTA an equal share of the call's 128-token tiles (in
 * sequence, head-group, tile order), so contexts are split wherever the shares
 * end and the combine kernel merges those.  partition_blocks does not apply to
 * it (pa_decode_partition_blocks reports max_blocks_per_seq); its workspace,
 * needed whenever more than one CTA runs, grows with the SM count (two slots
 * of partials per CTA) and the number of (sequence, head group) pairs.
 * Cites: no counterpart on the pages (a choice among this library's kernels);
 * each computes the decode of "vllmini", "The CUDA Block Kernel". */
enum {
    PA_DECODE_AUTO = 0,
    PA_DECODE_CUDA_CORES = 1,
    PA_DECODE_TENSOR_CORES = 2,
    PA_DECODE_TCGEN05 = 3
};
PA_API int pa_pool_set_decode_kernel(pa_pool* pool, int kind);

/* The decode kernel that a decode call with `num_heads` query heads runs on
 * this pool under its current choice: PA_DECODE_CUDA_CORES,
 * PA_DECODE_TENSOR_CORES or PA_DECODE_TCGEN05 in *kind.  PA_ERR_UNSUPPORTED
 * (with the reason) when no kernel serves the shape or the forced one cannot;
 * PA_ERR_INVALID_ARG when num_heads is not a positive multiple of the pool's
 * KV heads.  Host only: touches no device.
 * Cites: no counterpart on the pages (as pa_pool_set_decode_kernel). */
PA_API int pa_decode_kernel_choice(const pa_pool* pool, int num_heads, int* kind);

/* Bytes of one physical block: 2 * num_layers * num_kv_heads * block_size *
 * head_dim * element size (K and V of every layer and KV head).
 * Cites: mini-infer, "Memory Waste Analysis" (its block-size formula, which
 * omits the K/V factor and the element size) and "Python Implementation:
 * Physical Block Pool" (the tensor those factors come from). */
PA_API int pa_pool_block_bytes(const pa_pool* pool, size_t* bytes);

/* Replace the free stack by `order` (a permutation of 0..num_blocks-1, n ==
 * num_blocks); allowed only while every block is free.  The LAST entry is
 * handed out first.
 * Cites: mini-infer, "Python Implementation: Physical Block Pool" (the free
 * list that allocation pops from the end); the page always starts it as
 * range(num_blocks), seeding another order has no counterpart there. */
PA_API int pa_pool_seed_free_stack(pa_pool* pool, const int* order, int n);

/* Pop one block id from the free stack.  PA_ERR_NO_FREE_BLOCKS when empty
 * ("Out of KV-Cache Physical Blocks").
 * Cites: mini-infer, "Python Implementation: Physical Block Pool"
 * (allocate_block: pop from the end of the free list, MemoryError when empty);
 * "kv-cache" skill, section 2 (a block is taken as a sequence grows). */
PA_API int pa_alloc_block(pa_pool* pool, int* block_id);

/* Push `block_id` back; it becomes the next id handed out.  Ids outside the
 * pool are PA_ERR_INVALID_ARG, ids not currently allocated PA_ERR_DOUBLE_FREE.
 * Cites: mini-infer, "Python Implementation: Physical Block Pool" (free_block
 * appends the id to the free list); the page checks nothing, rejecting foreign
 * and double frees is this library's reading. */
PA_API int pa_free_block(pa_pool* pool, int block_id);

/* Number of ids on the free stack.
 * Cites: mini-infer, "Python Implementation: Physical Block Pool" (the length of
 * the free list). */
PA_API int pa_num_free(const pa_pool* pool, int* n);

/* ----------------------------------------------------------------------------
 * The free stack on the device ("kv-cache" skill, section 3.1 "Cache Block
 * Pool": one allocator hands out blocks as generation proceeds; mini-infer
 * BlockPool semantics).  A caller-owned int32 array of num_blocks + 1 entries
 * holds [height, id_0 (bottom), ..., id_{height-1} (top)].  While the stack is
 * on the device the host calls pa_alloc_block / pa_free_block /
 * pa_pool_seed_free_stack are refused.
 * ------------------------------------------------------------------------- */

/* Bytes of the device stack array: (num_blocks + 1) * 4.
 * Cites: as the section above. */
PA_API int pa_device_stack_bytes(const pa_pool* pool, size_t* bytes);

/* Copy the host free stack into dev_stack (waits for `stream`) and hand the
 * stack to the device.
 * Cites: as the section above (the same free list, moved to the device). */
PA_API int pa_device_stack_upload(pa_pool* pool, void* dev_stack, pa_stream_t stream);

/* Wait for `stream`, copy the device stack back into the host allocator
 * (validating every id) and return the stack to the host.
 * Cites: as the section above. */
PA_API int pa_device_stack_download(pa_pool* pool, const void* dev_stack, pa_stream_t stream);

/*
 * For every sequence b, in increasing b, whose next token starts a new block
 * (positions[b] % block_size == 0), pop the top id of the device stack and
 * store it at block_tables[b][positions[b] / block_size] -- the ids repeated
 * pa_alloc_block calls would hand out in that order.  When the stack runs dry
 * the remaining such entries are set to -1 and PA_STATUS_NO_FREE_BLOCKS is
 * raised.  One kernel launch; no host round trip.
 * Cites: mini-infer, "Python Implementation: Physical Block Pool"
 * (allocate_block, once per sequence that needs a block); "kv-cache" skill,
 * section 2 (a new block when a sequence crosses a block boundary).
 */
PA_API int pa_device_alloc_blocks(pa_pool* pool, void* dev_stack, int* block_tables,
                                  int max_blocks_per_seq, const int* positions, int batch,
                                  pa_stream_t stream);

/*
 * pa_device_alloc_blocks, and in the same launch next_lens[b] = positions[b] + 1
 * for every b: the context length once the token at positions[b] is appended,
 * i.e. the context_lens of the step's pa_write_kv_and_decode and the positions
 * of the next step.  A decode loop alternates two length arrays (this step's
 * next_lens is the next step's positions) and needs no kernel of its own to
 * advance them.  next_lens: device int32 [batch], 4-byte aligned, must not
 * overlap positions (PA_ERR_INVALID_ARG).
 * Cites: as pa_device_alloc_blocks; "kv-cache" skill, section 2 (each
 * generated token grows its sequence's context by one).
 */
PA_API int pa_device_alloc_blocks_step(pa_pool* pool, void* dev_stack, int* block_tables,
                                       int max_blocks_per_seq, const int* positions,
                                       int* next_lens, int batch, pa_stream_t stream);

/*
 * For every sequence b with finished[b] != 0, in increasing b, push the ids of
 * its ceil(context_lens[b] / block_size) blocks in table order (as repeated
 * pa_free_block calls) and set those table entries to -1.  Out-of-range ids are
 * skipped and flagged (PA_STATUS_BAD_BLOCK_ID); pushing an id that is already
 * free is not detected on the device (pa_device_stack_download rejects the
 * resulting stack).
 * Cites: mini-infer, "Python Implementation: Physical Block Pool" (free_block,
 * once per block of a finished sequence).
 */
PA_API int pa_device_free_blocks(pa_pool* pool, void* dev_stack, int* block_tables,
                                 int max_blocks_per_seq, const int* context_lens,
                                 const uint8_t* finished, int batch, pa_stream_t stream);

/* ----------------------------------------------------------------------------
 * KV append (reshape-and-cache).
 * ------------------------------------------------------------------------- */

/*
 * For every sequence b and KV head h, copy k[b][h][:] to pool[bt[b][p/B]][0]
 * [layer][h][p % B][:] and v[b][h][:] to the same slot with K/V index 1, where
 * p = positions[b] and B = block_size.  A bit copy: the stored bytes equal the
 * input bytes.
 *   k, v          device, [batch, num_kv_heads, head_dim] of the pool dtype,
 *                 16-byte aligned.
 *   block_tables  device int32 [batch, max_blocks_per_seq], row-major.
 *   positions     device int32 [batch]; p/B < max_blocks_per_seq required.
 * Rows whose position or block id is out of range are skipped and flagged in
 * the status word (PA_STATUS_BAD_LENGTH / PA_STATUS_BAD_BLOCK_ID).
 * Cites: mini-infer, "The Solution" (logical block p / B of a sequence is the
 * physical block its table names; the token sits at offset p % B) and "Python
 * Implementation: Physical Block Pool" (the K/V, layer and KV-head axes of the
 * pool tensor); "kv-cache" skill, section 2 "PagedAttention Architecture"
 * (blocks filled one token at a time as generation proceeds).
 */
PA_API int pa_write_kv(pa_pool* pool, int layer, const void* k, const void* v,
                const int* block_tables, int max_blocks_per_seq, const int* positions,
                int batch, pa_stream_t stream);

/* ----------------------------------------------------------------------------
 * Decode attention.
 * ------------------------------------------------------------------------- */

/*
 * out[b][h][:] = softmax_t(scale * q[b][h] . K_t) V_t over the n = context_lens[b]
 * cached tokens t of sequence b, where K_t / V_t are the rows of KV head
 * h / (num_heads / num_kv_heads) at slot (block_tables[b][t / B], t % B) of
 * `layer`.  n = 0 yields a zero vector.  Scores and sums are fp32.
 *   out           device fp32 [batch, num_heads, head_dim], 16-byte aligned.
 *   q             device [batch, num_heads, head_dim] of the pool dtype, 16-byte aligned.
 *   block_tables  device int32 [batch, max_blocks_per_seq]; entries past
 *                 ceil(n / B) do not affect the result (a kernel may load
 *                 them with the rest of its row; pad with -1).
 *   context_lens  device int32 [batch], 0 <= n <= max_blocks_per_seq * B.
 *   A table entry outside [0, num_blocks) among the first ceil(n / B) sets
 *   PA_STATUS_BAD_BLOCK_ID and that block's tokens get no weight (no valid
 *   token left: a zero vector); a length outside the range above sets
 *   PA_STATUS_BAD_LENGTH and the sequence is decoded as n = 0.  Neither is an
 *   error return: the kernels run before the lengths and tables are read.
 *   block_size, num_kv_heads, head_dim must equal the pool's; num_heads must be
 *   a multiple of num_kv_heads.
 *   workspace     device scratch of at least pa_decode_workspace_size() bytes,
 *                 256-byte aligned (may be NULL when that size is 0).  Contents
 *                 need no initialisation; concurrent calls need separate workspaces.
 * The context of each (sequence, KV head) is split into partitions of a
 * heuristically chosen number of blocks; with more than one partition a second
 * kernel merges the per-partition results (log-sum-exp combine).  The tcgen05
 * kernel instead cuts the batch's 128-token tiles into equal shares per SM
 * (see PA_DECODE_TCGEN05) and a combine merges the cut contexts.
 * Cites: "vllmini", "The CUDA Block Kernel" (the argument list out, q,
 * caches, block_tables, context_lens, block_size, num_heads, head_size; every
 * token resolved through the block table on the fly) and "PagedAttention
 * Metaphor" (logical block i of a sequence in physical block block_table[i]);
 * "vllmini", introduction (each decode step reads the K/V of all past tokens).
 * The scale argument, the query-to-KV-head grouping and the n = 0 result are
 * readings: the pages state none of them.
 */
PA_API int pa_decode_attention(float* out, const void* q, const pa_pool* pool, int layer,
                        const int* block_tables, int max_blocks_per_seq,
                        const int* context_lens, int batch, int block_size, int num_heads,
                        int num_kv_heads, int head_dim, float scale, void* workspace,
                        size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_attention with an explicit partition size: `partition_blocks`
 * physical blocks per partition (>= 1), or 0 for the heuristic choice.
 * A partition covering the whole table (partition_blocks >= max_blocks_per_seq)
 * runs a single kernel and needs no workspace.  The tcgen05 kernel ignores
 * partition_blocks (its split depends on the lengths only).
 * Cites: as pa_decode_attention; splitting a context into partitions has no
 * counterpart on the pages (it is this library's way to spread a few long
 * contexts over the whole GPU).
 */
PA_API int pa_decode_attention_partitioned(float* out, const void* q, const pa_pool* pool, int layer,
                                    const int* block_tables, int max_blocks_per_seq,
                                    const int* context_lens, int batch, int block_size,
                                    int num_heads, int num_kv_heads, int head_dim, float scale,
                                    int partition_blocks, void* workspace,
                                    size_t workspace_bytes, pa_stream_t stream);

/*
 * KV append fused into decode: one launch that first stores k[b][h] / v[b][h]
 * at slot (block_tables[b][p / B], p % B), p = positions[b] (exactly as
 * pa_write_kv), then computes pa_decode_attention_partitioned over
 * context_lens[b] tokens, which normally include the new one (n = p + 1).
 * Within a sequence the store is ordered before the decode reads it.  The
 * block receiving the new token must not be read by another sequence of the
 * same call.  Bad positions / ids are flagged in the status word as for
 * pa_write_kv.  Arguments as for pa_write_kv and pa_decode_attention_partitioned.
 * Cites: as pa_write_kv and pa_decode_attention (the pages run the two as
 * separate steps; doing them in one launch is this library's).
 */
PA_API int pa_write_kv_and_decode(float* out, const void* q, pa_pool* pool, int layer,
                                  const void* k, const void* v, const int* positions,
                                  const int* block_tables, int max_blocks_per_seq,
                                  const int* context_lens, int batch, int block_size,
                                  int num_heads, int num_kv_heads, int head_dim, float scale,
                                  int partition_blocks, void* workspace, size_t workspace_bytes,
                                  pa_stream_t stream);

/* The partition size (in blocks) that pa_decode_attention picks for these
 * sizes on the current device.  Queries the device's SM count.  On the
 * mma.sync kernel it is the whole table (max_blocks_per_seq: no workspace, no
 * combine) when the call's (sequence, KV head, head chunk) CTAs number between
 * a third of the SMs and all of them and the table holds at most 64 blocks
 * (head_dim 64) or 48 (head_dim 128): each context then runs in one wide CTA
 * of 16 (8) warps.  A partition covering the table that is passed explicitly
 * runs the same way under the same conditions.
 * Cites: no counterpart on the pages (see pa_decode_attention_partitioned). */
PA_API int pa_decode_partition_blocks(const pa_pool* pool, int batch, int num_heads,
                               int max_blocks_per_seq, int* partition_blocks);

/* Workspace bytes needed by pa_decode_attention_partitioned with the same
 * arguments (partition_blocks = 0: the heuristic choice, which queries the
 * current device; the tcgen05 kernel always queries it).  0 when a single
 * partition covers the table (tcgen05 kernel: when a single CTA runs).
 * Cites: no counterpart on the pages (the scratch of the split contexts). */
PA_API int pa_decode_workspace_size(const pa_pool* pool, int batch, int num_heads,
                             int max_blocks_per_seq, int partition_blocks, size_t* bytes);

/*
 * Decode attention for callers that cannot allocate device memory while they
 * run -- e.g. an operator called from another engine's execution step, where
 * that engine owns all device memory and forbids cudaMalloc (which can block on
 * the device and fails once the memory has been reserved).  The source pages
 * have no counterpart to this call; it exists for such callers only.
 *
 * Same arguments and results as pa_decode_attention_partitioned, without the
 * workspace: the split-K partials go to a fixed device array of
 * PA_NOALLOC_SCRATCH_BYTES compiled into the library, which every device that
 * loads the library's kernels holds until the process exits.  The call makes
 * no cudaMalloc/cudaFree and no allocating library call.
 *  - A call that needs more scratch than PA_NOALLOC_SCRATCH_BYTES (see
 *    pa_decode_workspace_size) fails with PA_ERR_WORKSPACE before any launch.
 *    On the mma.sync and CUDA-core kernels a larger partition_blocks needs
 *    less; the tcgen05 kernel ignores partition_blocks (its scratch follows the
 *    SM count and the number of (sequence, head group) pairs), so such a call
 *    needs pa_decode_attention with a caller-provided workspace instead.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it needs clearing: every partial a call reads was written
 *    earlier in the same call.  Calls that overlap on the GPU (other streams,
 *    other host threads) race on it: serialise them.
 */
#define PA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* Cites: no counterpart on the pages (see above). */
PA_API int pa_decode_attention_noalloc(float* out, const void* q, const pa_pool* pool, int layer,
                                const int* block_tables, int max_blocks_per_seq,
                                const int* context_lens, int batch, int block_size,
                                int num_heads, int num_kv_heads, int head_dim, float scale,
                                int partition_blocks, pa_stream_t stream);

/* ----------------------------------------------------------------------------
 * Batched gather (mini-infer "Zero-Copy Batched Attention Gather").
 * ------------------------------------------------------------------------- */

/*
 * Copy the first context_lens[b] K and V rows of every sequence of `layer`
 * into contiguous k_out / v_out [batch, max_len, num_kv_heads, head_dim] (pool
 * dtype) and set mask[b][t] = 1 for t < context_lens[b], else 0 (rows past the
 * length are zero-filled).  k_out, v_out 16-byte aligned; mask uint8
 * [batch, max_len].  Lengths above max_len or above the table are flagged
 * (PA_STATUS_BAD_LENGTH) and treated as 0.
 * Cites: mini-infer, "Zero-Copy Batched Attention Gather" (all active
 * sequences' past K/V of one layer into one [B, T, H, D] tensor plus a mask;
 * the listing stops after the call, so T = max_len, mask 1 = valid and the
 * zero rows past each length are readings).
 */
PA_API int pa_gather_kv(void* k_out, void* v_out, uint8_t* mask, const pa_pool* pool, int layer,
                 const int* block_tables, int max_blocks_per_seq, const int* context_lens,
                 int batch, int max_len, pa_stream_t stream);

/* ----------------------------------------------------------------------------
 * Device status.
 * ------------------------------------------------------------------------- */

/* Failure-detection self-test: launches one warp that waits on a shared-memory
 * barrier no copy or thread ever completes.  The bounded wait used by every
 * kernel of this library gives up (here after 20 ms), PA_STATUS_TIMEOUT is
 * raised in the status word and the kernel returns; the context stays usable.
 * No fault, trap or hang is involved.
 * Cites: no counterpart on the pages (this library's failure detection). */
PA_API int pa_selftest_wait_timeout(pa_stream_t stream);

/* Wait for `stream`, return the current device's status bits (PA_STATUS_*)
 * accumulated since the last call, and clear them.  Blocking.
 * The word is one per device, not per pool: every kernel of the library, of
 * any pool on that device, sets its bits in the same word, so the call takes
 * no pool argument.
 * Cites: no counterpart on the pages beyond the allocator's exhaustion error
 * (mini-infer, "Python Implementation: Physical Block Pool"); the bad-id and
 * bad-length bits report table entries and lengths the pages assume valid. */
PA_API int pa_get_status(unsigned int* status, pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
