// bf16 tensor-core decode in wide CTAs: the same kernel as pa_decode_mma.cu
// with many warps and one partition per context.
//
// For a batch whose (sequence, KV head) CTAs fill a third to all of one wave
// and whose contexts are short (a few blocks per warp), one CTA per (sequence,
// KV head) holds the
// whole context: its warps take every NW-th block, all their copies are in
// flight at once, and the warps' running (max, sum, O) merge in shared memory,
// so the output is written directly and no combine launch or partial round
// trip follows.  A split of the same context over several narrower CTAs pays
// that second launch and the partials' write and read after the decode.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_decode_mma.cuh"

namespace pa {

namespace {

// Warps per wide CTA and stages per warp: three stages per warp, 192 KB of
// stages per CTA (one CTA per SM).  GB300, graph-timed fused calls (us; the
// split path with 8-block partitions in brackets): mini-infer shape (32
// sequences x 2 KV heads, head_dim 64, lengths up to 800) 16 x 3: 7.51, 24 x 2:
// 7.76, 12 x 4: 7.69 (7.88); 16 x 8 KV heads at head_dim 128, lengths up to
// 768: 8 x 3: 10.76, 12 x 2: 11.02, 6 x 4: 11.70 (13.88).
template <int D>
constexpr int kWideWarps = D == 128 ? 8 : 16;
constexpr int kWideStages = 3;
// The longest table a wide CTA takes (4 blocks per warp at head_dim 64, 6 at
// 128), and the fewest CTAs: with fewer than a third of the SMs busy, a split
// over more CTAs is faster despite its combine (GB300: 4 to 16 CTAs at head_dim
// 64 took 7.2-7.5 us wide against 6.5-7.0 split; 32 CTAs at head_dim 128 9.4
// against 8.3).
template <int D>
constexpr int kWideMaxBlocks = D == 128 ? 6 * kWideWarps<128> : 4 * kWideWarps<64>;

template <int D, int B, int G>
cudaError_t launch_wide(const DecodeParams& p, const CUtensorMap* tm, cudaStream_t s) {
    return launch_mma_inst<D, B, G, kWideWarps<D>, kWideStages>(p, tm, s);
}

template <int D, int B>
cudaError_t launch_wide_g(const DecodeParams& p, const CUtensorMap* tm, int G, cudaStream_t s) {
    switch (G) {
        case 1: return launch_wide<D, B, 1>(p, tm, s);
        case 2: return launch_wide<D, B, 2>(p, tm, s);
        case 3: return launch_wide<D, B, 3>(p, tm, s);
        case 4: return launch_wide<D, B, 4>(p, tm, s);
        case 5: return launch_wide<D, B, 5>(p, tm, s);
        case 6: return launch_wide<D, B, 6>(p, tm, s);
        case 7: return launch_wide<D, B, 7>(p, tm, s);
        case 8: return launch_wide<D, B, 8>(p, tm, s);
        case 16: return launch_wide<D, B, 16>(p, tm, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool decode_mma_wide_fits(int D, int G, int maxb, long long ctas, int num_sms) {
    if ((D != 64 && D != 128) || decode_mma_chunk(G) == 0) return false;
    const int max_blocks = D == 128 ? kWideMaxBlocks<128> : kWideMaxBlocks<64>;
    return ctas <= num_sms && ctas * 3 >= num_sms && maxb <= max_blocks;
}

cudaError_t launch_decode_mma_wide(const DecodeParams& p_in, const void* tmaps, int D, int B,
                                   int Gtot, cudaStream_t s) {
    const CUtensorMap* tm = static_cast<const CUtensorMap*>(tmaps);
    const int G = decode_mma_chunk(Gtot);
    if (G == 0) return cudaErrorNotSupported;
    if (p_in.Cmax != 1) return cudaErrorInvalidValue;  // one partition per context
    DecodeParams p = p_in;
    p.gsize = Gtot;
    p.nchunks = (Gtot + G - 1) / G;
    p.chunk = G;
    if (D == 64) {
        if (B == 16) return launch_wide_g<64, 16>(p, tm, G, s);
        if (B == 32) return launch_wide_g<64, 32>(p, tm, G, s);
    } else if (D == 128) {
        if (B == 16) return launch_wide_g<128, 16>(p, tm, G, s);
        if (B == 32) return launch_wide_g<128, 32>(p, tm, G, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace pa
