// pa_decode_mma.cuh -- paged decode attention for bf16 pools on the tensor
// cores (mma.sync m16n8k16), K/V staged by 5-D tensor-map TMA with 128-byte
// swizzle.
//
// Computes the same thing as pa_decode_kernel (see pa_decode.cuh): for sequence
// b and query head h, out = softmax_t(scale * q . K_t) V_t over the tokens
// reached through the block table ("vllmini", "PagedAttention Metaphor" / "The
// CUDA Block Kernel"; mini-infer, "The Solution").
//
// Same work split as pa_decode_kernel: one CTA per (sequence, KV head,
// partition), each warp streams every NW-th block of the partition through its
// own S-stage pipeline.  What differs is the inner product machinery, chosen
// to cut the instruction count per token (the CUDA-core kernel is issue-bound):
//  * a stage holds 16 rows of K and 16 rows of V, each as D/64 TMA boxes of
//    16 x 64 bf16 with SWIZZLE_128B, so ldmatrix reads are bank-conflict free;
//  * S = K Q^T on mma.sync: M = 16 tokens, N = 8 query heads of the group per
//    tile (one tile for G <= 8, two for G <= 16; heads >= G are zero),
//    K = head_dim; the scale is applied to S in fp32;
//  * online softmax on the S fragments (a lane holds 2 tokens x 2 heads);
//  * P is split into bf16 hi + lo parts (|P - hi - lo| <= 2^-16 P), transposed
//    in registers with movmatrix, and O^T = V^T P accumulates on mma.sync with
//    M = 16 head-dim rows, N = 8 heads, K = 16 tokens (V^T via ldmatrix.trans).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_fused_append.cuh"
#include "pa_internal.h"

namespace pa {

template <int D_, int B_, int G_, int NW_, int S_>
struct MmaCfg {
    static constexpr int D = D_, B = B_, G = G_, NW = NW_, S = S_;
    static constexpr int R = 16;                   // rows per stage
    static constexpr int SPB = B / R;              // stages per block
    static constexpr int NBOX = D / 64;            // 64-element (128-byte) boxes per row
    static constexpr int BOX_BYTES = R * 128;      // one swizzled 16 x 128 B box
    static constexpr int TILE_BYTES = NBOX * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile, then V tile
    static constexpr int KS = D / 16;              // k-steps of S = K Q^T
    static constexpr int MT = D / 16;              // m-tiles of O^T = V^T P
    static constexpr int NT = (G + 7) / 8;         // 8-head mma tiles of the group
    // A warp's O in the merge area: one row of D floats per head, rows D + 4
    // apart, so that the four lanes of an mma group (heads 2cq, D columns
    // apart) write to different banks.
    static constexpr int ACC_LD = D + 4;
    static constexpr int WARP_STAGE_BYTES = S * STAGE_BYTES;
    static constexpr int META_BYTES = 64;          // per warp: nvalid[S], mbarriers[S]
    static constexpr int SMEM_BYTES = NW * WARP_STAGE_BYTES + NW * META_BYTES + 1024;

    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(B % R == 0, "block size must be a multiple of 16");
    static_assert(G >= 1 && G <= 16, "GQA group of at most 16 query heads");
    static_assert(S * 12 <= META_BYTES, "meta");
    static_assert((2 * G + G * ACC_LD) * 4 <= WARP_STAGE_BYTES, "merge area must fit in the stages");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// Byte offset of (row t, 16-byte chunk j) inside a K or V tile stored as D/64
// boxes of 16 rows x 128 bytes with the 128-byte swizzle (chunk j of row t sits
// at chunk j ^ (t % 8) of its 128-byte row).
__device__ __forceinline__ uint32_t swz_offset(int t, int j) {
    return (uint32_t)((j >> 3) * (16 * 128) + t * 128 + (((j & 7) ^ (t & 7)) << 4));
}

template <int D, int B, int G, int NW, int S>
__global__ void __launch_bounds__(NW * 32)
    pa_decode_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
    pdl_trigger();
    using C = MmaCfg<D, B, G, NW, S>;
    extern __shared__ unsigned char smem_raw[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;  // mma group id
    const int cq = lane & 3;  // thread within the group

    // CTA order: partition index slowest, so the end of the grid holds only the
    // last (partial) partitions of the longest sequences and empty slots --
    // a lighter tail than ending on full partitions (1-1.5% on GB300).
    // A group larger than G is split into head chunks of G (fastest index):
    // sibling chunks of one (sequence, KV head, partition) run side by side and
    // share each K/V tile through L2.
    int idx = blockIdx.x;
    const int hc = idx % p.nchunks;
    idx /= p.nchunks;
    const int nbh = p.batch * p.Hkv;
    const int c = idx / nbh;
    idx %= nbh;
    const int kvh = idx % p.Hkv;
    const int b = idx / p.Hkv;
    const int hbase = kvh * p.gsize + hc * G;  // first query head of this CTA in the sequence
    // this chunk's heads: G, fewer in the last chunk of a group that is not a
    // multiple of G (heads past them are masked like those past a small group)
    const int gact = min(G, p.gsize - hc * G);

    // 1024-byte aligned stage area (swizzle atoms), then per-warp metadata.
    // The barriers and the tensor maps read nothing the previous kernel
    // writes: they are set up before the programmatic-launch wait, while that
    // kernel drains.
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    unsigned char* smem = smem_raw + (base_addr - raw_addr);
    unsigned char* wbase = smem + warp * C::WARP_STAGE_BYTES;
    const uint32_t stage0 = base_addr + warp * C::WARP_STAGE_BYTES;
    unsigned char* meta = smem + NW * C::WARP_STAGE_BYTES + warp * C::META_BYTES;
    int* s_nvalid = reinterpret_cast<int*>(meta);
    const uint32_t bars = smem_addr(meta + 16);

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
        if (warp == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
    }
    __syncwarp();
    pdl_wait();

    // The first 32 block ids of this warp's share of the partition depend only
    // on the partition index (the table row holds maxb entries): their load
    // overlaps the length's instead of waiting for it.
    const int* bt_row = p.bt + (long long)b * p.maxb;
    const int k_first = c * p.PB + warp + lane * NW;
    const int id_first = k_first < p.maxb ? ld_dep(bt_row + k_first) : -1;
    // The fused append's position and new rows do not depend on the length
    // either: all four loads are in flight together.
    const bool fused = p.new_k != nullptr;
    const int pos = fused ? ld_dep(p.positions + b) : 0;
    const uint4 new_row = fused ? load_new_row<D * 2>(p, b, kvh, lane) : make_uint4(0u, 0u, 0u, 0u);

    int n = ld_dep(p.lens + b);
    if (n < 0 || n > p.maxb * B) {
        if (c == 0 && kvh == 0 && hc == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusBadLength);
        n = 0;
    }
    const int nblk = (n + B - 1) / B;
    const int nparts = nblk > 0 ? (nblk + p.PB - 1) / p.PB : 1;
    if (c >= nparts) return;
    const int pb0 = c * p.PB;
    const int pb1 = min(nblk, pb0 + p.PB);

    const int span = pb1 - pb0;
    const int nk = span > warp ? (span - warp + NW - 1) / NW : 0;
    int U = 0;
    if (nk > 0) {
        const int jb_last = pb0 + warp + (nk - 1) * NW;
        const int rows_last = min(B, n - jb_last * B);
        U = (nk - 1) * C::SPB + (rows_last + C::R - 1) / C::R;
    }


    // Fused append.  The partition that holds the new row's block (partition
    // 0 when the position lies past the context) stores it; every head chunk
    // of that partition stores the (identical) row itself.  The store is made
    // by the warp that copies that block, just before the copy, so its latency
    // hides behind the warp's earlier blocks and no other warp waits.
    int app_k = -1, app_blk = -1;
    if (fused) {
        if (pos < 0 || pos / B >= p.maxb) {
            if (c == 0 && kvh == 0 && hc == 0 && threadIdx.x == 0)
                atomicOr(p.status, kStatusBadLength);
        } else if (c == (pos < n ? (pos / B) / p.PB : 0)) {
            const int jb = pos / B;
            if (pos < n) {
                if (warp == (jb - pb0) % NW) {
                    // the block is this warp's k-th: among its prefetched ids
                    // when k < 32
                    const int k = (jb - pb0) / NW;
                    int blk = __shfl_sync(kFullMask, id_first, k & 31);
                    if (k >= 32) blk = ld_dep(bt_row + jb);
                    if (blk < 0 || blk >= p.num_blocks) {
                        if (lane == 0) atomicOr(p.status, kStatusBadBlock);
                    } else {
                        app_k = k;
                        app_blk = blk;
                    }
                }
            } else if (warp == 0) {
                // past the decoded context: no copy of this call needs the row
                const int blk = ld_dep(bt_row + jb);
                if (blk < 0 || blk >= p.num_blocks) {
                    if (lane == 0) atomicOr(p.status, kStatusBadBlock);
                } else {
                    store_new_row<D * 2, 2>(p, kvh, blk, pos, B, lane, new_row);
                }
            }
        }
    }

    const uint64_t policy = l2_policy_evict_first();
    int kbase = 0;
    int myid = (lane < nk) ? id_first : -1;

    auto issue = [&](int u) {
        const int k = u / C::SPB;
        const int sub = u % C::SPB;
        if (k >= kbase + 32) {
            kbase += 32;
            const int kk = kbase + lane;
            myid = (kk < nk) ? ld_dep(bt_row + pb0 + warp + kk * NW) : -1;
        }
        const int blk = __shfl_sync(kFullMask, myid, k - kbase);
        const int jb = pb0 + warp + k * NW;
        const int row0 = sub * C::R;
        const int rows = min(C::R, n - (jb * B + row0));
        const int stage = u % S;
        if (k == app_k && sub == 0) store_new_row<D * 2, 2>(p, kvh, app_blk, pos, B, lane, new_row);
        if (lane == 0) {
            const uint32_t bar = bars + 8 * stage;
            if (blk >= 0 && blk < p.num_blocks) {
                s_nvalid[stage] = rows;
                mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
                // outer coordinates in the tensor map's dimension order
                const int o2 = p.tma_slot_blk == 2 ? blk : (p.tma_slot_layer == 2 ? p.layer : kvh);
                const int o3 = p.tma_slot_blk == 3 ? blk : (p.tma_slot_layer == 3 ? p.layer : kvh);
                const int o4 = p.tma_slot_blk == 4 ? blk : (p.tma_slot_layer == 4 ? p.layer : kvh);
                const uint32_t dst = stage0 + stage * C::STAGE_BYTES;
#pragma unroll
                for (int bx = 0; bx < C::NBOX; ++bx) {
                    tma_load_5d(dst + bx * C::BOX_BYTES, &tmk, bar, bx * 64, row0, o2, o3, o4,
                                policy);
                    tma_load_5d(dst + C::TILE_BYTES + bx * C::BOX_BYTES, &tmv, bar, bx * 64, row0,
                                o2, o3, o4, policy);
                }
            } else {
                s_nvalid[stage] = 0;
                atomicOr(p.status, kStatusBadBlock);
                mbar_arrive(bar);
            }
        }
    };

    // q of the group as mma B fragments, one set per 8-head tile nt:
    // b0 = q[8nt+g][16ks+2cq..+1], b1 = q[8nt+g][16ks+8+2cq..+1] (zero past the group)
    uint32_t qb[C::NT][C::KS][2];
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
        const int hq = 8 * nt + g;
        const unsigned short* qrow =
            reinterpret_cast<const unsigned short*>(p.q) + ((long long)b * p.H + hbase + hq) * D;
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
            if (hq < gact) {
                qb[nt][ks][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * cq);
                qb[nt][ks][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * cq);
            } else {
                qb[nt][ks][0] = 0u;
                qb[nt][ks][1] = 0u;
            }
        }
    }

    float o[C::NT][C::MT][4];
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[nt][mt][i] = 0.f;
    // running max / sum of heads 8nt+2cq and 8nt+2cq+1 (the sum is this lane's share)
    float m0[C::NT], m1[C::NT], l0[C::NT], l1[C::NT];
    bool h0_ok[C::NT], h1_ok[C::NT];
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
        m0[nt] = -INFINITY;
        m1[nt] = -INFINITY;
        l0[nt] = 0.f;
        l1[nt] = 0.f;
        h0_ok[nt] = 8 * nt + 2 * cq < gact;
        h1_ok[nt] = 8 * nt + 2 * cq + 1 < gact;
    }

    int u_issue = 0;
    const int npro = U < S ? U : S;
    for (; u_issue < npro; ++u_issue) issue(u_issue);

    int u = 0;
    bool timed_out = false;
    for (; u < U; ++u) {
        const int stage = u % S;
        const bool ok = mbar_wait_bounded(bars + 8 * stage, (u / S) & 1);
        if (__any_sync(kFullMask, !ok)) {
            timed_out = true;
            break;
        }
        const int rows = s_nvalid[stage];
        if (rows > 0) {
            const uint32_t ktile = stage0 + stage * C::STAGE_BYTES;
            const uint32_t vtile = ktile + C::TILE_BYTES;
            if (rows < C::R) {
                // rows past the context are zeroed so that 0 * (stale value) stays 0
                unsigned char* vt = wbase + stage * C::STAGE_BYTES + C::TILE_BYTES;
                for (int i = lane; i < (C::R - rows) * 8 * C::NBOX; i += 32) {
                    const int t = rows + i / (8 * C::NBOX);
                    const int j = i % (8 * C::NBOX);
                    *reinterpret_cast<uint4*>(vt + swz_offset(t, j)) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }

            // ---- S = K Q^T (16 tokens x 8 heads per tile) ----
            float sacc[C::NT][4];
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.f;
            {
                const int mtx = lane >> 3;
                const int t = (lane & 7) + 8 * (mtx & 1);
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(ktile + swz_offset(t, 2 * ks + (mtx >> 1)), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < C::NT; ++nt)
                        mma_bf16_16816(sacc[nt], a0, a1, a2, a3, qb[nt][ks][0], qb[nt][ks][1]);
                }
            }
            // ---- online softmax: lane has tokens g, g+8 x heads 8nt+2cq, 8nt+2cq+1 ----
            const bool t0_ok = g < rows;
            const bool t1_ok = g + 8 < rows;
            uint32_t bh0[C::NT], bh1[C::NT], bl0[C::NT], bl1[C::NT];
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) {
                const float s00 = (t0_ok && h0_ok[nt]) ? sacc[nt][0] * p.qscale : -INFINITY;
                const float s01 = (t0_ok && h1_ok[nt]) ? sacc[nt][1] * p.qscale : -INFINITY;
                const float s10 = (t1_ok && h0_ok[nt]) ? sacc[nt][2] * p.qscale : -INFINITY;
                const float s11 = (t1_ok && h1_ok[nt]) ? sacc[nt][3] * p.qscale : -INFINITY;
                float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, off));
                }
                const float mn0 = fmaxf(m0[nt], mx0), mn1 = fmaxf(m1[nt], mx1);
                // (heads past the group keep O = 0, so their factor is left at 1)
                const float a0s =
                    !h0_ok[nt] ? 1.f : (m0[nt] == -INFINITY ? 0.f : exp2f(m0[nt] - mn0));
                const float a1s =
                    !h1_ok[nt] ? 1.f : (m1[nt] == -INFINITY ? 0.f : exp2f(m1[nt] - mn1));
                const float p00 = (s00 == -INFINITY) ? 0.f : exp2f(s00 - mn0);
                const float p01 = (s01 == -INFINITY) ? 0.f : exp2f(s01 - mn1);
                const float p10 = (s10 == -INFINITY) ? 0.f : exp2f(s10 - mn0);
                const float p11 = (s11 == -INFINITY) ? 0.f : exp2f(s11 - mn1);
                l0[nt] = l0[nt] * a0s + p00 + p10;
                l1[nt] = l1[nt] * a1s + p01 + p11;
                m0[nt] = mn0;
                m1[nt] = mn1;
                if (a0s != 1.f || a1s != 1.f) {
#pragma unroll
                    for (int mt = 0; mt < C::MT; ++mt) {
                        o[nt][mt][0] *= a0s;
                        o[nt][mt][1] *= a1s;
                        o[nt][mt][2] *= a0s;
                        o[nt][mt][3] *= a1s;
                    }
                }
                // ---- P -> bf16 hi + lo, transposed into mma B fragments ----
                const __nv_bfloat162 hi_t = __floats2bfloat162_rn(p00, p01);
                const __nv_bfloat162 hi_b = __floats2bfloat162_rn(p10, p11);
                const __nv_bfloat162 lo_t = __floats2bfloat162_rn(p00 - __low2float(hi_t),
                                                                  p01 - __high2float(hi_t));
                const __nv_bfloat162 lo_b = __floats2bfloat162_rn(p10 - __low2float(hi_b),
                                                                  p11 - __high2float(hi_b));
                bh0[nt] = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&hi_t));
                bh1[nt] = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&hi_b));
                bl0[nt] = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&lo_t));
                bl1[nt] = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&lo_b));
            }
            // ---- O^T += V^T P ----
            {
                const int mtx = lane >> 3;
                const int t = (lane & 7) + 8 * (mtx >> 1);
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    uint32_t v0, v1, v2, v3;
                    ldmatrix_x4_trans(vtile + swz_offset(t, 2 * mt + (mtx & 1)), v0, v1, v2, v3);
#pragma unroll
                    for (int nt = 0; nt < C::NT; ++nt) {
                        mma_bf16_16816(o[nt][mt], v0, v1, v2, v3, bh0[nt], bh1[nt]);
                        mma_bf16_16816(o[nt][mt], v0, v1, v2, v3, bl0[nt], bl1[nt]);
                    }
                }
            }
        }
        __syncwarp();
        if (u_issue < U) {
            fence_proxy_async_smem();
            issue(u_issue);
            ++u_issue;
        }
    }
    if (timed_out) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        for (int w = u; w < u_issue; ++w) (void)mbar_wait_bounded(bars + 8 * (w % S), (w / S) & 1);
    }

    // ---- warp totals: l over the 8 lanes sharing cq ----
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0[nt] += __shfl_xor_sync(kFullMask, l0[nt], off);
            l1[nt] += __shfl_xor_sync(kFullMask, l1[nt], off);
        }
    __syncwarp();
    float* w_m = reinterpret_cast<float*>(wbase);
    float* w_l = w_m + G;
    float* w_acc = w_l + G;  // [G][ACC_LD]
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
        const int h0 = 8 * nt + 2 * cq;
        if (g == 0) {
            if (h0_ok[nt]) {
                w_m[h0] = m0[nt];
                w_l[h0] = l0[nt];
            }
            if (h1_ok[nt]) {
                w_m[h0 + 1] = m1[nt];
                w_l[h0 + 1] = l1[nt];
            }
        }
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
            const int d = 16 * mt + g;
            if (h0_ok[nt]) {
                w_acc[h0 * C::ACC_LD + d] = o[nt][mt][0];
                w_acc[h0 * C::ACC_LD + d + 8] = o[nt][mt][2];
            }
            if (h1_ok[nt]) {
                w_acc[(h0 + 1) * C::ACC_LD + d] = o[nt][mt][1];
                w_acc[(h0 + 1) * C::ACC_LD + d + 8] = o[nt][mt][3];
            }
        }
    }
    __syncthreads();

    // ---- merge the NW warps (log-sum-exp) and write ----
    const long long head0 = (long long)b * p.H + hbase;
    for (int t = threadIdx.x; t < gact * D; t += NW * 32) {
        const int h = t / D;
        const int d = t % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            M = fmaxf(M, reinterpret_cast<const float*>(smem + w * C::WARP_STAGE_BYTES)[h]);
        float Lsum = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float* wm = reinterpret_cast<const float*>(smem + w * C::WARP_STAGE_BYTES);
            const float mw = wm[h];
            const float wt = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
            Lsum += wt * wm[G + h];
            O += wt * wm[2 * G + h * C::ACC_LD + d];
        }
        if (nparts == 1) {
            p.out[(head0 + h) * D + d] = Lsum > 0.f ? O / Lsum : 0.f;
        } else {
            const long long slot = (head0 + h) * p.Cmax + c;
            p.part_o[slot * D + d] = O;
            if (d == 0) {
                p.part_ml[slot * 2 + 0] = M;
                p.part_ml[slot * 2 + 1] = Lsum;
            }
        }
    }
}

// Host: sets the kernel's shared-memory limit once per device, then launches
// one CTA per (sequence, KV head, head chunk, partition) with programmatic
// serialisation.
template <int D, int B, int G, int NW, int S>
cudaError_t launch_mma_inst(const DecodeParams& p, const CUtensorMap* tm, cudaStream_t stream) {
    using Cfg = MmaCfg<D, B, G, NW, S>;
    auto kern = pa_decode_mma_kernel<D, B, G, NW, S>;
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
    const long long grid = (long long)p.batch * p.Hkv * p.nchunks * p.Cmax;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(NW * 32), Cfg::SMEM_BYTES, stream, p,
                      tm[0], tm[1]);
}

// The instantiation for head chunk G (the chunk sizes decode_mma_chunk gives).
template <int D, int B, int NW, int S>
cudaError_t launch_mma_g(const DecodeParams& p, const CUtensorMap* tm, int G, cudaStream_t s) {
    switch (G) {
        case 1: return launch_mma_inst<D, B, 1, NW, S>(p, tm, s);
        case 2: return launch_mma_inst<D, B, 2, NW, S>(p, tm, s);
        case 3: return launch_mma_inst<D, B, 3, NW, S>(p, tm, s);
        case 4: return launch_mma_inst<D, B, 4, NW, S>(p, tm, s);
        case 5: return launch_mma_inst<D, B, 5, NW, S>(p, tm, s);
        case 6: return launch_mma_inst<D, B, 6, NW, S>(p, tm, s);
        case 7: return launch_mma_inst<D, B, 7, NW, S>(p, tm, s);
        case 8: return launch_mma_inst<D, B, 8, NW, S>(p, tm, s);
        case 16: return launch_mma_inst<D, B, 16, NW, S>(p, tm, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
