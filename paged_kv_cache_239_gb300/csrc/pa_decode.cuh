// pa_decode.cuh -- paged decode attention for sm_103a (CUDA cores, fp32 math).
//
// What is computed ("vllmini", "The CUDA Block Kernel"; "kv-cache" skill,
// section 2 "Block Tables"; mini-infer, "The Solution"): for sequence b and
// query head h, the n = context_lens[b] cached tokens are reached through the
// block table -- token t lives in physical block bt[b][t / B] at offset t % B
// of the pool (the fused [num_blocks, 2, L, Hkv, B, D] tensor, or any layout
// whose B x D tiles are contiguous, see PoolGeom) -- and
//     out[b][h] = softmax_t(scale * q[b][h] . K_t) V_t .
//
// Work decomposition (GB300 design, not taken from the pages):
//  * one CTA per (sequence, KV head, partition of PB blocks); all G = H / Hkv
//    query heads of the GQA group are served from each K/V row load.
//  * each warp of the CTA owns every NW-th block of the partition and runs its
//    own pipeline: lane 0 issues 1-D bulk (TMA) copies of R contiguous K rows and
//    R contiguous V rows of a physical block into one of S shared-memory
//    stages, completion is tracked by one mbarrier per stage, so the warp never
//    waits on other warps inside the main loop.
//  * a lane owns E = 8 consecutive-in-chunk head-dim elements of a row; LR = D/8
//    lanes cover one row and a warp covers RP = 32/LR rows per pass.  q lives in
//    registers, pre-multiplied by scale*log2(e).  Partial dot products are summed
//    across the LR lanes of a row by a butterfly reduce-scatter (about one
//    shuffle per score), then an online softmax in base 2 updates each warp's
//    running max / sum, and P.V accumulates in packed fp32x2 FMAs.
//  * at the end the NW warp states are merged through shared memory
//    (log-sum-exp).  A CTA whose partition is the whole context writes the
//    normalised output; otherwise it writes (O, max, sum) for the combine kernel.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_fused_append.cuh"
#include "pa_internal.h"

namespace pa {

__host__ __device__ constexpr int round_up_int(int x, int m) { return (x + m - 1) / m * m; }

template <typename T, int D_, int B_, int G_, int NW_, int S_>
struct DecodeCfg {
    static constexpr int D = D_, B = B_, G = G_, NW = NW_, S = S_;
    static constexpr int ELT = sizeof(T);
    static constexpr int VE = 16 / ELT;         // elements per 16-byte vector
    static constexpr int E = 8;                 // elements a lane owns per row
    static constexpr int NV = E / VE;           // 16-byte vectors per lane per row
    static constexpr int LR = D / E;            // lanes per row
    static constexpr int RP = 32 / LR;          // rows per warp pass
    static constexpr int R = B < 16 ? B : 16;   // rows per pipeline stage (sub-tile)
    static constexpr int SPB = B / R;           // sub-tiles per block
    static constexpr int NPASS = R / RP;        // passes per sub-tile
    static constexpr int P = NPASS * G;         // partial scores per lane per sub-tile
    static constexpr int CF = P >= LR ? P / LR : 1;  // full scores per lane after reduce
    static constexpr int ROW_BYTES = D * ELT;
    static constexpr int TILE_BYTES = R * ROW_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int OFF_SCORES = S * STAGE_BYTES;
    static constexpr int OFF_ALPHA = OFF_SCORES + R * G * 4;
    static constexpr int OFF_NVALID = OFF_ALPHA + round_up_int(G * 4, 16);
    static constexpr int OFF_BARS = round_up_int(OFF_NVALID + S * 4, 8);
    static constexpr int WARP_BYTES = round_up_int(OFF_BARS + S * 8, 128);
    static constexpr int SMEM_BYTES = NW * WARP_BYTES;
    static constexpr int PAIRS = R * G;                 // (row, head) scores per sub-tile
    static constexpr int PPL = (PAIRS + 31) / 32;       // scores per lane in the softmax step

    static_assert(D % 8 == 0 && (D / 8) <= 32 && (32 % (D / 8)) == 0, "head_dim");
    static_assert(E % VE == 0, "vector split");
    static_assert(R % RP == 0, "rows per stage must be a multiple of rows per pass");
    static_assert(B % R == 0, "block size");
    static_assert(32 % G == 0, "group size must divide 32");
    static_assert((P & (P - 1)) == 0, "partials must be a power of two");
    static_assert((2 * G + G * D) * 4 <= S * STAGE_BYTES, "merge area must fit in the stages");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// Loads the lane's E elements of one row (NV vectors at chunk j, j+LR, ...) as fp32 pairs.
template <typename T, int NV, int LR>
__device__ __forceinline__ void load_row_slice(const T* row, int j, float2 (&f)[4]);

template <>
__device__ __forceinline__ void load_row_slice<unsigned short, 1, 8>(const unsigned short* row,
                                                                     int j, float2 (&f)[4]) {
    const uint4 v = reinterpret_cast<const uint4*>(row)[j];
    f[0] = bf16x2_to_float2(v.x);
    f[1] = bf16x2_to_float2(v.y);
    f[2] = bf16x2_to_float2(v.z);
    f[3] = bf16x2_to_float2(v.w);
}
template <>
__device__ __forceinline__ void load_row_slice<unsigned short, 1, 16>(const unsigned short* row,
                                                                      int j, float2 (&f)[4]) {
    const uint4 v = reinterpret_cast<const uint4*>(row)[j];
    f[0] = bf16x2_to_float2(v.x);
    f[1] = bf16x2_to_float2(v.y);
    f[2] = bf16x2_to_float2(v.z);
    f[3] = bf16x2_to_float2(v.w);
}
template <int LR>
__device__ __forceinline__ void load_row_slice_f32(const float* row, int j, float2 (&f)[4]) {
    const float4 a = reinterpret_cast<const float4*>(row)[j];
    const float4 b = reinterpret_cast<const float4*>(row)[j + LR];
    f[0] = make_float2(a.x, a.y);
    f[1] = make_float2(a.z, a.w);
    f[2] = make_float2(b.x, b.y);
    f[3] = make_float2(b.z, b.w);
}
template <>
__device__ __forceinline__ void load_row_slice<float, 2, 8>(const float* row, int j,
                                                           float2 (&f)[4]) {
    load_row_slice_f32<8>(row, j, f);
}
template <>
__device__ __forceinline__ void load_row_slice<float, 2, 16>(const float* row, int j,
                                                            float2 (&f)[4]) {
    load_row_slice_f32<16>(row, j, f);
}

// Head-dim index of element 2*i2 of a lane's slice (lane position j in its row).
template <int VE, int LR>
__device__ __forceinline__ int slice_dim(int j, int i2) {
    const int e = 2 * i2;          // 0..7
    const int k = e / VE;          // which of the lane's vectors
    return (j + k * LR) * VE + (e % VE);
}

// Butterfly reduce-scatter of P partial sums across the LR lanes of a row
// group.  Afterwards lane j (position in its row group) holds in v[0..CF) the
// full sums of partials j*CF .. j*CF+CF-1 (P >= LR), or of partial j/(LR/P)
// (P < LR, duplicated over LR/P lanes).
template <int P, int LR>
__device__ __forceinline__ void reduce_scatter(float (&v)[P], int lane) {
#pragma unroll
    for (int step = 0; (LR >> (step + 1)) >= 1; ++step) {
        const int o = LR >> (step + 1);
        const int cnt = P >> step;  // live values before this step (when >= 2)
        if (cnt >= 2) {
            const int half = cnt / 2;
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float send = upper ? v[i] : v[i + half];
                const float keep = upper ? v[i + half] : v[i];
                v[i] = keep + __shfl_xor_sync(kFullMask, send, o);
            }
        } else {
            v[0] += __shfl_xor_sync(kFullMask, v[0], o);
        }
    }
}

template <typename T, int D, int B, int G, int NW, int S>
__global__ void __launch_bounds__(NW * 32) pa_decode_kernel(const DecodeParams p) {
    pdl_trigger();
    pdl_wait();
    using C = DecodeCfg<T, D, B, G, NW, S>;
    constexpr int E2 = C::E / 2;
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rg = lane / C::LR;  // row group
    const int jl = lane % C::LR;  // position within the row

    // ---- CTA coordinates: head chunk fastest, then KV head, then sequence,
    //      partition slowest.  A group that is no power of two up to 8 runs
    //      in chunks of G heads (the next power of two, or 8), the heads past
    //      the group masked: zero q, nothing written. ----
    int idx = blockIdx.x;
    const int hc = idx % p.nchunks;
    idx /= p.nchunks;
    const int nbh = p.batch * p.Hkv;
    const int c = idx / nbh;
    idx %= nbh;
    const int kvh = idx % p.Hkv;
    const int b = idx / p.Hkv;
    const int hbase = kvh * p.gsize + hc * G;  // first query head of this CTA in the sequence
    const int gact = min(G, p.gsize - hc * G);

    // The first 32 block ids of this warp's share of the partition depend only
    // on the partition index (the table row holds maxb entries): their load
    // overlaps the length's instead of waiting for it.
    const int* bt_row = p.bt + (long long)b * p.maxb;
    const int k_first = c * p.PB + warp + lane * NW;
    const int id_first = k_first < p.maxb ? ld_dep(bt_row + k_first) : -1;

    int n = ld_dep(p.lens + b);
    if (n < 0 || n > p.maxb * B) {
        if (c == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusBadLength);
        n = 0;
    }
    const int nblk = (n + B - 1) / B;
    const int nparts = nblk > 0 ? (nblk + p.PB - 1) / p.PB : 1;
    if (c >= nparts) return;  // uniform for the whole CTA
    const int pb0 = c * p.PB;
    const int pb1 = min(nblk, pb0 + p.PB);

    unsigned char* wbase = smem + warp * C::WARP_BYTES;
    float* s_sc = reinterpret_cast<float*>(wbase + C::OFF_SCORES);
    float* s_alpha = reinterpret_cast<float*>(wbase + C::OFF_ALPHA);
    int* s_nvalid = reinterpret_cast<int*>(wbase + C::OFF_NVALID);
    const uint32_t bars = smem_addr(wbase + C::OFF_BARS);
    const uint32_t stage0 = smem_addr(wbase);

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- this warp's blocks: pb0 + warp + k*NW, k < nk; its sub-tiles: U ----
    const int span = pb1 - pb0;
    const int nk = span > warp ? (span - warp + NW - 1) / NW : 0;
    int U = 0;
    if (nk > 0) {
        const int jb_last = pb0 + warp + (nk - 1) * NW;
        const int rows_last = min(B, n - jb_last * B);
        U = (nk - 1) * C::SPB + (rows_last + C::R - 1) / C::R;
    }

    // This CTA's tiles: element offset of (block 0, layer, kvh) from each base.
    const long long tile0 = p.tile_off + (long long)kvh * p.s_head;
    const T* kpool = reinterpret_cast<const T*>(p.k_base) + tile0;
    const T* vpool = reinterpret_cast<const T*>(p.v_base) + tile0;

    // ---- fused append: the partition that holds the new token's block
    //      (partition 0 when the position lies past the context) stores this
    //      KV head's new K and V rows; the warp that copies that block makes
    //      the store, just before the copy (see pa_decode_mma_kernel). ----
    int app_k = -1, app_blk = -1, app_pos = 0;
    if (p.new_k != nullptr) {
        const int pos = ld_dep(p.positions + b);
        if (pos < 0 || pos / B >= p.maxb) {
            if (c == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusBadLength);
        } else if (c == (pos < n ? (pos / B) / p.PB : 0)) {
            const int jb = pos / B;
            const int blk = ld_dep(bt_row + jb);
            if (blk < 0 || blk >= p.num_blocks) {
                if (threadIdx.x == 0) atomicOr(p.status, kStatusBadBlock);
            } else if (pos < n) {
                if (warp == (jb - pb0) % NW) {
                    app_k = (jb - pb0) / NW;
                    app_blk = blk;
                    app_pos = pos;
                }
            } else if (warp == 0) {
                // past the decoded context: no copy of this call needs the row
                warp_store_new_row<C::ROW_BYTES, (int)sizeof(T)>(p, b, kvh, blk, pos, B, lane);
            }
        }
    }
    const uint64_t policy = l2_policy_evict_first();

    // Block ids of this warp's blocks kbase..kbase+31, one per lane.
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
        if (k == app_k && sub == 0)
            warp_store_new_row<C::ROW_BYTES, (int)sizeof(T)>(p, b, kvh, app_blk, app_pos, B, lane);
        if (lane == 0) {
            const uint32_t bar = bars + 8 * stage;
            if (blk >= 0 && blk < p.num_blocks) {
                s_nvalid[stage] = rows;
                const uint32_t bytes = (uint32_t)rows * C::ROW_BYTES;
                mbar_arrive_expect_tx(bar, 2 * bytes);
                const long long off = (long long)blk * p.s_blk + (long long)row0 * D;
                const uint32_t dst = stage0 + stage * C::STAGE_BYTES;
                bulk_copy_g2s(dst, kpool + off, bytes, bar, policy);
                bulk_copy_g2s(dst + C::TILE_BYTES, vpool + off, bytes, bar, policy);
            } else {
                s_nvalid[stage] = 0;
                atomicOr(p.status, kStatusBadBlock);
                mbar_arrive(bar);
            }
        }
    };

    // ---- q of the G heads, this lane's slice, scaled into the log2 domain ----
    float2 qf[G][E2];
    {
        const T* qb = reinterpret_cast<const T*>(p.q) + ((long long)b * p.H + hbase) * D;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float2 f[4] = {};
            if (h < gact) load_row_slice<T, C::NV, C::LR>(qb + h * D, jl, f);
#pragma unroll
            for (int i = 0; i < E2; ++i)
                qf[h][i] = make_float2(f[i].x * p.qscale, f[i].y * p.qscale);
        }
    }

    float2 acc[G][E2];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int i = 0; i < E2; ++i) acc[h][i] = make_float2(0.f, 0.f);
    float m_run = -INFINITY;  // running max of head (lane % G), log2 domain
    float l_run = 0.f;        // this lane's share of the running sum of weights

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
            const T* Ks = reinterpret_cast<const T*>(wbase + stage * C::STAGE_BYTES);
            const T* Vs = Ks + C::R * D;

            // 1. partial scores of this lane: part[pass * G + h]
            float part[C::P];
#pragma unroll
            for (int ps = 0; ps < C::NPASS; ++ps) {
                const int row = ps * C::RP + rg;
                float2 kf[4];
                load_row_slice<T, C::NV, C::LR>(Ks + row * D, jl, kf);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float2 a = __fmul2_rn(qf[h][0], kf[0]);
#pragma unroll
                    for (int i = 1; i < E2; ++i) a = __ffma2_rn(qf[h][i], kf[i], a);
                    part[ps * G + h] = a.x + a.y;
                }
            }
            // 2. full scores, scattered over the lanes of each row group
            reduce_scatter<C::P, C::LR>(part, lane);
            if constexpr (C::P >= C::LR) {
#pragma unroll
                for (int i = 0; i < C::CF; ++i) {
                    const int id = jl * C::CF + i;
                    s_sc[((id / G) * C::RP + rg) * G + (id % G)] = part[i];
                }
            } else {
                constexpr int DUP = C::LR / C::P;
                if (jl % DUP == 0) {
                    const int id = jl / DUP;
                    s_sc[((id / G) * C::RP + rg) * G + (id % G)] = part[0];
                }
            }
            __syncwarp();

            // 3. online softmax over the sub-tile: lane handles pairs lane + 32*i,
            //    all of head (lane % G); rows past `rows` are masked out.
            float sv[C::PPL];
            float mloc = -INFINITY;
#pragma unroll
            for (int i = 0; i < C::PPL; ++i) {
                const int k = lane + 32 * i;
                float s = -INFINITY;
                if (k < C::PAIRS && (k / G) < rows) s = s_sc[k];
                sv[i] = s;
                mloc = fmaxf(mloc, s);
            }
#pragma unroll
            for (int o = G; o < 32; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(kFullMask, mloc, o));
            const float m_new = fmaxf(m_run, mloc);
            const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
            l_run *= alpha;
#pragma unroll
            for (int i = 0; i < C::PPL; ++i) {
                const int k = lane + 32 * i;
                const float pw = (sv[i] == -INFINITY) ? 0.f : exp2f(sv[i] - m_new);
                l_run += pw;
                if (k < C::PAIRS) s_sc[k] = pw;
            }
            m_run = m_new;
            if (lane < G) s_alpha[lane] = alpha;
            __syncwarp();

            // 4. rescale the accumulators, then O += P V
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float a = s_alpha[h];
                if (a != 1.f) {
                    const float2 a2 = make_float2(a, a);
#pragma unroll
                    for (int i = 0; i < E2; ++i) acc[h][i] = __fmul2_rn(acc[h][i], a2);
                }
            }
#pragma unroll
            for (int ps = 0; ps < C::NPASS; ++ps) {
                const int row = ps * C::RP + rg;
                if (row < rows) {
                    float2 vf[4];
                    load_row_slice<T, C::NV, C::LR>(Vs + row * D, jl, vf);
                    float pr[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) pr[h] = s_sc[row * G + h];
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float2 p2 = make_float2(pr[h], pr[h]);
#pragma unroll
                        for (int i = 0; i < E2; ++i) acc[h][i] = __ffma2_rn(p2, vf[i], acc[h][i]);
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
        // Let copies still in flight land before the stage memory is reused.
        for (int w = u; w < u_issue; ++w) (void)mbar_wait_bounded(bars + 8 * (w % S), (w / S) & 1);
    }

    // ---- warp-level reductions ----
#pragma unroll
    for (int o = C::LR; o < 32; o <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < E2; ++i) {
                acc[h][i].x += __shfl_xor_sync(kFullMask, acc[h][i].x, o);
                acc[h][i].y += __shfl_xor_sync(kFullMask, acc[h][i].y, o);
            }
    }
#pragma unroll
    for (int o = G; o < 32; o <<= 1) l_run += __shfl_xor_sync(kFullMask, l_run, o);

    // ---- per-warp state into its own (now idle) stage memory ----
    __syncwarp();
    float* w_m = reinterpret_cast<float*>(wbase);
    float* w_l = w_m + G;
    float* w_acc = w_l + G;  // [G][D]
    if (lane < G) {
        w_m[lane] = m_run;
        w_l[lane] = l_run;
    }
    if (rg == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < E2; ++i)
                *reinterpret_cast<float2*>(w_acc + h * D + slice_dim<C::VE, C::LR>(jl, i)) =
                    acc[h][i];
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
            M = fmaxf(M, reinterpret_cast<const float*>(smem + w * C::WARP_BYTES)[h]);
        float Lsum = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float* wm = reinterpret_cast<const float*>(smem + w * C::WARP_BYTES);
            const float mw = wm[h];
            const float wt = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
            Lsum += wt * wm[G + h];
            O += wt * wm[2 * G + h * D + d];
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

// Merges the partials of one (sequence, query head) gh:
//   M = max_c m_c,  out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c .
// W warps (1, 2, 4 or 8) serve one head; a 256-thread CTA serves 8 / W of them
// (hl: this warp's head slot in the CTA, w: its warp within the head).  Warp w
// takes partials w, w + W, ... four at a time (four independent loads of
// (m, l, O) in flight per lane; a lane owns D/32 consecutive elements) and
// keeps a running maximum, rescaling its sums when it rises, so the partials
// are read in one pass; the W warps' (max, sum, O) are then merged through
// shared memory the same way.  Every thread of the CTA calls it (it
// synchronises the CTA); nparts <= 1 writes nothing.  slot_of(c) is the
// workspace slot of partial c.
template <int D, int W, typename SlotOf>
__device__ __forceinline__ void combine_head(const DecodeParams& p, long long gh, int nparts,
                                             SlotOf slot_of, int hl, int w) {
    constexpr int PL = D / 32;
    __shared__ float s_acc[8][D];
    __shared__ float s_l[8];
    __shared__ float s_m[8];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    float M = -INFINITY, L = 0.f;
    float acc[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) acc[i] = 0.f;
    if (nparts > 1) {
        for (int c0 = w; c0 < nparts; c0 += 4 * W) {
            float mv[4], lv[4], ov[4][PL];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + u * W;
                mv[u] = -INFINITY;
                lv[u] = 0.f;
#pragma unroll
                for (int i = 0; i < PL; ++i) ov[u][i] = 0.f;
                if (c < nparts) {
                    const long long sl = slot_of(c);
                    mv[u] = ld_dep(p.part_ml + 2 * sl);
                    lv[u] = ld_dep(p.part_ml + 2 * sl + 1);
                    const float* oc = p.part_o + sl * D + lane * PL;
                    if constexpr (PL == 4) {
                        const float4 v = ld_dep(reinterpret_cast<const float4*>(oc));
                        ov[u][0] = v.x;
                        ov[u][1] = v.y;
                        ov[u][2] = v.z;
                        ov[u][3] = v.w;
                    } else {
#pragma unroll
                        for (int i = 0; i < PL; ++i) ov[u][i] = ld_dep(oc + i);
                    }
                }
            }
            float mn = M;
#pragma unroll
            for (int u = 0; u < 4; ++u) mn = fmaxf(mn, mv[u]);
            if (mn == -INFINITY) continue;  // (nothing but empty partials so far)
            const float sc = (M == -INFINITY) ? 0.f : exp2f(M - mn);
            L *= sc;
#pragma unroll
            for (int i = 0; i < PL; ++i) acc[i] *= sc;
            M = mn;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float wt = (mv[u] == -INFINITY) ? 0.f : exp2f(mv[u] - M);
                L += wt * lv[u];
#pragma unroll
                for (int i = 0; i < PL; ++i) acc[i] += wt * ov[u][i];
            }
        }
    }
    if constexpr (W > 1) {
#pragma unroll
        for (int i = 0; i < PL; ++i) s_acc[warp][lane * PL + i] = acc[i];
        if (lane == 0) {
            s_l[warp] = L;
            s_m[warp] = M;
        }
    }
    __syncthreads();
    if (nparts > 1 && w == 0) {
        if constexpr (W > 1) {
            float Mt = -INFINITY;
#pragma unroll
            for (int k = 0; k < W; ++k) Mt = fmaxf(Mt, s_m[hl * W + k]);
            float wk[W];
            float Lt = 0.f;
#pragma unroll
            for (int k = 0; k < W; ++k) {
                const float mk = s_m[hl * W + k];
                wk[k] = (mk == -INFINITY) ? 0.f : exp2f(mk - Mt);
                Lt += wk[k] * s_l[hl * W + k];
            }
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                float a = 0.f;
#pragma unroll
                for (int k = 0; k < W; ++k) a += wk[k] * s_acc[hl * W + k][lane * PL + i];
                acc[i] = a;
            }
            L = Lt;
        }
        float* o = p.out + gh * D + lane * PL;
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int i = 0; i < PL; ++i) o[i] = acc[i] * inv;
    }
}

// Merges the fixed-size partitions of every (sequence, query head) with more
// than one (the mma.sync and CUDA-core kernels): partial c of head gh sits at
// slot gh * Cmax + c.
template <int D, int W>
__global__ void __launch_bounds__(256) pa_combine_kernel(const DecodeParams p, int B) {
    pdl_trigger();
    pdl_wait();
    constexpr int HPC = 8 / W;  // heads per CTA
    const int warp = threadIdx.x >> 5;
    const int hl = warp / W;
    const int w = warp % W;
    const long long gh = (long long)blockIdx.x * HPC + hl;  // b * H + h
    int nparts = 0;
    if (gh < (long long)p.batch * p.H) {
        int n = ld_dep(p.lens + gh / p.H);
        if (n < 0 || n > p.maxb * B) n = 0;
        const int nblk = (n + B - 1) / B;
        nparts = nblk > 0 ? (nblk + p.PB - 1) / p.PB : 1;
    }
    const long long base = gh * p.Cmax;
    combine_head<D, W>(p, gh, nparts, [&](int c) -> long long { return base + c; }, hl, w);
}

// Merges the pieces of the (sequence, head group) pairs the tcgen05 kernel
// cut at its CTAs' range ends.  CTA group k (ceil(chunk / (rounds * 8 / W))
// CTAs, each serving rounds * 8 / W heads of the chunk, 8 / W at a time) serves
// pair k (direct: fewer pairs than decode CTAs, so most are cut) or the pair
// tc_cut[k] whose first piece decode CTA k holds (pair -1: none), which carries
// the pair's descriptor {first CTA, pieces, slot of the first piece} itself
// (direct: the pair's descriptor).  Piece c sits at slot ((first + c nchunks) *
// 2 + (c == 0 ? slot0 : 0)) * chunk + head in chunk: piece c came from CTA
// first + c nchunks (the CTAs of one head chunk are every nchunks-th), and only
// the first piece can be a CTA's second.  (rounds > 1 when one head per warp
// would not fit the SMs in one wave of CTAs.)
template <int D, int W>
__global__ void __launch_bounds__(256) pa_combine_tc_kernel(const DecodeParams p, int direct,
                                                            int rounds) {
    pdl_trigger();
    pdl_wait();
    constexpr int HPC = 8 / W;
    const int warp = threadIdx.x >> 5;
    const int hl = warp / W;
    const int w = warp % W;
    const int chunk = p.chunk;                          // heads per chunk (slot width)
    const int per_cta = HPC * rounds;                  // heads of the chunk per CTA
    const int cpp = (chunk + per_cta - 1) / per_cta;   // CTAs per pair
    const long long k = blockIdx.x / cpp;
    const int h_first = (int)(blockIdx.x % cpp) * per_cta;
    const long long npairs = (long long)p.batch * p.Hkv * p.nchunks;
    long long pair = k;
    int4 d = make_int4(0, 0, 0, 0);
    if (direct) {
        if (k < npairs) d = p.tc_desc[k];
    } else {
        const int4 rec = p.tc_cut[k];
        pair = rec.x;
        d = make_int4(rec.y, rec.z, rec.w, 0);
    }
    int nparts = 0, first = 0, slot0 = 0;
    int hvalid = 0;     // the chunk's heads (fewer in the last chunk of some groups)
    long long gh0 = 0;  // the chunk's first head in the output
    if (pair >= 0 && pair < npairs) {
        first = d.x;
        nparts = d.y;
        slot0 = d.z;
        // (a descriptor the decode never wrote -- it stopped on a timeout --
        // must not send the loads outside the partial slots)
        if (first < 0 || nparts < 0 ||
            (long long)first + (long long)(nparts > 0 ? nparts - 1 : 0) * p.nchunks >= p.tc_grid ||
            (slot0 & ~1))
            nparts = 0;
        const long long gpairs = (long long)p.Hkv * p.nchunks;
        const int g = (int)(pair % gpairs);
        gh0 = (pair / gpairs) * p.H + (long long)(g / p.nchunks) * p.gsize +
              (long long)(g % p.nchunks) * chunk;
        hvalid = min(chunk, p.gsize - (g % p.nchunks) * chunk);
    }
    auto slot_of = [&](int hh, int c) -> long long {
        return ((long long)first + (long long)c * p.nchunks) * 2 * chunk +
               (long long)(c == 0 ? slot0 : 0) * chunk + hh;
    };
    if constexpr (W == 1 && D == 128) {
        if (rounds <= 2 && nparts <= 2) {
            // the common case (a pair cut once, one or two heads per warp):
            // every load of the warp's heads first, then the merges, so the
            // heads share one round trip (uniform per CTA: no barrier here)
            const int lane = threadIdx.x & 31;
            float mv[2][2], lv[2][2];
            float4 ov[2][2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int hh = h_first + r * HPC + hl;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    mv[r][c] = -INFINITY;
                    lv[r][c] = 0.f;
                    ov[r][c] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (r < rounds && hh < hvalid && nparts == 2) {
                        const long long sl = slot_of(hh, c);
                        mv[r][c] = ld_dep(p.part_ml + 2 * sl);
                        lv[r][c] = ld_dep(p.part_ml + 2 * sl + 1);
                        ov[r][c] = ld_dep(reinterpret_cast<const float4*>(p.part_o + sl * D) + lane);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int hh = h_first + r * HPC + hl;
                if (r < rounds && hh < hvalid && nparts == 2) {
                    const float M = fmaxf(mv[r][0], mv[r][1]);
                    const float w0 = mv[r][0] == -INFINITY ? 0.f : exp2f(mv[r][0] - M);
                    const float w1 = mv[r][1] == -INFINITY ? 0.f : exp2f(mv[r][1] - M);
                    const float L = w0 * lv[r][0] + w1 * lv[r][1];
                    const float inv = L > 0.f ? 1.f / L : 0.f;
                    float4 o;
                    o.x = (w0 * ov[r][0].x + w1 * ov[r][1].x) * inv;
                    o.y = (w0 * ov[r][0].y + w1 * ov[r][1].y) * inv;
                    o.z = (w0 * ov[r][0].z + w1 * ov[r][1].z) * inv;
                    o.w = (w0 * ov[r][0].w + w1 * ov[r][1].w) * inv;
                    reinterpret_cast<float4*>(p.out + (gh0 + hh) * D)[lane] = o;
                }
            }
            return;
        }
    }
    for (int r = 0; r < rounds; ++r) {  // (uniform: combine_head synchronises the CTA)
        const int hh = h_first + r * HPC + hl;  // head within the chunk
        combine_head<D, W>(
            p, gh0 + hh, hh < hvalid ? nparts : 0, [&](int c) { return slot_of(hh, c); }, hl, w);
    }
}

}  // namespace pa
