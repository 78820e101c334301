// pa_decode_umma.cuh -- paged decode attention for bf16 pools with large GQA
// groups (16, 32, 48, 64 or 128 query heads per CTA) on the 5th-generation
// tensor cores: tcgen05.mma with the accumulators in tensor memory (TMEM).
//
// Computes the same thing as the other decode kernels: for sequence b and query
// head h, out = softmax_t(scale * q . K_t) V_t over the tokens reached through
// the block table ("vllmini", "PagedAttention Metaphor" / "The CUDA Block
// Kernel"; mini-infer, "The Solution").
//
// Why a separate kernel: the work per K/V byte grows with the group (G flop per
// byte for S = K Q^T, twice that for P V with the hi + lo split of P).  Up to
// G = 8 mma.sync keeps pace with HBM; from G = 16 it does not, and a tile with
// 128 tokens x G heads is a real contraction.
//
// Structure: persistent CTAs (one per SM, ~225 KB of shared memory).  The
// call's work is cut into 128-token tiles of (sequence, head group) pairs and
// every CTA takes an equal contiguous share of them (see the schedule below),
// so ragged lengths cost no tail.  Warp-specialised roles connected by
// mbarriers:
//  * warp 0 (K producer): block-table walk (entries loaded a tile ahead, a
//    piece's first ones and its appended row a piece ahead), the fused
//    append's K row, q of each piece into a swizzled K-major tile (2-D
//    tensor-map TMA, two buffers; one for 128-head chunks), and 5-D
//    tensor-map TMA loads of 128-token
//    K tiles (8 boxes of 16 rows per 64-column half, SWIZZLE_128B) into the K
//    ring;
//  * warp 2 (V producer): computes the CTA's share at start; the same walk for
//    V tiles into the V ring, the fused append's V row, bad ids / lengths.
//    A K stage is free as soon as S = K Q^T is done, a V stage only after
//    P V, so the two rings are sized and released separately;
//  * warp 1 (MMA): allocates TMEM; one thread issues
//      S[128 tok x G]   = K[128 x 128] . Q^T          (A, B K-major in smem)
//      O^T[128 d x 2G] += V^T[128 x 128 tok] . [P_hi | P_lo]  (A, B MN-major)
//    polling the barriers of both without blocking on either, and signals
//    completion with tcgen05.commit.  S is double-buffered in TMEM, so S of
//    tile i+1 is computed while tile i's softmax runs;
//  * warps 3 .. (softmax, 8 or 16 warps): 2 or 4 head parts per TMEM lane
//    quarter.  They read S (thread = token), run the online softmax in base 2
//    with a lazily raised running max (the max is raised, and O and the sums
//    rescaled, only when a score exceeds it by more than 2^8 -- any reference
//    point gives the same normalised result), write P as bf16 hi + lo
//    (|P - hi - lo| <= 2^-16 P) into the one P buffer once the previous P V
//    has read it, and at the end of a piece read O^T (thread = head-dim
//    element), add the hi and lo halves and store the output or the partial.
// 128-head chunks (HM) swap the roles of the operands: S[128 heads x 128 tok]
// = Q K^T and O[128 heads x 128 d] += P_hi V + P_lo V with P written to TMEM
// by the softmax warps and read from there as the A operand; a softmax thread
// then owns one head's row (16 warps: 4 lane quarters of heads x 4 quarters of
// the tile's tokens, which agree on the running max at a named barrier).
// Groups of 80-112 heads fill one 128-head chunk; the rows past the group are
// computed and not written.
// Every wait is bounded (PA_STATUS_TIMEOUT); the roles then stop together,
// wait for their copies and MMAs in flight, and TMEM is freed.
#pragma once

#include <cfloat>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_schedule.cuh"

namespace pa {

// ---------------------------------------------------------------- tcgen05 --

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (all >> 4), the fixed version field (bits 46-48 = 0b001) and the
// 128-byte swizzle (layout type 2 in bits 61-63).  K-major operands: SBO is the
// distance between 8-row groups, LBO unused.  MN-major operands: LBO is the
// distance between 64-element column blocks, SBO between 8-row (K) groups.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B,
// operand majors (0 = K-major, 1 = MN-major), N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM) = A . B (+ D if accumulate), issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D (TMEM) = A . B (+ D), A read from tensor memory (M rows on the lanes, two
// 16-bit K elements per 32-bit column, the first in the low half), B from
// shared memory.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier receives one arrival once every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_addr, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     slot_addr),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (32x32b shape: lane
// 32 * (warp % 4) + laneid of the warp's quarter).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// N (8 or a multiple of 16) consecutive columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
    if constexpr (N == 8) {
        tmem_ld8(taddr, r);
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 16)
            tmem_ld16(taddr + c, *reinterpret_cast<uint32_t(*)[16]>(r + c));
    }
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* r) {
    if constexpr (N == 8) {
        tmem_st8(taddr, r);
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 16)
            tmem_st16(taddr + c, *reinterpret_cast<const uint32_t(*)[16]>(r + c));
    }
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barriers over the 128 softmax threads of one head part (four warps,
// one per TMEM lane quarter): id 1 + 2 * part plain, 2 + 2 * part with an OR
// reduction of `v` (separate ids, so the two forms never share one).
__device__ __forceinline__ void part_bar(int part) {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + 2 * part) : "memory");
}
__device__ __forceinline__ bool part_bar_or(int part, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(2 + 2 * part)
        : "memory");
    return r != 0;
}

// HM softmax: named barriers over the four warps of one TMEM lane quarter (the
// four token parts of the same 32 heads): id 1 + 2 * quarter plain, 2 + 2 *
// quarter with an OR reduction (the ids of the head parts' barriers above,
// which an HM kernel does not use).
__device__ __forceinline__ void quarter_bar(int qd) {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + 2 * qd) : "memory");
}
__device__ __forceinline__ bool quarter_bar_or(int qd, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(2 + 2 * qd)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ config --

template <int B_, int G_>
struct UmmaCfg {
    static constexpr int D = 128, B = B_, G = G_;
    // 128-head chunks put the heads on the rows of the accumulators (HM):
    // S[128 heads x 128 tok] = Q K^T and O[128 heads x 128 d] += P V, with P
    // written to tensor memory and read from there as the A operand -- no P
    // buffer in shared memory, and one row of S and O per softmax thread.
    static constexpr bool HM = G == 128;
    static constexpr int TT = 128;                  // tokens per tile (M of S = K Q^T)
    static constexpr int NBOX = TT / 16;            // 16-row boxes per 64-column half
    static constexpr int HALF = TT * 128;           // one 64-column half of a tile (bytes)
    static constexpr int TILE = 2 * HALF;           // a K or a V tile
    // Separate K and V rings: a K stage is free once S = K Q^T has read it, a V
    // stage only after P V; so K runs ahead and the V ring covers the long
    // chain (copy, S, softmax, P V).
    static constexpr int SK = G >= 48 ? 2 : 3;      // K stages
    static constexpr int SV = 3;                    // V stages
    // P of a tile: [64-column block][token][128 B] rows of hi heads | lo heads
    // | zeros up to a whole block, in one buffer: the softmax of tile i + 1
    // overlaps P V of tile i and waits for it only before writing P.  (HM: in
    // tensor memory instead.)
    static constexpr int PW = HM ? 0 : (2 * G + 63) / 64 * 64;
    static constexpr int P_BYTES = (PW / 64) * HALF;
    static constexpr int Q_BYTES = 2 * G * 128;     // q of one piece, two 64-column halves
    // q buffers: two (the next piece's q lands while this piece's S runs); HM
    // one, for the third V stage (the next q is loaded once this piece's last
    // S is done, while its last tiles' softmax and P V still run)
    static constexpr int NQ = HM ? 1 : 2;
    // TMEM: S0 [0, G), S1 [G, 2G), O^T after; HM: S0 [0, 128), S1 [128, 256),
    // P [256, 384) (hi, tokens packed in pairs, then lo), O [384, 512).  (P in
    // the tile's own S buffer, which the next S but one overwrites behind this
    // tile's P V, measured the same on GB300: 78.2 against 78.3 us per call.)
    static constexpr int S_COLS = HM ? TT : G;
    static constexpr int P_COL = 256;
    static constexpr int O_COL = HM ? 384 : 2 * G;
    static constexpr int TMEM_USED = HM ? 512 : 2 * G + PW;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64
                                   : TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
    static constexpr int OFF_V = SK * TILE;
    static constexpr int OFF_P = OFF_V + SV * TILE;
    static constexpr int OFF_Q = OFF_P + P_BYTES;
    static constexpr int OFF_CTRL = OFF_Q + NQ * Q_BYTES;
    // ctrl: mbarriers [0, 224) | TMEM address | abort flag | m[G] | alpha[G] |
    // red[4][G] | this CTA's schedule (48 bytes)
    static constexpr int SCHED_OFF = 256 + 6 * G * 4;
    static constexpr int CTRL_BYTES = SCHED_OFF + 48;
    static constexpr int TMEM_SLOT_OFF = 224, ABORT_OFF = 228;
    static constexpr int SMEM_BYTES = OFF_CTRL + CTRL_BYTES + 1024;
    // warps: 0 K producer (+ q), 1 MMA, 2 V producer, 3 .. softmax (4 lane
    // quarters x 2, 3 or 4 head parts: more than one warp per scheduler, so
    // the dependent latencies of the per-token work overlap; HM: 4 lane
    // quarters of heads x 4 parts of the tile's tokens)
    static constexpr int NPART = G == 48 ? 3 : (G >= 64 ? 4 : 2);   // head (HM: token) parts
    static constexpr int HG = HM ? 8 : G / NPART;   // heads per softmax warp (not HM)
    static constexpr int TP = TT / NPART;           // HM: tokens per softmax warp
    static constexpr int SM_WARP0 = 3;
    static constexpr int NSW = 4 * NPART;           // softmax warps
    static constexpr int NSM = NSW * 32;            // softmax threads
    static constexpr int THREADS = (SM_WARP0 + NSW) * 32;
    // barrier indices
    static constexpr int K_FULL = 0, K_EMPTY = SK, V_FULL = 2 * SK, V_EMPTY = 2 * SK + SV,
                         Q_FULL = 2 * SK + 2 * SV, Q_EMPTY = Q_FULL + 2, S_FULL = Q_FULL + 4,
                         P_FULL = Q_FULL + 6, PV_DONE = Q_FULL + 8, FINAL = Q_FULL + 10,
                         NBAR = Q_FULL + 11;
    // Q_FULL / Q_EMPTY pairs follow the two q buffers; S_FULL, P_FULL and
    // PV_DONE are pairs used by tile parity, so that no barrier ever runs two
    // phases ahead of a waiter (parity waits would alias); every other
    // barrier's next phase needs the waiter's own progress.

    static_assert(G == 16 || G == 32 || G == 48 || G == 64 || G == 128,
                  "head chunk of 16, 32, 48, 64 or 128");
    static_assert(B == 16 || B == 32, "block size 16 or 32");
    static_assert(NBAR * 8 <= TMEM_SLOT_OFF, "barriers");
    static_assert(TMEM_USED <= TMEM_COLS, "TMEM columns");
    static_assert(HG == 8 || HG % 16 == 0, "TMEM loads of 8 or 16k columns");
    static_assert(!HM || TP == 32, "HM: 32 tokens per softmax warp");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Work schedule: equal shares of 128-token tiles per persistent CTA (see
// pa_schedule.cuh), each (sequence, head group) pair charged extra units for a
// piece's fixed cost (q, the first tile's maximum, the output, the next
// copies' latency).  GB300, once a piece's inputs were loaded a piece ahead:
// two units ahead of three by 1-2 % at 16, 32 and 48 heads, and by 1.5 % at
// 64 (0 and 1 slower); three for 128-head chunks (128 heads: 74.7 us per call
// against 76.5 with two and 75.7 with four).
template <int G>
constexpr int kUmmaPieceUnits = G == 128 ? 3 : 2;
using UItem = SPiece;
using UWalk = SWalk;

template <int B, int G>
__device__ __forceinline__ void umma_schedule(const DecodeParams& p, unsigned char* sched,
                                              int lane) {
    sched_compute<B, 128, kUmmaPieceUnits<G>>(p, sched, lane);
}
template <int B>
__device__ __forceinline__ void umma_walk_begin(const DecodeParams& p, const unsigned char* sched,
                                                UWalk& w) {
    sched_walk_begin<B, 128>(p, sched, w);
}
template <int B, int G>
__device__ __forceinline__ bool umma_walk_next(const DecodeParams& p, UWalk& w, UItem& it) {
    return sched_walk_next<B, 128, kUmmaPieceUnits<G>, G>(p, w, it);
}

// Non-blocking test of an mbarrier phase (try_wait may suspend the thread for
// a while; a thread that polls several barriers must not be parked on one).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for an mbarrier phase, suspending the thread (no issue slots used)
// until the phase completes or about `ns` nanoseconds have passed.
__device__ __forceinline__ bool mbar_try_wait_for(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool umma_wait(uint32_t bar, uint32_t parity, volatile int* abort_all,
                                          unsigned* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_all) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
    *abort_all = 1;
    atomicOr(status, kStatusTimeout);
    return false;
}

// Byte offset of 16-byte chunk j of row r in a 1024-byte-aligned stack of
// 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128(int r, int j) {
    return (uint32_t)(r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

// Max (or sum) of v[j] over the warp's 32 lanes for each of N = 2^k values,
// as a reduce-scatter butterfly: at each step a lane sends the half of its
// values it does not keep, so N + N/2 + ... shuffles become N - 1 + 5 - log2 N
// (16 values: 16 shuffles instead of 80).  Lane l ends with value
// l / (32 / N)'s result (lanes that differ in their low 5 - log2 N bits hold
// the same one).
template <int N, bool MAX>
__device__ __forceinline__ float warp_scatter_reduce(const float (&in)[N], int lane) {
    static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "a power of two up to 32");
    float v[N];
#pragma unroll
    for (int j = 0; j < N; ++j) v[j] = in[j];
#pragma unroll
    for (int k = N, o = 16; k > 1; k >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < k / 2; ++j) {
            const float send = up ? v[j] : v[j + k / 2];
            const float keep = up ? v[j + k / 2] : v[j];
            const float got = __shfl_xor_sync(kFullMask, send, o);
            v[j] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    float r = v[0];
#pragma unroll
    for (int o = 16 / N; o > 0; o >>= 1) {
        const float got = __shfl_xor_sync(kFullMask, r, o);
        r = MAX ? fmaxf(r, got) : r + got;
    }
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <int B, int G>
__global__ void __launch_bounds__(UmmaCfg<B, G>::THREADS, 1)
    pa_decode_umma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv,
                          const __grid_constant__ CUtensorMap tmq) {
    pdl_trigger();
    using C = UmmaCfg<B, G>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
    unsigned char* smem = smem_raw + (sbase - raw_addr);
    unsigned char* ctrl = smem + C::OFF_CTRL;
    const uint32_t bar0 = sbase + C::OFF_CTRL;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + C::TMEM_SLOT_OFF);
    volatile int* abort_all = reinterpret_cast<volatile int*>(ctrl + C::ABORT_OFF);
    float* m_sh = reinterpret_cast<float*>(ctrl + 256);             // running max per head
    float* a_sh = m_sh + G;                                         // rescale factor per head
    float* red = a_sh + G;                                          // [4][G] cross-warp partials

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NBAR; ++i)
            mbar_init(bar0 + 8 * i, (i == C::P_FULL || i == C::P_FULL + 1) ? C::NSW : 1);
        *abort_all = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        prefetch_tensormap(&tmq);
    }
    // (nothing above reads what the previous kernel may have written: the
    // set-up overlaps its tail)
    pdl_wait();
    if (warp == 2) umma_schedule<B, G>(p, ctrl + C::SCHED_OFF, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == 2) {
        // ============================= producers: warp 0 K (and q), warp 2 V
        // Both walk the same pieces and table entries.  Everything a piece
        // needs from global memory before its first copy (its first table
        // entries, the appended row's position and bytes) is loaded one piece
        // ahead: under a full HBM stream a dependent load costs microseconds.
        // The fused append's new row is stored by each producer for its own
        // half (K or V) right before the copy of the tile that holds it; warp
        // 2 reports bad ids and lengths.
        const bool is_v = (warp == 2);
        const CUtensorMap* tm = is_v ? &tmv : &tmk;
        const int NS = is_v ? C::SV : C::SK;
        const uint32_t full0 = bar0 + 8 * (is_v ? C::V_FULL : C::K_FULL);
        const uint32_t empty0 = bar0 + 8 * (is_v ? C::V_EMPTY : C::K_EMPTY);
        const uint32_t ring = sbase + (is_v ? C::OFF_V : 0);
        // (streamed once: evict first; a group served in chunks is streamed by
        // the sibling CTAs side by side, all but the first from L2)
        const uint64_t policy = p.nchunks > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
        const bool append = p.new_k != nullptr;
        const unsigned char* new_rows =
            static_cast<const unsigned char*>(is_v ? p.new_v : p.new_k);
        unsigned short* pool_rows = const_cast<unsigned short*>(
            reinterpret_cast<const unsigned short*>(is_v ? p.v_base : p.k_base));
        int kt = 0, qi = 0, q_last = -1;
        bool aborted = false;
        // block-table entry of box `lane` of tile i of a piece (0 if none)
        auto box_block = [&](const UItem& pc, int i) {
            const int tok = pc.t0 + i * C::TT + 16 * lane;
            return (i < pc.ntiles && lane < C::NBOX && tok < pc.t1)
                       ? ld_dep(p.bt + (long long)pc.b * p.maxb + tok / B)
                       : 0;
        };
        // the appended row of a piece's (sequence, KV head): its position and
        // (lanes < 16) one 16-byte chunk of its 256 bytes
        auto row_pos = [&](const UItem& pc) { return append ? ld_dep(p.positions + pc.b) : -1; };
        auto row_val = [&](const UItem& pc) {
            return (append && lane < 16)
                       ? ld_dep(reinterpret_cast<const uint4*>(
                                   new_rows + ((long long)pc.b * p.Hkv + pc.kvh) * 256) +
                               lane)
                       : make_uint4(0, 0, 0, 0);
        };
        // (this CTA's cut pair, if any, is recorded as its pieces are walked;
        // none so far)
        if (is_v && lane == 0 && p.tc_cut != nullptr) p.tc_cut[blockIdx.x] = make_int4(-1, 0, 0, 0);
        UWalk w;
        umma_walk_begin<B>(p, ctrl + C::SCHED_OFF, w);
        UItem it, nx;
        bool have = umma_walk_next<B, G>(p, w, it);
        int blk_first = have ? box_block(it, 0) : 0;
        int pos = have ? row_pos(it) : -1;
        uint4 rowv = have ? row_val(it) : make_uint4(0, 0, 0, 0);
        while (have && !aborted) {
            const bool have_nx = umma_walk_next<B, G>(p, w, nx);
            const int blk_first_nx = have_nx ? box_block(nx, 0) : 0;
            const int pos_nx = have_nx ? row_pos(nx) : -1;
            const uint4 rowv_nx = have_nx ? row_val(nx) : make_uint4(0, 0, 0, 0);
            // (the piece at tile 0 of head group 0 reports for the sequence)
            const bool reporter = is_v && it.g == 0 && it.u == 0 && lane == 0;
            if (reporter && it.bad_len) atomicOr(p.status, kStatusBadLength);
            if (is_v && it.u == 0 && lane == 0 && p.tc_desc != nullptr) {
                // where the combine finds this pair's pieces: CTAs first ..
                // first + pieces - 1 (the owners of its first and last unit); a
                // pair that continues past this CTA is its cut pair (at most
                // one: the range's last piece).  (Written here, a piece ahead of
                // the softmax warps: the count takes a 64-bit division.)
                const int pieces = sched_pieces(p, it, w);
                const long long pair = (long long)it.b * p.Hkv * p.nchunks + it.g;
                p.tc_desc[pair] = make_int4((int)blockIdx.x, pieces, it.first ? 0 : 1, 0);
                if (!it.whole)
                    p.tc_cut[blockIdx.x] =
                        make_int4((int)pair, (int)blockIdx.x, pieces, it.first ? 0 : 1);
            }
            // stores the appended row into block `blk` (every head chunk its
            // own identical copy), ordered before this warp's later copies
            auto store_row = [&](int blk) {
                if (blk < 0 || blk >= p.num_blocks) {
                    if (is_v && lane == 0) atomicOr(p.status, kStatusBadBlock);
                } else if (lane < 16) {
                    const long long off = (long long)blk * p.s_blk + p.tile_off +
                                          (long long)it.kvh * p.s_head + (long long)(pos % B) * 128;
                    reinterpret_cast<uint4*>(pool_rows + off)[lane] = rowv;
                    fence_proxy_async_global();
                }
                __syncwarp();
            };
            // the piece holding the row's tile stores it before that tile's
            // copy; a row past the context is stored by the pair's first piece
            int store_tile = -1;
            if (append) {
                if (pos < 0 || pos / B >= p.maxb) {
                    if (reporter) atomicOr(p.status, kStatusBadLength);
                } else if (pos < it.n) {
                    if (pos >= it.t0 && pos < it.t1) store_tile = (pos - it.t0) / C::TT;
                } else if (it.u == 0) {
                    store_row(ld_dep(p.bt + (long long)it.b * p.maxb + pos / B));
                }
            }

            // 128-token tiles: lane r < 8 walks box r (16 rows) of the tile; the
            // block-table entries of tile i + 1 are loaded while tile i waits
            // for its stage
            int blk_next = blk_first;
            for (int i = 0; i < it.ntiles; ++i, ++kt) {
                const int stage = kt % NS;
                const int use = kt / NS;
                const int tok = it.t0 + i * C::TT + 16 * lane;
                bool valid = lane < C::NBOX && tok < it.t1;
                const int blk = blk_next;
                blk_next = box_block(it, i + 1);
                // (every lane waits and votes: the warp leaves the loop together)
                if (use > 0 && !__all_sync(kFullMask, umma_wait(empty0 + 8 * stage, (use - 1) & 1,
                                                                abort_all, p.status))) {
                    aborted = true;
                    break;
                }
                if (i == store_tile)  // (the row's box lane holds its block id)
                    store_row(__shfl_sync(kFullMask, blk, ((pos - it.t0) % C::TT) / 16));
                const bool bad = valid && (blk < 0 || blk >= p.num_blocks);
                valid = valid && !bad;
                const unsigned vmask = __ballot_sync(kFullMask, valid);
                const unsigned bmask = __ballot_sync(kFullMask, bad);
                const uint32_t fb = full0 + 8 * stage;
                if (lane == 0) {
                    if (is_v && bmask) atomicOr(p.status, kStatusBadBlock);
                    mbar_arrive_expect_tx(fb, (uint32_t)__popc(vmask) * 2u * 2048u);
                }
                __syncwarp();
                if (valid) {
                    const int row0 = tok % B;
                    const int o2 = p.tma_slot_blk == 2 ? blk
                                   : (p.tma_slot_layer == 2 ? p.layer : it.kvh);
                    const int o3 = p.tma_slot_blk == 3 ? blk
                                   : (p.tma_slot_layer == 3 ? p.layer : it.kvh);
                    const int o4 = p.tma_slot_blk == 4 ? blk
                                   : (p.tma_slot_layer == 4 ? p.layer : it.kvh);
                    const uint32_t dst = ring + stage * C::TILE + lane * 2048;
                    tma_load_5d(dst, tm, fb, 0, row0, o2, o3, o4, policy);
                    tma_load_5d(dst + C::HALF, tm, fb, 64, row0, o2, o3, o4, policy);
                }
                if (!is_v && i == 0) {
                    // q of the piece's G heads -> K-major swizzled tile
                    // [half][G][128 B] by two tensor-map copies, once its first
                    // K copy is on its way (buffer qi % NQ: free once the last S
                    // of piece qi - NQ is done)
                    if (qi >= C::NQ &&
                        !__all_sync(kFullMask, umma_wait(bar0 + 8 * (C::Q_EMPTY + qi % C::NQ),
                                                         ((qi / C::NQ) - 1) & 1, abort_all,
                                                         p.status))) {
                        aborted = true;
                        ++kt;  // (tile 0's copy is in flight: the exit path waits for it)
                        break;
                    }
                    if (lane == 0) {
                        const uint32_t qbuf = sbase + C::OFF_Q + (qi % C::NQ) * C::Q_BYTES;
                        const uint32_t qbar = bar0 + 8 * (C::Q_FULL + qi % C::NQ);
                        const int qrow = it.b * p.H + it.hbase;
                        mbar_arrive_expect_tx(qbar, (uint32_t)C::Q_BYTES);
                        tma_load_2d(qbuf, &tmq, qbar, 0, qrow);
                        tma_load_2d(qbuf + G * 128, &tmq, qbar, 64, qrow);
                    }
                    q_last = qi;
                    __syncwarp();
                }
            }
            if (!aborted && it.ntiles > 0) ++qi;
            it = nx;
            have = have_nx;
            blk_first = blk_first_nx;
            pos = pos_nx;
            rowv = rowv_nx;
        }
        if (aborted || *abort_all) {
            // copies still in flight land before the CTA can exit
            for (int k = kt > NS ? kt - NS : 0; k < kt; ++k)
                (void)mbar_wait_bounded(full0 + 8 * (k % NS), (k / NS) & 1);
            for (int k = q_last >= C::NQ - 1 ? q_last - (C::NQ - 1) : 0; !is_v && k <= q_last; ++k)
                (void)mbar_wait_bounded(bar0 + 8 * (C::Q_FULL + k % C::NQ), (k / C::NQ) & 1);
        }
    } else if (warp == 1) {
        // ============================================ MMA issuer (warp 1, lane 0)
        if (lane == 0) {
            // Two cursors: S = K Q^T of tile kt_q (once its K and q are in and an
            // S buffer is free: at most two tiles ahead of P V; the K stage is
            // released when S completes) and O^T += V^T [P_hi | P_lo] of tile
            // kt_pv (once its P is written and its V is in; the V stage is
            // released when P V completes).  Tested without blocking on either;
            // with nothing to issue the thread suspends on the barrier it
            // expects next (it shares a scheduler with softmax warps, which
            // need the issue slots a spinning loop would take).
            // Descriptors: each buffer's base is encoded once; a K-step adds its
            // byte offset / 16 to the start-address field (no carry: shared
            // addresses stay below 256 KB).
            constexpr uint32_t IDQ = umma_idesc_bf16(128, C::HM ? C::TT : G, 0, 0);
            constexpr uint32_t IDP = umma_idesc_bf16(128, C::HM ? 128 : C::PW, 1, 1);
            const uint64_t dP0 = umma_desc_sw128(sbase + C::OFF_P, C::HALF, 1024);
            const uint64_t dV0 = umma_desc_sw128(sbase + C::OFF_V, C::HALF, 1024);
            const uint64_t dK0 = umma_desc_sw128(sbase, 0, 1024);
            const uint64_t dQ0 = umma_desc_sw128(sbase + C::OFF_Q, 0, 1024);
            UWalk wq;
            umma_walk_begin<B>(p, ctrl + C::SCHED_OFF, wq);
            int tiles_left = 0;       // tiles of the current piece still without S
            int i_q = 0, qi = -1;     // tile within the piece; piece (with tiles) count
            bool q_ready = false, done_q = false;
            int kt_q = 0, kt_pv = 0;
            unsigned first_bits = 0;  // bit (tile & 1): the tile is its piece's first
            unsigned long long idle_since = 0;
            while (true) {
                bool progressed = false;
                if (kt_pv < kt_q &&
                    mbar_test(bar0 + 8 * (C::P_FULL + (kt_pv & 1)), (kt_pv >> 1) & 1) &&
                    mbar_test(bar0 + 8 * (C::V_FULL + kt_pv % C::SV), (kt_pv / C::SV) & 1)) {
                    tc_fence_after();
                    const int vs = kt_pv % C::SV;
                    const bool first = (first_bits >> (kt_pv & 1)) & 1u;
                    const uint64_t a0 = dV0 + (uint64_t)((vs * C::TILE) >> 4);
                    if constexpr (C::HM) {
                        // O[128 heads x 128 d] += P_hi V, then += P_lo V: A = P in
                        // TMEM (a K-step of 16 tokens is 8 columns), B = V
                        // (MN-major, the same descriptor as V^T as A below)
                        constexpr uint32_t IDV = umma_idesc_bf16(128, 128, 0, 1);
                        constexpr int KS = C::TT / 16;
#pragma unroll
                        for (int k = 0; k < 2 * KS; ++k)
                            umma_bf16_ts(tmem + C::O_COL,
                                         tmem + C::P_COL + (k / KS) * 64 + (k % KS) * 8,
                                         a0 + (uint64_t)((k % KS) * (2048 >> 4)), IDV,
                                         (k > 0 || !first) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < C::TT / 16; ++k)
                            umma_bf16(tmem + C::O_COL, a0 + (uint64_t)(k * (2048 >> 4)),
                                      dP0 + (uint64_t)(k * (2048 >> 4)), IDP,
                                      (k > 0 || !first) ? 1u : 0u);
                    }
                    umma_commit(bar0 + 8 * (C::PV_DONE + (kt_pv & 1)));
                    umma_commit(bar0 + 8 * (C::V_EMPTY + vs));
                    ++kt_pv;
                    progressed = true;
                }
                if (!done_q && kt_q < kt_pv + 2) {
                    while (tiles_left == 0) {
                        UItem it;
                        if (!umma_walk_next<B, G>(p, wq, it)) break;
                        if (it.ntiles > 0) {
                            tiles_left = it.ntiles;
                            i_q = 0;
                            ++qi;
                            q_ready = false;
                        }
                    }
                    if (tiles_left == 0) {
                        done_q = true;
                    } else {
                        if (!q_ready)
                            q_ready = mbar_test(bar0 + 8 * (C::Q_FULL + qi % C::NQ), (qi / C::NQ) & 1);
                        const int ks = kt_q % C::SK;
                        if (q_ready &&
                            mbar_test(bar0 + 8 * (C::K_FULL + ks), (kt_q / C::SK) & 1)) {
                            tc_fence_after();
                            const uint64_t a0 = dK0 + (uint64_t)((ks * C::TILE) >> 4);
                            const uint64_t b0 = dQ0 + (uint64_t)(((qi % C::NQ) * C::Q_BYTES) >> 4);
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const int h = k >> 2, kk = k & 3;
                                const uint64_t kdesc = a0 + (uint64_t)((h * C::HALF + kk * 32) >> 4);
                                const uint64_t qdesc =
                                    b0 + (uint64_t)((h * (G * 128) + kk * 32) >> 4);
                                if constexpr (C::HM)   // S[128 heads x 128 tok] = Q K^T
                                    umma_bf16(tmem + (kt_q & 1) * C::S_COLS, qdesc, kdesc, IDQ,
                                              k > 0 ? 1u : 0u);
                                else                   // S[128 tok x G] = K Q^T
                                    umma_bf16(tmem + (kt_q & 1) * C::S_COLS, kdesc, qdesc, IDQ,
                                              k > 0 ? 1u : 0u);
                            }
                            umma_commit(bar0 + 8 * (C::S_FULL + (kt_q & 1)));
                            umma_commit(bar0 + 8 * (C::K_EMPTY + ks));
                            first_bits = (first_bits & ~(1u << (kt_q & 1))) |
                                         ((i_q == 0 ? 1u : 0u) << (kt_q & 1));
                            ++i_q;
                            if (--tiles_left == 0) umma_commit(bar0 + 8 * (C::Q_EMPTY + qi % C::NQ));
                            ++kt_q;
                            progressed = true;
                        }
                    }
                }
                if (done_q && kt_pv == kt_q) break;
                if (progressed) {
                    idle_since = 0;
                    continue;
                }
                if (*abort_all) break;
                // suspend on what gates the next step: the next S (its q, then
                // its K) while it may run ahead, else the pending P V's P
                if (!done_q && tiles_left > 0 && kt_q < kt_pv + 2) {
                    if (!q_ready)
                        (void)mbar_try_wait_for(bar0 + 8 * (C::Q_FULL + qi % C::NQ), (qi / C::NQ) & 1,
                                                200);
                    else
                        (void)mbar_try_wait_for(bar0 + 8 * (C::K_FULL + kt_q % C::SK),
                                                (kt_q / C::SK) & 1, 200);
                } else if (kt_pv < kt_q) {
                    (void)mbar_try_wait_for(bar0 + 8 * (C::P_FULL + (kt_pv & 1)),
                                            (kt_pv >> 1) & 1, 200);
                }
                const unsigned long long now = globaltimer_ns();
                if (idle_since == 0) {
                    idle_since = now;
                } else if (now - idle_since > kWaitLimitNs) {
                    *abort_all = 1;
                    atomicOr(p.status, kStatusTimeout);
                    break;
                }
            }
            // every MMA issued so far completes before TMEM is released
            umma_commit(bar0 + 8 * C::FINAL);
            (void)mbar_wait_bounded(bar0 + 8 * C::FINAL, 0);
        }
        __syncwarp();
    } else if constexpr (C::HM) {
        // ========== softmax, heads on the rows (128-head chunks): warp w reads
        // TMEM lane quarter w % 4 (heads 32 * (w % 4) + lane) and the tile's
        // tokens [32 * part, 32 * part + 32) of S; O's head-dim columns are
        // split the same way.  A thread holds one head's running max (the four
        // parts of a quarter agree on it at the quarter's barrier) and its
        // part's share of the sum.
        const int part = (warp - C::SM_WARP0) >> 2;
        const int qd = warp & 3;
        const int hrow = qd * 32 + lane;       // head within the chunk (TMEM lane)
        const int c0 = part * C::TP;           // the part's first token / head-dim column
        const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
        int kt = 0;
        bool stop = false;
        bool failed = false;   // (as below: the threads stop together at a barrier)
        auto swait = [&](uint32_t bar, uint32_t parity) {
            return umma_wait(bar, parity, abort_all, p.status);
        };
        // block ids of the part's 32 tokens in tile i of a piece (two boxes of
        // 16 tokens; one block when B = 32), -1 past the piece; loaded a tile
        // ahead
        auto part_blocks = [&](const UItem& pc, int i, int& b0, int& b1) {
            const int tok = pc.t0 + i * C::TT + c0;
            const int* row = p.bt + (long long)pc.b * p.maxb;
            b0 = (i < pc.ntiles && tok < pc.t1) ? ld_dep(row + tok / B) : -1;
            if constexpr (B == 16)
                b1 = (i < pc.ntiles && tok + 16 < pc.t1) ? ld_dep(row + (tok + 16) / B) : -1;
            else
                b1 = b0;
        };
        UWalk w;
        umma_walk_begin<B>(p, ctrl + C::SCHED_OFF, w);
        UItem it;
        bool have = umma_walk_next<B, G>(p, w, it);
        int nb0 = -1, nb1 = -1;
        if (have) part_blocks(it, 0, nb0, nb1);
        while (!stop && have) {
            // this thread's head is one of the chunk's (a group of 80-112 heads
            // fills 128 rows: the rows past it are computed and not written)
            const bool own = hrow < p.gsize - it.hc * G;
            if (it.ntiles == 0) {  // empty context: output 0 (always a whole piece)
                const long long head0 = (long long)it.b * p.H + it.hbase;
                float4* o4 = reinterpret_cast<float4*>(p.out + (head0 + hrow) * 128 + c0);
#pragma unroll
                for (int j = 0; j < C::TP / 4; ++j)
                    if (own) o4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                have = umma_walk_next<B, G>(p, w, it);
                if (have) part_blocks(it, 0, nb0, nb1);
                continue;
            }
            float m_run = -INFINITY;   // this head's running max (the floor -FLT_MAX
            float l_run = 0.f;         // once a tile has passed), this part's sum
            for (int i = 0; i < it.ntiles; ++i, ++kt) {
                const int stage = kt % C::SV;  // V stage
                const int b0 = nb0, b1 = nb1;
                part_blocks(it, i + 1, nb0, nb1);
                // the part's valid tokens: before the piece's end, in a good block
                uint32_t vm;
                {
                    const int nv = it.t1 - (it.t0 + i * C::TT + c0);
                    vm = nv >= 32 ? 0xffffffffu : (nv > 0 ? (1u << nv) - 1u : 0u);
                    if (b0 < 0 || b0 >= p.num_blocks) vm &= 0xffff0000u;
                    if (b1 < 0 || b1 >= p.num_blocks) vm &= 0x0000ffffu;
                }
                const bool ok = swait(bar0 + 8 * (C::S_FULL + (kt & 1)), (kt >> 1) & 1);
                failed = failed || !ok;
                __syncwarp();
                tc_fence_after();
                float x[C::TP];
                {
                    uint32_t v[C::TP];
                    tmem_ld_cols<C::TP>(trow + (kt & 1) * C::S_COLS + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < C::TP; ++j)
                        x[j] = ((vm >> j) & 1u) ? __uint_as_float(v[j]) * p.qscale : -INFINITY;
                }
                float mloc = -INFINITY;
#pragma unroll
                for (int j = 0; j < C::TP; ++j) mloc = fmaxf(mloc, x[j]);
                // the running max is raised (to the tile's max over the four
                // parts) only when a score exceeds it by more than 2^8; every
                // part of the head takes the same decision from the same values
                float alpha = 1.f;
                bool raised = false;
                if (quarter_bar_or(qd, i == 0 || mloc - m_run > 8.f || failed)) {
                    red[part * G + hrow] = mloc;
                    if (quarter_bar_or(qd, failed)) {
                        stop = true;
                        break;
                    }
                    const float mt = fmaxf(fmaxf(red[hrow], red[G + hrow]),
                                           fmaxf(red[2 * G + hrow], red[3 * G + hrow]));
                    if (i == 0 || mt - m_run > 8.f) {
                        // (a head with no valid score yet keeps the finite floor
                        // -FLT_MAX: its scores minus the max are -inf, p = 0)
                        const float mn = fmaxf(fmaxf(m_run, mt), -FLT_MAX);
                        alpha = (i == 0) ? 0.f : exp2f(m_run - mn);
                        m_run = mn;
                        raised = i > 0;
                    }
                }
                float lsum = 0.f;
#pragma unroll
                for (int j = 0; j < C::TP; ++j) {
                    const float pv = ex2_approx(x[j] - m_run);
                    lsum += pv;
                    x[j] = pv;
                }
                l_run = l_run * alpha + lsum;
                // the P columns and O are free once the previous tile's P V is
                // done
                if (kt > 0 &&
                    !swait(bar0 + 8 * (C::PV_DONE + ((kt - 1) & 1)), ((kt - 1) >> 1) & 1))
                    failed = true;
                // V of this tile must have landed before its invalid rows are
                // zeroed (0 * a stale value must stay 0); warp (part, quarter)
                // takes the part's rows 8 * quarter .. + 8, each row's 16 chunks
                // over four lanes
                if (!swait(bar0 + 8 * (C::V_FULL + stage), (kt / C::SV) & 1)) failed = true;
                {
                    const int rr = 8 * qd + (lane >> 2);
                    if (!((vm >> rr) & 1u)) {
                        unsigned char* vrow = smem + C::OFF_V + stage * C::TILE + (c0 + rr) * 128;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int ch = (lane & 3) * 4 + k;   // half ch / 8, chunk ch % 8
                            *reinterpret_cast<uint4*>(vrow + (ch >> 3) * C::HALF + (ch & 7) * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                // P of the part's tokens as bf16 hi, then lo, two tokens per
                // column (the first in the low half): columns P_COL + 16 * part
                // and P_COL + 64 + 16 * part (in two halves of 16 tokens: fewer
                // registers live at once)
                const uint32_t sbuf = trow + C::P_COL;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float a = x[16 * hf + 2 * c], b = x[16 * hf + 2 * c + 1];
                        hi[c] = pack_bf16x2(a, b);
                        const float ha = __uint_as_float(hi[c] << 16);
                        const float hb = __uint_as_float(hi[c] & 0xffff0000u);
                        lo[c] = pack_bf16x2(a - ha, b - hb);
                    }
                    tmem_st8(sbuf + c0 / 2 + 8 * hf, hi);
                    tmem_st8(sbuf + 64 + c0 / 2 + 8 * hf, lo);
                }
                if (raised) {
                    // O (this piece's earlier tiles) by the same factor: the
                    // part's 32 of the row's 128 head-dim columns
                    tc_fence_after();
                    uint32_t v[C::TP];
                    tmem_ld_cols<C::TP>(trow + C::O_COL + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < C::TP; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
                    tmem_st_cols<C::TP>(trow + C::O_COL + c0, v);
                }
                tmem_wait_st();
                // one arrival per warp, after all its lanes' writes
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar0 + 8 * (C::P_FULL + (kt & 1)));
            }
            if (stop) break;

            // ---- piece epilogue: the four parts' sums, the O row, output ----
            if (!swait(bar0 + 8 * (C::PV_DONE + ((kt - 1) & 1)), ((kt - 1) >> 1) & 1))
                failed = true;
            // (every part has read the last tile's maxima before the sums
            // replace them)
            if (quarter_bar_or(qd, failed)) {
                stop = true;
                break;
            }
            red[part * G + hrow] = l_run;
            quarter_bar(qd);
            const float L = (red[hrow] + red[G + hrow]) + (red[2 * G + hrow] + red[3 * G + hrow]);
            __syncwarp();
            tc_fence_after();
            {
                uint32_t v[C::TP];
                tmem_ld_cols<C::TP>(trow + C::O_COL + c0, v);
                tmem_wait_ld();
                if (!own) {
                } else if (it.whole) {
                    const float inv = L > 0.f ? 1.f / L : 0.f;
                    const long long head0 = (long long)it.b * p.H + it.hbase;
                    float4* o4 = reinterpret_cast<float4*>(p.out + (head0 + hrow) * 128 + c0);
#pragma unroll
                    for (int j = 0; j < C::TP / 4; ++j)
                        o4[j] = make_float4(__uint_as_float(v[4 * j]) * inv,
                                            __uint_as_float(v[4 * j + 1]) * inv,
                                            __uint_as_float(v[4 * j + 2]) * inv,
                                            __uint_as_float(v[4 * j + 3]) * inv);
                } else {
                    const long long slot =
                        ((long long)blockIdx.x * 2 + (it.first ? 0 : 1)) * G + hrow;
                    float4* o4 = reinterpret_cast<float4*>(p.part_o + slot * 128 + c0);
#pragma unroll
                    for (int j = 0; j < C::TP / 4; ++j)
                        o4[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                            __uint_as_float(v[4 * j + 2]),
                                            __uint_as_float(v[4 * j + 3]));
                    if (part == 0) {
                        p.part_ml[slot * 2 + 0] = m_run == -FLT_MAX ? -INFINITY : m_run;
                        p.part_ml[slot * 2 + 1] = L;
                    }
                }
            }
            tc_fence_before();
            // the next piece, and its first tile's block ids
            have = umma_walk_next<B, G>(p, w, it);
            if (have) part_blocks(it, 0, nb0, nb1);
        }
    } else {
        // ====================== softmax (warps SM_WARP0 .. SM_WARP0 + NSW - 1)
        // Warp w works on TMEM lane quarter w % 4 (token / head-dim rows
        // 32 * (w % 4) + lane) and on heads [h0, h0 + HG).
        // The head parts are independent (own barriers, heads, sums and
        // maxima); they meet only at P_FULL.
        constexpr int HG = C::HG;
        const int part = (warp - C::SM_WARP0) >> 2;
        const int qd = warp & 3;
        const int sp = ((warp - C::SM_WARP0) & 3) * 32 + lane;  // thread within the part, 0 .. 127
        const int h0 = part * HG;
        const int r = qd * 32 + lane;            // token of the tile (S) / head-dim element (O)
        const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
        unsigned char* pbuf = smem + C::OFF_P;
        if (C::PW > 2 * G && part == 0) {
            // the P buffer's zero columns (past the hi and lo heads, up to a
            // whole 64-column block) are written once
#pragma unroll
            for (int c8 = (2 * G) / 8; c8 < C::PW / 8; ++c8)
                *reinterpret_cast<uint4*>(pbuf + (c8 / 8) * C::HALF + sw128(r, c8 % 8)) =
                    make_uint4(0, 0, 0, 0);
        }
        int kt = 0;
        bool stop = false;
        // A failed wait only marks this thread; the softmax threads decide to
        // stop together at the next barrier reduction, so none is left waiting
        // at a named barrier the others have abandoned.
        bool failed = false;
        float lp[HG];  // this thread's share of the softmax denominators
        auto swait = [&](uint32_t bar, uint32_t parity) {
            return umma_wait(bar, parity, abort_all, p.status);
        };
        UWalk w;
        umma_walk_begin<B>(p, ctrl + C::SCHED_OFF, w);
        // the block id of this thread's token in a piece's first tile, loaded
        // one piece ahead (later tiles' ids are loaded a tile ahead)
        auto first_block = [&](const UItem& pc) {
            const int tok = pc.t0 + r;
            return (pc.ntiles > 0 && tok < pc.t1) ? ld_dep(p.bt + (long long)pc.b * p.maxb + tok / B)
                                                  : -1;
        };
        UItem it;
        bool have = umma_walk_next<B, G>(p, w, it);
        int blk0 = have ? first_block(it) : -1;
        while (!stop && have) {
            const long long head0 = (long long)it.b * p.H + it.hbase + h0;
            if (it.ntiles == 0) {  // empty context: output 0 (always a whole piece)
#pragma unroll
                for (int g = 0; g < HG; ++g) p.out[(head0 + g) * 128 + r] = 0.f;
                have = umma_walk_next<B, G>(p, w, it);
                blk0 = have ? first_block(it) : -1;
                continue;
            }
#pragma unroll
            for (int g = 0; g < HG; ++g) lp[g] = 0.f;
            // this thread's token's block id, a tile ahead: a token past the
            // context or in a bad block gets no weight (the producers skip the
            // same boxes)
            const int* bt_row = p.bt + (long long)it.b * p.maxb;
            auto tok_block = [&](int i) {
                const int tok = it.t0 + i * C::TT + r;
                return (i < it.ntiles && tok < it.t1) ? ld_dep(bt_row + tok / B) : -1;
            };
            int blk_next = blk0;
            for (int i = 0; i < it.ntiles; ++i, ++kt) {
                const int stage = kt % C::SV;  // V stage
                const int blk = blk_next;
                blk_next = tok_block(i + 1);
                const bool ok = swait(bar0 + 8 * (C::S_FULL + (kt & 1)), (kt >> 1) & 1);
                failed = failed || !ok;
                __syncwarp();
                tc_fence_after();
                const int tok = it.t0 + i * C::TT + r;
                const bool valid = tok < it.t1 && blk >= 0 && blk < p.num_blocks;
                // this thread's scaled scores (-inf for a token past the
                // context or in a bad block), read from the tile's S buffer
                // (which stays in place until every warp has written P)
                float x[HG];
                auto load_scores = [&]() {
                    uint32_t v[HG];
                    tmem_ld_cols<HG>(trow + (kt & 1) * G + h0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < HG; ++j)
                        x[j] = valid ? __uint_as_float(v[j]) * p.qscale : -INFINITY;
                };
                load_scores();
                // x becomes score - running max, the exponent of p unless the
                // max is raised (the running maxima are read from shared
                // memory: no thread of the part changes them before every
                // thread has passed this tile's vote, and registers are short)
                float dmax = -INFINITY;  // largest score - running max (NaN-free)
#pragma unroll
                for (int g = 0; g < HG; g += 4) {
                    const float4 m4 = *reinterpret_cast<const float4*>(m_sh + h0 + g);
                    const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        x[g + e] -= mv[e];
                        dmax = fmaxf(dmax, x[g + e]);
                    }
                }
                const bool need = i == 0 || dmax > 8.f;
                bool rescale = false;
                if (part_bar_or(part, need | failed)) {
                    // raise the running max to this tile's max (per head); the
                    // barrier that publishes the warps' maxima also decides
                    // whether the part stops.  The scores are read again (x
                    // holds them minus the old max, which may be the floor).
                    load_scores();
                    {
                        const float v = warp_scatter_reduce<HG, true>(x, lane);
                        if ((lane & (32 / HG - 1)) == 0) red[qd * G + h0 + lane / (32 / HG)] = v;
                    }
                    if (part_bar_or(part, failed)) {
                        stop = true;
                        break;
                    }
                    if (sp < HG) {
                        const int h = h0 + sp;
                        const float mt = fmaxf(fmaxf(red[h], red[G + h]),
                                               fmaxf(red[2 * G + h], red[3 * G + h]));
                        const float old = (i == 0) ? -INFINITY : m_sh[h];
                        const float mn = fmaxf(old, mt);
                        a_sh[h] = (old == -INFINITY) ? 0.f : exp2f(old - mn);
                        // (a head with no valid score yet keeps the finite
                        // floor -FLT_MAX: its scores minus the max are then
                        // -inf, and 2^-inf = 0, with no special case below)
                        m_sh[h] = fmaxf(mn, -FLT_MAX);
                    }
                    part_bar(part);
#pragma unroll
                    for (int g = 0; g < HG; ++g) lp[g] *= a_sh[h0 + g];
#pragma unroll
                    for (int g = 0; g < HG; g += 4) {
                        const float4 m4 = *reinterpret_cast<const float4*>(m_sh + h0 + g);
                        x[g] -= m4.x;
                        x[g + 1] -= m4.y;
                        x[g + 2] -= m4.z;
                        x[g + 3] -= m4.w;
                    }
                    // O (this piece's earlier tiles) is scaled by the same
                    // factors once P is written (the scores are dead there)
                    rescale = i > 0;
                }
                // p = 2^(score - m) for this thread's token and heads (a head
                // whose max is still the floor has only -inf scores: p = 0)
#pragma unroll
                for (int g = 0; g < HG; ++g) {
                    const float pv = ex2_approx(x[g]);
                    lp[g] += pv;
                    x[g] = pv;
                }
                // the one P buffer (and O) is free once the previous tile's P V
                // is done
                if (kt > 0 &&
                    !swait(bar0 + 8 * (C::PV_DONE + ((kt - 1) & 1)), ((kt - 1) >> 1) & 1))
                    failed = true;
                // V of this tile must have landed before its invalid rows are
                // zeroed (only the rows' own threads need it, but all wait so
                // that the tile's stage is in place before P is published)
                if (!swait(bar0 + 8 * (C::V_FULL + stage), (kt / C::SV) & 1))
                    failed = true;
                if (!valid && h0 == 0) {
                    // rows past the context (or of a bad block) hold stale or
                    // foreign values: zero V so that 0 * V stays 0.  The lanes
                    // of a shared-memory phase (rows r .. r + 7) start at
                    // different 16-byte columns, one bank group each; the loop
                    // stays rolled (unrolled, the eight column offsets were
                    // hoisted out of the tile loop into registers)
                    unsigned char* vrow = smem + C::OFF_V + stage * C::TILE + r * 128;
#pragma unroll 1
                    for (int j = 0; j < 8; ++j) {
                        const int col = j ^ (r & 7);
                        *reinterpret_cast<uint4*>(vrow + col * 16) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4*>(vrow + C::HALF + col * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                // P row (MN-major, 64-column blocks): hi heads, then lo heads
#pragma unroll
                for (int g8 = 0; g8 < HG; g8 += 8) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float a = x[g8 + 2 * j], b = x[g8 + 2 * j + 1];
                        hi[j] = pack_bf16x2(a, b);
                        const float ha = __uint_as_float(hi[j] << 16);
                        const float hb = __uint_as_float(hi[j] & 0xffff0000u);
                        lo[j] = pack_bf16x2(a - ha, b - hb);
                    }
                    const int nh = h0 + g8, nl = G + h0 + g8;  // element index in the row
                    *reinterpret_cast<uint4*>(pbuf + (nh >> 6) * C::HALF +
                                              sw128(r, (nh & 63) >> 3)) =
                        make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(pbuf + (nl >> 6) * C::HALF +
                                              sw128(r, (nl & 63) >> 3)) =
                        make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
                if (rescale) {
                    __syncwarp();
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 2 * HG; c += 8) {   // hi heads, then lo heads
                        uint32_t v[8];
                        const int hc = c % HG;
                        const uint32_t col = trow + C::O_COL + (c / HG) * G + h0 + hc;
                        tmem_ld_cols<8>(col, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            v[j] = __float_as_uint(__uint_as_float(v[j]) * a_sh[h0 + hc + j]);
                        tmem_st_cols<8>(col, v);
                    }
                    tmem_wait_st();
                }
                // one arrival per warp, after all its lanes' writes
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar0 + 8 * (C::P_FULL + (kt & 1)));
            }
            if (stop) break;
            // the next piece, and its first tile's block id (loaded while this
            // piece's output is finished)
            UItem nx;
            const bool have_nx = umma_walk_next<B, G>(p, w, nx);
            const int blk0_nx = have_nx ? first_block(nx) : -1;

            // ---- piece epilogue: denominators, O = O_hi + O_lo, output ----
            {
                const float v = warp_scatter_reduce<HG, false>(lp, lane);
                if ((lane & (32 / HG - 1)) == 0) red[qd * G + h0 + lane / (32 / HG)] = v;
            }
            if (!swait(bar0 + 8 * (C::PV_DONE + ((kt - 1) & 1)), ((kt - 1) >> 1) & 1))
                failed = true;
            if (part_bar_or(part, failed)) {
                stop = true;
                break;
            }
            if (sp < HG) {
                const int h = h0 + sp;
                const float L = (red[h] + red[G + h]) + (red[2 * G + h] + red[3 * G + h]);
                a_sh[h] = L;
                red[h] = L > 0.f ? 1.f / L : 0.f;  // one division per head
            }
            part_bar(part);
            __syncwarp();
            tc_fence_after();
            {
                uint32_t vh[HG], vl[HG];
                tmem_ld_cols<HG>(trow + C::O_COL + h0, vh);
                tmem_ld_cols<HG>(trow + C::O_COL + G + h0, vl);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < HG; ++g) {
                    const float o = __uint_as_float(vh[g]) + __uint_as_float(vl[g]);
                    const float L = a_sh[h0 + g];
                    if (it.whole) {
                        p.out[(head0 + g) * 128 + r] = o * red[h0 + g];
                    } else {
                        const long long slot =
                            ((long long)blockIdx.x * 2 + (it.first ? 0 : 1)) * G + h0 + g;
                        p.part_o[slot * 128 + r] = o;
                        if (r == 0) {
                            const float m = m_sh[h0 + g];
                            p.part_ml[slot * 2 + 0] = m == -FLT_MAX ? -INFINITY : m;
                            p.part_ml[slot * 2 + 1] = L;
                        }
                    }
                }
            }
            tc_fence_before();
            it = nx;
            have = have_nx;
            blk0 = blk0_nx;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace pa
