// pa_schedule.cuh -- equal shares of a decode call's work for persistent CTAs.
//
// The unit of work is TU tokens (the tcgen05 kernel: one 128-token tile) of
// one (sequence b, KV head) pair; a context of n tokens has max(1, ceil(n /
// TU)) units (an empty one still owes its zero output).  A group served as
// nchunks head chunks splits the grid into nchunks groups of CTAs (CTA j serves
// chunk j % nchunks): every group takes the same ranges below over the same
// units, so sibling CTAs j, j + 1, ... stream the same K/V tiles side by side
// and all but the first find them in L2.  Head group g = kv head * nchunks +
// chunk.  Every pair is charged
// OV more units for the fixed cost of starting and finishing a piece of it,
// placed before its real units and doing no work.  Units are ordered by b, then
// KV head, then position, and CTA j of a group of the persistent grid takes the
// contiguous range [ceil(j T / grid), ceil((j + 1) T / grid)) of the T units
// (grid: CTAs per group, <= T):
// every CTA gets the same share of the work, whatever the mix of lengths.  A
// range covers whole pairs, except that its first and last piece may be parts
// of one that neighbouring CTAs share; those write unnormalised partials into
// the CTA's two slots (first piece slot 0, last slot 1) and the combine kernel
// merges them, told where by the descriptor the piece holding unit 0 writes
// ({first CTA, pieces, slot of the first piece}: piece k came from CTA first +
// k * nchunks, and only the first piece can be a CTA's second).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// One piece: units [u, u + units) of pair (b, g), tokens [t0, t1).
struct SPiece {
    int b, g, kvh, hc, hbase, n, c, u, units, t0, t1, ntiles;
    long long gpos;          // global index of the piece's first unit
    bool bad_len, whole, first;
};

template <int TU>
__device__ __forceinline__ int sched_units(int n, int maxtok) {
    return (n <= 0 || n > maxtok) ? 1 : (int)(((long long)n + TU - 1) / TU);
}

// Units (real + charged) of the pairs of sequences b0 + 8 lane + k, k < 8.
template <int B, int TU, int OV>
__device__ __forceinline__ void sched_pair_units(const DecodeParams& p, int b0, int lane,
                                                 int (&cu)[8]) {
    int nv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int b = b0 + 8 * lane + k;
        nv[k] = b < p.batch ? ld_dep(p.lens + b) : 0;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
        cu[k] = b0 + 8 * lane + k < p.batch ? OV + sched_units<TU>(nv[k], p.maxb * B) : 0;
}

// Computes this CTA's range (warp-wide; lane 0 stores it in `sched`, 48 bytes,
// 8-byte aligned): [0] T, [8] grid (min(gridDim, T)), [16] first unit, [24]
// unit count, [32] its b, [36] its g, [40] its offset within the pair.  A
// batch of up to 256 sequences takes one round of loads (8 per lane).
template <int B, int TU, int OV>
__device__ __forceinline__ void sched_compute(const DecodeParams& p, unsigned char* sched,
                                              int lane) {
    const long long Gq = p.Hkv;
    int cu[8];
    long long T = 0;
    for (int b0 = 0; b0 < p.batch; b0 += 256) {
        sched_pair_units<B, TU, OV>(p, b0, lane, cu);
#pragma unroll
        for (int k = 0; k < 8; ++k) T += cu[k];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) T += __shfl_xor_sync(kFullMask, T, off);
    T *= Gq;
    const long long grid = min((long long)(gridDim.x / p.nchunks), T);
    const long long j = blockIdx.x / p.nchunks;
    long long lo = 0, cnt = 0;
    int b_sel = 0, g_sel = 0, o_sel = 0;
    if (j < grid) {
        lo = (j * T + grid - 1) / grid;
        cnt = ((j + 1) * T + grid - 1) / grid - lo;
        long long P = 0;  // units before sequence b0
        for (int b0 = 0; b0 < p.batch; b0 += 256) {
            if (p.batch > 256) sched_pair_units<B, TU, OV>(p, b0, lane, cu);
            long long mine = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) mine += cu[k];
            mine *= Gq;
            long long incl = mine;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const long long v = __shfl_up_sync(kFullMask, incl, off);
                if (lane >= off) incl += v;
            }
            const unsigned hit =
                __ballot_sync(kFullMask, mine > 0 && P + incl - mine <= lo && lo < P + incl);
            if (hit) {
                const int f = __ffs(hit) - 1;
                if (lane == f) {
                    long long pos = P + incl - mine;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const long long pc = (long long)cu[k] * Gq;
                        if (cu[k] > 0 && lo < pos + pc) {
                            const long long off = lo - pos;
                            b_sel = b0 + 8 * lane + k;
                            g_sel = (int)(off / cu[k]);
                            o_sel = (int)(off % cu[k]);
                            break;
                        }
                        pos += pc;
                    }
                }
                b_sel = __shfl_sync(kFullMask, b_sel, f);
                g_sel = __shfl_sync(kFullMask, g_sel, f);
                o_sel = __shfl_sync(kFullMask, o_sel, f);
                break;
            }
            P += __shfl_sync(kFullMask, incl, 31);
        }
    }
    if (lane == 0) {
        long long* s64 = reinterpret_cast<long long*>(sched);
        int* s32 = reinterpret_cast<int*>(sched + 32);
        s64[0] = T;
        s64[1] = grid;
        s64[2] = lo;
        s64[3] = cnt;
        s32[0] = b_sel;
        s32[1] = g_sel;
        s32[2] = o_sel;
    }
}

// Walks the pieces of this CTA's range.  Every role walks it the same way; the
// length of the next sequence is loaded one sequence ahead (under a full HBM
// stream a dependent global load costs microseconds).
struct SWalk {
    int b, g, o, n, c, n_next;  // g: KV head; o: offset within the pair, charged units first
    bool bad, emitted;
    long long gpos, left;
    const long long* sched;  // T, grid, first unit (read where needed: registers are short)
};

template <int B, int TU>
__device__ __forceinline__ void sched_walk_seq(const DecodeParams& p, SWalk& w, int n_raw) {
    const int maxtok = p.maxb * B;
    w.bad = n_raw < 0 || n_raw > maxtok;
    w.n = w.bad ? 0 : n_raw;
    w.c = sched_units<TU>(w.n, maxtok);
    w.n_next = w.b + 1 < p.batch ? ld_dep(p.lens + w.b + 1) : 0;
}

template <int B, int TU>
__device__ __forceinline__ void sched_walk_begin(const DecodeParams& p,
                                                 const unsigned char* sched, SWalk& w) {
    const long long* s64 = reinterpret_cast<const long long*>(sched);
    const int* s32 = reinterpret_cast<const int*>(sched + 32);
    w.sched = s64;
    w.left = s64[3];
    w.gpos = s64[2];
    w.b = s32[0];
    w.g = s32[1];
    w.o = s32[2];
    w.emitted = false;
    if (w.left > 0) sched_walk_seq<B, TU>(p, w, ld_dep(p.lens + w.b));
}

template <int B, int TU, int OV, int G>
__device__ __forceinline__ bool sched_walk_next(const DecodeParams& p, SWalk& w, SPiece& it) {
    if (w.left <= 0) return false;
    if (w.o < OV) {  // the pair's charged units: nothing to do
        const long long skip = min((long long)(OV - w.o), w.left);
        w.o += (int)skip;
        w.gpos += skip;
        w.left -= skip;
        if (w.left <= 0) return false;
    }
    const int u = w.o - OV;
    const int units = (int)min((long long)(w.c - u), w.left);
    it.b = w.b;
    it.kvh = w.g;
    it.hc = (int)(blockIdx.x % p.nchunks);
    it.g = w.g * p.nchunks + it.hc;
    it.hbase = it.kvh * p.gsize + it.hc * G;
    it.n = w.n;
    it.c = w.c;
    it.u = u;
    it.units = units;
    it.gpos = w.gpos;
    it.bad_len = w.bad;
    it.whole = u == 0 && units == w.c;
    it.first = !w.emitted;
    w.emitted = true;
    it.t0 = (int)min((long long)u * TU, (long long)w.n);
    it.t1 = (int)min((long long)(u + units) * TU, (long long)w.n);
    it.ntiles = (it.t1 - it.t0 + TU - 1) / TU;
    w.left -= units;
    w.gpos += units;
    w.o += units;
    if (w.o == OV + w.c) {
        w.o = 0;
        if (++w.g == p.Hkv) {
            w.g = 0;
            ++w.b;
            if (w.left > 0) sched_walk_seq<B, TU>(p, w, w.n_next);
        }
    }
    return true;
}

// Pieces of a pair cut at CTA ranges: this CTA .. the owner of its last unit
// (within the CTA's group).
__device__ __forceinline__ int sched_pieces(const DecodeParams& p, const SPiece& it,
                                            const SWalk& w) {
    return it.whole ? 1
                    : (int)((it.gpos + it.c - 1) * w.sched[1] / w.sched[0] -
                            blockIdx.x / p.nchunks + 1);
}

}  // namespace pa
