// Device-side helpers shared by the attention kernels: mask bands, packed-row
// bookkeeping and the packed-batch block numbering.
#pragma once
#include "kernels.h"
#include "ptx.cuh"

namespace fa {

// Allowed key interval [lo(i), hi(i)] of query position i in a sequence of nq queries
// and nk keys, bottom-right aligned (off = nk - nq).  A causal call arrives here with
// right = 0, so the causal mask is the right edge of the window.
struct Band {
    int off, left, right, nk;
    __device__ __forceinline__ int lo(int i) const { return left >= 0 ? max(0, i + off - left) : 0; }
    __device__ __forceinline__ int hi(int i) const {
        return right >= 0 ? min(nk - 1, i + off + right) : nk - 1;
    }
};

// Range [t0, t1) of `bn`-key tiles that intersect the band of query positions
// [i0, i1] (inclusive); empty (t0 == t1) when no key is allowed.
__device__ __forceinline__ void kv_tile_range(const Band& bd, int i0, int i1, int bn, int& t0, int& t1) {
    int jlo = bd.lo(i0);
    int jhi = bd.hi(i1);
    if (bd.nk <= 0 || jhi < jlo || i1 < i0) {
        t0 = t1 = 0;
        return;
    }
    t0 = jlo / bn;
    t1 = jhi / bn + 1;
}

// Packed-batch block numbering: sequence s owns blocks starting at cu[s] / bs + s, so a
// sequence of n tokens has at least ceil(n / bs) blocks and an empty one costs a single
// idle block.  Returns the sequence that owns block g (binary search over the offsets).
__device__ __forceinline__ int owner_sequence(const int32_t* cu, int nseq, int g, int bs) {
    int lo = 0, hi = nseq - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cu[mid] / bs + mid <= g)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Largest sequence s in [0, nseq) with cu[s] <= row: the sequence that holds packed row
// `row` (empty sequences at the same offset come before it).
__device__ __forceinline__ int row_sequence(const int32_t* cu, int nseq, int row) {
    int lo = 0, hi = nseq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= row)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Banded work order over hb (batch, key/value head) units of per_unit items each: the
// units form n_bands bands of near-equal size (the first hb % n_bands bands one unit
// larger), taken one after the other; inside a band the unit varies fastest, so the items
// running at one time share few units' data in L2.  Gives the unit of item idx and the
// item's index x within its unit.  n_bands = 1 is the plain unit-fastest order.
__device__ __forceinline__ void band_order(int idx, int hb, int n_bands, int per_unit, int& unit, int& x) {
    const int base = hb / n_bands, big = hb % n_bands;  // band sizes base + 1 (first big), base
    const int big_items = big * (base + 1) * per_unit;
    int ub, unit0, r;
    if (idx < big_items) {
        ub = base + 1;
        const int band = idx / (ub * per_unit);
        r = idx - band * ub * per_unit;
        unit0 = band * ub;
    } else {
        ub = base;
        const int y = idx - big_items;
        const int band = y / (ub * per_unit);
        r = y - band * ub * per_unit;
        unit0 = big * (base + 1) + band * ub;
    }
    unit = unit0 + r % ub;
    x = r / ub;
}

// Global view of one sequence's rows.
struct SeqView {
    int b;        // batch index (dense) or sequence index (packed)
    int q0, nq;   // first token row of the sequence and its query count
    int k0, nk;   // first key row and key count
    int tma_b;    // 4th TMA coordinate: batch index (dense) or 0 (packed)
};

__device__ __forceinline__ SeqView seq_view(const Problem& p, int b) {
    SeqView v;
    v.b = b;
    if (p.cu_q) {
        v.q0 = p.cu_q[b];
        v.nq = p.cu_q[b + 1] - v.q0;
        v.k0 = p.cu_k[b];
        v.nk = p.cu_k[b + 1] - v.k0;
        v.tma_b = 0;
    } else {
        v.q0 = 0;
        v.nq = p.s_q;
        v.k0 = 0;
        v.nk = p.s_kv;
        v.tma_b = b;
    }
    // a slot filled only up to seqused_q[b] / seqused_k[b]: the rest of the slot takes no part
    if (p.seqused_q) v.nq = min(v.nq, max(0, p.seqused_q[b]));
    if (p.seqused_k) v.nk = min(v.nk, max(0, p.seqused_k[b]));
    return v;
}

// Tensor-map coordinates of the key tile that starts at key j (a multiple of the tile
// size) of sequence sv: the key row and the outer (batch or page) coordinate.  A paged
// cache keeps key j in row j % page_size of page block_table[b][j / page_size]; page_size
// is a multiple of every key tile, so a tile never straddles two pages.
__device__ __forceinline__ void kv_tile_coord(const Problem& p, const SeqView& sv, int j, int& row, int& outer) {
    if (p.block_table) {
        outer = p.block_table[(long)sv.b * p.max_blocks + j / p.page_size];
        row = j % p.page_size;
    } else {
        row = sv.k0 + j;
        outer = sv.tma_b;
    }
}

// Index of (sequence b, local row i, head h) in the LSE output.
__device__ __forceinline__ long lse_index(const Problem& p, const SeqView& sv, int i, int h) {
    if (p.cu_q) return (long)h * p.T_q + sv.q0 + i;
    return ((long)sv.b * p.h_q + h) * p.s_q + i;
}

// Token row (global) of local row i.
__device__ __forceinline__ long token_row(const Problem& p, const SeqView& sv, int i) {
    return p.cu_q ? (long)sv.q0 + i : (long)sv.b * p.s_q + i;
}

__device__ __forceinline__ long key_row(const Problem& p, const SeqView& sv, int j) {
    return p.cu_q ? (long)sv.k0 + j : (long)sv.b * p.s_kv + j;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace fa
