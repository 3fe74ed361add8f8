// Work items of the persistent forward kernels (bf16 and e4m3): decoding an item index
// into its sequence, key/value head, two query tiles and their key-tile ranges, and the
// order in which the persistent CTAs take the items.
#pragma once
#include "common.cuh"

namespace fa {
namespace {

constexpr int BN = 128;  // keys per KV tile

struct TileInfo {
    int s0;       // first query position of the tile
    int t0, t1;   // KV tile range [t0, t1)
    bool active;  // the tile holds at least one valid query row
};

// One work item: the two query tiles [2 blk P, 2 blk P + 2P) of key/value head g of a
// sequence (and one key split in split mode), numbered heaviest first: the key/value head
// (and batch) vary fastest, the query block slowest, latest (longest causal band) first.
// Key tiles are `bn` keys long (BN unless the kernel takes shorter ones).
struct FwdItem {
    SeqView sv;
    Band band;
    int g, split;
    TileInfo ti[2];
    int u0, u1;  // union key-tile range of the two tiles
    bool live;   // false for an idle block of a packed batch
    bool tail;   // a piece of a tail-split unit: its rows go to the partials
};

__device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, int idx, int bn = BN) {
    const Problem& p = a.p;
    FwdItem w;
    int seq, blk;
    w.split = 0;
    w.tail = false;
    if (p.cu_q && a.tokens) {
        // token tiles: query tile k of block blk holds packed rows [(2 blk + k) P, + P), whatever
        // sequences they belong to; key coordinates are packed rows too.  The key-tile ranges
        // follow from the rows' own bands (fwd_row_band), so they are left empty here.
        w.g = idx % p.h_kv;
        blk = a.n_blocks - 1 - idx / p.h_kv;  // later tokens first
        w.sv = SeqView{0, 0, p.T_q, 0, p.T_k, 0};
        w.band = Band{0, p.left, p.right, p.T_k};
        w.u0 = w.u1 = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            w.ti[k].s0 = (2 * blk + k) * p.P;
            w.ti[k].active = w.ti[k].s0 < p.T_q;
            w.ti[k].t0 = w.ti[k].t1 = 0;
        }
        w.live = blk * 2 * p.P < p.T_q;
        return w;
    }
    if (a.tail_k > 1 && idx >= a.tail_item0) {
        // tail split (dense, unit-major): the last units' items, each cut into tail_k key
        // ranges, numbered unit by unit after the whole items
        const int t = idx - a.tail_item0;
        const int per_unit = a.n_blocks * a.tail_k;
        const int unit = a.tail_item0 / a.n_blocks + t / per_unit;
        const int x = t % per_unit;
        w.g = unit % p.h_kv;
        seq = unit / p.h_kv;
        w.split = x % a.tail_k;
        blk = a.n_blocks - 1 - x / a.tail_k;
        w.tail = true;
    } else if (p.cu_q) {
        w.g = idx % p.h_kv;
        const int bs = 2 * p.P;
        blk = idx / p.h_kv;
        seq = owner_sequence(p.cu_q, p.B, blk, bs);
        blk -= p.cu_q[seq] / bs + seq;
    } else {
        const int hb = p.h_kv * p.B;
        const int per_unit = a.n_blocks * a.n_splits;
        const int unit = a.unit_major ? idx / per_unit : idx % hb;
        const int x = a.unit_major ? idx % per_unit : idx / hb;
        w.g = unit % p.h_kv;
        seq = unit / p.h_kv;
        w.split = x % a.n_splits;
        blk = a.n_blocks - 1 - x / a.n_splits;
    }
    w.sv = seq_view(p, seq);
    w.band = Band{w.sv.nk - w.sv.nq, p.left, p.right, w.sv.nk};
    w.u0 = 0x7fffffff;
    w.u1 = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        w.ti[k].s0 = (2 * blk + k) * p.P;
        w.ti[k].active = w.ti[k].s0 < w.sv.nq;
        const int i1 = min(w.ti[k].s0 + p.P, w.sv.nq) - 1;
        if (w.ti[k].active) {
            kv_tile_range(w.band, w.ti[k].s0, i1, bn, w.ti[k].t0, w.ti[k].t1);
            if (a.n_splits > 1 || w.tail) {
                const int st = w.tail ? a.tail_split_tiles : a.split_tiles;
                w.ti[k].t0 = max(w.ti[k].t0, w.split * st);
                w.ti[k].t1 = min(w.ti[k].t1, (w.split + 1) * st);
                if (w.ti[k].t1 < w.ti[k].t0) w.ti[k].t1 = w.ti[k].t0;
            }
        } else {
            w.ti[k].t0 = w.ti[k].t1 = 0;
        }
        if (w.ti[k].t1 > w.ti[k].t0) {
            w.u0 = min(w.u0, w.ti[k].t0);
            w.u1 = max(w.u1, w.ti[k].t1);
        }
    }
    if (w.u1 == 0) w.u0 = 0;
    w.live = blk * 2 * p.P < w.sv.nq;
    return w;
}

// Allowed keys of row r (TMEM lane) of query tile k of item w, in the key coordinates of
// the item's key tiles (sequence-local, or packed rows in token mode): [jlo, jhi].  A row
// that holds no query (padding past P G rows, past the sequence or its used length) gets
// jlo = kNoRow; a query with no allowed key gets jlo = kNoKeys; both get jhi = -1.
constexpr int kNoRow = 0x7fffffff;
constexpr int kNoKeys = 0x7ffffffe;
__device__ __forceinline__ void fwd_row_band(const FwdArgs& a, const FwdItem& w, int k, int r, int& jlo, int& jhi) {
    const Problem& p = a.p;
    jlo = kNoRow;
    jhi = -1;
    if (!w.ti[k].active || r >= p.P * p.G) return;
    const int i = w.ti[k].s0 + r / p.G;
    int lo, hi;
    if (p.cu_q && a.tokens) {
        if (i >= p.T_q) return;
        const SeqView sv = seq_view(p, row_sequence(p.cu_q, p.B, i));
        const int il = i - sv.q0;
        if (il >= sv.nq) return;
        const Band bd{sv.nk - sv.nq, p.left, p.right, sv.nk};
        lo = sv.k0 + bd.lo(il);
        hi = sv.k0 + bd.hi(il);
    } else {
        if (i >= w.sv.nq) return;
        lo = w.band.lo(i);
        hi = w.band.hi(i);
    }
    if (hi < lo) {
        jlo = kNoKeys;
        return;
    }
    jlo = lo;
    jhi = hi;
}

// The persistent loop's items: a plain grid stride (idx = c, c + G, c + 2G, ...), or with
// `snake` rounds that alternate direction across the grid (c, 2G - 1 - c, 2G + c, ...,
// strides 2G - 1 - 2c and 1 + 2c in turn).  Under a causal mask the dense items come
// heaviest first, so the CTA that takes the heaviest item of one round takes the lightest
// of the next, which evens out the CTAs' totals that a plain stride leaves skewed toward
// the low CTA indices.  The loop advances with step' = 2G - step.
__device__ __forceinline__ int first_step(int snake) {
    return snake ? 2 * ((int)gridDim.x - (int)blockIdx.x) - 1 : (int)gridDim.x;
}

}  // namespace
}  // namespace fa
