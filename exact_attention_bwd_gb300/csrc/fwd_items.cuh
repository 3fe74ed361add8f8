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
struct FwdItem {
    SeqView sv;
    Band band;
    int g, split;
    TileInfo ti[2];
    int u0, u1;  // union key-tile range of the two tiles
    bool live;   // false for an idle block of a packed batch
};

__device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, int idx) {
    const Problem& p = a.p;
    FwdItem w;
    int seq, blk;
    w.split = 0;
    if (p.cu_q) {
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
            kv_tile_range(w.band, w.ti[k].s0, i1, BN, w.ti[k].t0, w.ti[k].t1);
            if (a.n_splits > 1) {
                w.ti[k].t0 = max(w.ti[k].t0, w.split * a.split_tiles);
                w.ti[k].t1 = min(w.ti[k].t1, (w.split + 1) * a.split_tiles);
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
