// Forward attention on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
//
// One CTA owns two 128-row query tiles of one key/value head.  A tile's rows are
// "packed": the G query heads that share the key/value head are interleaved, row
// r = (position s0 + r / G, head g*G + r % G), so one pass over K/V serves all of them
// (grouped-query heads; vllm-project/flash-attention README, flash_attn_func docstring).
//
// Warp roles (384 threads):
//   warp 0       TMA producer: Q tiles once, then K and V tiles through a STAGES-deep ring
//   warp 1       MMA issuer (one thread): S_k = Q_k K^T into TMEM, O_k += P_k V with P_k
//                read back from TMEM
//   warp 2       owns the TMEM allocation
//   warp 3       tile scheduler: decodes this CTA's work items ahead of the other roles into
//                a small ring in shared memory (the item, each row's allowed key interval),
//                so that no role spends its own latency on the decode
//   warps 4..7   softmax of tile 0, warps 8..11 softmax of tile 1: each thread owns one
//                row (one TMEM lane); exp2-based online softmax with lazy rescaling
//
// The online softmax follows the recurrence of the "Flash Attention Tutorial" README
// (GitHub search results page, sections 3 to 5): a running max m and running sum l per
// row, with the accumulated output rescaled when the max moves.  Here the output stays
// un-normalised in TMEM and is divided by l once at the end, and the running max is only
// moved when it grows by more than 2^8 (the stale max keeps every exponential below 256,
// and the final division uses the same max, so the result is unchanged).
//
// Key tiles that lie wholly outside a tile's causal / sliding-window band are skipped
// (fa4-jax PyPI page, "Native two-sided sliding windows"); only tiles that cut the band
// edge evaluate the mask per element.
//
// Scheduling is persistent: one CTA per SM walks the work items (a key/value head's two
// query tiles, and a key range in split mode) in heaviest-first order with a grid stride
// (alternating direction from round to round under a causal mask, see first_step);
// a packed batch's items are found by binary search over its offsets (dew-flash-attn PyPI
// page, "Packed sequences"), and idle items cost only their decode.  When the queries and
// keys are packed alike (cu_seqlens_q and cu_seqlens_k the same array) the query tiles run
// over the packed token axis instead: a tile holds P consecutive tokens, which may belong
// to several short sequences, each row masked to its own sequence's band, so a batch of
// short sequences costs only its tokens rather than a tile per sequence.  Barrier phases carry
// over from item to item, so the next item's Q load and first S = Q K^T overlap the
// previous item's epilogue; two barriers hand the shared resources over: q_empty (the
// previous item's S MMAs, which read the Q tiles, have completed) and o_free[k] (the
// epilogue has read O_k out of tensor memory before the next P V overwrites it).
#include "fwd_items.cuh"
#include "trace.cuh"

namespace fa {
namespace {

constexpr int kThreadsFwd = 384;
#ifndef FA_FWD_EXP_POLY_PAIRS
#define FA_FWD_EXP_POLY_PAIRS 0
#endif
// of every 4 column pairs of an unmasked tile, this many take the polynomial exp2
constexpr int kExpPolyPairs = FA_FWD_EXP_POLY_PAIRS;

// KT keys per key tile: 128, or 64 at d = 64 for narrow bands (sliding windows), where an
// item sees only a few key tiles and its chain of waits, not the tensor pipe, sets the pace.
// With 64-key tiles the tensor memory of a CTA halves to 256 columns and its shared memory
// to about 100 KB, so two CTAs share an SM and twice as many query tiles are in flight.
template <int D, int KT>
struct FwdCfg {
    static_assert(KT == 128 || (KT == 64 && D == 64), "64-key tiles only at d = 64");
    static constexpr int KCH = D / 64;                  // 64-column chunks of a row
    static constexpr int TILE_BYTES = 128 * D * 2;      // one Q tile (128 rows)
    static constexpr int CHUNK_BYTES = 128 * 128;       // one [128 rows][64 cols] chunk of Q
    static constexpr int KV_BYTES = KT * D * 2;         // one K / V tile (KT rows)
    static constexpr int KV_CHUNK = KT * 128;           // one [KT rows][64 cols] chunk of K / V
    static constexpr int STAGES = (D == 64) ? 4 : 2;
    static constexpr int TMEM_COLS = KT == 128 ? 512 : 256;
    static constexpr int CTAS_PER_SM = KT == 128 ? 1 : 2;
    // TMEM columns: S_k at KT k (P_k is written over its first KT / 2), O_k at 2 KT + OW k
    static constexpr int OW = KT == 128 ? 128 : D;
    __host__ __device__ static constexpr uint32_t s_col(int k) { return (uint32_t)(KT * k); }
    __host__ __device__ static constexpr uint32_t o_col(int k) { return (uint32_t)(2 * KT + OW * k); }
    // registers per thread after setmaxnreg: producer / MMA / TMEM owner / scheduler group,
    // and the two softmax groups; 128 REG_LOW + 256 REG_HIGH stays within what the CTA is
    // launched with (checked before every launch)
    static constexpr int REG_LOW = KT == 128 ? 56 : 48;
    static constexpr int REG_HIGH = KT == 128 ? 224 : 96;
};

// One decoded work item, as the scheduler warp hands it to the other roles.
struct ItemInfo {
    int idx, end;       // item index; end = 1: no more items for this CTA
    int g, split, b;    // key/value head, key split, batch or sequence
    int tail;           // 1: a tail-split piece (rows to the partials from tail_row0 on)
    int q0, k0, tma_b;  // first query / key row of the sequence, outer TMA coordinate
    int u0, u1;         // union key-tile range of the two tiles (u1 <= u0: none)
    int s0[2], t0[2], t1[2];  // first query position and key-tile range of each tile
};
constexpr int kItemSlots = 3;
// arrivals that free an item slot: producer, MMA issuer and the eight softmax warps
constexpr int kItemReaders = 10;

template <int D, int KT>
struct __align__(1024) FwdSmem {
    using C = FwdCfg<D, KT>;
    uint8_t q[2][C::TILE_BYTES];
    uint8_t k[C::STAGES][C::KV_BYTES];
    uint8_t v[C::STAGES][C::KV_BYTES];
    uint64_t q_full;
    uint64_t k_full[C::STAGES], k_empty[C::STAGES];
    uint64_t v_full[C::STAGES], v_empty[C::STAGES];
    uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
    uint64_t q_empty;
    uint64_t drain;
    uint64_t item_full[kItemSlots], item_empty[kItemSlots];
    ItemInfo item[kItemSlots];
    int2 band[kItemSlots][2][128];  // (jlo, jhi) of every row of both query tiles
    uint32_t tmem_base;
    int abort_flag;
};

template <int D, bool F16, int KT>
__global__ void __launch_bounds__(kThreadsFwd, FwdCfg<D, KT>::CTAS_PER_SM)
    fwd_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
               const __grid_constant__ CUtensorMap tmv) {
    using C = FwdCfg<D, KT>;
    extern __shared__ uint8_t smem_raw[];
    FwdSmem<D, KT>& s =
        *reinterpret_cast<FwdSmem<D, KT>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Problem& p = a.p;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // an earlier CTA of this launch gave up: do not start
    if (a.status && *reinterpret_cast<volatile int*>(a.status) != 0) return;

    // ---------------- setup ----------------
    Abort ab{&s.abort_flag, a.status, p.wait_ns};
    if (tid == 0) {
        s.abort_flag = 0;
        mbar_init(&s.q_full, 1);
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&s.k_full[i], 1);
            mbar_init(&s.k_empty[i], 1);
            mbar_init(&s.v_full[i], 1);
            mbar_init(&s.v_empty[i], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s.s_full[k], 1);
            mbar_init(&s.p_full[k], 4);  // one arrive per softmax warp
            mbar_init(&s.o_full[k], 1);
            mbar_init(&s.o_free[k], 4);  // one arrive per softmax warp
        }
        mbar_init(&s.q_empty, 1);
        mbar_init(&s.drain, 1);
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(&s.item_full[i], 1);
            mbar_init(&s.item_empty[i], kItemReaders);
        }
        fence_mbar_init();
    }
    if (p.P * p.G < 128) {
        // rows past P*G of a Q tile are never written by TMA: zero them once
        for (int k = 0; k < 2; ++k)
            for (int c = 0; c < C::KCH; ++c)
                for (int x = p.P * p.G * 128 + tid * 16; x < 128 * 128; x += kThreadsFwd * 16)
                    *reinterpret_cast<uint4*>(&s.q[k][c * C::CHUNK_BYTES + x]) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == 2) {
        tmem_alloc(&s.tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    // registers: 384 x 168 at launch (one CTA per SM; 384 x 80 with two); the producer/MMA
    // group hands part of its share to the two softmax groups (128 x 56 + 256 x 224 = 64512;
    // 128 x 48 + 256 x 96 = 30720).  The change is made at the top of each warp group's
    // branch so the register allocator sees it on every path.
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" :: "n"(C::REG_LOW) : "memory");
    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            Tracer tr;
            tr.init(a.trace, 0);
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            const uint32_t qbox = (uint32_t)(p.P * p.G) * 128u;  // bytes of one 64-col Q box
            int gt = 0, n_q = 0, k_issued = 0, v_issued = 0;    // key tiles, Q loads, copies issued
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int slot = n % kItemSlots;
                if (!(ok = mbar_wait(&s.item_full[slot], (n / kItemSlots) & 1, ab))) break;
                const ItemInfo& it = s.item[slot];
                const int end = it.end, idx = it.idx, g = it.g, u0 = it.u0, u1 = it.u1;
                const SeqView sv{it.b, it.q0, 0, it.k0, 0, it.tma_b};
                const int qr0 = it.q0 + it.s0[0], qr1 = it.q0 + it.s0[1];
                const bool on0 = it.t1[0] > it.t0[0], on1 = it.t1[1] > it.t0[1];
                mbar_arrive(&s.item_empty[slot]);
                if (end) break;
                if (u1 <= u0) continue;
                tr.item(idx);
                // the previous item's Q tiles are free once its S MMAs have completed
                if (n_q > 0 && !(ok = twait(tr, kBQEmpty, &s.q_empty, (n_q - 1) & 1, ab))) break;
                mbar_expect_tx(&s.q_full, qbox * C::KCH * ((on0 ? 1u : 0u) + (on1 ? 1u : 0u)));
                for (int c = 0; c < C::KCH; ++c) {
                    if (on0) tma_load_4d(&s.q[0][c * C::CHUNK_BYTES], &tmq, &s.q_full, c * 64, g * p.G, qr0, sv.tma_b);
                    if (on1) tma_load_4d(&s.q[1][c * C::CHUNK_BYTES], &tmq, &s.q_full, c * 64, g * p.G, qr1, sv.tma_b);
                }
                ++n_q;
                for (int j = u0; j < u1; ++j, ++gt) {
                    const int st = gt % C::STAGES;
                    const uint32_t ph = (gt / C::STAGES) & 1;
                    int krow, kouter;
                    kv_tile_coord(p, sv, j * KT, krow, kouter);
                    if (!(ok = twait(tr, kBKEmpty, &s.k_empty[st], ph ^ 1, ab))) break;
                    mbar_expect_tx(&s.k_full[st], C::KV_BYTES);
                    for (int c = 0; c < C::KCH; ++c)
                        tma_load_4d(&s.k[st][c * C::KV_CHUNK], &tmk, &s.k_full[st], c * 64, g, krow, kouter);
                    ++k_issued;
                    if (!(ok = twait(tr, kBVEmpty, &s.v_empty[st], ph ^ 1, ab))) break;
                    mbar_expect_tx(&s.v_full[st], C::KV_BYTES);
                    for (int c = 0; c < C::KCH; ++c)
                        tma_load_4d(&s.v[st][c * C::KV_CHUNK], &tmv, &s.v_full[st], c * 64, g, krow, kouter);
                    ++v_issued;
                }
            }
            // wait for every copy still in flight before the CTA may exit
            for (int back = 1; back <= C::STAGES; ++back) {
                if (k_issued - back >= 0) {
                    const int i2 = k_issued - back;
                    mbar_wait_quiet(&s.k_full[i2 % C::STAGES], (i2 / C::STAGES) & 1);
                }
                if (v_issued - back >= 0) {
                    const int i2 = v_issued - back;
                    mbar_wait_quiet(&s.v_full[i2 % C::STAGES], (i2 / C::STAGES) & 1);
                }
            }
            if (n_q > 0) mbar_wait_quiet(&s.q_full, (n_q - 1) & 1);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        // Everything the issue path touches lives in registers (no per-tile arrays indexed
        // at run time), so consecutive MMAs go out back to back.
        if (lane == 0) {
            Tracer tr;
            tr.init(a.trace, 1);
            constexpr uint32_t idS = idesc_16(128, KT, false, false, F16);
            constexpr uint32_t idO = idesc_16(128, D, false, true, F16);
            constexpr uint32_t kStageStep = (uint32_t)C::KV_BYTES >> 4;  // descriptor units per stage
            // a descriptor's start-address field is addr >> 4 in its low bits, so stepping
            // through a tile is a plain add to a base descriptor (no carry: addr < 256 KB)
            const uint64_t qd0 = sdesc_sw128(smem_u32(s.q[0]), 16, 1024);
            const uint64_t qd1 = sdesc_sw128(smem_u32(s.q[1]), 16, 1024);
            const uint64_t kd_base = sdesc_sw128(smem_u32(s.k[0]), 16, 1024);
            const uint64_t vd_base = sdesc_sw128(smem_u32(s.v[0]), C::KV_CHUNK, 1024);
            auto issue_s = [&](uint64_t qd, uint32_t scol, uint64_t kd) {
                if constexpr (D == 128) mma_ss_kk16_x8(tmem + scol, qd, kd, idS, 0u);
                else mma_ss_kk16_x4(tmem + scol, qd, kd, idS, 0u);
            };
            auto issue_pv = [&](uint32_t ocol, uint32_t pcol, uint64_t vd, uint32_t acc0) {
                if constexpr (KT == 128) mma_ts_lin_mn_x8(tmem + ocol, tmem + pcol, vd, idO, acc0);
                else mma_ts_lin_mn_x4(tmem + ocol, tmem + pcol, vd, idO, acc0);
            };
            uint32_t pc0 = 0, pc1 = 0;  // P tiles consumed per query tile
            uint32_t oc0 = 0, oc1 = 0;  // O tiles completed per query tile (o_full commits)
            int gt = 0, n_q = 0;        // key tiles, items consumed
            bool ok = true;
            for (int n = 0; ok; ++n) {
                // the item's key-tile ranges are all the issue loop needs
                const int slot = n % kItemSlots;
                if (!(ok = mbar_wait(&s.item_full[slot], (n / kItemSlots) & 1, ab))) break;
                const ItemInfo& itm = s.item[slot];
                const int end = itm.end, idx = itm.idx;
                const int ta0 = itm.t0[0], ta1 = itm.t1[0], tb0 = itm.t0[1], tb1 = itm.t1[1];
                const int u0 = itm.u0, u1 = itm.u1;
                mbar_arrive(&s.item_empty[slot]);
                if (end) break;
                if (u1 <= u0) continue;
                tr.item(idx);
                ok = twait(tr, kBQFull, &s.q_full, n_q & 1, ab);
                ++n_q;
                tc_fence_after();
                {
                    const int st0 = gt % C::STAGES;
                    if (ok && (ok = twait(tr, kBKFull, &s.k_full[st0], (gt / C::STAGES) & 1, ab))) {
                        // prologue: S_k for the first KV tile (the S columns held the previous
                        // item's last P, read by P V MMAs issued earlier)
                        tc_fence_after();
                        const uint64_t kd0 = kd_base + (uint64_t)(st0 * kStageStep);
                        if (u0 >= ta0 && u0 < ta1) {
                            issue_s(qd0, C::s_col(0), kd0);
                            tc_commit(&s.s_full[0]);
                        }
                        if (u0 >= tb0 && u0 < tb1) {
                            issue_s(qd1, C::s_col(1), kd0);
                            tc_commit(&s.s_full[1]);
                        }
                        tc_commit(&s.k_empty[st0]);
                        if (u1 - u0 == 1) tc_commit(&s.q_empty);  // the item's last S
                    }
                }
                int it = gt;
                for (int j = u0; ok && j < u1; ++j, ++it) {
                    const int st = it % C::STAGES;
                    const uint32_t ph = (it / C::STAGES) & 1;
                    const int st1 = (it + 1) % C::STAGES;
                    const uint32_t ph1 = ((it + 1) / C::STAGES) & 1;
                    const uint64_t vd = vd_base + (uint64_t)(st * kStageStep);
                    const uint64_t kd1 = kd_base + (uint64_t)(st1 * kStageStep);
                    const bool next = j + 1 < u1;
                    bool k_ready = false;
                    ok = twait(tr, kBVFull, &s.v_full[st], ph, ab);
                    tc_fence_after();
                    // tile 0: O_0 += P_0 V_j, then S_0 for the next key tile
                    if (ok && j >= ta0 && j < ta1) {
                        ok = twait(tr, kBPFull, &s.p_full[0], pc0 & 1, ab);
                        ++pc0;
                        // the first P V of the item overwrites O_0: the previous item's
                        // epilogue must have read it
                        if (ok && j == ta0 && oc0 > 0) ok = twait(tr, kBOFree, &s.o_free[0], (oc0 - 1) & 1, ab);
                        tc_fence_after();
                        if (ok) {
                            issue_pv(C::o_col(0), C::s_col(0), vd, j > ta0 ? 1u : 0u);
                            if (j == ta1 - 1) {
                                tc_commit(&s.o_full[0]);
                                ++oc0;
                            }
                        }
                    }
                    if (ok && next && j + 1 >= ta0 && j + 1 < ta1) {
                        ok = twait(tr, kBKFull, &s.k_full[st1], ph1, ab);
                        tc_fence_after();
                        k_ready = true;
                        if (ok) {
                            issue_s(qd0, C::s_col(0), kd1);
                            tc_commit(&s.s_full[0]);
                        }
                    }
                    // tile 1
                    if (ok && j >= tb0 && j < tb1) {
                        ok = twait(tr, kBPFull, &s.p_full[1], pc1 & 1, ab);
                        ++pc1;
                        if (ok && j == tb0 && oc1 > 0) ok = twait(tr, kBOFree, &s.o_free[1], (oc1 - 1) & 1, ab);
                        tc_fence_after();
                        if (ok) {
                            issue_pv(C::o_col(1), C::s_col(1), vd, j > tb0 ? 1u : 0u);
                            if (j == tb1 - 1) {
                                tc_commit(&s.o_full[1]);
                                ++oc1;
                            }
                        }
                    }
                    if (ok && next && j + 1 >= tb0 && j + 1 < tb1) {
                        if (!k_ready) {
                            ok = twait(tr, kBKFull, &s.k_full[st1], ph1, ab);
                            tc_fence_after();
                            k_ready = true;
                        }
                        if (ok) {
                            issue_s(qd1, C::s_col(1), kd1);
                            tc_commit(&s.s_full[1]);
                        }
                    }
                    if (!ok) break;
                    // the last S of the item has been issued: the Q tiles are free when it
                    // completes, so the next item's Q load overlaps this item's last P V
                    if (j + 2 == u1) tc_commit(&s.q_empty);
                    tc_commit(&s.v_empty[st]);
                    if (next) {
                        // the next K tile always feeds an S of this CTA (the union of two bands is
                        // contiguous); wait for it here if neither tile did
                        if (!k_ready) ok = mbar_wait(&s.k_full[st1], ph1, ab);
                        if (ok) tc_commit(&s.k_empty[st1]);
                    }
                }
                gt += u1 - u0;
            }
            // let every issued MMA finish before the CTA tears down
            tc_commit(&s.drain);
            mbar_wait_quiet(&s.drain, 0);
        }
    } else if (warp == 3) {
        // ================= tile scheduler =================
        // Walks the CTA's items (a grid stride, alternating direction under `snake`; taking
        // items from a shared counter instead measured slower on most shapes) and hands each
        // live one to the other roles through the item ring: lane 0 writes the item, every
        // lane the allowed key interval of 8 of its 256 rows.  In token mode the key-tile ranges
        // come from those intervals (their hull), since a tile's rows may span sequences.
        int n = 0;
        bool ok = true;
        for (int idx = blockIdx.x, step = first_step(a.snake); idx < a.n_items;
             idx += step, step = 2 * (int)gridDim.x - step) {
            FwdItem w = fwd_item(a, idx, KT);
            if (!w.live) continue;
            const int slot = n % kItemSlots;
            if (n >= kItemSlots) {
                const bool wt = mbar_wait(&s.item_empty[slot], ((n / kItemSlots) - 1) & 1, ab);
                if (!__all_sync(0xffffffffu, wt)) {
                    ok = false;
                    break;
                }
            }
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                int lo_min = kNoRow, hi_max = -1;
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
                    const int r = lane + 32 * m;
                    int jlo, jhi;
                    fwd_row_band(a, w, k, r, jlo, jhi);
                    s.band[slot][k][r] = make_int2(jlo, jhi);
                    if (jlo <= jhi) {
                        lo_min = min(lo_min, jlo);
                        hi_max = max(hi_max, jhi);
                    }
                }
                if (a.tokens) {
                    lo_min = __reduce_min_sync(0xffffffffu, lo_min);
                    hi_max = __reduce_max_sync(0xffffffffu, hi_max);
                    w.ti[k].t0 = lo_min <= hi_max ? lo_min / KT : 0;
                    w.ti[k].t1 = lo_min <= hi_max ? hi_max / KT + 1 : 0;
                }
            }
            if (a.tokens) {
                w.u0 = 0x7fffffff;
                w.u1 = 0;
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (w.ti[k].t1 > w.ti[k].t0) {
                        w.u0 = min(w.u0, w.ti[k].t0);
                        w.u1 = max(w.u1, w.ti[k].t1);
                    }
                if (w.u1 == 0) w.u0 = 0;
            }
            if (lane == 0) {
                ItemInfo& it = s.item[slot];
                it.idx = idx;
                it.end = 0;
                it.g = w.g;
                it.split = w.split;
                it.tail = w.tail ? 1 : 0;
                it.b = w.sv.b;
                it.q0 = w.sv.q0;
                it.k0 = w.sv.k0;
                it.tma_b = w.sv.tma_b;
                it.u0 = w.u0;
                it.u1 = w.u1;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    it.s0[k] = w.ti[k].s0;
                    it.t0[k] = w.ti[k].t0;
                    it.t1[k] = w.ti[k].t1;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.item_full[slot]);
            ++n;
        }
        if (ok) {
            // the end marker
            const int slot = n % kItemSlots;
            bool wt = true;
            if (n >= kItemSlots) wt = mbar_wait(&s.item_empty[slot], ((n / kItemSlots) - 1) & 1, ab);
            if (__all_sync(0xffffffffu, wt)) {
                if (lane == 0) s.item[slot].end = 1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.item_full[slot]);
            }
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" :: "n"(C::REG_HIGH) : "memory");
        // ================= softmax: one thread per row =================
        const int k = (warp - 4) >> 2;           // query tile
        const int r = ((warp & 3) << 5) | lane;  // row = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_base + C::s_col(k);
        const uint32_t tO = tmem + lane_base + C::o_col(k);
        const float c = p.scale_log2;
        uint32_t scount = 0, ocount = 0;  // S tiles and O tiles received (carried across items)
        bool ok = true;
        Tracer tr;
        tr.init((warp & 3) == 0 ? a.trace : nullptr, 2 + k);
        for (int n = 0; ok; ++n) {
        // the item comes decoded from the scheduler warp; only the loop bounds, the row's key
        // band and its sink stay live across the key loop, the epilogue reads the rest again
        // from the item slot (held until the epilogue is done)
        const int slot = n % kItemSlots;
        {
            const bool wt = mbar_wait(&s.item_full[slot], (n / kItemSlots) & 1, ab);
            if (!__all_sync(0xffffffffu, wt)) {
                ok = false;
                break;
            }
        }
        if (s.item[slot].end) break;
        tr.item(s.item[slot].idx);
        const int my_t0 = s.item[slot].t0[k], my_t1 = s.item[slot].t1[k];
        const int2 rb = s.band[slot][k][r];
        const int jlo = rb.x, jhi = rb.y;
        // the sink's logit, fetched now so that its latency hides behind the key loop
        float sink2 = 0.f;
        if (p.sinks && a.n_splits == 1 && jlo != kNoRow) sink2 = p.sinks[s.item[slot].g * p.G + r % p.G] * kLog2e;
        float m_used = -INFINITY, l = 0.f;
        for (int j = my_t0; j < my_t1; ++j) {
            const bool w = twait(tr, kBSFull, &s.s_full[k], scount & 1, ab);
            if (!__all_sync(0xffffffffu, w)) {
                ok = false;
                break;
            }
            ++scount;
            tc_fence_after();
            // one TMEM read of the whole S row (KT fp32 columns)
            const int j0 = j * KT;
            const bool edge = (j0 < jlo || j0 + KT - 1 > jhi);
            uint32_t sr[KT];
            if constexpr (KT == 128) tmem_ld_32x32b_x128(tS, sr);
            else tmem_ld_32x32b_x64(tS, sr);
            if (edge) {
                // the row's allowed columns [lo, hi] of this tile (a row without keys has
                // lo > KT - 1 and hi < 0) as a bit mask per 32-column chunk, applied without
                // branches: one bit test and one select per element
                const int lo = jlo - j0, hi = jhi - j0;
#pragma unroll
                for (int cb = 0; cb < KT; cb += 32) {
                    const int c0 = max(lo - cb, 0), c1 = min(hi - cb, 31);
                    const uint32_t keep = c0 > c1 ? 0u : (0xffffffffu >> (31 - c1)) & (0xffffffffu << c0);
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (!(keep & (1u << t))) sr[cb + t] = __float_as_uint(-INFINITY);
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < KT; cc += 4) {
                mx0 = max3(mx0, __uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1]));
                mx1 = max3(mx1, __uint_as_float(sr[cc + 2]), __uint_as_float(sr[cc + 3]));
            }
            const float m_new = fmaxf(m_used, fmaxf(mx0, mx1) * c);
            float alpha = 1.f;
            bool rescale = false;
            if (m_used == -INFINITY) {
                m_used = m_new;  // nothing accumulated yet (O is exactly 0)
            } else if (m_new > m_used + 8.f) {
                alpha = ex2(m_used - m_new);
                m_used = m_new;
                l *= alpha;
                rescale = true;
            }
            // O_k row *= alpha (warp-wide TMEM access; alpha = 1 on the other lanes); with
            // 64-key tiles after P is out of the registers (the softmax has fewer of them), the
            // P V that accumulates into O_k waits for p_full below
            auto rescale_o = [&]() {
#pragma unroll
                for (int cb = 0; cb < D; cb += 32) {
                    uint32_t orr[32];
                    tmem_ld_32x32b_x32(tO + cb, orr);
#pragma unroll
                    for (int t = 0; t < 32; ++t) orr[t] = __float_as_uint(__uint_as_float(orr[t]) * alpha);
                    tmem_st_32x32b_x32(tO + cb, orr);
                }
            };
            if (KT == 128 && __any_sync(0xffffffffu, rescale)) rescale_o();
            // P = exp2(S*c - m) as 16-bit pairs (the inputs' type), packed in place (slot cc/2 is already consumed).
            // On tiles without masked entries a fraction of the exponentials runs on the FMA
            // pipe (exp2_poly2) to share the load with the MUFU unit.
            const float base = (m_used == -INFINITY) ? 0.f : m_used;
            const bool poly_ok = !__any_sync(0xffffffffu, edge);
            const float2 c2 = make_float2(c, c), nb2 = make_float2(-base, -base);
            float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < KT; cc += 2) {
                float2 xv = __ffma2_rn(make_float2(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])), c2, nb2);
                float2 pv;
                if (kExpPolyPairs > 0 && ((cc >> 1) & 3) < kExpPolyPairs && poly_ok) {
                    xv.x = fmaxf(xv.x, -125.f);
                    xv.y = fmaxf(xv.y, -125.f);
                    pv = exp2_poly2(xv);
                } else {
                    pv = make_float2(ex2(xv.x), ex2(xv.y));
                }
                sum2 = __fadd2_rn(sum2, pv);
                sr[cc / 2] = pack16<F16>(pv.x, pv.y);
            }
            const float sum = sum2.x + sum2.y;
            if constexpr (KT == 128) tmem_st_32x32b_x64(tS, sr);
            else tmem_st_32x32b_x32(tS, sr);
            l += sum;
            if (KT == 64 && __any_sync(0xffffffffu, rescale)) rescale_o();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.p_full[k]);
            tr.mark(kMSoftmaxDone);
        }
        // ---------------- epilogue ----------------
        const ItemInfo& itm = s.item[slot];
        const SeqView sv{itm.b, itm.q0, 0, 0, 0, 0};
        const int g = itm.g, split = itm.split;
        const int i = itm.s0[k] + r / p.G;  // query position (a packed row in token mode)
        const int h = g * p.G + r % p.G;    // query head
        const bool row_valid = jlo != kNoRow;
        const bool has_o = my_t1 > my_t0;  // uniform over the warp group
        if (has_o && ok) {
            const bool wt = twait(tr, kBOFull, &s.o_full[k], ocount & 1, ab);
            ++ocount;
            ok = __all_sync(0xffffffffu, wt);
            tc_fence_after();
        }
        const bool split_mode = a.n_splits > 1 || itm.tail;
        // 32-byte stores where the base allows (the rows, 128 or more bytes, keep the alignment)
        const bool o_al32 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;
        const bool part_al32 = (reinterpret_cast<uintptr_t>(a.o_part) & 31u) == 0;
        float oscale = 0.f, lse = -INFINITY;
        if (!split_mode && p.sinks && row_valid) {
            const float s2 = sink2;
            const float mf = fmaxf(m_used, s2);
            const float wgt = (m_used == -INFINITY) ? 0.f : ex2(m_used - mf);
            const float lt = l * wgt + ex2(s2 - mf);
            oscale = wgt / lt;
            lse = (mf + log2f(lt)) * kLn2;
        } else if (l > 0.f) {
            oscale = 1.f / l;
            lse = (m_used + log2f(l)) * kLn2;
        }
        // split-mode rows (dense only): all B h_q s_q rows, or (tail split) those from
        // tail_row0 on
        const long row_base = itm.tail ? a.tail_row0 : 0;
        const long nrows = (long)p.B * p.h_q * p.s_q - row_base;
        const long prow = ((long)sv.b * p.h_q + h) * p.s_q + i - row_base;
        if (row_valid) {
            if (!split_mode) {
                if (a.lse) a.lse[lse_index(p, sv, i, h)] = lse;
            } else {
                a.lse_part[(long)split * nrows + prow] = lse;
            }
        }
        if (has_o && ok) {
            // the whole O row into registers (warp-collective TMEM reads), then O_k is free for
            // the next item's P V while the row is scaled and stored; only valid rows store
            uint32_t orr[D];
            if constexpr (D == 128) tmem_ld_32x32b_x128(tO, orr);
            else tmem_ld_32x32b_x64(tO, orr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.o_free[k]);
            if (row_valid) {
                if (!split_mode) {
                    uint16_t* orow = a.o + (token_row(p, sv, i) * p.h_q + h) * D;
                    if (o_al32) {
                        // 32-byte stores (half the instructions; each row is 128 or 256 bytes)
#pragma unroll
                        for (int t = 0; t < D / 16; ++t) {
                            uint32_t wv[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                wv[u] = pack16<F16>(__uint_as_float(orr[16 * t + 2 * u]) * oscale,
                                                    __uint_as_float(orr[16 * t + 2 * u + 1]) * oscale);
                            st_global_v8(orow + 16 * t, wv);
                        }
                    } else {
#pragma unroll
                        for (int t = 0; t < D / 8; ++t) {
                            uint4 wv;
                            wv.x = pack16<F16>(__uint_as_float(orr[8 * t + 0]) * oscale, __uint_as_float(orr[8 * t + 1]) * oscale);
                            wv.y = pack16<F16>(__uint_as_float(orr[8 * t + 2]) * oscale, __uint_as_float(orr[8 * t + 3]) * oscale);
                            wv.z = pack16<F16>(__uint_as_float(orr[8 * t + 4]) * oscale, __uint_as_float(orr[8 * t + 5]) * oscale);
                            wv.w = pack16<F16>(__uint_as_float(orr[8 * t + 6]) * oscale, __uint_as_float(orr[8 * t + 7]) * oscale);
                            reinterpret_cast<uint4*>(orow)[t] = wv;
                        }
                    }
                } else {
                    float* op = a.o_part + ((long)split * nrows + prow) * D;
                    if (part_al32) {
#pragma unroll
                        for (int t = 0; t < D / 8; ++t) {
                            uint32_t wv[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) wv[u] = __float_as_uint(__uint_as_float(orr[8 * t + u]) * oscale);
                            st_global_v8(op + 8 * t, wv);
                        }
                    } else {
#pragma unroll
                        for (int t = 0; t < D / 4; ++t)
                            reinterpret_cast<float4*>(op)[t] =
                                make_float4(__uint_as_float(orr[4 * t]) * oscale, __uint_as_float(orr[4 * t + 1]) * oscale,
                                            __uint_as_float(orr[4 * t + 2]) * oscale, __uint_as_float(orr[4 * t + 3]) * oscale);
                    }
                }
            }
            tr.mark(kMEpilogueDone);
        } else if (row_valid) {
            if (!split_mode) {
                uint16_t* orow = a.o + (token_row(p, sv, i) * p.h_q + h) * D;
#pragma unroll
                for (int t = 0; t < D / 8; ++t) reinterpret_cast<uint4*>(orow)[t] = make_uint4(0, 0, 0, 0);
            } else {
                float* op = a.o_part + ((long)split * nrows + prow) * D;
#pragma unroll
                for (int t = 0; t < D / 4; ++t) reinterpret_cast<float4*>(op)[t] = make_float4(0, 0, 0, 0);
            }
        }
        // the item slot is read for the last time: hand it back to the scheduler
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.item_empty[slot]);
        }  // items
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace

template <int D, bool F16, int KT>
static cudaError_t launch_fwd_k(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t st) {
    using C = FwdCfg<D, KT>;
    const size_t smem = sizeof(FwdSmem<D, KT>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, F16, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // the warp groups' setmaxnreg shares must fit in the registers the CTA is launched with
    // (an increase beyond them would never be granted)
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, fwd_kernel<D, F16, KT>)) != cudaSuccess) return e;
    if (fa.numRegs * kThreadsFwd < 128 * C::REG_LOW + 256 * C::REG_HIGH) return cudaErrorLaunchOutOfResources;
    if (a.n_items <= 0 || a.n_ctas <= 0) return cudaSuccess;
    fwd_kernel<D, F16, KT><<<(unsigned)a.n_ctas, kThreadsFwd, smem, st>>>(a, tq, tk, tv);
    return cudaGetLastError();
}

template <int D, bool F16>
static cudaError_t launch_fwd_d(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t st) {
    if constexpr (D == 64)
        if (a.kt == 64) return launch_fwd_k<D, F16, 64>(a, tq, tk, tv, st);
    return launch_fwd_k<D, F16, 128>(a, tq, tk, tv, st);
}

cudaError_t launch_fwd(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t st) {
    const bool f16 = a.p.dtype == FA_DTYPE_F16;
    switch (a.p.d) {
        case 64: return f16 ? launch_fwd_d<64, true>(a, tq, tk, tv, st) : launch_fwd_d<64, false>(a, tq, tk, tv, st);
        case 128: return f16 ? launch_fwd_d<128, true>(a, tq, tk, tv, st) : launch_fwd_d<128, false>(a, tq, tk, tv, st);
        case 192:
        case 256: return launch_fwd256(a, tq, tk, tv, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
