// Backward attention on the 5th-generation tensor cores, sm_103a.
//
// The derivation is the one of the "Flash Attention Tutorial" README (GitHub search
// results page, section 6 "Flash Attention Backward Pass", "Key derivations"), with the
// softmax scale kept where the chain rule puts it:
//   P = exp(scale Q K^T - LSE)         recomputed from the saved per-row LSE
//   dV = P^T dO
//   D_i = rowsum(dO_i * O_i)           (preprocess kernel)
//   dS = P * (dO V^T - D)
//   dQ = scale dS K,   dK = scale dS^T Q
// The tiled loop is the tutorial's: the outer loop runs over key/value tiles (one CTA
// each, dK and dV accumulated on chip), the inner loop over the query tiles that can see
// the key tile, with dQ summed across key tiles.  Here the inner loop runs over packed
// query tiles that hold all G query heads of the key/value head, so the grouped-query
// reduction of dK and dV happens in the fp32 TMEM accumulators (fa4-jax PyPI page,
// Restrictions: GQA backward accumulates dK/dV in fp32).  dQ is accumulated in an fp32
// workspace with atomic adds and converted by the postprocess kernel.
//
// Main-kernel warp roles (d <= 128, 512 threads):
//   warp 0      TMA producer: K and V once, then Q_i and dO_i through a two-stage ring
//   warp 1      MMA issuer: S^T = K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q,
//               dQ_i (dQ^T_i = K^T dS^T at d = 128), all into TMEM
//   warp 2      owns the TMEM allocation
//   warps 4-11  two groups of 128: thread = key row; group c takes query columns
//               [64c, 64c+64): P^T = exp2(S^T * c - LSE2), dS^T = P^T (dP^T - D) into
//               shared memory
//   warps 12-15 drain dQ_i and reduce it into the workspace: d = 128 as dQ^T_i (thread =
//               column of d), d = 64 as dQ_i (thread = query row)
// d = 256 has its own kernel (bwd256_kernel below).
#include "common.cuh"
#include "trace.cuh"

namespace fa {
namespace {

constexpr int kThreadsBwd = 512;
constexpr int kRows = 128;

template <int D>
struct BwdCfg {
    static constexpr int KCH = D / 64;
    static constexpr int TILE = 128 * D * 2;     // Q / K / V / dO tile bytes
    static constexpr int CHUNK = 128 * 128;      // one [128 rows][64 cols] chunk
    static constexpr int TMEM_COLS = 512;
    // TMEM columns
    static constexpr uint32_t C_S = 0;           // S^T (fp32); P^T (16-bit) in [0, 32) and [64, 96)
    static constexpr uint32_t C_DP = 128;        // dP^T
    static constexpr uint32_t C_DV = 256;
    static constexpr uint32_t C_DK = 256 + D;
    static constexpr uint32_t C_DQ = (D == 128) ? 128 : 384;  // dQ^T_i (lanes = d, columns = query rows)
    static constexpr bool DQ_OVER_DP = (D == 128);             // dQ_i reuses the dP^T columns
    static constexpr bool DQ_T = (D == 128);                   // dQ computed transposed (lanes = d)
};

// The work-unit ring of the d <= 128 main kernel: slots, and the arrivals that free one
// (producer, MMA issuer, the eight compute warps and the four dQ warps).
constexpr int kUnitSlots = 4;
constexpr int kUnitReaders = 14;

template <int D>
struct __align__(1024) BwdSmem {
    uint8_t k[BwdCfg<D>::TILE];
    uint8_t v[BwdCfg<D>::TILE];
    uint8_t q[2][BwdCfg<D>::TILE];
    uint8_t dO[2][BwdCfg<D>::TILE];
    uint8_t dst[2][128 * 128];   // dS^T: [key row][query col], two 64-column chunks
    float stat[2][2][128];       // per Q stage: LSE * log2(e) and D of the tile's 128 rows
    uint64_t kv_full;
    uint64_t q_full[2], q_empty[2], do_full[2], do_empty[2];
    uint64_t s_full, dp_full, p_full, ds_full, ds_free, dq_full, dq_free, dkv_full, dkv_free, drain;
    uint64_t unit_full[kUnitSlots], unit_empty[kUnitSlots];
    int unit[kUnitSlots];  // work units handed out by the scheduler warp (-1: no more)
    uint32_t tmem_base;
    int abort_flag;
};

// First tiled-layout index of the query tiles of sequence `seq` (see the workspace
// layout in the planner): dense = seq * ceil(s_q / P), packed = cu_q[seq] / P + seq.
__device__ __forceinline__ int qtile_base(const Problem& p, int seq) {
    if (p.cu_q) return p.cu_q[seq] / p.P + seq;
    return seq * cdiv(p.s_q, p.P);
}

// Query tiles [qt0, qt1) whose positions have a band reaching key block `blk` of the
// sequence (qt0 == qt1 when no query sees the block).  Over the blocks that some query
// sees, both ends are non-decreasing in the block index.
__device__ __forceinline__ void block_qtiles(const Problem& p, const SeqView& sv, const Band& band, int blk, int& qt0,
                                             int& qt1) {
    const int j0 = blk * kRows;
    const int j1 = min(j0 + kRows, sv.nk) - 1;
    int i_lo = 0, i_hi = sv.nq - 1;
    if (p.right >= 0) i_lo = max(i_lo, j0 - band.off - p.right);
    if (p.left >= 0) i_hi = min(i_hi, j1 - band.off + p.left);
    qt0 = (i_hi >= i_lo) ? i_lo / p.P : 0;
    qt1 = (i_hi >= i_lo) ? i_hi / p.P + 1 : 0;
}

// Token mode: the packed query rows [qlo, qhi] whose band holds packed key row j (qlo > qhi
// when none: a key past the batch, past its sequence's used keys, or seen by no query).
__device__ __forceinline__ void token_key_queries(const Problem& p, int j, int& qlo, int& qhi) {
    qlo = 1;
    qhi = 0;
    if (j >= p.T_k) return;
    const SeqView sv = seq_view(p, row_sequence(p.cu_k, p.B, j));
    const int jl = j - sv.k0;
    if (jl >= sv.nk) return;
    const int off = sv.nk - sv.nq;
    const int i_min = p.right >= 0 ? max(0, jl - off - p.right) : 0;
    const int i_max = p.left >= 0 ? min(sv.nq - 1, jl - off + p.left) : sv.nq - 1;
    if (i_min > i_max) return;
    qlo = sv.q0 + i_min;
    qhi = sv.q0 + i_max;
}

// Token mode: the query tiles [qt0, qt1) (P packed rows each) that some key of the block
// [j0, j1] sees.  Within a sequence a key's first and last query rise with the key, and a
// later sequence's rows follow an earlier one's, so the first key's first query and the last
// key's last query bound the rest; when either key sees no query, its sequence's first (or
// last) row stands in.
__device__ __forceinline__ void token_block_qtiles(const Problem& p, int j0, int j1, int& qt0, int& qt1) {
    int a_lo, a_hi, b_lo, b_hi;
    token_key_queries(p, j0, a_lo, a_hi);
    token_key_queries(p, j1, b_lo, b_hi);
    const int qstart = a_lo <= a_hi ? a_lo : p.cu_q[row_sequence(p.cu_k, p.B, j0)];
    const int qend = b_lo <= b_hi ? b_hi : p.cu_q[row_sequence(p.cu_k, p.B, j1) + 1] - 1;
    qt0 = qend >= qstart ? qstart / p.P : 0;
    qt1 = qend >= qstart ? qend / p.P + 1 : 0;
}

// Deterministic dQ order.  Every query tile receives the contributions of the key blocks
// that see it in descending block order, each block's contribution complete before the
// next one starts, so the fp32 sums are formed in the same order on every run.  A key
// block's CTA walks its query tiles in ascending order; before adding into tile t it
// waits until the tile's counter shows every later block's contribution (one count per
// adding warp).  The launch puts a sequence's later blocks at lower CTA indices, so each
// CTA waits only on CTAs dispatched before it (and, run after run, on ones that are a
// step ahead of it: the later block reached tile t one query tile earlier).
struct DqOrder {
    int next = 0;  // next later key block to examine
    int n = 0;     // later blocks seen so far whose query tiles start at or before the tile
};

// Number of later key blocks whose contributions precede this block's in query tile t;
// t never decreases between calls (the cursor only moves forward).
__device__ __forceinline__ int dq_predecessors(const Problem& p, const SeqView& sv, const Band& band, DqOrder& o,
                                               int t) {
    while (o.next * kRows < sv.nk) {
        int a0, a1;
        block_qtiles(p, sv, band, o.next, a0, a1);
        if (a1 > a0) {
            if (a0 > t) break;  // later blocks start later still; each earlier one reaches t
            ++o.n;
        }
        ++o.next;
    }
    return o.n;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* ptr) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// Lane 0 waits until the counter reaches `need`; the warp learns the outcome.  Bounded
// like every other wait: false when the limit passes, the CTA gave up, or another CTA of
// the launch recorded a failure (its contributions may never come).
__device__ __forceinline__ bool dq_turn_wait(const int* cnt, int need, const Abort& ab) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0 && ld_acquire_gpu(cnt) < need) {
        const unsigned long long t0 = globaltimer();
        while (ld_acquire_gpu(cnt) < need) {
            if (ab.raised() || (ab.status && *reinterpret_cast<volatile int*>(ab.status) != 0)) {
                ab.raise(kStatusTimeout);
                ok = false;
                break;
            }
            if (globaltimer() - t0 > ab.limit) {
                ab.raise(kStatusTimeout);
                ok = false;
                break;
            }
        }
    }
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// After a warp's reductions into a tile: make them visible, then count the warp in.
__device__ __forceinline__ void dq_turn_done(int* cnt) {
    __threadfence();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) atomicAdd(cnt, 1);
}

// One key block of the d <= 128 backward: its (key/value head, sequence, block), the
// sequence view and band, its keys [j0, j1] and the query tiles [qt0, qt0 + nsteps) that
// see it.  Work unit idx is numbered as the grid was before the kernel became persistent:
// dense units in L2-sized bands (see band_order), packed blocks over cu_k, token blocks over
// the packed key axis; with the fixed dQ order a sequence's later blocks come first.
struct BwdBlock {
    int g, blk, seq, qt0, nsteps, tbase, j0, j1;
    SeqView sv;
    Band band;
    bool live;  // false: an idle block of a packed batch (nothing to compute or write)
};

// The n-th work unit this role takes from the scheduler's ring (-1: none left, or a failed
// wait, which also clears ok).  Every thread of a calling warp (or the single calling thread
// of the producer / MMA roles) reads the slot; lane 0 frees it.
template <class Smem>
__device__ __forceinline__ int take_unit(Smem& s, int n, const Abort& ab, bool& ok) {
    const int slot = n % kUnitSlots;
    const bool w = mbar_wait(&s.unit_full[slot], (n / kUnitSlots) & 1, ab);
    if (!__all_sync(__activemask(), w)) {
        ok = false;
        return -1;
    }
    const int idx = s.unit[slot];
    __syncwarp(__activemask());
    if ((threadIdx.x & 31) == 0) mbar_arrive(&s.unit_empty[slot]);
    return idx;
}

template <bool DET, bool TOK>
__device__ __forceinline__ BwdBlock bwd_block(const BwdArgs& a, int idx) {
    const Problem& p = a.p;
    BwdBlock b;
    if (TOK) {
        // token mode: key block blk holds packed key rows [128 blk, 128 blk + 128)
        b.g = idx % p.h_kv;
        b.blk = idx / p.h_kv;
        b.seq = 0;
    } else if (p.cu_q) {
        b.g = idx % p.h_kv;
        int blk = idx / p.h_kv;
        if (DET) blk = a.n_kvblocks - 1 - blk;
        b.seq = owner_sequence(p.cu_k, p.B, blk, kRows);
        b.blk = blk - (p.cu_k[b.seq] / kRows + b.seq);
    } else {
        int unit, blk;
        band_order(idx, p.h_kv * p.B, a.n_bands, a.n_kvblocks, unit, blk);
        b.g = unit % p.h_kv;
        b.seq = unit / p.h_kv;
        b.blk = DET ? a.n_kvblocks - 1 - blk : blk;
    }
    b.sv = TOK ? SeqView{0, 0, p.T_q, 0, p.T_k, 0} : seq_view(p, b.seq);
    b.j0 = b.blk * kRows;
    b.live = b.j0 < b.sv.nk;
    b.j1 = min(b.j0 + kRows, b.sv.nk) - 1;
    b.band = Band{b.sv.nk - b.sv.nq, p.left, p.right, b.sv.nk};
    int qt1 = 0;
    b.qt0 = 0;
    if (b.live) {
        if (TOK)
            token_block_qtiles(p, b.j0, b.j1, b.qt0, qt1);
        else
            block_qtiles(p, b.sv, b.band, b.blk, b.qt0, qt1);
    }
    b.nsteps = qt1 - b.qt0;
    b.tbase = TOK ? 0 : qtile_base(p, b.seq);
    return b;
}

template <int D, bool DET, bool F16, bool TOK>
__global__ void __launch_bounds__(kThreadsBwd, 1)
    bwd_main_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo) {
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the layout needs 1024-byte alignment (128-byte swizzle atoms) and fills the whole
    // 227 KB, so there is no room to realign by hand: refuse to run if the window is not
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0 && a.status) atomicCAS(a.status, 0, kStatusDeviceCheck);
        return;
    }
    BwdSmem<D>& s = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
    const Problem& p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // an earlier kernel or CTA of the call failed (a device check of the offsets, a
    // timeout): do not start, and read nothing the offsets point at
    if (a.status && *reinterpret_cast<volatile int*>(a.status) != 0) return;
    // token mode (TOK): key blocks and query tiles over the packed token axis; never with DET
    constexpr bool tokens = TOK;
    static_assert(!(DET && TOK), "the fixed dQ order uses blocks per sequence");
    // Persistent (a.persist): one CTA per SM, whose scheduler warp walks the work units with a
    // grid stride (units are numbered heaviest first, in L2-sized bands for dense batches)
    // and hands them to the other roles through a small ring.  Otherwise the launch has one
    // CTA per unit (unit = CTA index): always with the fixed dQ order, so that a CTA waits
    // only on CTAs dispatched before it, and for long causal dense problems, where one unit
    // per CTA measured faster (the hardware's dispatch of CTAs as SMs free up).  Every role keeps a running
    // count of the steps (query tiles) and blocks it has been through, so that the barrier
    // phases carry on from block to block; two barriers hand a block's resources to the next:
    // dkv_full (the block's last MMAs, which read K and V and finish dK and dV, have
    // completed: the next K/V may load) and dkv_free (the compute groups have read dK and
    // dV out of tensor memory: the next block's first dV / dK may overwrite them).
    const int n_units = a.n_units;

    Abort ab{&s.abort_flag, a.status, p.wait_ns};
    if (tid == 0) {
        s.abort_flag = 0;
        mbar_init(&s.kv_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.q_full[i], 1);
            mbar_init(&s.q_empty[i], 1);
            mbar_init(&s.do_full[i], 1);
            mbar_init(&s.do_empty[i], 1);
        }
        mbar_init(&s.s_full, 1);
        mbar_init(&s.dp_full, 1);
        mbar_init(&s.p_full, 256);
        mbar_init(&s.ds_full, 256);
        mbar_init(&s.ds_free, 1);
        mbar_init(&s.dq_full, 1);
        mbar_init(&s.dq_free, 128);  // the dQ group's threads
        mbar_init(&s.dkv_full, 1);
        mbar_init(&s.dkv_free, 256);  // the compute groups' threads
        mbar_init(&s.drain, 1);
        for (int i = 0; i < kUnitSlots; ++i) {
            mbar_init(&s.unit_full[i], 1);
            mbar_init(&s.unit_empty[i], kUnitReaders);
        }
        fence_mbar_init();
    }
    if (p.P * p.G < 128) {
        // rows past P*G of a query tile are never written by TMA: zero them once
        for (int st = 0; st < 2; ++st)
            for (int c = 0; c < C::KCH; ++c)
                for (int x = p.P * p.G * 128 + tid * 16; x < 128 * 128; x += kThreadsBwd * 16) {
                    *reinterpret_cast<uint4*>(&s.q[st][c * C::CHUNK + x]) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(&s.dO[st][c * C::CHUNK + x]) = make_uint4(0, 0, 0, 0);
                }
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

    // registers: 512 x 128 at launch, redistributed per warp group (the change is made at
    // the top of each group's branch): the two compute groups 160; d = 128: producer/MMA 48
    // and the dQ group, which holds a whole 128-row dQ^T column in registers, 144
    // (128*48 + 256*160 + 128*144 = 65536); d = 64 (a 64-column dQ row per thread): 64 and
    // 128.  Splits that leave a group short make it spill, which costs more than the
    // registers save.
    if (warp >= 12) {
        if constexpr (D == 128) asm volatile("setmaxnreg.inc.sync.aligned.u32 144;\n" ::: "memory");
        else asm volatile("setmaxnreg.dec.sync.aligned.u32 128;\n" ::: "memory");
        // ================= dQ group: drains dQ_i and reduces it into the workspace =================
        // d = 128: dQ^T_i (TMEM lane = column of d); d = 64: dQ_i (TMEM lane = query row of the
        // tile, 64 columns of d per row), drained here so the compute groups go on meanwhile
        const int tl = ((warp & 3) << 5) | lane;  // this thread's TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
        Tracer tr;
        tr.init(warp == 12 ? a.trace : nullptr, 3);
        int gs = 0;  // steps of earlier blocks
        bool ok = true;
        for (int n = 0; ok; ++n) {
            const int idx = take_unit(s, n, ab, ok);
            if (idx < 0) break;
            const BwdBlock bk = bwd_block<DET, TOK>(a, idx);
            if (bk.nsteps <= 0) continue;
            tr.item(idx);
            DqOrder order;
            order.next = bk.blk + 1;
            for (int it = 0; it < bk.nsteps; ++it) {
                const int i = gs + it;
                const int t = bk.qt0 + it;
                const long trow = ((long)bk.g * a.n_qtiles + bk.tbase + t) * 128;
                int need = 0;
                if constexpr (DET) need = 4 * dq_predecessors(p, bk.sv, bk.band, order, t);
                {
                    const bool w = twait(tr, kBDqFull, &s.dq_full, i & 1, ab);
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                }
                tc_fence_after();
                int* cnt = DET ? a.dq_count + (long)bk.g * a.n_qtiles + bk.tbase + t : nullptr;
                if constexpr (C::DQ_T) {
                    uint32_t qa[64], qb[64];
                    tmem_ld_32x32b_x64(tmem + lane_base + C::C_DQ, qa);
                    tmem_ld_32x32b_x64(tmem + lane_base + C::C_DQ + 64, qb);
                    // the columns are free as soon as they are in registers
                    tc_fence_before();
                    mbar_arrive(&s.dq_free);
                    if (DET && !dq_turn_wait(cnt, need, ab)) { ok = false; break; }
                    // for each query row the 32 lanes of a warp add to 32 consecutive floats
                    // (the accumulator lines are kept in L2 ahead of streamed data: each is added to
                    // by every key block that sees the tile)
                    float* acc = a.dq_acc + trow * D + tl;
                    const uint64_t keep = policy_evict_last();
#pragma unroll
                    for (int r = 0; r < 64; ++r) red_add_hint(acc + (long)r * D, __uint_as_float(qa[r]), keep);
#pragma unroll
                    for (int r = 0; r < 64; ++r) red_add_hint(acc + (long)(64 + r) * D, __uint_as_float(qb[r]), keep);
                } else {
                    uint32_t qv[D];
                    tmem_ld_32x32b_x64(tmem + lane_base + C::C_DQ, qv);
                    tc_fence_before();
                    mbar_arrive(&s.dq_free);
                    if (DET && !dq_turn_wait(cnt, need, ab)) { ok = false; break; }
                    float* acc = a.dq_acc + (trow + tl) * D;
                    const uint64_t keep = policy_evict_last();
#pragma unroll
                    for (int t4 = 0; t4 < D / 4; ++t4)
                        red_add4_hint(acc + 4 * t4, __uint_as_float(qv[4 * t4]), __uint_as_float(qv[4 * t4 + 1]),
                                      __uint_as_float(qv[4 * t4 + 2]), __uint_as_float(qv[4 * t4 + 3]), keep);
                }
                if constexpr (DET) dq_turn_done(cnt);
                tr.mark(kMDqReduced);
            }
            gs += bk.nsteps;
        }
    } else if (warp < 4) {
    if constexpr (D == 128) asm volatile("setmaxnreg.dec.sync.aligned.u32 48;\n" ::: "memory");
    else asm volatile("setmaxnreg.dec.sync.aligned.u32 64;\n" ::: "memory");
    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            Tracer tr;
            tr.init(a.trace, 0);
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            tma_prefetch_desc(&tmdo);
            const uint32_t tile_bytes = (uint32_t)(p.P * p.G) * 128u * C::KCH;  // one Q or dO tile
            const uint32_t qbytes = tile_bytes + 2 * 128 * 4;                       // Q plus LSE2, D rows
            int q_issued = 0, do_issued = 0, kv_issued = 0;  // copies issued (also the step / block counts)
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int idx = take_unit(s, n, ab, ok);
                if (idx < 0) break;
                const BwdBlock bk = bwd_block<DET, TOK>(a, idx);
                if (bk.nsteps <= 0) continue;
                tr.item(idx);
                for (int it = 0; it < bk.nsteps; ++it) {
                    const int i = q_issued;  // global step
                    const int st = i & 1;
                    const uint32_t ph = (i >> 1) & 1;
                    const int row = bk.sv.q0 + (bk.qt0 + it) * p.P;
                    if (!(ok = twait(tr, kBQEmpty, &s.q_empty[st], ph ^ 1, ab))) break;
                    mbar_expect_tx(&s.q_full[st], qbytes);
                    for (int c = 0; c < C::KCH; ++c)
                        tma_load_4d(s.q[st] + c * C::CHUNK, &tmq, &s.q_full[st], c * 64, bk.g * p.G, row, bk.sv.tma_b);
                    {
                        const long trow = ((long)bk.g * a.n_qtiles + bk.tbase + bk.qt0 + it) * 128;
                        bulk_load(s.stat[st][0], a.lse2_t + trow, 512, &s.q_full[st]);
                        bulk_load(s.stat[st][1], a.delta_t + trow, 512, &s.q_full[st]);
                    }
                    ++q_issued;
                    if (it == 0) {
                        // this block's K and V, once the previous block's last MMAs (which read
                        // them) have completed; the first Q went out before, as its ring slot
                        // frees while the previous block still runs
                        if (kv_issued > 0 && !(ok = twait(tr, kBDkvFull, &s.dkv_full, (kv_issued - 1) & 1, ab))) break;
                        mbar_expect_tx(&s.kv_full, 2 * C::TILE);
                        // a block's K and V are read once: at d = 128 they leave L2 first (measured
                        // faster there, slightly slower at d = 64)
                        const uint64_t once = policy_evict_first();
                        for (int c = 0; c < C::KCH; ++c) {
                            if constexpr (D == 128) {
                                tma_load_4d_hint(s.k + c * C::CHUNK, &tmk, &s.kv_full, c * 64, bk.g, bk.sv.k0 + bk.j0,
                                                 bk.sv.tma_b, once);
                                tma_load_4d_hint(s.v + c * C::CHUNK, &tmv, &s.kv_full, c * 64, bk.g, bk.sv.k0 + bk.j0,
                                                 bk.sv.tma_b, once);
                            } else {
                                tma_load_4d(s.k + c * C::CHUNK, &tmk, &s.kv_full, c * 64, bk.g, bk.sv.k0 + bk.j0, bk.sv.tma_b);
                                tma_load_4d(s.v + c * C::CHUNK, &tmv, &s.kv_full, c * 64, bk.g, bk.sv.k0 + bk.j0, bk.sv.tma_b);
                            }
                        }
                        ++kv_issued;
                    }
                    if (!(ok = twait(tr, kBDoEmpty, &s.do_empty[st], ph ^ 1, ab))) break;
                    mbar_expect_tx(&s.do_full[st], tile_bytes);
                    for (int c = 0; c < C::KCH; ++c)
                        tma_load_4d(s.dO[st] + c * C::CHUNK, &tmdo, &s.do_full[st], c * 64, bk.g * p.G, row, bk.sv.tma_b);
                    ++do_issued;
                }
            }
            // the copies still in flight: the latest phase of each ring stage and of K/V
            for (int back = 1; back <= 2; ++back) {
                if (q_issued - back >= 0) mbar_wait_quiet(&s.q_full[(q_issued - back) & 1], ((q_issued - back) >> 1) & 1);
                if (do_issued - back >= 0)
                    mbar_wait_quiet(&s.do_full[(do_issued - back) & 1], ((do_issued - back) >> 1) & 1);
            }
            if (kv_issued > 0) mbar_wait_quiet(&s.kv_full, (kv_issued - 1) & 1);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_16(128, 128, false, false, F16);  // S^T, dP^T: K-major both
            constexpr uint32_t id_dv = idesc_16(128, D, false, true, F16);    // A from TMEM, B MN-major
            constexpr uint32_t id_dk = idesc_16(128, D, false, true, F16);    // A K-major, B MN-major
            // dQ^T (M = d, N = query rows) when d = 128; dQ (M = query rows, N = d) when d = 64,
            // whose 64-row accumulator would need the M = 64 lane layout
            constexpr uint32_t id_dq = C::DQ_T ? idesc_16(128, 128, true, true, F16) : idesc_16(128, D, true, true, F16);
            const uint32_t ka = smem_u32(s.k), va = smem_u32(s.v);
            Tracer tr;
            tr.init(a.trace, 1);
            // each GEMM goes out as one MMA burst (ptx.cuh): base descriptors only, the step
            // offsets are immediates inside the asm block
            const uint64_t kd_k = sdesc_sw128(ka, 16, 1024), vd_k = sdesc_sw128(va, 16, 1024);
            const uint64_t kd_mn = sdesc_sw128(ka, C::CHUNK, 1024);
            const uint32_t sa = smem_u32(s.dst[0]);
            const uint64_t sd_k = sdesc_sw128(sa, 16, 1024), sd_mn = sdesc_sw128(sa, 128 * 128, 1024);
            auto issue_st = [&](int i) {  // S^T_i = K Q_i^T into the S^T columns
                const uint64_t qd = sdesc_sw128(smem_u32(s.q[i & 1]), 16, 1024);
                if constexpr (D == 128) mma_ss_kk16_x8(tmem + C::C_S, kd_k, qd, id_s, 0u);
                else mma_ss_kk16_x4(tmem + C::C_S, kd_k, qd, id_s, 0u);
                tc_commit(&s.s_full);
            };
            int gs = 0, nb = 0;  // steps and blocks of earlier blocks
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int idx = take_unit(s, n, ab, ok);
                if (idx < 0) break;
                const int nsteps = bwd_block<DET, TOK>(a, idx).nsteps;
                if (nsteps <= 0) continue;
                tr.item(idx);
                if (!(ok = twait(tr, kBKvFull, &s.kv_full, nb & 1, ab))) break;
                tc_fence_after();
                // issue order per step i:  dP^T_i, dV_i, S^T_{i+1}, dQ^T_i, dK_i  (S^T_0 first);
                // S^T_{i+1} goes before dQ^T_i / dK_i so that the next step's P^T overlaps them
                if (!(ok = twait(tr, kBQFull, &s.q_full[gs & 1], (gs >> 1) & 1, ab))) break;
                tc_fence_after();
                issue_st(gs);
                for (int it = 0; ok && it < nsteps; ++it) {
                    const int i = gs + it;  // global step
                    const int st = i & 1;
                    const uint32_t ph = (i >> 1) & 1;
                    const uint32_t par = i & 1;
                    const uint32_t qa = smem_u32(s.q[st]), da = smem_u32(s.dO[st]);
                    // dP^T = V dO_i^T (its columns held dQ^T_{i-1} when D == 128)
                    if (!(ok = twait(tr, kBDoFull, &s.do_full[st], ph, ab))) break;
                    if (C::DQ_OVER_DP && i > 0) {
                        if (!(ok = twait(tr, kBDqFree, &s.dq_free, par ^ 1, ab))) break;
                    }
                    tc_fence_after();
                    if constexpr (D == 128) mma_ss_kk16_x8(tmem + C::C_DP, vd_k, sdesc_sw128(da, 16, 1024), id_s, 0u);
                    else mma_ss_kk16_x4(tmem + C::C_DP, vd_k, sdesc_sw128(da, 16, 1024), id_s, 0u);
                    tc_commit(&s.dp_full);
                    // dV += P^T dO_i (query pairs of group c sit at columns 64c + 8k, k < 4); the
                    // block's first dV overwrites the accumulators, which the compute groups
                    // must have read out for the previous block
                    if (!(ok = twait(tr, kBPFull, &s.p_full, par, ab))) break;
                    if (it == 0 && nb > 0 && !(ok = twait(tr, kBDkvFree, &s.dkv_free, (nb - 1) & 1, ab))) break;
                    tc_fence_after();
                    mma_ts_p_mn_x8(tmem + C::C_DV, tmem + C::C_S, sdesc_sw128(da, C::CHUNK, 1024), id_dv, it > 0 ? 1u : 0u);
                    tc_commit(&s.do_empty[st]);
                    // S^T_{i+1}: its columns held P^T_i, read by dV_i issued just above
                    if (it + 1 < nsteps) {
                        if (!(ok = twait(tr, kBQFull, &s.q_full[st ^ 1], ((i + 1) >> 1) & 1, ab))) break;
                        tc_fence_after();
                        issue_st(i + 1);
                    }
                    // dQ^T_i = K^T dS^T, then dK += dS^T Q_i: dQ goes first so that its drain by the
                    // dQ warps (which frees the dP^T columns for the next step) overlaps dK
                    if (!(ok = twait(tr, kBDsFull, &s.ds_full, par, ab))) break;
                    if (!C::DQ_OVER_DP && i > 0) {
                        if (!(ok = twait(tr, kBDqFree, &s.dq_free, par ^ 1, ab))) break;
                    }
                    tc_fence_after();
                    if constexpr (C::DQ_T)  // dQ^T = K^T dS^T: A = K tile (MN-major), B = dS^T (MN-major)
                        mma_ss_mnmn_x8(tmem + C::C_DQ, kd_mn, sd_mn, id_dq, 0u);
                    else                    // dQ = dS K: A = dS (MN-major), B = K tile (MN-major)
                        mma_ss_mnmn_x8(tmem + C::C_DQ, sd_mn, kd_mn, id_dq, 0u);
                    tc_commit(&s.dq_full);
                    mma_ss_kmn16_x8(tmem + C::C_DK, sd_k, sdesc_sw128(qa, C::CHUNK, 1024), id_dk, it > 0 ? 1u : 0u);
                    tc_commit(&s.q_empty[st]);
                    tc_commit(&s.ds_free);
                }
                if (!ok) break;
                // dK and dV of the block are final, and K and V are read, once these complete
                tc_commit(&s.dkv_full);
                gs += nsteps;
                ++nb;
            }
            // let every issued MMA finish before the CTA tears down
            tc_commit(&s.drain);
            mbar_wait_quiet(&s.drain, 0);
        }
    } else if (warp == 3) {
        // ================= scheduler: hands out the work units =================
        if (lane == 0) {
            for (int n = 0;; ++n) {
                // a grid stride over the units (a launch with one CTA per unit takes one)
                const int idx = (int)blockIdx.x + n * (int)gridDim.x;
                const int slot = n % kUnitSlots;
                if (n >= kUnitSlots && !mbar_wait(&s.unit_empty[slot], ((n / kUnitSlots) - 1) & 1, ab)) break;
                s.unit[slot] = idx < n_units ? idx : -1;
                mbar_arrive(&s.unit_full[slot]);
                if (idx >= n_units) break;
            }
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 160;\n" ::: "memory");
        // ================= compute groups =================
        const int cg = (warp - 4) >> 2;            // column group
        const int wq = warp & 3;
        const bool dkv_al32 = ((reinterpret_cast<uintptr_t>(a.dk) | reinterpret_cast<uintptr_t>(a.dv)) & 31u) == 0;
        const int jr = (wq << 5) | lane;           // key row of this thread (TMEM lane)
        const uint32_t lane_base = (uint32_t)(wq << 5) << 16;
        const float c = p.scale_log2;
        bool ok = true;
        Tracer tr;
        tr.init(warp == 4 ? a.trace : nullptr, 2);
        int gs = 0, nb = 0;  // steps and blocks of earlier blocks
        for (int n = 0; ok; ++n) {
            const int idx = take_unit(s, n, ab, ok);
            if (idx < 0) break;
            const BwdBlock bk = bwd_block<DET, TOK>(a, idx);
            if (!bk.live) continue;  // an idle block of a packed batch writes nothing
            tr.item(idx);
            const int j = bk.j0 + jr;
            // token mode: this key's queries as packed rows (its own sequence's band)
            int tq_lo = 1, tq_hi = 0;
            if (tokens) token_key_queries(p, j, tq_lo, tq_hi);
            for (int it = 0; it < bk.nsteps; ++it) {
                const int i = gs + it;                  // global step
                const uint32_t par = i & 1;
                const int t = bk.qt0 + it;              // query tile within the sequence
                const int s0 = t * p.P;                 // its first query position
                const int st = i & 1;
                const float* lse2 = s.stat[st][0] + 64 * cg;
                const float* dlt = s.stat[st][1] + 64 * cg;
                // edge test: does the band cut this (query tile, key tile) pair?
                const int iq_first = s0, iq_last = min(s0 + p.P, bk.sv.nq) - 1;
                const bool interior =
                    !tokens && bk.j0 >= bk.band.lo(iq_last) && bk.j0 + kRows - 1 <= bk.band.hi(iq_first);
                // ---- P^T ----
                {
                    // the stage's LSE / D rows landed with Q_i (already complete by the time S^T is)
                    bool w = twait(tr, kBQFull, &s.q_full[st], (i >> 1) & 1, ab);
                    w = w && twait(tr, kBSFull, &s.s_full, par, ab);
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                }
                tc_fence_after();
                float pf[64];
                {
                    uint32_t sr[64];
                    tmem_ld_32x32b_x64(tmem + lane_base + C::C_S + 64 * cg, sr);
#pragma unroll
                    for (int cc = 0; cc < 64; cc += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(lse2 + cc);
                        pf[cc + 0] = ex2(fmaf(__uint_as_float(sr[cc + 0]), c, -l4.x));
                        pf[cc + 1] = ex2(fmaf(__uint_as_float(sr[cc + 1]), c, -l4.y));
                        pf[cc + 2] = ex2(fmaf(__uint_as_float(sr[cc + 2]), c, -l4.z));
                        pf[cc + 3] = ex2(fmaf(__uint_as_float(sr[cc + 3]), c, -l4.w));
                    }
                    if (!interior) {
                        // the query positions whose band holds key j form one interval
                        // [i_min, i_max] (lo and hi are monotone in the position); in this tile's
                        // packed columns (column = G (i - s0) + head) it is the column range
                        // [G (i_min - s0), G (i_max + 1 - s0)), taken relative to this group's
                        // first column
                        int c_lo, c_hi;
                        if constexpr (TOK) {
                            // the key's queries as packed rows (none: an empty column range)
                            c_lo = tq_lo > tq_hi ? 0 : (tq_lo - s0) * p.G - 64 * cg;
                            c_hi = tq_lo > tq_hi ? 0 : (tq_hi + 1 - s0) * p.G - 64 * cg;
                        } else {
                            const int i_min = p.right >= 0 ? j - bk.band.off - p.right : 0;
                            const int i_max =
                                j >= bk.sv.nk ? i_min - 1 : (p.left >= 0 ? j - bk.band.off + p.left : bk.sv.nq - 1);
                            c_lo = (i_min - s0) * p.G - 64 * cg;
                            c_hi = (i_max + 1 - s0) * p.G - 64 * cg;
                        }
#pragma unroll
                        for (int cc = 0; cc < 64; ++cc)
                            if (cc < c_lo || cc >= c_hi) pf[cc] = 0.f;
                    }
                    uint32_t pk[32];
#pragma unroll
                    for (int cc = 0; cc < 64; cc += 2) pk[cc / 2] = pack16<F16>(pf[cc], pf[cc + 1]);
                    // P^T of query columns [64cg, 64cg+64) goes over the first half of the S^T
                    // columns this group has just read (the other group never touches them)
                    tmem_st_32x32b_x32(tmem + lane_base + C::C_S + 64 * cg, pk);
                }
                tc_fence_before();
                mbar_arrive(&s.p_full);
                // ---- dS^T = P^T (dP^T - D) -> shared memory ----
                {
                    const bool w = twait(tr, kBDpFull, &s.dp_full, par, ab);
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                }
                if (i > 0) {
                    const bool w = twait(tr, kBDsFree, &s.ds_free, par ^ 1, ab);
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                }
                tc_fence_after();
                {
                    uint8_t* drow = s.dst[cg] + jr * 128;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t dr[32];
                        tmem_ld_32x32b_x32(tmem + lane_base + C::C_DP + 64 * cg + 32 * hf, dr);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {  // 16-byte units of 8 columns
                            const int cb = 32 * hf + 8 * u;
                            const float4 d0 = *reinterpret_cast<const float4*>(dlt + cb);
                            const float4 d1 = *reinterpret_cast<const float4*>(dlt + cb + 4);
                            uint4 w;
                            w.x = pack16<F16>(pf[cb + 0] * (__uint_as_float(dr[8 * u + 0]) - d0.x),
                                            pf[cb + 1] * (__uint_as_float(dr[8 * u + 1]) - d0.y));
                            w.y = pack16<F16>(pf[cb + 2] * (__uint_as_float(dr[8 * u + 2]) - d0.z),
                                            pf[cb + 3] * (__uint_as_float(dr[8 * u + 3]) - d0.w));
                            w.z = pack16<F16>(pf[cb + 4] * (__uint_as_float(dr[8 * u + 4]) - d1.x),
                                            pf[cb + 5] * (__uint_as_float(dr[8 * u + 5]) - d1.y));
                            w.w = pack16<F16>(pf[cb + 6] * (__uint_as_float(dr[8 * u + 6]) - d1.z),
                                            pf[cb + 7] * (__uint_as_float(dr[8 * u + 7]) - d1.w));
                            const int unit = (cb >> 3) ^ (jr & 7);
                            *reinterpret_cast<uint4*>(drow + unit * 16) = w;
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&s.ds_full);
                tr.mark(kMStepDone);
            }
            if (!ok) break;
            // ---- epilogue: dK, dV for this key block ----
            const bool have = bk.nsteps > 0;  // uniform over the CTA
            if (have) {
                const bool w = twait(tr, kBDkvFull, &s.dkv_full, nb & 1, ab);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                tc_fence_after();
            }
            tr.mark(kMEpilogue);
            // rows past the block's keys, or (token mode) past the key's sequence's used keys,
            // are not written
            bool row_ok = j <= bk.j1;
            if (tokens && row_ok && p.seqused_k) {
                const SeqView ks = seq_view(p, row_sequence(p.cu_k, p.B, j));
                row_ok = j - ks.k0 < ks.nk;
            }
            const long krow = key_row(p, bk.sv, j);
            // this group's half of the dV and dK row into registers; then the accumulators are
            // free for the next block while the rows are scaled and stored
            uint32_t vv[D / 2], kk[D / 2];
            if (have) {
                if constexpr (D == 128) {
                    tmem_ld_32x32b_x64(tmem + lane_base + C::C_DV + (D / 2) * cg, vv);
                    tmem_ld_32x32b_x64(tmem + lane_base + C::C_DK + (D / 2) * cg, kk);
                } else {
                    tmem_ld_32x32b_x32(tmem + lane_base + C::C_DV + (D / 2) * cg, vv);
                    tmem_ld_32x32b_x32(tmem + lane_base + C::C_DK + (D / 2) * cg, kk);
                }
                tc_fence_before();
                mbar_arrive(&s.dkv_free);
            } else {
#pragma unroll
                for (int t = 0; t < D / 2; ++t) vv[t] = kk[t] = 0u;
            }
            if (row_ok && dkv_al32) {
                // 32-byte stores (the half rows are 64 or 128 bytes)
                uint16_t* dvp = a.dv + (krow * p.h_kv + bk.g) * D + (D / 2) * cg;
                uint16_t* dkp = a.dk + (krow * p.h_kv + bk.g) * D + (D / 2) * cg;
                const float mul = p.scale;
#pragma unroll
                for (int t = 0; t < D / 32; ++t) {
                    uint32_t w[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        w[u] = pack16<F16>(__uint_as_float(vv[16 * t + 2 * u]), __uint_as_float(vv[16 * t + 2 * u + 1]));
                    st_global_v8(dvp + 16 * t, w);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        w[u] = pack16<F16>(__uint_as_float(kk[16 * t + 2 * u]) * mul,
                                           __uint_as_float(kk[16 * t + 2 * u + 1]) * mul);
                    st_global_v8(dkp + 16 * t, w);
                }
            } else if (row_ok) {
                uint4* dvp = reinterpret_cast<uint4*>(a.dv + (krow * p.h_kv + bk.g) * D + (D / 2) * cg);
                uint4* dkp = reinterpret_cast<uint4*>(a.dk + (krow * p.h_kv + bk.g) * D + (D / 2) * cg);
                const float mul = p.scale;
#pragma unroll
                for (int t = 0; t < D / 16; ++t) {
                    uint4 w;
                    w.x = pack16<F16>(__uint_as_float(vv[8 * t + 0]), __uint_as_float(vv[8 * t + 1]));
                    w.y = pack16<F16>(__uint_as_float(vv[8 * t + 2]), __uint_as_float(vv[8 * t + 3]));
                    w.z = pack16<F16>(__uint_as_float(vv[8 * t + 4]), __uint_as_float(vv[8 * t + 5]));
                    w.w = pack16<F16>(__uint_as_float(vv[8 * t + 6]), __uint_as_float(vv[8 * t + 7]));
                    dvp[t] = w;
                    w.x = pack16<F16>(__uint_as_float(kk[8 * t + 0]) * mul, __uint_as_float(kk[8 * t + 1]) * mul);
                    w.y = pack16<F16>(__uint_as_float(kk[8 * t + 2]) * mul, __uint_as_float(kk[8 * t + 3]) * mul);
                    w.z = pack16<F16>(__uint_as_float(kk[8 * t + 4]) * mul, __uint_as_float(kk[8 * t + 5]) * mul);
                    w.w = pack16<F16>(__uint_as_float(kk[8 * t + 6]) * mul, __uint_as_float(kk[8 * t + 7]) * mul);
                    dkp[t] = w;
                }
            }
            if (have) {
                gs += bk.nsteps;
                ++nb;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------------------------------
// backward at d = 192 and 256: one CTA per 64-key block, query rows on the tensor-memory lanes
// ------------------------------------------------------------------------------------------
// The d <= 128 layout (128-key block, the key rows on the lanes, dK and dV accumulated in
// tensor memory at full width) does not fit at d = 256: the two 256-column accumulators
// alone fill the 512 columns (and at d = 192 the two 192-column ones, with S and dP,
// leave no room for dQ).  Here a CTA owns 64 keys and the GEMMs are oriented so that
// every accumulator has M = 128 on the lanes:
//   S = Q K^T, dP = dO V^T          M = 128 query rows, N = 64 keys       (64 + 64 columns)
//   dV^T += dO^T P, dK^T += Q^T dS  M = 128 of d (two halves), N = 64     (128 + 128 columns)
//   dQ^T = K^T dS^T                 M = 128 of d (two halves, one after the other), N = 128
//                                   query rows, drained between the halves (128 columns)
// P and dS go through shared memory ([query row][64 keys], 128-byte swizzle), where they
// serve as the MN-major B operand of dV^T / dK^T and the K-major B operand of dQ^T.  Shared
// memory holds Q, dO (64 KB each, one buffer), K, V (32 KB each) and P, dS (16 KB each).
//
// Warp roles (256 threads): warp 0 TMA producer, warp 1 MMA issuer, warp 2 owns the TMEM
// allocation, warps 4-7 the compute group (thread = TMEM lane: a query row for P / dS, a
// column of d for the dQ^T drain and the dK / dV epilogue).
//
// d = 192 runs the same layout with three 64-column chunks of Q, dO, K and V: S and dP
// take K = 192 (no padding), while the GEMMs with d on the lanes keep their two 128-row
// halves, the second of which reads a fourth chunk of Q, dO and K that is zero in shared
// memory (written once, never loaded); its rows 192..255 come out zero and are neither
// reduced nor stored.
constexpr int kThreadsBwd256 = 256;
constexpr int kKeys256 = 64;  // keys per block

struct __align__(1024) BwdSmem256 {
    uint8_t q[4][128 * 128];       // [128 packed rows][64 cols] x 4 chunks of d
    uint8_t dO[4][128 * 128];
    uint8_t k[4][kKeys256 * 128];  // [64 keys][64 cols] x 4 chunks of d
    uint8_t v[4][kKeys256 * 128];
    uint8_t p[128 * 128];          // P:  [128 query rows][64 keys]
    uint8_t ds[128 * 128];         // dS: [128 query rows][64 keys]
    float stat[2][128];            // LSE * log2(e) and D of the tile's rows
    uint64_t kv_full, q_full, q_empty, do_full, do_empty, s_full, dp_full, pds_full, pds_free, dq_full, dq_free,
        dkv_full;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(BwdSmem256) <= 232448, "d = 256 backward: shared memory over the 227 KB limit");

// Query tiles [qt0, qt1) whose positions have a band reaching 64-key block `blk`.
__device__ __forceinline__ void block_qtiles64(const Problem& p, const SeqView& sv, const Band& band, int blk,
                                               int& qt0, int& qt1) {
    const int j0 = blk * kKeys256;
    const int j1 = min(j0 + kKeys256, sv.nk) - 1;
    int i_lo = 0, i_hi = sv.nq - 1;
    if (p.right >= 0) i_lo = max(i_lo, j0 - band.off - p.right);
    if (p.left >= 0) i_hi = min(i_hi, j1 - band.off + p.left);
    qt0 = (i_hi >= i_lo) ? i_lo / p.P : 0;
    qt1 = (i_hi >= i_lo) ? i_hi / p.P + 1 : 0;
}

// dq_predecessors for the 64-key blocks of the wide-head kernel.
__device__ __forceinline__ int dq_predecessors64(const Problem& p, const SeqView& sv, const Band& band, DqOrder& o,
                                                 int t) {
    while (o.next * kKeys256 < sv.nk) {
        int a0, a1;
        block_qtiles64(p, sv, band, o.next, a0, a1);
        if (a1 > a0) {
            if (a0 > t) break;
            ++o.n;
        }
        ++o.next;
    }
    return o.n;
}

// DET: the fixed dQ order of the d <= 128 kernel (DqOrder): a sequence's later 64-key
// blocks take lower CTA indices, and the compute group adds its two dQ^T halves into query
// tile t only after every later block that sees t has added (one count per warp).
template <int D, bool F16, bool DET>
__global__ void __launch_bounds__(kThreadsBwd256, 1)
    bwd256_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo) {
    static_assert(D == 192 || D == 256, "wide-head backward: d = 192 or 256");
    constexpr int KCH = D / 64;  // chunks loaded; a zero fourth chunk pads d = 192
    // TMEM columns
    constexpr uint32_t C_S = 0, C_DP = 64, C_DV = 128, C_DK = 256, C_DQ = 384;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the layout fills the shared memory: no room to realign by hand
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0 && a.status) atomicCAS(a.status, 0, kStatusDeviceCheck);
        return;
    }
    BwdSmem256& s = *reinterpret_cast<BwdSmem256*>(smem_raw);
    const Problem& p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (a.status && *reinterpret_cast<volatile int*>(a.status) != 0) return;  // the call already failed
    int g, seq, blk;
    {
        const int idx = blockIdx.x;
        if (p.cu_q) {
            g = idx % p.h_kv;
            blk = idx / p.h_kv;
            if (DET) blk = a.n_kvblocks - 1 - blk;
            seq = owner_sequence(p.cu_k, p.B, blk, kKeys256);
            blk -= p.cu_k[seq] / kKeys256 + seq;
        } else {
            int unit;
            band_order(idx, p.h_kv * p.B, a.n_bands, a.n_kvblocks, unit, blk);
            g = unit % p.h_kv;
            seq = unit / p.h_kv;
            if (DET) blk = a.n_kvblocks - 1 - blk;
        }
    }
    const SeqView sv = seq_view(p, seq);
    const int j0 = blk * kKeys256;
    if (j0 >= sv.nk) return;  // idle packed-batch block
    const Band band{sv.nk - sv.nq, p.left, p.right, sv.nk};
    int qt0, qt1;
    block_qtiles64(p, sv, band, blk, qt0, qt1);
    const int nsteps = qt1 - qt0;
    const int tbase = qtile_base(p, seq);

    Abort ab{&s.abort_flag, a.status, p.wait_ns};
    if (tid == 0) {
        s.abort_flag = 0;
        mbar_init(&s.kv_full, 1);
        mbar_init(&s.q_full, 1);
        mbar_init(&s.q_empty, 1);
        mbar_init(&s.do_full, 1);
        mbar_init(&s.do_empty, 1);
        mbar_init(&s.s_full, 1);
        mbar_init(&s.dp_full, 1);
        mbar_init(&s.pds_full, 128);
        mbar_init(&s.pds_free, 1);
        mbar_init(&s.dq_full, 1);
        mbar_init(&s.dq_free, 128);
        mbar_init(&s.dkv_full, 1);
        fence_mbar_init();
    }
    if (p.P * p.G < 128) {
        // rows past P*G of a query tile are never written by TMA: zero them once
        for (int c = 0; c < KCH; ++c)
            for (int x = p.P * p.G * 128 + tid * 16; x < 128 * 128; x += kThreadsBwd256 * 16) {
                *reinterpret_cast<uint4*>(&s.q[c][x]) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(&s.dO[c][x]) = make_uint4(0, 0, 0, 0);
            }
    }
    if constexpr (KCH < 4) {
        // d = 192: the fourth chunk of Q, dO and K (read by the second d-half GEMMs) is zero
        for (int x = tid * 16; x < 128 * 128; x += kThreadsBwd256 * 16) {
            *reinterpret_cast<uint4*>(&s.q[3][x]) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(&s.dO[3][x]) = make_uint4(0, 0, 0, 0);
        }
        for (int x = tid * 16; x < kKeys256 * 128; x += kThreadsBwd256 * 16)
            *reinterpret_cast<uint4*>(&s.k[3][x]) = make_uint4(0, 0, 0, 0);
    }
    if (p.P * p.G < 128 || KCH < 4) fence_proxy_async_smem();
    if (warp == 2) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0 && nsteps > 0) {
            Tracer tr;
            tr.init(a.trace, 0);
            tr.item(blockIdx.x);
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            tma_prefetch_desc(&tmdo);
            mbar_expect_tx(&s.kv_full, 2 * KCH * kKeys256 * 128);
            for (int c = 0; c < KCH; ++c) {
                tma_load_4d(s.k[c], &tmk, &s.kv_full, c * 64, g, sv.k0 + j0, sv.tma_b);
                tma_load_4d(s.v[c], &tmv, &s.kv_full, c * 64, g, sv.k0 + j0, sv.tma_b);
            }
            const uint32_t tile_bytes = (uint32_t)(p.P * p.G) * 128u * KCH;  // one Q or dO tile
            int q_issued = 0, do_issued = 0;
            for (int it = 0; it < nsteps; ++it) {
                const uint32_t ph = it & 1;
                const int row = sv.q0 + (qt0 + it) * p.P;
                if (!twait(tr, kBQEmpty, &s.q_empty, ph ^ 1, ab)) break;
                mbar_expect_tx(&s.q_full, tile_bytes + 2 * 128 * 4);
                for (int c = 0; c < KCH; ++c) tma_load_4d(s.q[c], &tmq, &s.q_full, c * 64, g * p.G, row, sv.tma_b);
                {
                    const long trow = ((long)g * a.n_qtiles + tbase + qt0 + it) * 128;
                    bulk_load(s.stat[0], a.lse2_t + trow, 512, &s.q_full);
                    bulk_load(s.stat[1], a.delta_t + trow, 512, &s.q_full);
                }
                ++q_issued;
                if (!twait(tr, kBDoEmpty, &s.do_empty, ph ^ 1, ab)) break;
                mbar_expect_tx(&s.do_full, tile_bytes);
                for (int c = 0; c < KCH; ++c) tma_load_4d(s.dO[c], &tmdo, &s.do_full, c * 64, g * p.G, row, sv.tma_b);
                ++do_issued;
            }
            // the copies still in flight: the last phase of each buffer
            if (q_issued > 0) mbar_wait_quiet(&s.q_full, (q_issued - 1) & 1);
            if (do_issued > 0) mbar_wait_quiet(&s.do_full, (do_issued - 1) & 1);
            mbar_wait_quiet(&s.kv_full, 0);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0 && nsteps > 0) {
            constexpr uint32_t id_s = idesc_16(128, kKeys256, false, false, F16);   // S, dP: K-major both
            constexpr uint32_t id_kv = idesc_16(128, kKeys256, true, true, F16);    // dV^T, dK^T: MN-major both
            constexpr uint32_t id_dq = idesc_16(128, 128, true, false, F16);        // dQ^T: A MN-major, B K-major
            const uint64_t qd_k = sdesc_sw128(smem_u32(s.q[0]), 16, 1024);
            const uint64_t dod_k = sdesc_sw128(smem_u32(s.dO[0]), 16, 1024);
            const uint64_t kd_k = sdesc_sw128(smem_u32(s.k[0]), 16, 1024);
            const uint64_t vd_k = sdesc_sw128(smem_u32(s.v[0]), 16, 1024);
            const uint64_t pd_mn = sdesc_sw128(smem_u32(s.p), 128 * 128, 1024);
            const uint64_t dsd_mn = sdesc_sw128(smem_u32(s.ds), 128 * 128, 1024);
            const uint64_t dsd_k = sdesc_sw128(smem_u32(s.ds), 16, 1024);
            Tracer tr;
            tr.init(a.trace, 1);
            tr.item(blockIdx.x);
            bool ok = twait(tr, kBKvFull, &s.kv_full, 0, ab);
            int ndq = 0;  // dQ^T halves issued so far
            for (int it = 0; ok && it < nsteps; ++it) {
                const uint32_t par = it & 1;
                if (!(ok = twait(tr, kBQFull, &s.q_full, par, ab))) break;
                if (!(ok = twait(tr, kBDoFull, &s.do_full, par, ab))) break;
                tc_fence_after();
                // S = Q K^T, dP = dO V^T (K = d: KCH 64-column chunks of each operand)
                if constexpr (KCH == 4) {
                    mma_ss_k16k8_x16(tmem + C_S, qd_k, kd_k, id_s, 0u);
                    tc_commit(&s.s_full);
                    mma_ss_k16k8_x16(tmem + C_DP, dod_k, vd_k, id_s, 0u);
                } else {
                    mma_ss_k16k8_x12(tmem + C_S, qd_k, kd_k, id_s, 0u);
                    tc_commit(&s.s_full);
                    mma_ss_k16k8_x12(tmem + C_DP, dod_k, vd_k, id_s, 0u);
                }
                tc_commit(&s.dp_full);
                // P and dS in shared memory (the compute group has also read S and dP out)
                if (!(ok = twait(tr, kBPdsFull, &s.pds_full, par, ab))) break;
                tc_fence_after();
                const uint32_t acc = it > 0 ? 1u : 0u;
                // dQ^T_h = K_h^T dS^T into the one dQ^T column block, drained between the halves
                auto issue_dq = [&](int h) -> bool {
                    if (ndq > 0 && !twait(tr, kBDqFree, &s.dq_free, (ndq - 1) & 1, ab)) return false;
                    tc_fence_after();
                    mma_ss_mnk_x4(tmem + C_DQ, sdesc_sw128(smem_u32(s.k[2 * h]), kKeys256 * 128, 1024), dsd_k, id_dq,
                                  0u);
                    tc_commit(&s.dq_full);
                    ++ndq;
                    return true;
                };
                // the first dQ^T half goes first, so that its drain overlaps dV^T and dK^T
                if (!(ok = issue_dq(0))) break;
                for (int h = 0; h < 2; ++h) {
                    // dV^T_h += dO_h^T P, dK^T_h += Q_h^T dS (the h-th 128 columns of d)
                    mma_ss_mnmn_x8(tmem + C_DV + 64 * h, sdesc_sw128(smem_u32(s.dO[2 * h]), 128 * 128, 1024), pd_mn,
                                   id_kv, acc);
                    mma_ss_mnmn_x8(tmem + C_DK + 64 * h, sdesc_sw128(smem_u32(s.q[2 * h]), 128 * 128, 1024), dsd_mn,
                                   id_kv, acc);
                }
                // Q and dO of this step are read once these complete (dQ^T reads K and dS only):
                // the next step's copies start while the second dQ^T half runs and drains
                tc_commit(&s.q_empty);
                tc_commit(&s.do_empty);
                if (!(ok = issue_dq(1))) break;
                // P and dS are read once the second dQ^T half completes
                tc_commit(&s.pds_free);
            }
            tc_commit(&s.dkv_full);
            mbar_wait_quiet(&s.dkv_full, 0);
        }
    } else if (warp >= 4) {
        // ================= compute group =================
        const int wq = warp & 3;
        const int r = (wq << 5) | lane;  // TMEM lane: query row (P, dS) or column of d (drains)
        const uint32_t lane_base = (uint32_t)(wq << 5) << 16;
        const float c = p.scale_log2;
        bool ok = true;
        int ndq = 0;
        DqOrder order;  // DET: the later blocks examined so far
        order.next = blk + 1;
        Tracer tr;
        tr.init(warp == 4 ? a.trace : nullptr, 2);
        tr.item(blockIdx.x);
        for (int it = 0; it < nsteps; ++it) {
            const uint32_t par = it & 1;
            const int t = qt0 + it;
            const long trow = ((long)g * a.n_qtiles + tbase + t) * 128;
            {
                bool w = twait(tr, kBQFull, &s.q_full, par, ab);  // the LSE / D rows land with Q
                w = w && twait(tr, kBSFull, &s.s_full, par, ab);
                w = w && twait(tr, kBDpFull, &s.dp_full, par, ab);
                if (it > 0) w = w && twait(tr, kBPdsFree, &s.pds_free, par ^ 1, ab);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            }
            tc_fence_after();
            // ---- P = exp2(S c - LSE2) on the allowed keys, dS = P (dP - D); row r ----
            {
                const int i = t * p.P + r / p.G;  // query position of this row
                const bool row_ok = r < p.P * p.G && i < sv.nq;
                // allowed keys of the row, as columns [c_lo, c_hi) of this block
                const int c_lo = row_ok ? band.lo(i) - j0 : 0;
                const int c_hi = row_ok ? band.hi(i) + 1 - j0 : 0;
                const float l2 = s.stat[0][r], dl = s.stat[1][r];
                uint32_t sr[64], dr[64];
                tmem_ld_32x32b_x64(tmem + lane_base + C_S, sr);
                tmem_ld_32x32b_x64(tmem + lane_base + C_DP, dr);
                // S and dP are in registers: the next step's S / dP may overwrite them once
                // this step's P and dS are handed over (pds_full)
                uint8_t* prow = s.p + r * 128;
                uint8_t* drow = s.ds + r * 128;
#pragma unroll
                for (int u = 0; u < 8; ++u) {  // 16-byte units of 8 keys
                    float pv[8], dv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int cc = 8 * u + e;
                        const float pe = (cc >= c_lo && cc < c_hi) ? ex2(fmaf(__uint_as_float(sr[cc]), c, -l2)) : 0.f;
                        pv[e] = pe;
                        dv[e] = pe * (__uint_as_float(dr[cc]) - dl);
                    }
                    const int unit = (u ^ (r & 7)) << 4;
                    *reinterpret_cast<uint4*>(prow + unit) = make_uint4(
                        pack16<F16>(pv[0], pv[1]), pack16<F16>(pv[2], pv[3]), pack16<F16>(pv[4], pv[5]),
                        pack16<F16>(pv[6], pv[7]));
                    *reinterpret_cast<uint4*>(drow + unit) = make_uint4(
                        pack16<F16>(dv[0], dv[1]), pack16<F16>(dv[2], dv[3]), pack16<F16>(dv[4], dv[5]),
                        pack16<F16>(dv[6], dv[7]));
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s.pds_full);
            tr.mark(kMSoftmaxDone);
            // ---- dQ^T halves: lane = column of d within the half, columns = query rows ----
            int* cnt = DET ? a.dq_count + (long)g * a.n_qtiles + tbase + t : nullptr;
            for (int h = 0; h < 2; ++h) {
                {
                    const bool w = twait(tr, kBDqFull, &s.dq_full, ndq & 1, ab);
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                }
                ++ndq;
                tc_fence_after();
                uint32_t qa[64], qb[64];
                tmem_ld_32x32b_x64(tmem + lane_base + C_DQ, qa);
                tmem_ld_32x32b_x64(tmem + lane_base + C_DQ + 64, qb);
                tc_fence_before();
                mbar_arrive(&s.dq_free);
                if (DET && h == 0 && !dq_turn_wait(cnt, 4 * dq_predecessors64(p, sv, band, order, t), ab)) {
                    ok = false;
                    break;
                }
                // for each query row the 32 lanes of a warp add to 32 consecutive floats
                // (at d = 192 the second half's lanes 64..127 hold the zero padding rows)
                if (128 * h + r < D) {
                    float* acc = a.dq_acc + trow * D + 128 * h + r;
#pragma unroll
                    for (int x = 0; x < 64; ++x) atomicAdd(acc + (long)x * D, __uint_as_float(qa[x]));
#pragma unroll
                    for (int x = 0; x < 64; ++x) atomicAdd(acc + (long)(64 + x) * D, __uint_as_float(qb[x]));
                }
                tr.mark(kMDqReduced);
            }
            if (!ok) break;
            if constexpr (DET) dq_turn_done(cnt);
        }
        // ---- epilogue: dV, dK of the block's 64 keys (lane = column of d within a half) ----
        if (nsteps > 0 && ok) {
            const bool w = mbar_wait(&s.dkv_full, 0, ab);
            ok = __all_sync(0xffffffffu, w);
            tc_fence_after();
        }
        const int nkeys = min(kKeys256, sv.nk - j0);
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
            uint16_t* base = which == 0 ? a.dv : a.dk;
            const float mul = which == 0 ? 1.f : p.scale;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t v[64];
                if (nsteps > 0 && ok) {
                    tmem_ld_32x32b_x64(tmem + lane_base + (which == 0 ? C_DV : C_DK) + 64 * h, v);
                } else {
#pragma unroll
                    for (int x = 0; x < 64; ++x) v[x] = 0u;
                }
                if (128 * h + r >= D) continue;  // d = 192: a padding row of the second half
                // key rows are consecutive within a sequence: one stride of h_kv * d elements
                uint16_t* dst = base + (key_row(p, sv, j0) * p.h_kv + g) * D + 128 * h + r;
                const long stride = (long)p.h_kv * D;
#pragma unroll
                for (int x = 0; x < 64; ++x, dst += stride)
                    if (x < nkeys) *dst = round16<F16>(__uint_as_float(v[x]) * mul);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------------------------
// preprocess: one CTA (128 threads) per (tiled query tile, key/value head)
// ------------------------------------------------------------------------------------------
// Decodes a tiled query-tile index into (sequence, tile within it); false for an idle tile.
// Token mode: the tile is the packed rows [idx P, idx P + P) (sequence 0's view spans them all).
__device__ __forceinline__ bool decode_qtile(const BwdArgs& a, int idx, int& seq, int& t) {
    const Problem& p = a.p;
    if (p.cu_q && a.tokens) {
        seq = 0;
        t = idx;
        return idx * p.P < p.T_q;
    }
    if (p.cu_q) {
        seq = owner_sequence(p.cu_q, p.B, idx, p.P);
        t = idx - (p.cu_q[seq] / p.P + seq);
        return t * p.P < p.cu_q[seq + 1] - p.cu_q[seq];
    }
    const int per = cdiv(p.s_q, p.P);
    seq = idx / per;
    t = idx % per;
    return true;
}

// The view the pre- and postprocess index a query tile's rows with, and whether local row
// i of it holds a query: in token mode the view spans the packed rows, and a row past its
// own sequence's used queries (seqused_q) holds none.
__device__ __forceinline__ SeqView qtile_view(const BwdArgs& a, int seq) {
    const Problem& p = a.p;
    return (p.cu_q && a.tokens) ? SeqView{0, 0, p.T_q, 0, p.T_k, 0} : seq_view(p, seq);
}
__device__ __forceinline__ bool query_row_used(const BwdArgs& a, const SeqView& sv, int i) {
    const Problem& p = a.p;
    if (i >= sv.nq) return false;
    if (p.cu_q && a.tokens && p.seqused_q) {
        const SeqView own = seq_view(p, row_sequence(p.cu_q, p.B, i));
        return i - own.q0 < own.nq;
    }
    return true;
}

template <int D, bool F16>
__global__ void __launch_bounds__(128) bwd_pre_kernel(const BwdArgs a) {
    const Problem& p = a.p;
    const int idx = blockIdx.x, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the offset check (FA_FLAG_VALIDATE_CU) ran first on this stream: when it failed,
    // touch nothing (the later kernels of the call skip as well)
    if (*reinterpret_cast<volatile const int*>(a.status) != 0) return;
    int seq, t;
    const bool live = decode_qtile(a, idx, seq, t);
    const long trow = ((long)g * a.n_qtiles + idx) * 128;
    if (a.dq_count && threadIdx.x == 0) a.dq_count[(long)g * a.n_qtiles + idx] = 0;
    if (!live) {
        a.lse2_t[trow + threadIdx.x] = INFINITY;
        a.delta_t[trow + threadIdx.x] = 0.f;
        if (a.sink_t) a.sink_t[trow + threadIdx.x] = 0.f;
        return;
    }
    const SeqView sv = qtile_view(a, seq);
    // a warp takes its 32 rows RPI at a time: LPR lanes per row (a power of two), VPL
    // 16-byte units (8 elements) of O and dO each per lane, so every load instruction moves
    // whole 128-byte lines
    constexpr int LPR = D == 192 ? 8 : D / 8, RPI = 32 / LPR, VPL = D / (8 * LPR);
    static_assert(LPR * RPI == 32 && VPL * 8 * LPR == D, "row split of the preprocess");
    const int sub = lane / LPR, ch = lane % LPR;
#pragma unroll 4
    for (int rr = 0; rr < 32; rr += RPI) {
        const int r = warp * 32 + rr + sub;
        const int i = t * p.P + r / p.G;
        const int h = g * p.G + r % p.G;
        const bool valid = r < p.P * p.G && query_row_used(a, sv, i);
        float dsum = 0.f;
        long tok = 0;
        if (valid) {
            tok = token_row(p, sv, i);
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                const long off = (tok * p.h_q + h) * D + 8 * ch + 8 * LPR * u;
                const uint4 ov = *reinterpret_cast<const uint4*>(a.o + off);
                const uint4 dv = *reinterpret_cast<const uint4*>(a.dout + off);
                dsum = fmaf(lo16<F16>(ov.x), lo16<F16>(dv.x), dsum);
                dsum = fmaf(hi16<F16>(ov.x), hi16<F16>(dv.x), dsum);
                dsum = fmaf(lo16<F16>(ov.y), lo16<F16>(dv.y), dsum);
                dsum = fmaf(hi16<F16>(ov.y), hi16<F16>(dv.y), dsum);
                dsum = fmaf(lo16<F16>(ov.z), lo16<F16>(dv.z), dsum);
                dsum = fmaf(hi16<F16>(ov.z), hi16<F16>(dv.z), dsum);
                dsum = fmaf(lo16<F16>(ov.w), lo16<F16>(dv.w), dsum);
                dsum = fmaf(hi16<F16>(ov.w), hi16<F16>(dv.w), dsum);
            }
        }
        // sum over the row's LPR lanes (all lanes take part: rows differ in validity)
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
        if (ch == 0) {
            float l2 = INFINITY, sterm = 0.f;
            if (valid) {
                const float lse = a.lse[lse_index(p, sv, i, h)];
                l2 = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
                // d(sum O.dO)/d(sink_h) = - exp(sink_h - LSE_i) * D_i, summed per head later
                if (p.sinks && lse > -INFINITY) sterm = -__expf(p.sinks[h] - lse) * dsum;
            }
            a.delta_t[trow + r] = valid ? dsum : 0.f;
            a.lse2_t[trow + r] = l2;
            if (a.sink_t) a.sink_t[trow + r] = sterm;
        }
    }
    // zero this tile's dQ accumulator rows
    float4* acc = reinterpret_cast<float4*>(a.dq_acc + trow * D);
    for (int x = threadIdx.x; x < 128 * D / 4; x += 128) acc[x] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Sink gradient of one query head (one CTA each): the sum of its rows' terms, over the
// tiles of its key/value head, in a fixed order (strided per-thread sums, then a tree).
__global__ void __launch_bounds__(256) bwd_dsink_kernel(const BwdArgs a) {
    const Problem& p = a.p;
    if (*reinterpret_cast<volatile const int*>(a.status) != 0) return;  // the call failed: dsinks stay 0
    const int h = blockIdx.x, g = h / p.G, hh = h % p.G;
    // head h holds rows hh + G k (k < P) of every tile of its key/value head
    const long n = (long)a.n_qtiles * p.P;
    float acc = 0.f;
    for (long x = threadIdx.x; x < n; x += 256) {
        const long tile = x / p.P;
        const int k = (int)(x - tile * p.P);
        acc += a.sink_t[((long)g * a.n_qtiles + tile) * 128 + hh + p.G * k];
    }
    __shared__ float part[256];
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) a.dsinks[h] = part[0];
}

// postprocess: dQ = scale * acc -> rows of the inputs' 16-bit type
template <int D, bool F16>
__global__ void __launch_bounds__(128) bwd_post_kernel(const BwdArgs a) {
    const Problem& p = a.p;
    const int idx = blockIdx.x, g = blockIdx.y;
    if (*reinterpret_cast<volatile const int*>(a.status) != 0) return;  // the call failed: dQ not written
    int seq, t;
    if (!decode_qtile(a, idx, seq, t)) return;
    const SeqView sv = qtile_view(a, seq);
    const long trow = ((long)g * a.n_qtiles + idx) * 128;
    constexpr int V = 8;  // columns per thread step
    for (int x = threadIdx.x; x < 128 * D / V; x += 128) {
        const int r = x / (D / V), cb = (x % (D / V)) * V;
        const int i = t * p.P + r / p.G;
        const int h = g * p.G + r % p.G;
        if (r >= p.P * p.G || !query_row_used(a, sv, i)) continue;
        const float4 u0 = *reinterpret_cast<const float4*>(a.dq_acc + (trow + r) * D + cb);
        const float4 u1 = *reinterpret_cast<const float4*>(a.dq_acc + (trow + r) * D + cb + 4);
        const float sc = p.scale;
        uint4 w;
        w.x = pack16<F16>(u0.x * sc, u0.y * sc);
        w.y = pack16<F16>(u0.z * sc, u0.w * sc);
        w.z = pack16<F16>(u1.x * sc, u1.y * sc);
        w.w = pack16<F16>(u1.z * sc, u1.w * sc);
        *reinterpret_cast<uint4*>(a.dq + (token_row(p, sv, i) * p.h_q + h) * D + cb) = w;
    }
}

}  // namespace

template <int D, bool DET, bool TOK>
static cudaError_t launch_main_d(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, cudaStream_t st) {
    const size_t smem = sizeof(BwdSmem<D>);
    static_assert(sizeof(BwdSmem<D>) <= 232448, "backward: shared memory over the 227 KB limit");
    auto kernel = a.p.dtype == FA_DTYPE_F16 ? bwd_main_kernel<D, DET, true, TOK> : bwd_main_kernel<D, DET, false, TOK>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // persistent CTAs (at most one per SM), or one CTA per unit
    const long n = (DET || !a.persist) ? (long)a.n_units : (long)a.n_ctas;
    if (n <= 0) return cudaSuccess;
    kernel<<<(unsigned)n, kThreadsBwd, smem, st>>>(a, tq, tk, tv, tdo);
    return cudaGetLastError();
}

template <int D, bool DET>
static cudaError_t launch_main256(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const CUtensorMap& tdo, cudaStream_t st) {
    const size_t smem = sizeof(BwdSmem256);
    auto kernel = a.p.dtype == FA_DTYPE_F16 ? bwd256_kernel<D, true, DET> : bwd256_kernel<D, false, DET>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long n = (long)a.n_kvblocks * a.p.h_kv * (a.p.cu_q ? 1 : a.p.B);
    kernel<<<(unsigned)n, kThreadsBwd256, smem, st>>>(a, tq, tk, tv, tdo);
    return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, cudaStream_t st) {
    switch (a.p.d) {
        case 192:
            return a.dq_count ? launch_main256<192, true>(a, tq, tk, tv, tdo, st)
                              : launch_main256<192, false>(a, tq, tk, tv, tdo, st);
        case 256:
            return a.dq_count ? launch_main256<256, true>(a, tq, tk, tv, tdo, st)
                              : launch_main256<256, false>(a, tq, tk, tv, tdo, st);
        case 64:
            if (a.dq_count) return launch_main_d<64, true, false>(a, tq, tk, tv, tdo, st);
            return a.tokens ? launch_main_d<64, false, true>(a, tq, tk, tv, tdo, st)
                            : launch_main_d<64, false, false>(a, tq, tk, tv, tdo, st);
        case 128:
            if (a.dq_count) return launch_main_d<128, true, false>(a, tq, tk, tv, tdo, st);
            return a.tokens ? launch_main_d<128, false, true>(a, tq, tk, tv, tdo, st)
                            : launch_main_d<128, false, false>(a, tq, tk, tv, tdo, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t st) {
    dim3 grid(a.n_qtiles, a.p.h_kv);
    if (a.n_qtiles == 0) return cudaSuccess;
    const bool f16 = a.p.dtype == FA_DTYPE_F16;
    auto kernel = a.p.d == 64    ? (f16 ? bwd_pre_kernel<64, true> : bwd_pre_kernel<64, false>)
                  : a.p.d == 128 ? (f16 ? bwd_pre_kernel<128, true> : bwd_pre_kernel<128, false>)
                  : a.p.d == 192 ? (f16 ? bwd_pre_kernel<192, true> : bwd_pre_kernel<192, false>)
                                 : (f16 ? bwd_pre_kernel<256, true> : bwd_pre_kernel<256, false>);
    kernel<<<grid, 128, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_post(const BwdArgs& a, cudaStream_t st) {
    dim3 grid(a.n_qtiles, a.p.h_kv);
    if (a.n_qtiles == 0) return cudaSuccess;
    const bool f16 = a.p.dtype == FA_DTYPE_F16;
    auto kernel = a.p.d == 64    ? (f16 ? bwd_post_kernel<64, true> : bwd_post_kernel<64, false>)
                  : a.p.d == 128 ? (f16 ? bwd_post_kernel<128, true> : bwd_post_kernel<128, false>)
                  : a.p.d == 192 ? (f16 ? bwd_post_kernel<192, true> : bwd_post_kernel<192, false>)
                                 : (f16 ? bwd_post_kernel<256, true> : bwd_post_kernel<256, false>);
    kernel<<<grid, 128, 0, st>>>(a);
    if (a.dsinks) bwd_dsink_kernel<<<a.p.h_q, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace fa
