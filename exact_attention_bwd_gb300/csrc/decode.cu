// Decode-shaped forward (few query rows per key/value head) and the split-KV combine.
//
// With s_q * (h_q / h_kv) <= 8 query rows per key/value head (4 at d = 192, 256) the work is a stream over
// the key/value cache: about 2 multiply-adds per byte read, far below what the tensor
// cores would need, so this path runs on the CUDA cores and is sized to keep HBM busy.
// The cache of one (batch, key/value head) is split across CTAs, each CTA writes a
// partial (O, LSE) for its key range, and a second kernel merges the partials by their
// log-sum-exp (vllm-project/flash-attention README, changelog 2.2 "Optimize for
// inference": split the KV load across thread blocks, combine in a separate kernel).
#include "common.cuh"

namespace fa {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kThreadsDec = 32 * (kComputeWarps + 1);  // + one producer warp
constexpr int BK = 64;                                 // keys per tile
constexpr int KPW = BK / kComputeWarps;                // keys per warp per tile (8)

template <int D, int RG>
struct DecCfg {
    static constexpr int KCH = D / 64;
    static constexpr int CHUNK = BK * 128;             // [64 rows][64 cols] 16-bit, swizzled
    static constexpr int TILE = BK * D * 2;            // one K (or V) tile
    static constexpr int EPL = D / 32;                 // head-dim elements per lane
    static constexpr int R = 4 * RG;                   // query rows held (padded)
    // two CTAs per SM where the stages fit in half the shared memory
    static constexpr int STAGES = (D >= 128) ? 3 : 6;
    static constexpr int MIN_BLOCKS = (D >= 192 || RG > 1) ? 1 : 2;
};

template <int D, int RG>
struct __align__(1024) DecSmem {
    uint8_t k[DecCfg<D, RG>::STAGES][DecCfg<D, RG>::TILE];
    uint8_t v[DecCfg<D, RG>::STAGES][DecCfg<D, RG>::TILE];
    float mw[kComputeWarps][4 * RG], lw[kComputeWarps][4 * RG];
    float4 pbuf[kComputeWarps][KPW];  // a warp's P of the current tile: [key][row of the group]
    uint64_t full[DecCfg<D, RG>::STAGES], empty[DecCfg<D, RG>::STAGES];
    int abort_flag;
};

// Byte offset of element (row, col) of a [rows][64] 16-bit chunk written by a TMA load with
// 128-byte swizzle: the 16-byte unit index is XORed with row % 8.
__device__ __forceinline__ int sw128(int row, int col) {
    return row * 128 + ((((col >> 3) ^ row) & 7) << 4) + ((col & 7) << 1);
}

// EPL consecutive 16-bit values (fp16 if F16, else bf16) of row `row` starting at column
// `col` of a swizzled tile, widened to fp32 (EPL = 2, 4 or 8: one 4-, 8- or 16-byte load
// that stays in a unit; EPL = 6, at d = 192: three 4-byte loads, since six values starting
// at an even column can straddle a 16-byte unit or a 64-column chunk).
template <int EPL, int CHUNK, bool F16>
__device__ __forceinline__ void load_row_slice(const uint8_t* tile, int row, int col, float* out) {
    const uint8_t* src = tile + (col >> 6) * CHUNK + sw128(row, col & 63);
    if constexpr (EPL == 6) {
#pragma unroll
        for (int e = 0; e < 6; e += 2) {
            const int c = col + e;
            const uint32_t w = *reinterpret_cast<const uint32_t*>(tile + (c >> 6) * CHUNK + sw128(row, c & 63));
            out[e] = lo16<F16>(w);
            out[e + 1] = hi16<F16>(w);
        }
    } else if constexpr (EPL == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
        out[0] = lo16<F16>(w);
        out[1] = hi16<F16>(w);
    } else if constexpr (EPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(src);
        out[0] = lo16<F16>(w.x); out[1] = hi16<F16>(w.x); out[2] = lo16<F16>(w.y); out[3] = hi16<F16>(w.y);
    } else {
        const uint4 w = *reinterpret_cast<const uint4*>(src);
        out[0] = lo16<F16>(w.x); out[1] = hi16<F16>(w.x); out[2] = lo16<F16>(w.y); out[3] = hi16<F16>(w.y);
        out[4] = lo16<F16>(w.z); out[5] = hi16<F16>(w.z); out[6] = lo16<F16>(w.w); out[7] = hi16<F16>(w.w);
    }
}

// Each compute warp streams its own 8 keys of every 64-key tile and keeps a private online
// softmax (running max m, running sum l, un-normalised output) for every query row; lane
// L holds head-dim elements [EPL L, EPL L + EPL).  Per tile and group of 4 rows, the 32
// (key, row) dot products are formed by a reduce-scatter across the lanes, so lane L ends
// with item L = 4 * key + row.  The warps' states are merged by their log-sum-exp at the
// end and the CTA writes the partial (O, LSE) of its key range.
template <int D, int RG, bool F16>
__global__ void __launch_bounds__(kThreadsDec, DecCfg<D, RG>::MIN_BLOCKS)
    decode_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using C = DecCfg<D, RG>;
    constexpr int EPL = C::EPL;
    extern __shared__ uint8_t smem_raw[];
    DecSmem<D, RG>& s =
        *reinterpret_cast<DecSmem<D, RG>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Problem& p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x % a.n_splits;
    const int unit = blockIdx.x / a.n_splits;
    const int g = unit % p.h_kv, b = unit / p.h_kv;
    const int R = p.s_q * p.G;
    if (a.status && *reinterpret_cast<volatile int*>(a.status) != 0) return;
    const SeqView sv = seq_view(p, b);  // dense; nq, nk below s_q, s_kv when the slot is partly filled
    const Band band{sv.nk - sv.nq, p.left, p.right, sv.nk};

    int j_begin = split * a.split_keys, j_end = min(sv.nk, (split + 1) * a.split_keys);
    j_begin = max(j_begin, band.lo(0));
    j_end = sv.nq > 0 ? min(j_end, band.hi(sv.nq - 1) + 1) : 0;
    const int t_begin = j_begin / BK;
    const int n_tiles = j_end > j_begin ? (j_end - 1) / BK + 1 - t_begin : 0;
    // keys every query row may see, whether its position is used or not (the band bounds are
    // monotone in the position, positions 0 .. s_q - 1): a tile inside [in_lo, in_hi] needs
    // no per-key mask
    const int in_lo = max(j_begin, band.lo(p.s_q - 1));
    const int in_hi = min(j_end - 1, band.hi(0));

    Abort ab{&s.abort_flag, a.status, p.wait_ns};
    if (tid == 0) {
        s.abort_flag = 0;
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], kComputeWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // per-lane state of a compute warp: un-normalised output, running max and sum per row
    float acc[C::R][EPL], m[C::R], l[C::R];
#pragma unroll
    for (int r = 0; r < C::R; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[r][e] = 0.f;
    }

    if (warp == kComputeWarps) {
        // ================= producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % C::STAGES;
                if (!mbar_wait(&s.empty[st], ((t / C::STAGES) & 1) ^ 1, ab)) break;
                int row, outer;
                kv_tile_coord(p, sv, (t_begin + t) * BK, row, outer);
                mbar_expect_tx(&s.full[st], 2 * C::TILE);
                for (int c = 0; c < C::KCH; ++c) {
                    tma_load_4d(&s.k[st][c * C::CHUNK], &tmk, &s.full[st], c * 64, g, row, outer);
                    tma_load_4d(&s.v[st][c * C::CHUNK], &tmv, &s.full[st], c * 64, g, row, outer);
                }
                ++issued;
            }
            // wait for the copies still in flight (the latest phase of each used stage)
            for (int back = 1; back <= C::STAGES && back <= issued; ++back) {
                const int t = issued - back;
                mbar_wait_quiet(&s.full[t % C::STAGES], (t / C::STAGES) & 1);
            }
        }
    } else {
        // ================= compute warps =================
        const int e0 = EPL * lane;
        float q[C::R][EPL];
#pragma unroll
        for (int r = 0; r < C::R; ++r) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                float val = 0.f;
                if (r < R) {
                    const int i = r / p.G, h = g * p.G + r % p.G;
                    val = lo16<F16>(a.q[(((long)b * p.s_q + i) * p.h_q + h) * D + e0 + e]) * p.scale_log2;
                }
                q[r][e] = val;
            }
        }
        for (int t = 0; t < n_tiles; ++t) {
            const int st = t % C::STAGES;
            {
                const bool w = mbar_wait(&s.full[st], (t / C::STAGES) & 1, ab);
                if (!__all_sync(0xffffffffu, w)) break;
            }
            const int jw = (t_begin + t) * BK + KPW * warp;  // first key of this warp
            const bool interior = (t_begin + t) * BK >= in_lo && (t_begin + t) * BK + BK - 1 <= in_hi;
            float kv[KPW][EPL];
#pragma unroll
            for (int k = 0; k < KPW; ++k) load_row_slice<EPL, C::CHUNK, F16>(s.k[st], KPW * warp + k, e0, kv[k]);
            const int kk = lane >> 2, rr = lane & 3;   // item of this lane after the reduction
            const int j = jw + kk;
#pragma unroll
            for (int rg = 0; rg < RG; ++rg) {
                // 32 partial dot products: item 4k + rr
                float v32[32];
#pragma unroll
                for (int k = 0; k < KPW; ++k)
#pragma unroll
                    for (int r4 = 0; r4 < 4; ++r4) {
                        float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < EPL; e += 2)
                            acc2 = __ffma2_rn(make_float2(q[4 * rg + r4][e], q[4 * rg + r4][e + 1]),
                                              make_float2(kv[k][e], kv[k][e + 1]), acc2);
                        v32[4 * k + r4] = acc2.x + acc2.y;
                    }
                // reduce-scatter: lane L ends with the full sum of item L
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
                    for (int i = 0; i < o; ++i) {
                        const bool up = (lane & o) != 0;
                        const float send = up ? v32[i] : v32[i + o];
                        const float keep = up ? v32[i + o] : v32[i];
                        v32[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                }
                const int r = 4 * rg + rr;
                float sc = v32[0];
                if (!interior || r >= R) {
                    const int i = r / p.G;
                    const bool keep = r < R && j >= j_begin && j < j_end && j >= band.lo(i) && j <= band.hi(i);
                    if (!keep) sc = -INFINITY;
                }
                // per-row max and sum over the warp's 8 keys (lanes with equal lane % 4)
                float mt = sc;
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
                const float m_old = (rr == 0) ? m[4 * rg] : (rr == 1) ? m[4 * rg + 1] : (rr == 2) ? m[4 * rg + 2] : m[4 * rg + 3];
                // the running max moves only when it grows by more than 2^8 (exact: every
                // exponential stays below 256 and the final division uses the same max)
                const bool grow = m_old == -INFINITY ? mt > -INFINITY : mt > m_old + 8.f;
                const bool any_grow = __any_sync(0xffffffffu, grow);
                const float m_new = grow ? mt : m_old;
                const float base = (m_new == -INFINITY) ? 0.f : m_new;
                const float pr = ex2(sc - base);
                float ps = pr;
                ps += __shfl_xor_sync(0xffffffffu, ps, 4);
                ps += __shfl_xor_sync(0xffffffffu, ps, 8);
                ps += __shfl_xor_sync(0xffffffffu, ps, 16);
                if (any_grow) {
                    // some row's max moved: every lane takes the new state of the group's 4 rows
                    // from lanes 0..3 and rescales its accumulators
                    const float alpha = (m_old == -INFINITY) ? 0.f : (grow ? ex2(m_old - base) : 1.f);
#pragma unroll
                    for (int r4 = 0; r4 < 4; ++r4) {
                        const float al = __shfl_sync(0xffffffffu, alpha, r4);
                        m[4 * rg + r4] = __shfl_sync(0xffffffffu, m_new, r4);
                        l[4 * rg + r4] = l[4 * rg + r4] * al + __shfl_sync(0xffffffffu, ps, r4);
#pragma unroll
                        for (int e = 0; e < EPL; ++e) acc[4 * rg + r4][e] *= al;
                    }
                } else {
#pragma unroll
                    for (int r4 = 0; r4 < 4; ++r4) l[4 * rg + r4] += __shfl_sync(0xffffffffu, ps, r4);
                }
                // P of the warp's 8 keys to every lane: lane 4k + r holds (key k, row r)
                reinterpret_cast<float*>(s.pbuf[warp])[lane] = pr;
                __syncwarp();
                // O += P V over the warp's 8 keys
#pragma unroll
                for (int k = 0; k < KPW; ++k) {
                    float vv[EPL];
                    load_row_slice<EPL, C::CHUNK, F16>(s.v[st], KPW * warp + k, e0, vv);
                    const float4 p4 = s.pbuf[warp][k];
                    const float pk4[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                    for (int r4 = 0; r4 < 4; ++r4) {
                        const float pk = pk4[r4];
#pragma unroll
                        for (int e = 0; e < EPL; e += 2) {
                            const float2 o2 = __ffma2_rn(make_float2(pk, pk), make_float2(vv[e], vv[e + 1]),
                                                         make_float2(acc[4 * rg + r4][e], acc[4 * rg + r4][e + 1]));
                            acc[4 * rg + r4][e] = o2.x;
                            acc[4 * rg + r4][e + 1] = o2.y;
                        }
                    }
                }
                __syncwarp();  // pbuf is rewritten by the next row group or tile
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.empty[st]);
        }
    }
    // every tile is consumed and the producer has drained: the stages become the merge buffer
    __syncthreads();
    float* red = reinterpret_cast<float*>(s.k[0]);  // [warp][row][D], spans the K and V stages
    if (warp < kComputeWarps) {
        const int e0 = EPL * lane;
#pragma unroll
        for (int r = 0; r < C::R; ++r)
#pragma unroll
            for (int e = 0; e < EPL; ++e) red[(warp * C::R + r) * D + e0 + e] = acc[r][e];
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < C::R; ++r) {
                s.mw[warp][r] = m[r];
                s.lw[warp][r] = l[r];
            }
        }
    }
    __syncthreads();
    // merge the warps' states by their running max, write the CTA's partial (O / l, LSE)
    const long nrows = (long)p.B * p.h_q * p.s_q;
    for (int x = tid; x < R * D; x += kThreadsDec) {
        const int r = x / D, c = x % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, s.mw[w][r]);
        float L = 0.f, O = 0.f;
        if (M > -INFINITY) {
#pragma unroll
            for (int w = 0; w < kComputeWarps; ++w) {
                const float mw = s.mw[w][r];
                if (mw == -INFINITY) continue;
                const float sc = ex2(mw - M);
                L += s.lw[w][r] * sc;
                O += red[(w * C::R + r) * D + c] * sc;
            }
        }
        const int i = r / p.G, h = g * p.G + r % p.G;
        const long row = ((long)b * p.h_q + h) * p.s_q + i;
        a.o_part[((long)split * nrows + row) * D + c] = L > 0.f ? O / L : 0.f;
        if (c == 0) a.lse_part[(long)split * nrows + row] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
}

// Merges the splits' partials of each output row by their log-sum-exp and folds in the
// sink, which joins the denominator exactly once.  A row is taken by L lanes (32, or 16 at
// d = 64), each holding 4 consecutive columns per step (two steps at d = 256), so every
// warp instruction reads whole 128-byte lines; a lane group takes RL rows.  The splits are
// merged in one pass, four at a time with a running maximum: every load of a batch (the
// splits' log-sum-exps and partial rows of all RL rows) is independent of the others, so
// a lane has them all in flight at once instead of waiting for the statistics first.
constexpr int kCombineWarps = 8;

template <int D>
struct CombineCfg {
    static constexpr int L = D == 192 ? 16 : (D >= 128 ? 32 : D / 4);  // lanes per row (a power of two)
    static constexpr int V = D / (4 * L);             // float4 columns per lane
    static constexpr int RL = D >= 192 ? 1 : 2;       // rows per lane group
    static constexpr int ROWS_PER_BLOCK = kCombineWarps * (32 / L) * RL;
};

template <int D, bool F16>
__global__ void __launch_bounds__(kCombineWarps * 32, 3) combine_kernel(const CombineArgs a) {
    using C = CombineCfg<D>;
    constexpr int L = C::L, V = C::V, RL = C::RL;
    const Problem& p = a.p;
    // an earlier kernel of the call failed: its partials are incomplete, write nothing
    if (a.status && *reinterpret_cast<volatile const int*>(a.status) != 0) return;
    const long nrows = a.nrows ? a.nrows : (long)p.B * p.h_q * p.s_q;  // rows of the partials
    const int lane = threadIdx.x & 31, l = lane % L;
    const long row0 = (((long)blockIdx.x * kCombineWarps + threadIdx.x / 32) * (32 / L) + lane / L) * RL;
    const int n = a.n_splits;
    float m[RL], den[RL];
    float4 acc[RL][V];
#pragma unroll
    for (int q = 0; q < RL; ++q) {
        m[q] = -INFINITY;
        den[q] = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) acc[q][v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int sp0 = 0; sp0 < n; sp0 += 4) {
        float lk[RL][4];
        float4 x[RL][4][V];
#pragma unroll
        for (int q = 0; q < RL; ++q) {
            const long r = min(row0 + q, nrows - 1);  // rows past the end read the last row, store nothing
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int sp = sp0 + k;
                const bool in = sp < n;
                lk[q][k] = in ? a.lse_part[(long)sp * nrows + r] : -INFINITY;
                const float* src = a.o_part + ((long)sp * nrows + r) * D + 4 * l;
#pragma unroll
                for (int v = 0; v < V; ++v)
                    x[q][k][v] = in ? *reinterpret_cast<const float4*>(src + 4 * L * v) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int q = 0; q < RL; ++q) {
            const float mn = fmaxf(m[q], fmaxf(fmaxf(lk[q][0], lk[q][1]), fmaxf(lk[q][2], lk[q][3])));
            if (mn == -INFINITY) continue;  // no keys in any split so far
            const float sc = m[q] == -INFINITY ? 0.f : __expf(m[q] - mn);
            den[q] *= sc;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                acc[q][v].x *= sc;
                acc[q][v].y *= sc;
                acc[q][v].z *= sc;
                acc[q][v].w *= sc;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // an empty split (-inf) adds nothing; its partial row may never have been
                // written, so it is skipped rather than multiplied by zero
                if (lk[q][k] == -INFINITY) continue;
                const float w = __expf(lk[q][k] - mn);
                den[q] += w;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    acc[q][v].x = fmaf(w, x[q][k][v].x, acc[q][v].x);
                    acc[q][v].y = fmaf(w, x[q][k][v].y, acc[q][v].y);
                    acc[q][v].z = fmaf(w, x[q][k][v].z, acc[q][v].z);
                    acc[q][v].w = fmaf(w, x[q][k][v].w, acc[q][v].w);
                }
            }
            m[q] = mn;
        }
    }
    // (batch, head, position) of the lane group's first output row; the next rows follow by
    // carrying (rows are ordered batch, head, position)
    int i, h, b;
    {
        const long row = a.row0 + row0;
        if (row < 0x7fffffffL) {
            const unsigned r = (unsigned)row, hb = r / (unsigned)p.s_q;
            i = (int)(r - hb * (unsigned)p.s_q);
            b = (int)(hb / (unsigned)p.h_q);
            h = (int)(hb - (unsigned)b * (unsigned)p.h_q);
        } else {
            i = (int)(row % p.s_q);
            h = (int)((row / p.s_q) % p.h_q);
            b = (int)(row / ((long)p.s_q * p.h_q));
        }
    }
#pragma unroll
    for (int q = 0; q < RL; ++q) {
        if (row0 + q >= nrows) break;
        if (q > 0 && ++i == p.s_q) {
            i = 0;
            if (++h == p.h_q) {
                h = 0;
                ++b;
            }
        }
        const long row = a.row0 + row0 + q;  // the output row
        const float sink = p.sinks ? p.sinks[h] : -INFINITY;
        const float m_all = fmaxf(m[q], sink);
        const float sc = m[q] == -INFINITY ? 0.f : __expf(m[q] - m_all);
        const float den_keys = den[q] * sc;
        const float dn = den_keys + (p.sinks && m_all != -INFINITY ? __expf(sink - m_all) : 0.f);
        const float lse = dn > 0.f ? m_all + __logf(dn) : -INFINITY;
        const float f = den_keys > 0.f ? sc / dn : 0.f;
        uint16_t* out = a.o + (((long)b * p.s_q + i) * p.h_q + h) * D + 4 * l;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            uint2 packed;
            packed.x = pack16<F16>(acc[q][v].x * f, acc[q][v].y * f);
            packed.y = pack16<F16>(acc[q][v].z * f, acc[q][v].w * f);
            *reinterpret_cast<uint2*>(out + 4 * L * v) = packed;
        }
        if (l == 0 && a.lse) a.lse[row] = lse;  // [B, h_q, s_q]: the row index itself
    }
}

}  // namespace

template <int D, int RG>
static cudaError_t launch_decode_dr(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    const size_t smem = sizeof(DecSmem<D, RG>) + 1024;
    auto kernel = a.p.dtype == FA_DTYPE_F16 ? decode_kernel<D, RG, true> : decode_kernel<D, RG, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long n = (long)a.n_splits * a.p.h_kv * a.p.B;
    kernel<<<(unsigned)n, kThreadsDec, smem, st>>>(a, tk, tv);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_decode_d(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    const int R = a.p.s_q * a.p.G;
    if (R <= 4) return launch_decode_dr<D, 1>(a, tk, tv, st);
    if constexpr (D <= 128) {
        if (R <= 8) return launch_decode_dr<D, 2>(a, tk, tv, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    switch (a.p.d) {
        case 64: return launch_decode_d<64>(a, tk, tv, st);
        case 128: return launch_decode_d<128>(a, tk, tv, st);
        case 192: return launch_decode_d<192>(a, tk, tv, st);
        case 256: return launch_decode_d<256>(a, tk, tv, st);
        default: return cudaErrorInvalidValue;
    }
}

// The per-lane state (query rows and output accumulators) grows with the rows; past these
// counts the registers spill, and the tensor-core path takes the problem instead.
int decode_rows_max(int d) { return d >= 192 ? 4 : 8; }
int decode_ctas_per_sm(int d, int rows) { return (d >= 192 || rows > 4) ? 1 : 2; }

template <int D>
static cudaError_t launch_combine_d(const CombineArgs& a, cudaStream_t st) {
    const long nrows = a.nrows ? a.nrows : (long)a.p.B * a.p.h_q * a.p.s_q;
    const long rows_per_block = CombineCfg<D>::ROWS_PER_BLOCK;
    const long blocks = (nrows + rows_per_block - 1) / rows_per_block;
    if (blocks == 0) return cudaSuccess;
    auto kernel = a.p.dtype == FA_DTYPE_F16 ? combine_kernel<D, true> : combine_kernel<D, false>;
    kernel<<<(unsigned)blocks, kCombineWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
    switch (a.p.d) {
        case 64: return launch_combine_d<64>(a, st);
        case 128: return launch_combine_d<128>(a, st);
        case 192: return launch_combine_d<192>(a, st);
        case 256: return launch_combine_d<256>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
