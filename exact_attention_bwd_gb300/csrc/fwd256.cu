// Forward attention for head dimensions 192 and 256 on the tcgen05 tensor cores.
//
// The accumulator of one 128-row query tile is d TMEM columns wide, so a CTA holds a
// single query tile.  Tensor memory: O in columns [0, d), two 64-column S buffers in
// [256, 384), and the Q tile itself from column 384 on (16-bit pairs, one row per lane,
// d / 2 columns), so S = Q K^T takes its A operand from tensor memory and reads only K
// from shared memory.  Q arrives by TMA in the first ring slot (a Q tile is as large as a
// K plus a V tile); the softmax warps copy their rows into tensor memory, after which that
// slot joins the key/value ring.  Keys and values stream in 64-row tiles (32 KB each at
// d = 256, 24 KB at d = 192, which leaves room for a fourth slot).  d = 192 is one of the
// head sizes the pages pad to (dew-flash-attn PyPI page, the FA3 head-dim padding to
// 64 / 128 / 192 / 256); here it runs as three 64-column chunks, not padded.  The MMA thread runs one
// tile ahead: S(j+1) is computed while the softmax group works on S(j), then
// O += P(j) V(j).  Rows are packed across the G query heads of the key/value head exactly
// as in the d <= 128 kernel, and the online softmax is the same (running max / running
// sum with lazy rescaling, "Flash Attention Tutorial" README, sections 3 to 5); key tiles
// outside the causal / sliding-window band are skipped.
#include "common.cuh"

namespace fa {
namespace {

constexpr int kThreads256 = 256;
constexpr int BN = 64;               // keys per KV tile
constexpr int Q_CHUNK = 128 * 128;   // [128 rows][64 cols] 16-bit
constexpr int KV_CHUNK = BN * 128;   // [64 rows][64 cols] 16-bit
constexpr uint32_t C_O = 0;
constexpr uint32_t C_S = 256;        // S buffer b at columns 256 + 64 b
constexpr uint32_t C_Q = 384;        // Q: column c holds elements 2c, 2c+1 of the row

template <int D>
struct Cfg256 {
    static constexpr int KCH = D / 64;              // 64-column chunks
    static constexpr int KV_BYTES = KCH * KV_CHUNK; // one K or V tile (32 KB at d = 256)
    static constexpr int SLOT_BYTES = 2 * KV_BYTES; // ring slot: K then V; slot 0 first holds Q
    static constexpr int STAGES = D == 256 ? 3 : 4;
    static_assert(KCH * Q_CHUNK == SLOT_BYTES, "the Q tile fills one ring slot");
    static_assert(C_Q + D / 2 <= 512 && C_O + D <= C_S, "tensor-memory columns overlap");
    // ring slot and use count of KV tile `it`: tiles 0 .. STAGES-2 take slots 1 .. STAGES-1,
    // tile STAGES-1 the slot Q came in, and so on round the ring
    static __device__ __forceinline__ int slot_of(int it) { return (it + 1) % STAGES; }
    static __device__ __forceinline__ uint32_t use_parity(int it) { return (uint32_t)(it / STAGES) & 1u; }
};

template <int D>
struct __align__(1024) Smem256 {
    uint8_t ring[Cfg256<D>::STAGES][Cfg256<D>::SLOT_BYTES];  // K at 0, V at KV_BYTES
    uint64_t q_full, q_tmem;
    uint64_t k_full[Cfg256<D>::STAGES], k_empty[Cfg256<D>::STAGES], v_full[Cfg256<D>::STAGES],
        v_empty[Cfg256<D>::STAGES];
    uint64_t s_full[2], p_full[2], pv_done, o_full, drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D, bool F16>
__global__ void __launch_bounds__(kThreads256, 1)
    fwd256_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
    using C = Cfg256<D>;
    constexpr int KCH = C::KCH, KV_BYTES = C::KV_BYTES, SLOT_BYTES = C::SLOT_BYTES, STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    Smem256<D>& s = *reinterpret_cast<Smem256<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Problem& p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // an earlier kernel or CTA of the call failed (a device check, a timeout): read nothing
    // the offsets point at
    if (a.status && *reinterpret_cast<volatile int*>(a.status) != 0) return;

    // ---------------- work unit ----------------
    // 1-D grid, heaviest work first (see the d <= 128 kernel); the last (batch, kv head)
    // units may be cut into tail_k key ranges each (the tail split, see FwdArgs)
    int g, seq, blk, split = 0;
    bool tail = false;
    {
        const int idx = blockIdx.x;
        if (a.tail_k > 1 && idx >= a.tail_item0) {
            const int t = idx - a.tail_item0;
            const int per_unit = a.n_blocks * a.tail_k;
            const int unit = a.tail_item0 / a.n_blocks + t / per_unit;
            const int x = t % per_unit;
            g = unit % p.h_kv;
            seq = unit / p.h_kv;
            split = x % a.tail_k;
            blk = a.n_blocks - 1 - x / a.tail_k;
            tail = true;
        } else if (p.cu_q) {
            g = idx % p.h_kv;
            blk = idx / p.h_kv;
            seq = owner_sequence(p.cu_q, p.B, blk, p.P);
            blk -= p.cu_q[seq] / p.P + seq;
        } else {
            const int hb = p.h_kv * p.B;
            const int per_unit = a.n_blocks * a.n_splits;
            const int unit = a.unit_major ? idx / per_unit : idx % hb;
            const int x = a.unit_major ? idx % per_unit : idx / hb;
            g = unit % p.h_kv;
            seq = unit / p.h_kv;
            split = x % a.n_splits;
            blk = a.n_blocks - 1 - x / a.n_splits;
        }
    }
    const SeqView sv = seq_view(p, seq);
    const int s0 = blk * p.P;
    if (s0 >= sv.nq) return;  // idle packed-batch block
    const Band band{sv.nk - sv.nq, p.left, p.right, sv.nk};
    int t0, t1;
    kv_tile_range(band, s0, min(s0 + p.P, sv.nq) - 1, BN, t0, t1);
    if (a.n_splits > 1 || tail) {
        const int st = tail ? a.tail_split_tiles : a.split_tiles;
        t0 = max(t0, split * st);
        t1 = min(t1, (split + 1) * st);
        if (t1 < t0) t1 = t0;
    }
    const int ntiles = t1 - t0;

    Abort ab{&s.abort_flag, a.status, p.wait_ns};
    if (tid == 0) {
        s.abort_flag = 0;
        mbar_init(&s.q_full, 1);
        mbar_init(&s.q_tmem, 4);  // one arrive per softmax warp once its Q rows are in TMEM
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&s.k_full[i], 1);
            mbar_init(&s.k_empty[i], 1);
            mbar_init(&s.v_full[i], 1);
            mbar_init(&s.v_empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s.s_full[b], 1);
            mbar_init(&s.p_full[b], 4);  // one arrive per softmax warp
        }
        mbar_init(&s.pv_done, 1);
        mbar_init(&s.o_full, 1);
        mbar_init(&s.drain, 1);
        fence_mbar_init();
    }
    if (p.P * p.G < 128) {
        for (int c = 0; c < KCH; ++c)
            for (int x = p.P * p.G * 128 + tid * 16; x < 128 * 128; x += kThreads256 * 16)
                *reinterpret_cast<uint4*>(&s.ring[0][c * Q_CHUNK + x]) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
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
        if (lane == 0 && ntiles > 0) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            mbar_expect_tx(&s.q_full, (uint32_t)(p.P * p.G) * 128u * KCH);
            for (int c = 0; c < KCH; ++c)
                tma_load_4d(&s.ring[0][c * Q_CHUNK], &tmq, &s.q_full, c * 64, g * p.G, sv.q0 + s0, sv.tma_b);
            int k_issued = 0, v_issued = 0;
            for (int it = 0; it < ntiles; ++it) {
                const int st = C::slot_of(it);
                const uint32_t ph = C::use_parity(it);
                int row, outer;
                kv_tile_coord(p, sv, (t0 + it) * BN, row, outer);
                // slot 0 is free for keys once the softmax warps have copied Q out of it
                if (it == STAGES - 1 && !mbar_wait(&s.q_tmem, 0, ab)) break;
                if (!mbar_wait(&s.k_empty[st], ph ^ 1, ab)) break;
                mbar_expect_tx(&s.k_full[st], KV_BYTES);
                for (int c = 0; c < KCH; ++c)
                    tma_load_4d(&s.ring[st][c * KV_CHUNK], &tmk, &s.k_full[st], c * 64, g, row, outer);
                ++k_issued;
                if (!mbar_wait(&s.v_empty[st], ph ^ 1, ab)) break;
                mbar_expect_tx(&s.v_full[st], KV_BYTES);
                for (int c = 0; c < KCH; ++c)
                    tma_load_4d(&s.ring[st][KV_BYTES + c * KV_CHUNK], &tmv, &s.v_full[st], c * 64, g, row, outer);
                ++v_issued;
            }
            // wait for every copy still in flight before the CTA may exit
            for (int back = 1; back <= STAGES; ++back) {
                if (k_issued - back >= 0)
                    mbar_wait_quiet(&s.k_full[C::slot_of(k_issued - back)], C::use_parity(k_issued - back));
                if (v_issued - back >= 0)
                    mbar_wait_quiet(&s.v_full[C::slot_of(v_issued - back)], C::use_parity(v_issued - back));
            }
            mbar_wait_quiet(&s.q_full, 0);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idS = idesc_16(128, BN, false, false, F16);  // A = Q from TMEM, B = K K-major
            constexpr uint32_t idO = idesc_16(128, D, false, true, F16);    // A = P from TMEM, B = V MN-major
            // descriptors: base values plus (byte offset >> 4) in the start-address field
            const uint64_t kd0 = sdesc_sw128(smem_u32(s.ring[0]), 16, 1024);
            const uint64_t vd0 = sdesc_sw128(smem_u32(s.ring[0] + KV_BYTES), KV_CHUNK, 1024);
            constexpr uint32_t kSlot = SLOT_BYTES >> 4;
            auto issue_s = [&](int it) {  // S(it) = Q K(it)^T into buffer it & 1
                const int st = C::slot_of(it);
                if constexpr (D == 256)
                    mma_ts_lin_k8_x16(tmem + C_S + 64 * (it & 1), tmem + C_Q, kd0 + (uint64_t)(st * kSlot), idS, 0u);
                else
                    mma_ts_lin_k8_x12(tmem + C_S + 64 * (it & 1), tmem + C_Q, kd0 + (uint64_t)(st * kSlot), idS, 0u);
                tc_commit(&s.s_full[it & 1]);
                tc_commit(&s.k_empty[st]);
            };
            bool ok = mbar_wait(&s.q_tmem, 0, ab);
            if (ok && (ok = mbar_wait(&s.k_full[C::slot_of(0)], 0, ab))) {
                tc_fence_after();
                issue_s(0);
            }
            for (int it = 0; ok && it < ntiles; ++it) {
                if (it + 1 < ntiles) {
                    if (!(ok = mbar_wait(&s.k_full[C::slot_of(it + 1)], C::use_parity(it + 1), ab))) break;
                    tc_fence_after();
                    issue_s(it + 1);  // its buffer held P(it-1), read by PV(it-1) issued earlier
                }
                const int st = C::slot_of(it), b = it & 1;
                if (!(ok = mbar_wait(&s.v_full[st], C::use_parity(it), ab))) break;
                // buffer b is used at iterations b, b + 2, ...: this is its (it >> 1)-th phase
                if (!(ok = mbar_wait(&s.p_full[b], (it >> 1) & 1, ab))) break;
                tc_fence_after();
                mma_ts_lin_mn_x4(tmem + C_O, tmem + C_S + 64 * b, vd0 + (uint64_t)(st * kSlot), idO, it > 0 ? 1u : 0u);
                tc_commit(&s.pv_done);
                tc_commit(&s.v_empty[st]);
                if (it == ntiles - 1) tc_commit(&s.o_full);  // single-phase: O is final
            }
            tc_commit(&s.drain);
            mbar_wait_quiet(&s.drain, 0);
        }
    } else if (warp >= 4) {
        // ================= softmax: one thread per row =================
        const int r = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
        const uint32_t tO = tmem + lane_base + C_O;
        const int i = s0 + r / p.G;
        const int h = g * p.G + r % p.G;
        const bool row_valid = (r < p.P * p.G) && i < sv.nq;
        const int jlo = row_valid ? band.lo(i) : 1;
        const int jhi = row_valid ? band.hi(i) : 0;
        const float c = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        if (ntiles > 0) {
            // copy this thread's Q row (TMEM lane r) out of the swizzled TMA layout: 16-byte
            // unit u of a [128][64] chunk row sits at position u ^ (r & 7)
            {
                const bool w = mbar_wait(&s.q_full, 0, ab);
                if (!__all_sync(0xffffffffu, w)) ok = false;
            }
            if (ok) {
#pragma unroll
                for (int cch = 0; cch < KCH; ++cch) {
                    const uint8_t* qrow = &s.ring[0][cch * Q_CHUNK + r * 128];
                    uint32_t qr[32];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint4 x = *reinterpret_cast<const uint4*>(qrow + ((u ^ (r & 7)) << 4));
                        qr[4 * u + 0] = x.x;
                        qr[4 * u + 1] = x.y;
                        qr[4 * u + 2] = x.z;
                        qr[4 * u + 3] = x.w;
                    }
                    tmem_st_32x32b_x32(tmem + lane_base + C_Q + 32 * cch, qr);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.q_tmem);
            }
        }
        for (int it = 0; ok && it < ntiles; ++it) {
            const int b = it & 1;
            {
                const bool w = mbar_wait(&s.s_full[b], (it >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            }
            tc_fence_after();
            const uint32_t tS = tmem + lane_base + C_S + 64 * b;
            const int j0 = (t0 + it) * BN;
            const bool edge = (j0 < jlo || j0 + BN - 1 > jhi);
            uint32_t sr[64];
            tmem_ld_32x32b_x64(tS, sr);
            if (edge) {
#pragma unroll
                for (int cc = 0; cc < BN; ++cc)
                    if (j0 + cc < jlo || j0 + cc > jhi) sr[cc] = __float_as_uint(-INFINITY);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < BN; ++cc) mx = fmaxf(mx, __uint_as_float(sr[cc]));
            const float m_new = fmaxf(m_used, mx * c);
            float alpha = 1.f;
            bool rescale = false;
            if (m_used == -INFINITY) {
                m_used = m_new;
            } else if (m_new > m_used + 8.f) {
                alpha = ex2(m_used - m_new);
                m_used = m_new;
                l *= alpha;
                rescale = true;
            }
            if (__any_sync(0xffffffffu, rescale)) {
                // O must hold PV(it-1) before it is rescaled
                const bool w = mbar_wait(&s.pv_done, (it - 1) & 1, ab);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < D; cb += 32) {
                    uint32_t orr[32];
                    tmem_ld_32x32b_x32(tO + cb, orr);
#pragma unroll
                    for (int t = 0; t < 32; ++t) orr[t] = __float_as_uint(__uint_as_float(orr[t]) * alpha);
                    tmem_st_32x32b_x32(tO + cb, orr);
                }
            }
            const float base = (m_used == -INFINITY) ? 0.f : m_used;
            float sum = 0.f;
#pragma unroll
            for (int cc = 0; cc < BN; cc += 2) {
                const float p0 = ex2(fmaf(__uint_as_float(sr[cc]), c, -base));
                const float p1 = ex2(fmaf(__uint_as_float(sr[cc + 1]), c, -base));
                sum += p0 + p1;
                sr[cc / 2] = pack16<F16>(p0, p1);
            }
            l += sum;
            tmem_st_32x32b_x32(tS, sr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.p_full[b]);
        }
        // ---------------- epilogue ----------------
        const bool has_o = ntiles > 0;
        if (has_o && ok) {
            // pv_done can lag two phases behind here (S(last) was issued before
            // PV(last-1)), which a parity wait cannot tell apart: use the one-shot barrier
            const bool w = mbar_wait(&s.o_full, 0, ab);
            ok = __all_sync(0xffffffffu, w);
            tc_fence_after();
        }
        const bool split_mode = a.n_splits > 1 || tail;
        const bool o_al32 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;  // rows keep the alignment (D * 2 bytes)
        float oscale = 0.f, lse = -INFINITY;
        if (!split_mode && p.sinks && row_valid) {
            const float s2 = p.sinks[h] * kLog2e;
            const float mf = fmaxf(m_used, s2);
            const float wgt = (m_used == -INFINITY) ? 0.f : ex2(m_used - mf);
            const float lt = l * wgt + ex2(s2 - mf);
            oscale = wgt / lt;
            lse = (mf + log2f(lt)) * kLn2;
        } else if (l > 0.f) {
            oscale = 1.f / l;
            lse = (m_used + log2f(l)) * kLn2;
        }
        // the partials' rows: all B h_q s_q rows, or (tail split) those from tail_row0 on
        const long row_base = tail ? a.tail_row0 : 0;
        const long nrows = (long)p.B * p.h_q * p.s_q - row_base;
        const long prow = ((long)sv.b * p.h_q + h) * p.s_q + i - row_base;
        if (row_valid) {
            if (!split_mode) {
                if (a.lse) a.lse[lse_index(p, sv, i, h)] = lse;
            } else {
                a.lse_part[(long)split * nrows + prow] = lse;
            }
        }
        for (int cb = 0; cb < D; cb += 32) {
            uint32_t orr[32];
            if (has_o && ok) {
                tmem_ld_32x32b_x32(tO + cb, orr);
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) orr[t] = 0u;
            }
            if (!row_valid) continue;
            if (!split_mode && o_al32) {
                // 32-byte stores (a 32-column chunk of the row is 64 bytes)
                uint16_t* orow = a.o + (token_row(p, sv, i) * p.h_q + h) * D + cb;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    uint32_t wv[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        wv[u] = pack16<F16>(__uint_as_float(orr[16 * t + 2 * u]) * oscale,
                                            __uint_as_float(orr[16 * t + 2 * u + 1]) * oscale);
                    st_global_v8(orow + 16 * t, wv);
                }
            } else if (!split_mode) {
                uint16_t* orow = a.o + (token_row(p, sv, i) * p.h_q + h) * D + cb;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    uint4 wv;
                    wv.x = pack16<F16>(__uint_as_float(orr[8 * t + 0]) * oscale, __uint_as_float(orr[8 * t + 1]) * oscale);
                    wv.y = pack16<F16>(__uint_as_float(orr[8 * t + 2]) * oscale, __uint_as_float(orr[8 * t + 3]) * oscale);
                    wv.z = pack16<F16>(__uint_as_float(orr[8 * t + 4]) * oscale, __uint_as_float(orr[8 * t + 5]) * oscale);
                    wv.w = pack16<F16>(__uint_as_float(orr[8 * t + 6]) * oscale, __uint_as_float(orr[8 * t + 7]) * oscale);
                    reinterpret_cast<uint4*>(orow)[t] = wv;
                }
            } else {
                float* op = a.o_part + ((long)split * nrows + prow) * D + cb;
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    reinterpret_cast<float4*>(op)[t] =
                        make_float4(__uint_as_float(orr[4 * t]) * oscale, __uint_as_float(orr[4 * t + 1]) * oscale,
                                    __uint_as_float(orr[4 * t + 2]) * oscale, __uint_as_float(orr[4 * t + 3]) * oscale);
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

}  // namespace

template <int D>
static cudaError_t launch_fwd_wide(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, cudaStream_t st) {
    const size_t smem = sizeof(Smem256<D>) + 1024;
    auto kernel = a.p.dtype == FA_DTYPE_F16 ? fwd256_kernel<D, true> : fwd256_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    long n = a.p.cu_q ? (long)a.n_blocks * a.p.h_kv : (long)a.n_blocks * a.n_splits * a.p.h_kv * a.p.B;
    if (a.tail_k > 1) n = a.tail_item0 + (n - a.tail_item0) * a.tail_k;
    kernel<<<(unsigned)n, kThreads256, smem, st>>>(a, tq, tk, tv);
    return cudaGetLastError();
}

cudaError_t launch_fwd256(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          cudaStream_t st) {
    switch (a.p.d) {
        case 192: return launch_fwd_wide<192>(a, tq, tk, tv, st);
        case 256: return launch_fwd_wide<256>(a, tq, tk, tv, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
