// Forward attention with e4m3 (fp8) inputs on the 5th-generation tensor cores, sm_103a.
//
// The FP8 forward is one of the variants the vllm-project/flash-attention README lists for
// FlashAttention-3 ("FP16 / BF16 forward and backward, FP8 forward").  Here Q, K and V are
// e4m3 with a per-(batch, key/value head) descale factor each (true value = stored value x
// descale); both GEMMs run as tcgen05.mma kind::f8f6f4 with fp32 accumulation, the
// probabilities P are rounded to e4m3 for the second GEMM, and O (bf16) and the LSE
// (fp32, natural log) are those of the descaled problem.
//
// Differences from the bf16 kernel (same work items, persistent scheduling, masks and
// online softmax with lazy rescaling):
//  - P goes to shared memory (two buffers per query tile) instead of over S in tensor
//    memory, so the S tile is free as soon as the softmax has read it into registers and
//    the next S = Q K^T is issued while the softmax still works: the softmax warps run back
//    to back instead of waiting for each P V to finish.
//  - Both GEMMs use K-major operands only: each V tile arrives by TMA as it is stored
//    ([keys][d], like K) into a staging slot, and warps 2 and 3 transpose it into a V^T tile
//    ([d][keys]) of the ring the MMA reads, so P V reads V^T tiles exactly as S = Q K^T reads
//    K tiles (no pass over V in memory).
//  - A 128-element e4m3 row is one 128-byte swizzle atom: Q, K, V, V^T and P tiles are 16 KB.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 2 and 3 the V
// transpose (warp 2 also owns the TMEM allocation), warps 4..7 and 8..11 the softmax of
// query tiles 0 and 1 (one thread per row).
#include "fwd_items.cuh"

namespace fa {
namespace {

constexpr int kThreads8 = 384;
constexpr int kTile8 = 128 * 128;  // bytes of one e4m3 tile (128 rows of 128 bytes)
constexpr int kStagesK = 4;   // K ring
constexpr int kStagesVt = 2;  // V^T ring (written by the transpose warps)
constexpr int kStagesV = 2;   // V staging ring (written by TMA)

struct __align__(1024) Smem8 {
    uint8_t q[2][kTile8];
    uint8_t k[kStagesK][kTile8];
    uint8_t vt[kStagesVt][kTile8];  // V^T tiles: [128 d rows][128 keys]
    uint8_t v[kStagesV][kTile8];    // V tiles as stored: [128 keys][128 d]
    uint8_t p[2][2][kTile8];        // [query tile][buffer]: P rows of 128 keys
    uint64_t q_full, q_empty;
    uint64_t k_full[kStagesK], k_empty[kStagesK], v_full[kStagesVt], v_empty[kStagesVt];
    uint64_t vin_full[kStagesV], vin_empty[kStagesV];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full[2][2], p_free[2][2];
    uint64_t o_full[2], o_free[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
// the dynamic shared memory window (1024 bytes of slack for the manual alignment) must fit
// the 227 KB a CTA may use
static_assert(sizeof(Smem8) + 1024 <= 232448, "e4m3 forward shared memory exceeds 227 KB");

// ------------------------------------------------------------------------------------------
// V -> V^T inside the CTA: warp w (0 or 1) of the two transpose warps takes the 16-byte units
// U = 4w .. 4w + 3 of d, lane l the keys 4l .. 4l + 3.  For each U the lane loads its four
// keys' 16 bytes (one 16-byte load per key row of the swizzled V tile), transposes each of
// the four 4 x 4 byte blocks in registers with byte permutes and stores one 4-byte word into
// each of the 16 d rows of the V^T tile, so a warp store covers one whole 128-byte row.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void transpose_v_tile(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt, int w,
                                                 int lane) {
#pragma unroll 1
    for (int U = 4 * w; U < 4 * w + 4; ++U) {
        uint32_t x[4][4];  // [key 4 lane + i][word c]: bytes 16 U + 4 c .. + 3 of d
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int key = 4 * lane + i;
            const uint4 u = *reinterpret_cast<const uint4*>(v + key * 128 + ((U ^ (key & 7)) << 4));
            x[i][0] = u.x, x[i][1] = u.y, x[i][2] = u.z, x[i][3] = u.w;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            // d rows 16 U + 4 c + 0..3, keys 4 lane .. 4 lane + 3 (lowest byte first)
            const uint32_t t0 = __byte_perm(x[0][c], x[1][c], 0x5140), t1 = __byte_perm(x[2][c], x[3][c], 0x5140);
            const uint32_t t2 = __byte_perm(x[0][c], x[1][c], 0x7362), t3 = __byte_perm(x[2][c], x[3][c], 0x7362);
            const uint32_t row_words[4] = {__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632),
                                           __byte_perm(t2, t3, 0x5410), __byte_perm(t2, t3, 0x7632)};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int d = 16 * U + 4 * c + m;
                *reinterpret_cast<uint32_t*>(vt + d * 128 + (((lane >> 2) ^ (d & 7)) << 4) + 4 * (lane & 3)) =
                    row_words[m];
            }
        }
    }
}

// Row r of a K-major 128-byte-swizzled tile (the layout TMA writes with SWIZZLE_128B):
// 16-byte unit u of the row lives at unit u ^ (r % 8) of the row's 128 bytes.
__device__ __forceinline__ uint32_t sw128_unit(int r, int u) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kThreads8, 1)
    fwd_e4m3_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv) {
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    Smem8& s = *reinterpret_cast<Smem8*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Problem& p = a.p;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    if (a.status && *reinterpret_cast<volatile int*>(a.status) != 0) return;

    Abort ab{&s.abort_flag, a.status, p.wait_ns};
    if (tid == 0) {
        s.abort_flag = 0;
        mbar_init(&s.q_full, 1);
        mbar_init(&s.q_empty, 1);
        for (int i = 0; i < kStagesK; ++i) {
            mbar_init(&s.k_full[i], 1);
            mbar_init(&s.k_empty[i], 1);
        }
        for (int i = 0; i < kStagesVt; ++i) {
            mbar_init(&s.v_full[i], 2);  // one arrive per transpose warp
            mbar_init(&s.v_empty[i], 1);
        }
        for (int i = 0; i < kStagesV; ++i) {
            mbar_init(&s.vin_full[i], 1);
            mbar_init(&s.vin_empty[i], 2);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s.s_full[k], 1);
            mbar_init(&s.s_free[k], 4);  // one arrive per softmax warp
            for (int b = 0; b < 2; ++b) {
                mbar_init(&s.p_full[k][b], 4);
                mbar_init(&s.p_free[k][b], 1);
            }
            mbar_init(&s.o_full[k], 1);
            mbar_init(&s.o_free[k], 4);
        }
        mbar_init(&s.drain, 1);
        fence_mbar_init();
    }
    if (p.P * p.G < 128) {
        // rows past P*G of a Q tile are never written by TMA: zero them once
        for (int k = 0; k < 2; ++k)
            for (int x = p.P * p.G * 128 + tid * 16; x < kTile8; x += kThreads8 * 16)
                *reinterpret_cast<uint4*>(&s.q[k][x]) = make_uint4(0, 0, 0, 0);
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
    // registers: 384 x 168 at launch; the producer / MMA / transpose group hands part of
    // its share to the softmax groups (128 x 72 + 256 x 216 = 64512)
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;\n" ::: "memory");
    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            const uint32_t qbox = (uint32_t)(p.P * p.G) * 128u;  // bytes of one Q box
            int gt = 0, n_q = 0, k_issued = 0, v_issued = 0;
            bool ok = true;
            for (int idx = blockIdx.x, step = first_step(a.snake); ok && idx < a.n_items;
                 idx += step, step = 2 * (int)gridDim.x - step) {
                const FwdItem w = fwd_item(a, idx);
                if (!w.live || w.u1 <= w.u0) continue;
                if (n_q > 0 && !(ok = mbar_wait(&s.q_empty, (n_q - 1) & 1, ab))) break;
                uint32_t qbytes = 0;
                for (int k = 0; k < 2; ++k)
                    if (w.ti[k].t1 > w.ti[k].t0) qbytes += qbox;
                mbar_expect_tx(&s.q_full, qbytes);
                for (int k = 0; k < 2; ++k)
                    if (w.ti[k].t1 > w.ti[k].t0)
                        tma_load_4d(s.q[k], &tmq, &s.q_full, 0, w.g * p.G, w.sv.q0 + w.ti[k].s0, w.sv.tma_b);
                ++n_q;
                for (int j = w.u0; j < w.u1; ++j, ++gt) {
                    const int st = gt % kStagesK;
                    int row, outer;  // the key tile's map coordinates (dense or packed)
                    kv_tile_coord(p, w.sv, j * BN, row, outer);
                    if (!(ok = mbar_wait(&s.k_empty[st], ((gt / kStagesK) & 1) ^ 1, ab))) break;
                    mbar_expect_tx(&s.k_full[st], kTile8);
                    tma_load_4d(s.k[st], &tmk, &s.k_full[st], 0, w.g, row, outer);
                    ++k_issued;
                    const int sv = gt % kStagesV;
                    if (!(ok = mbar_wait(&s.vin_empty[sv], ((gt / kStagesV) & 1) ^ 1, ab))) break;
                    mbar_expect_tx(&s.vin_full[sv], kTile8);
                    tma_load_4d(s.v[sv], &tmv, &s.vin_full[sv], 0, w.g, row, outer);
                    ++v_issued;
                }
            }
            for (int back = 1; back <= kStagesK; ++back) {
                if (k_issued - back >= 0) {
                    const int i2 = k_issued - back;
                    mbar_wait_quiet(&s.k_full[i2 % kStagesK], (i2 / kStagesK) & 1);
                }
            }
            for (int back = 1; back <= kStagesV; ++back) {
                if (v_issued - back >= 0) {
                    const int i2 = v_issued - back;
                    mbar_wait_quiet(&s.vin_full[i2 % kStagesV], (i2 / kStagesV) & 1);
                }
            }
            if (n_q > 0) mbar_wait_quiet(&s.q_full, (n_q - 1) & 1);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idS = idesc_e4m3(128, BN);  // S = Q K^T
            constexpr uint32_t idO = idesc_e4m3(128, D);   // O += P V  (B = V^T tile, K-major)
            constexpr uint32_t kStep = (uint32_t)kTile8 >> 4;  // descriptor units per tile
            const uint64_t qd[2] = {sdesc_sw128(smem_u32(s.q[0]), 16, 1024), sdesc_sw128(smem_u32(s.q[1]), 16, 1024)};
            const uint64_t kd_base = sdesc_sw128(smem_u32(s.k[0]), 16, 1024);
            const uint64_t vd_base = sdesc_sw128(smem_u32(s.vt[0]), 16, 1024);
            const uint64_t pd_base = sdesc_sw128(smem_u32(s.p[0][0]), 16, 1024);  // p[k][b] = base + (2k + b) tiles
            uint32_t sc[2] = {0, 0};  // S tiles issued per query tile
            uint32_t pc[2] = {0, 0};  // P V issued per query tile
            uint32_t oc[2] = {0, 0};  // O tiles completed per query tile
            int gt = 0, n_q = 0;
            bool ok = true;
            // S_k into its TMEM columns once the softmax has read the previous S_k
            auto issue_s = [&](int k, uint64_t kd) -> bool {
                if (sc[k] > 0 && !mbar_wait(&s.s_free[k], (sc[k] - 1) & 1, ab)) return false;
                tc_fence_after();
                mma_f8_ss_k128(tmem + 128u * k, qd[k], kd, idS, 0u);
                tc_commit(&s.s_full[k]);
                ++sc[k];
                return true;
            };
            for (int idx = blockIdx.x, step = first_step(a.snake); ok && idx < a.n_items;
                 idx += step, step = 2 * (int)gridDim.x - step) {
                int t0[2], t1[2], u0, u1;
                {
                    const FwdItem w = fwd_item(a, idx);
                    t0[0] = w.ti[0].t0;
                    t1[0] = w.ti[0].t1;
                    t0[1] = w.ti[1].t0;
                    t1[1] = w.ti[1].t1;
                    u0 = w.u0;
                    u1 = w.u1;
                    if (!w.live) u1 = u0;
                }
                if (u1 <= u0) continue;
                ok = mbar_wait(&s.q_full, n_q & 1, ab);
                ++n_q;
                tc_fence_after();
                // prologue: S for the item's first key tile
                {
                    const int st0 = gt % kStagesK;
                    if (ok && (ok = mbar_wait(&s.k_full[st0], (gt / kStagesK) & 1, ab))) {
                        tc_fence_after();
                        const uint64_t kd0 = kd_base + (uint64_t)(st0 * kStep);
                        for (int k = 0; ok && k < 2; ++k)
                            if (u0 >= t0[k] && u0 < t1[k]) ok = issue_s(k, kd0);
                        tc_commit(&s.k_empty[st0]);
                        if (u1 - u0 == 1) tc_commit(&s.q_empty);
                    }
                }
                int it = gt;
                for (int j = u0; ok && j < u1; ++j, ++it) {
                    // S for key tile j + 1 first: the softmax can go on while P V of tile j runs
                    if (j + 1 < u1) {
                        const int st1 = (it + 1) % kStagesK;
                        if (!(ok = mbar_wait(&s.k_full[st1], ((it + 1) / kStagesK) & 1, ab))) break;
                        tc_fence_after();
                        const uint64_t kd1 = kd_base + (uint64_t)(st1 * kStep);
                        for (int k = 0; ok && k < 2; ++k)
                            if (j + 1 >= t0[k] && j + 1 < t1[k]) ok = issue_s(k, kd1);
                        if (!ok) break;
                        if (j + 2 == u1) tc_commit(&s.q_empty);  // the item's last S
                        tc_commit(&s.k_empty[st1]);
                    }
                    const int st = it % kStagesVt;
                    if (!(ok = mbar_wait(&s.v_full[st], (it / kStagesVt) & 1, ab))) break;
                    const uint64_t vd = vd_base + (uint64_t)(st * kStep);
                    for (int k = 0; ok && k < 2; ++k) {
                        if (j < t0[k] || j >= t1[k]) continue;
                        const uint32_t b = pc[k] & 1;
                        if (!(ok = mbar_wait(&s.p_full[k][b], (pc[k] >> 1) & 1, ab))) break;
                        // the first P V of the item overwrites O_k: the previous epilogue must have read it
                        if (j == t0[k] && oc[k] > 0 && !(ok = mbar_wait(&s.o_free[k], (oc[k] - 1) & 1, ab))) break;
                        tc_fence_after();
                        mma_f8_ss_k128(tmem + 256u + 128u * k, pd_base + (uint64_t)((2 * k + b) * kStep), vd, idO,
                                       j > t0[k] ? 1u : 0u);
                        tc_commit(&s.p_free[k][b]);
                        ++pc[k];
                        if (j == t1[k] - 1) {
                            tc_commit(&s.o_full[k]);
                            ++oc[k];
                        }
                    }
                    if (!ok) break;
                    tc_commit(&s.v_empty[st]);
                }
                gt += u1 - u0;
            }
            tc_commit(&s.drain);
            mbar_wait_quiet(&s.drain, 0);
        }
    } else {
        // ================= V transpose (warps 2, 3) =================
        const int wt = warp - 2;
        int gt = 0;
        bool ok = true;
        for (int idx = blockIdx.x, step = first_step(a.snake); ok && idx < a.n_items;
             idx += step, step = 2 * (int)gridDim.x - step) {
            const FwdItem w = fwd_item(a, idx);
            if (!w.live || w.u1 <= w.u0) continue;
            for (int j = w.u0; j < w.u1; ++j, ++gt) {
                const int sv = gt % kStagesV, st = gt % kStagesVt;
                {
                    // the V tile has landed, and the P V that read this V^T slot last is done
                    bool wv = mbar_wait(&s.vin_full[sv], (gt / kStagesV) & 1, ab);
                    wv = wv && mbar_wait(&s.v_empty[st], ((gt / kStagesVt) & 1) ^ 1, ab);
                    if (!__all_sync(0xffffffffu, wv)) { ok = false; break; }
                }
                transpose_v_tile(s.v[sv], s.vt[st], wt, lane);
                fence_proxy_async_smem();  // the V^T words, for the tensor core's reads
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&s.vin_empty[sv]);
                    mbar_arrive(&s.v_full[st]);
                }
            }
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 216;\n" ::: "memory");
        // ================= softmax: one thread per row =================
        const int k = (warp - 4) >> 2;           // query tile
        const int r = ((warp & 3) << 5) | lane;  // row = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_base + 128 * k;
        const uint32_t tO = tmem + lane_base + 256 + 128 * k;
        uint32_t scount = 0, pcount = 0, ocount = 0;  // carried across items
        bool ok = true;
        for (int idx = blockIdx.x, step = first_step(a.snake); ok && idx < a.n_items;
             idx += step, step = 2 * (int)gridDim.x - step) {
        int my_t0, my_t1, jlo, jhi;
        float c;  // softmax scale x log2(e) x the item's Q and K descales
        {
            const FwdItem w = fwd_item(a, idx);
            if (!w.live) continue;
            my_t0 = k ? w.ti[1].t0 : w.ti[0].t0;
            my_t1 = k ? w.ti[1].t1 : w.ti[0].t1;
            const int i = (k ? w.ti[1].s0 : w.ti[0].s0) + r / p.G;
            const bool rv = (k ? w.ti[1].active : w.ti[0].active) && (r < p.P * p.G) && i < w.sv.nq;
            jlo = rv ? w.band.lo(i) : 1;
            jhi = rv ? w.band.hi(i) : 0;
            const long u = (long)w.sv.b * p.h_kv + w.g;
            c = p.scale_log2 * (a.q_descale ? a.q_descale[u] : 1.f) * (a.k_descale ? a.k_descale[u] : 1.f);
        }
        float m_used = -INFINITY, l = 0.f;
        uint8_t* prow_base = nullptr;
        for (int j = my_t0; j < my_t1; ++j) {
            {
                const bool w = mbar_wait(&s.s_full[k], scount & 1, ab);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
            }
            ++scount;
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld_32x32b_x128(tS, sr);
            // S_k is in registers: its columns may take the next S = Q K^T
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.s_free[k]);
            const int j0 = j * BN;
            const bool edge = (j0 < jlo || j0 + BN - 1 > jhi);
            if (edge) {
#pragma unroll
                for (int cc = 0; cc < BN; ++cc)
                    if (j0 + cc < jlo || j0 + cc > jhi) sr[cc] = __float_as_uint(-INFINITY);
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < BN; cc += 4) {
                mx0 = max3(mx0, __uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1]));
                mx1 = max3(mx1, __uint_as_float(sr[cc + 2]), __uint_as_float(sr[cc + 3]));
            }
            const float m_new = fmaxf(m_used, fmaxf(mx0, mx1) * c);
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
                // O_k may still be the target of the previous P V (tile j - 1 of this item,
                // buffer (pcount - 1) & 1): wait for it, then O_k row *= alpha
                const uint32_t pb = (pcount - 1) & 1;
                const bool w = mbar_wait(&s.p_free[k][pb], ((pcount - 1) >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < D; cb += 32) {
                    uint32_t orr[32];
                    tmem_ld_32x32b_x32(tO + cb, orr);
#pragma unroll
                    for (int t = 0; t < 32; ++t) orr[t] = __float_as_uint(__uint_as_float(orr[t]) * alpha);
                    tmem_st_32x32b_x32(tO + cb, orr);
                }
                tc_fence_before();
            }
            // the P buffer of this step was last read by the P V two steps back
            const uint32_t b = pcount & 1;
            if (pcount >= 2) {
                const bool w = mbar_wait(&s.p_free[k][b], ((pcount - 2) >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
            }
            prow_base = s.p[k][b];
            // P = exp2(S*c - m) -> e4m3, 16 keys (one 16-byte unit) at a time, into the row's
            // swizzled slots of the K-major P tile
            const float base = (m_used == -INFINITY) ? 0.f : m_used;
            const float2 c2 = make_float2(c, c), nb2 = make_float2(-base, -base);
            float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                uint32_t wv[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int cc = 16 * u + 4 * q4;
                    const float2 x0 =
                        __ffma2_rn(make_float2(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])), c2, nb2);
                    const float2 x1 =
                        __ffma2_rn(make_float2(__uint_as_float(sr[cc + 2]), __uint_as_float(sr[cc + 3])), c2, nb2);
                    const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
                    const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
                    sum2 = __fadd2_rn(sum2, p0);
                    sum2 = __fadd2_rn(sum2, p1);
                    wv[q4] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
                }
                *reinterpret_cast<uint4*>(prow_base + sw128_unit(r, u)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
            l += sum2.x + sum2.y;
            // make the generic-proxy writes visible to the MMA, then hand the buffer over
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.p_full[k][b]);
            ++pcount;
        }
        // ---------------- epilogue ----------------
        int idx2 = idx;
        asm volatile("" : "+r"(idx2));
        const FwdItem w = fwd_item(a, idx2);
        const SeqView& sv = w.sv;
        const int g = w.g, split = w.split;
        const int i = (k ? w.ti[1].s0 : w.ti[0].s0) + r / p.G;
        const int h = g * p.G + r % p.G;
        const bool row_valid = (k ? w.ti[1].active : w.ti[0].active) && (r < p.P * p.G) && i < sv.nq;
        const bool has_o = my_t1 > my_t0;
        if (has_o && ok) {
            const bool wt = mbar_wait(&s.o_full[k], ocount & 1, ab);
            ++ocount;
            ok = __all_sync(0xffffffffu, wt);
            tc_fence_after();
        }
        const float vds = a.v_descale ? a.v_descale[(long)sv.b * p.h_kv + g] : 1.f;
        const bool split_mode = a.n_splits > 1 || w.tail;
        float oscale = 0.f, lse = -INFINITY;
        if (!split_mode && p.sinks && row_valid) {
            const float s2 = p.sinks[h] * kLog2e;
            const float mf = fmaxf(m_used, s2);
            const float wgt = (m_used == -INFINITY) ? 0.f : ex2(m_used - mf);
            const float lt = l * wgt + ex2(s2 - mf);
            oscale = wgt / lt * vds;
            lse = (mf + log2f(lt)) * kLn2;
        } else if (l > 0.f) {
            oscale = vds / l;
            lse = (m_used + log2f(l)) * kLn2;
        }
        // split-mode rows: all B h_q s_q rows, or (tail split) those from tail_row0 on
        const long row_base = w.tail ? a.tail_row0 : 0;
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
#pragma unroll
            for (int cb = 0; cb < D; cb += 32) {
                uint32_t orr[32];
                tmem_ld_32x32b_x32(tO + cb, orr);
                if (!row_valid) continue;
                if (!split_mode) {
                    uint16_t* orow = a.o + (token_row(p, sv, i) * p.h_q + h) * D + cb;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        uint4 wv;
                        wv.x = pack_bf16(__uint_as_float(orr[8 * t + 0]) * oscale, __uint_as_float(orr[8 * t + 1]) * oscale);
                        wv.y = pack_bf16(__uint_as_float(orr[8 * t + 2]) * oscale, __uint_as_float(orr[8 * t + 3]) * oscale);
                        wv.z = pack_bf16(__uint_as_float(orr[8 * t + 4]) * oscale, __uint_as_float(orr[8 * t + 5]) * oscale);
                        wv.w = pack_bf16(__uint_as_float(orr[8 * t + 6]) * oscale, __uint_as_float(orr[8 * t + 7]) * oscale);
                        reinterpret_cast<uint4*>(orow)[t] = wv;
                    }
                } else {
                    float* op = a.o_part + ((long)split * nrows + prow) * D + cb;
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        reinterpret_cast<float4*>(op)[t] = make_float4(
                            __uint_as_float(orr[4 * t]) * oscale, __uint_as_float(orr[4 * t + 1]) * oscale,
                            __uint_as_float(orr[4 * t + 2]) * oscale, __uint_as_float(orr[4 * t + 3]) * oscale);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.o_free[k]);
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
        }  // items
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_fwd_e4m3(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            cudaStream_t st) {
    const size_t smem = sizeof(Smem8) + 1024;
    cudaError_t e = cudaFuncSetAttribute(fwd_e4m3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (a.n_items <= 0 || a.n_ctas <= 0) return cudaSuccess;
    fwd_e4m3_kernel<<<(unsigned)a.n_ctas, kThreads8, smem, st>>>(a, tq, tk, tv);
    return cudaGetLastError();
}

}  // namespace fa
