// Decode-shaped forward (few query rows per key/value head) and the split-KV combine.
//
// With s_q * (h_q / h_kv) <= 16 query rows per key/value head the work is a stream over
// the key/value cache: about 2 multiply-adds per byte read, far below what the tensor
// cores would need, so this path runs on the CUDA cores and is sized to keep HBM busy.
// The cache of one (batch, key/value head) is split across CTAs, each CTA writes a
// partial (O, LSE) for its key range, and a second kernel merges the partials by their
// log-sum-exp (vllm-project/flash-attention README, changelog 2.2 "Optimize for
// inference": split the KV load across thread blocks, combine in a separate kernel).
#include "common.cuh"

namespace fa {
namespace {

constexpr int kThreadsDec = 256;
constexpr int BK = 64;        // keys per tile
constexpr int RMAX = 16;      // query rows per CTA

template <int D>
struct DecCfg {
    static constexpr int KCH = D / 64;
    static constexpr int CHUNK = BK * 128;             // [64 rows][64 cols] bf16, swizzled
    static constexpr int TILE = BK * D * 2;            // one K (or V) tile
    static constexpr int STAGES = (D == 256) ? 3 : 4;
    static constexpr int DP = D / 2;                   // column pairs
    static constexpr int KG = kThreadsDec / DP;        // key groups in the P.V phase
};

template <int D>
struct __align__(1024) DecSmem {
    uint8_t k[DecCfg<D>::STAGES][DecCfg<D>::TILE];
    uint8_t v[DecCfg<D>::STAGES][DecCfg<D>::TILE];
    float q[RMAX][D];        // query rows pre-multiplied by scale * log2(e)
    float sc[RMAX][BK];      // scores, then probabilities
    float alpha[RMAX];
    float m[RMAX], l[RMAX];
    uint64_t full[DecCfg<D>::STAGES];
    int abort_flag;
};

// Byte offset of element (row, col) of a [rows][64] bf16 chunk written by a TMA load with
// 128-byte swizzle: the 16-byte unit index is XORed with row % 8.
__device__ __forceinline__ int sw128(int row, int col) {
    return row * 128 + ((((col >> 3) ^ row) & 7) << 4) + ((col & 7) << 1);
}

template <int D>
__global__ void __launch_bounds__(kThreadsDec) decode_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                                                             const __grid_constant__ CUtensorMap tmv) {
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    DecSmem<D>& s = *reinterpret_cast<DecSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Problem& p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int R = p.s_q * p.G;
    const Band band{p.s_kv - p.s_q, p.left, p.right, p.s_kv};

    // key range of this split, clipped to the union of the rows' bands
    int j_begin = split * a.split_keys, j_end = min(p.s_kv, (split + 1) * a.split_keys);
    {
        const int lo = band.lo(0), hi = band.hi(p.s_q - 1);
        j_begin = max(j_begin, lo);
        j_end = min(j_end, hi + 1);
    }
    const int t_begin = j_begin / BK;
    const int n_tiles = j_end > j_begin ? (j_end - 1) / BK + 1 - t_begin : 0;

    // an earlier CTA of this launch gave up: do not start new work
    if (a.status && *reinterpret_cast<volatile int*>(a.status) != 0) return;
    Abort ab{&s.abort_flag, a.status};
    if (tid == 0) {
        s.abort_flag = 0;
        for (int i = 0; i < C::STAGES; ++i) mbar_init(&s.full[i], 1);
        fence_mbar_init();
    }
    for (int x = tid; x < RMAX * D; x += kThreadsDec) {
        const int r = x / D, c = x % D;
        float val = 0.f;
        if (r < R) {
            const int i = r / p.G, h = g * p.G + r % p.G;
            val = __bfloat162float(a.q[(((long)b * p.s_q + i) * p.h_q + h) * D + c]) * p.scale_log2;
        }
        s.q[r][c] = val;
    }
    if (tid < RMAX) {
        s.m[tid] = -INFINITY;
        s.l[tid] = 0.f;
    }
    __syncthreads();

    auto issue = [&](int t) {  // tile t (relative) into stage t % STAGES
        const int st = t % C::STAGES;
        const int j0 = (t_begin + t) * BK;
        mbar_expect_tx(&s.full[st], 2 * C::TILE);
        for (int c = 0; c < C::KCH; ++c) {
            tma_load_4d(&s.k[st][c * C::CHUNK], &tmk, &s.full[st], c * 64, g, j0, b);
            tma_load_4d(&s.v[st][c * C::CHUNK], &tmv, &s.full[st], c * 64, g, j0, b);
        }
    };
    if (tid == 0) {
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        for (int t = 0; t < C::STAGES && t < n_tiles; ++t) issue(t);
    }

    // P.V accumulators: column pair dp, key group kg, all rows
    const int dp = tid % C::DP, kg = tid / C::DP;
    float acc[RMAX][2];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) acc[r][0] = acc[r][1] = 0.f;

    int issued = min(C::STAGES, n_tiles);
    int consumed = 0;  // tiles whose copies have landed and been waited for
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % C::STAGES;
        const bool w = mbar_wait(&s.full[st], (t / C::STAGES) & 1, ab);
        if (!__syncthreads_and(w)) {
            ok = false;
            break;
        }
        consumed = t + 1;
        const int j0 = (t_begin + t) * BK;
        // ---- scores: thread = (key, row group) ----
        {
            const int jj = tid & (BK - 1);
            const int rg = tid / BK;  // 0..3
            const uint8_t* kb = s.k[st];
            float dots[RMAX / 4];
#pragma unroll
            for (int u = 0; u < RMAX / 4; ++u) dots[u] = 0.f;
#pragma unroll 4
            for (int c8 = 0; c8 < D; c8 += 8) {
                const uint4 kv = *reinterpret_cast<const uint4*>(kb + (c8 >> 6) * C::CHUNK + sw128(jj, c8 & 63));
                const float k0 = bf16_lo(kv.x), k1 = bf16_hi(kv.x), k2 = bf16_lo(kv.y), k3 = bf16_hi(kv.y);
                const float k4 = bf16_lo(kv.z), k5 = bf16_hi(kv.z), k6 = bf16_lo(kv.w), k7 = bf16_hi(kv.w);
#pragma unroll
                for (int u = 0; u < RMAX / 4; ++u) {
                    const int r = rg + 4 * u;
                    if (r < R) {
                        const float4 qa = *reinterpret_cast<const float4*>(&s.q[r][c8]);
                        const float4 qb = *reinterpret_cast<const float4*>(&s.q[r][c8 + 4]);
                        float d0 = dots[u];
                        d0 = fmaf(qa.x, k0, d0);
                        d0 = fmaf(qa.y, k1, d0);
                        d0 = fmaf(qa.z, k2, d0);
                        d0 = fmaf(qa.w, k3, d0);
                        d0 = fmaf(qb.x, k4, d0);
                        d0 = fmaf(qb.y, k5, d0);
                        d0 = fmaf(qb.z, k6, d0);
                        d0 = fmaf(qb.w, k7, d0);
                        dots[u] = d0;
                    }
                }
            }
            const int j = j0 + jj;
#pragma unroll
            for (int u = 0; u < RMAX / 4; ++u) {
                const int r = rg + 4 * u;
                if (r < R) {
                    const int i = r / p.G;
                    const bool keep = j >= j_begin && j < j_end && j >= band.lo(i) && j <= band.hi(i);
                    s.sc[r][jj] = keep ? dots[u] : -INFINITY;
                }
            }
        }
        __syncthreads();
        // ---- online softmax: warp w owns rows w and w + 8 ----
        for (int r = warp; r < R; r += kThreadsDec / 32) {
            const float x0 = s.sc[r][lane], x1 = s.sc[r][lane + 32];
            float mx = fmaxf(x0, x1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_old = s.m[r];
            const float m_new = fmaxf(m_old, mx);
            const float base = (m_new == -INFINITY) ? 0.f : m_new;
            const float p0 = ex2(x0 - base), p1 = ex2(x1 - base);
            float sum = p0 + p1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            s.sc[r][lane] = p0;
            s.sc[r][lane + 32] = p1;
            __syncwarp();
            if (lane == 0) {
                const float al = (m_old == -INFINITY) ? 0.f : ex2(m_old - base);
                s.alpha[r] = al;
                s.l[r] = s.l[r] * al + sum;
                s.m[r] = m_new;
            }
        }
        __syncthreads();
        // ---- O += P V: thread = (column pair, key group) ----
        {
#pragma unroll
            for (int r = 0; r < RMAX; ++r) {
                if (r < R) {
                    const float al = s.alpha[r];
                    acc[r][0] *= al;
                    acc[r][1] *= al;
                }
            }
            const uint8_t* vb = s.v[st];
            const int c = 2 * dp;
            constexpr int KPG = BK / C::KG;  // keys per group
            for (int kk = 0; kk < KPG; ++kk) {
                const int jj = kg * KPG + kk;
                const uint32_t vv = *reinterpret_cast<const uint32_t*>(vb + (c >> 6) * C::CHUNK + sw128(jj, c & 63));
                const float v0 = bf16_lo(vv), v1 = bf16_hi(vv);
#pragma unroll
                for (int r = 0; r < RMAX; ++r) {
                    if (r < R) {
                        const float pr = s.sc[r][jj];
                        acc[r][0] = fmaf(pr, v0, acc[r][0]);
                        acc[r][1] = fmaf(pr, v1, acc[r][1]);
                    }
                }
            }
        }
        __syncthreads();  // stage st and the scores are free again
        if (tid == 0 && issued < n_tiles) {
            issue(issued);
            ++issued;
        }
    }
    // abort path: wait for the copies issued but never waited for (at most STAGES of
    // them, each the latest phase of its stage) before the shared memory goes away
    if (tid == 0) {
        for (int t = consumed; t < issued; ++t) mbar_wait_quiet(&s.full[t % C::STAGES], (t / C::STAGES) & 1);
    }
    __syncthreads();

    // ---- reduce the key groups and write the partial (O / l, LSE) ----
    float* red = reinterpret_cast<float*>(s.k[0]);  // [KG][RMAX][D] floats, fits in the K stages
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        if (r < R) {
            red[(kg * RMAX + r) * D + 2 * dp] = acc[r][0];
            red[(kg * RMAX + r) * D + 2 * dp + 1] = acc[r][1];
        }
    }
    __syncthreads();
    const long nrows = (long)p.B * p.h_q * p.s_q;
    for (int x = tid; x < R * D; x += kThreadsDec) {
        const int r = x / D, c = x % D;
        float sum = 0.f;
        for (int q = 0; q < C::KG; ++q) sum += red[(q * RMAX + r) * D + c];
        const int i = r / p.G, h = g * p.G + r % p.G;
        const long row = ((long)b * p.h_q + h) * p.s_q + i;
        const float l = s.l[r];
        a.o_part[((long)split * nrows + row) * D + c] = (l > 0.f && ok) ? sum / l : 0.f;
        if (c == 0) a.lse_part[(long)split * nrows + row] = (l > 0.f && ok) ? (s.m[r] + log2f(l)) * kLn2 : -INFINITY;
    }
}

// One warp per output row: merge the splits' partials by their log-sum-exp and fold in
// the sink, which joins the denominator exactly once.
__global__ void combine_kernel(const CombineArgs a) {
    const Problem& p = a.p;
    const long nrows = (long)p.B * p.h_q * p.s_q;
    const long row = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= nrows) return;
    const int i = (int)(row % p.s_q);
    const int h = (int)((row / p.s_q) % p.h_q);
    const int b = (int)(row / ((long)p.s_q * p.h_q));
    float mx = -INFINITY;
    for (int sp = 0; sp < a.n_splits; ++sp) mx = fmaxf(mx, a.lse_part[sp * nrows + row]);
    const float sink = p.sinks ? p.sinks[h] : -INFINITY;
    const float m_all = fmaxf(mx, sink);
    float den = 0.f;
    for (int sp = 0; sp < a.n_splits; ++sp) {
        const float x = a.lse_part[sp * nrows + row];
        den += (x == -INFINITY) ? 0.f : __expf(x - m_all);
    }
    const float den_keys = den;
    if (p.sinks) den += __expf(sink - m_all);
    const float lse = den > 0.f ? m_all + __logf(den) : -INFINITY;
    const int D = p.d;
    __nv_bfloat16* out = a.o + (((long)b * p.s_q + i) * p.h_q + h) * D;
    for (int c = lane * 4; c < D; c += 128) {
        float4 o = make_float4(0, 0, 0, 0);
        if (den_keys > 0.f) {
            for (int sp = 0; sp < a.n_splits; ++sp) {
                const float x = a.lse_part[sp * nrows + row];
                if (x == -INFINITY) continue;
                const float w = __expf(x - m_all) / den;
                const float4 v = *reinterpret_cast<const float4*>(a.o_part + (sp * nrows + row) * D + c);
                o.x += w * v.x;
                o.y += w * v.y;
                o.z += w * v.z;
                o.w += w * v.w;
            }
        }
        uint2 packed;
        packed.x = pack_bf16(o.x, o.y);
        packed.y = pack_bf16(o.z, o.w);
        *reinterpret_cast<uint2*>(out + c) = packed;
    }
    if (lane == 0 && a.lse) a.lse[((long)b * p.h_q + h) * p.s_q + i] = lse;
}

}  // namespace

template <int D>
static cudaError_t launch_decode_d(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    const size_t smem = sizeof(DecSmem<D>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.n_splits, a.p.h_kv, a.p.B);
    decode_kernel<D><<<grid, kThreadsDec, smem, st>>>(a, tk, tv);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    switch (a.p.d) {
        case 64: return launch_decode_d<64>(a, tk, tv, st);
        case 128: return launch_decode_d<128>(a, tk, tv, st);
        case 256: return launch_decode_d<256>(a, tk, tv, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
    const long nrows = (long)a.p.B * a.p.h_q * a.p.s_q;
    const int rows_per_block = 8;
    const long blocks = (nrows + rows_per_block - 1) / rows_per_block;
    combine_kernel<<<(unsigned)blocks, rows_per_block * 32, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace fa
