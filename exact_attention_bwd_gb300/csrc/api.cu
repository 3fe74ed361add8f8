// C ABI of the library (include/fa.h): argument checks, planning, TMA descriptors and
// launches on the caller's stream.  Nothing here allocates device memory: every
// scratch buffer is carved out of the caller's workspace.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "kernels.h"
#include "trace.cuh"

namespace fa {
namespace {

// ------------------------------------------------------------------------------------------
// device properties and the driver's tensor-map encoder
// ------------------------------------------------------------------------------------------
int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cached[dev] = n;
    }
    return cached[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 4-D tensor map of 16-bit elements (fp16 if f16, else bf16) over [b][s][h][d] (innermost
// first: d, h, s, b) with a (64, box_h, box_s, 1) box and 128-byte swizzle.  Out-of-range
// rows read as zero.
bool encode_bhsd(CUtensorMap* m, const void* base, int d, int h, int s, int b, int box_h, int box_s, bool f16) {
    auto fn = encoder();
    if (!fn) return false;
    if (s <= 0 || b <= 0) {
        std::memset(m, 0, sizeof(*m));  // never dereferenced: no tile of this tensor is loaded
        return true;
    }
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)h, (cuuint64_t)s, (cuuint64_t)b};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)h * d * 2, (cuuint64_t)s * h * d * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)box_h, (cuuint32_t)box_s, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D tensor map over one-byte (e4m3) elements, 128-byte swizzle.  dims innermost first;
// strides in bytes for dims 1..3.  Out-of-range elements read as zero.
bool encode_u8_4d(CUtensorMap* m, const void* base, const cuuint64_t dims[4], const cuuint64_t strides[3],
                  const cuuint32_t box[4]) {
    auto fn = encoder();
    if (!fn) return false;
    if (dims[2] == 0 || dims[3] == 0 || dims[0] == 0) {
        std::memset(m, 0, sizeof(*m));  // never dereferenced: no tile of this tensor is loaded
        return true;
    }
    cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
    cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), d, st, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------------------------------
// profiling hooks
// ------------------------------------------------------------------------------------------
const char* const kKernelNames[] = {"fwd", "decode", "combine", "bwd_pre", "bwd_main", "bwd_post"};
enum KernelId { kFwd = 0, kDecode, kCombine, kBwdPre, kBwdMain, kBwdPost, kNumKernels };

struct Profiler {
    std::mutex mu;
    bool on = false;
    cudaEvent_t ev[kNumKernels][2] = {};
    bool recorded[kNumKernels] = {};
};
Profiler& prof() {
    static Profiler p;
    return p;
}

template <class F>
cudaError_t timed(KernelId id, cudaStream_t st, F&& launch) {
    Profiler& P = prof();
    bool on;
    {
        std::lock_guard<std::mutex> g(P.mu);
        on = P.on;
    }
    if (!on) return launch();
    cudaEventRecord(P.ev[id][0], st);
    cudaError_t e = launch();
    cudaEventRecord(P.ev[id][1], st);
    std::lock_guard<std::mutex> g(P.mu);
    P.recorded[id] = (e == cudaSuccess);
    return e;
}

// ------------------------------------------------------------------------------------------
// argument normalisation
// ------------------------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Default bound on each pipeline wait of a kernel (2 s; fa_params.wait_limit_ns = 0).
constexpr unsigned long long kWaitLimitNsDefault = 2000000000ull;

// Host-visible total token counts of a packed call are not known without reading the
// offsets; the caller passes them as s_q / s_kv (T_q, T_k).
fa_status normalise(const fa_params* in, Problem& p) {
    if (!in) return FA_ERR_INVALID_ARG;
    const fa_params& a = *in;
    if (a.B < 0 || a.s_q < 0 || a.s_kv < 0 || a.h_q <= 0 || a.h_kv <= 0 || a.d <= 0) return FA_ERR_INVALID_ARG;
    if (a.h_q % a.h_kv != 0) return FA_ERR_INVALID_ARG;
    if ((a.cu_seqlens_q == nullptr) != (a.cu_seqlens_k == nullptr)) return FA_ERR_INVALID_ARG;
    if (a.window_left < -1 || a.window_right < -1) return FA_ERR_INVALID_ARG;
    if (a.d % 8 != 0 || a.d > 256) return FA_ERR_UNSUPPORTED;
    if (a.dtype != FA_DTYPE_BF16 && a.dtype != FA_DTYPE_F16 && a.dtype != FA_DTYPE_E4M3) return FA_ERR_INVALID_ARG;
    // e4m3: d = 128 (dense, packed or a paged cache)
    if (a.dtype == FA_DTYPE_E4M3 && a.d != 128) return FA_ERR_UNSUPPORTED;
    std::memset(&p, 0, sizeof(p));
    p.B = a.B;
    p.s_q = a.s_q;
    p.s_kv = a.s_kv;
    p.h_q = a.h_q;
    p.h_kv = a.h_kv;
    p.d = a.d;
    p.G = a.h_q / a.h_kv;
    if (p.G > 128) return FA_ERR_UNSUPPORTED;
    p.P = 128 / p.G;
    p.scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / std::sqrt((float)a.d);
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.causal = a.causal ? 1 : 0;
    p.left = a.window_left;
    p.right = a.window_right;
    if (p.causal) p.right = 0;  // intersection of the causal mask with any right window
    p.sinks = a.sinks;
    p.cu_q = a.cu_seqlens_q;
    p.cu_k = a.cu_seqlens_k;
    if (p.cu_q) {
        p.T_q = a.s_q;
        p.T_k = a.s_kv;
    }
    p.dtype = a.dtype;
    p.wait_ns = a.wait_limit_ns ? a.wait_limit_ns : kWaitLimitNsDefault;
    // KV-cache forms: a per-sequence used length, and a paged cache (dense q only)
    p.seqused_q = a.seqused_q;
    p.seqused_k = a.seqused_k;
    p.block_table = a.block_table;
    if (a.block_table) {
        if (p.cu_q) return FA_ERR_UNSUPPORTED;
        if (a.page_size <= 0 || a.page_size % 128 != 0 || a.max_blocks_per_seq <= 0 || a.num_pages <= 0)
            return FA_ERR_INVALID_ARG;
        if ((long)a.max_blocks_per_seq * a.page_size < (long)a.s_kv) return FA_ERR_INVALID_ARG;
        p.page_size = a.page_size;
        p.max_blocks = a.max_blocks_per_seq;
    }
    return FA_OK;
}

// ------------------------------------------------------------------------------------------
// forward plan
// ------------------------------------------------------------------------------------------
enum class FwdPath { kEmpty, kTensor, kDecode };

constexpr int kDecodeKeys = 64;     // keys per decode tile
constexpr double kBandBytes = 64.0 * (1 << 20);  // L2 share for one band of backward units
constexpr size_t kStatusBytes = 256;

struct FwdPlan {
    FwdPath path = FwdPath::kEmpty;
    int n_blocks = 0, n_splits = 1, split_tiles = 0;
    int unit_major = 0;
    int tokens = 0;        // packed batch with cu_seqlens_q == cu_seqlens_k: token tiles
    int kt = 128;          // keys per key tile of the d <= 128 kernel (64: two CTAs per SM)
    int tail_units = 0, tail_k = 0, tail_split_tiles = 0;  // tail split (d = 192 / 256)
    size_t part_rows = 0;  // rows of the split partials
    size_t off_trace = 0;  // trace builds: the per-role event records (tensor-core path)
    size_t ws_bytes = kStatusBytes;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Head dimensions with kernels: 64 and 128 (two query tiles per CTA), 192 and 256 (one).
bool supported_d(int d) { return d == 64 || d == 128 || d == 192 || d == 256; }

// Chooses the number of KV splits that minimises (waves) x (tiles per split), with a
// small charge per split for the partial results written and read back.
int choose_splits(long ctas, int tiles, int slots, double part_cost_per_split) {
    int best = 1;
    double best_cost = 1e300;
    for (int s = 1; s <= 64 && s <= tiles; ++s) {
        const int per = (tiles + s - 1) / s;
        const long waves = (ctas * s + slots - 1) / slots;
        const double cost = (double)waves * per * (1.0 + (s > 1 ? part_cost_per_split * s : 0.0));
        if (cost < best_cost * 0.98) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

fa_status plan_fwd(const Problem& p, unsigned flags, FwdPlan& pl) {
    pl = FwdPlan();
    const long rows_total = p.cu_q ? (long)p.T_q : (long)p.B * p.s_q;
    if (p.B == 0 || rows_total == 0) return FA_OK;  // nothing to compute
    const bool dense = p.cu_q == nullptr;
    const int R = p.s_q * p.G;  // query rows per key/value head (dense)
    if (dense && p.dtype != FA_DTYPE_E4M3 && supported_d(p.d) && R <= decode_rows_max(p.d)) {
        pl.path = FwdPath::kDecode;
        const int tiles = (p.s_kv + kDecodeKeys - 1) / kDecodeKeys;
        const long units = (long)p.B * p.h_kv;
        const int slots = sm_count() * decode_ctas_per_sm(p.d, R);
        // partials: R rows x (d + 1) floats per split, written and read, against the
        // unit's 2 * s_kv * d 16-bit elements of keys and values
        const double part = p.s_kv > 0 ? (double)R * (p.d + 1) * 8.0 / ((double)p.s_kv * p.d * 4.0) : 1.0;
        pl.n_splits = tiles > 0 ? choose_splits(units, tiles, slots, part) : 1;
        pl.split_tiles = tiles > 0 ? (tiles + pl.n_splits - 1) / pl.n_splits : 0;
        pl.n_splits = pl.split_tiles > 0 ? (tiles + pl.split_tiles - 1) / pl.split_tiles : 1;
        pl.part_rows = (size_t)p.B * p.h_q * p.s_q;
        pl.ws_bytes = kStatusBytes + align256(pl.part_rows * pl.n_splits * p.d * 4) +
                      align256(pl.part_rows * pl.n_splits * 4);
        return FA_OK;
    }
    if (!supported_d(p.d)) return FA_ERR_UNSUPPORTED;
    pl.path = FwdPath::kTensor;
    // d <= 128: two 128-row query tiles and 128-key tiles per CTA; d = 192 / 256: one query
    // tile and 64-key tiles (the d-column accumulator fills much of the tensor memory)
    const int rows_per_cta = (p.d >= 192 ? 1 : 2) * p.P;
    const int kv_tile = p.d >= 192 ? 64 : kTileRows;
    if (dense) {
        pl.n_blocks = (p.s_q + rows_per_cta - 1) / rows_per_cta;
        const int tiles = (p.s_kv + kv_tile - 1) / kv_tile;
        const long ctas = (long)pl.n_blocks * p.h_kv * p.B;
        pl.n_splits = 1;
        if (!(flags & FA_FLAG_NO_SPLIT) && !p.causal && p.left < 0 && p.right < 0 && tiles >= 8 &&
            ctas < 4L * sm_count()) {
            const double part = (double)(2 * 128) * (p.d + 1) * 8.0 / ((double)p.s_kv * p.d * 4.0);
            pl.n_splits = choose_splits(ctas, tiles, sm_count(), part);
        } else if (!(flags & FA_FLAG_NO_SPLIT) && tiles >= 8 && ctas < 4L * sm_count() && p.s_q * 4 <= p.s_kv) {
            // masked decode-like shapes: every query block sees (almost) every key
            const double part = (double)(2 * 128) * (p.d + 1) * 8.0 / ((double)p.s_kv * p.d * 4.0);
            pl.n_splits = choose_splits(ctas, tiles, sm_count(), part);
        }
        if (pl.n_splits > 1) {
            pl.split_tiles = (tiles + pl.n_splits - 1) / pl.n_splits;
            pl.n_splits = (tiles + pl.split_tiles - 1) / pl.split_tiles;
        }
        // few queries against a long key range: every query block does about the same work,
        // so launch the blocks of one (batch, kv head) together and let them share K/V in L2
        pl.unit_major = (p.s_q * 4 <= p.s_kv) ? 1 : 0;
        // Tail split.  Where every item takes about as long (few queries against a long key
        // range), a last partial round of items leaves the other SMs idle for a whole item;
        // the last units' items are cut into k key ranges instead (k chosen so that the
        // pieces fill the last round best) and their rows merged by the combine.  d = 192 /
        // 256 (one CTA per item and per SM) takes it in place of no split; d <= 128 (the
        // persistent kernels, 16-bit and e4m3) in place of splitting every unit's keys when it
        // is as short (only the tail's rows then go through the fp32 partials), or in place of
        // no split when it is shorter.
        const bool wide = p.d >= 192;
        const bool tail_ok = wide ? pl.n_splits == 1 : true;
        if (tail_ok && pl.unit_major && p.left < 0 && tiles >= (wide ? 64 : 8)) {
            const long units = (long)p.h_kv * p.B, items = units * pl.n_blocks, slots = sm_count();
            const long rem = items % slots;
            if (items > slots && rem > 0) {
                const long tail_units = (rem + pl.n_blocks - 1) / pl.n_blocks;
                const long tail = tail_units * pl.n_blocks;
                // the tail's duration in whole items: ceil(k tail / slots) / k (1 without a split)
                double best = (double)((tail + slots - 1) / slots);
                int best_k = 1;
                for (int k = 2; k <= 8; ++k) {
                    const double len = (double)((k * tail + slots - 1) / slots) / k;
                    if (len < best - 1e-9) {
                        best = len;
                        best_k = k;
                    }
                }
                bool take = best_k > 1 && best <= 0.8;
                if (take && !wide) {
                    // in item-rounds, against every unit split n ways (ceil(n items / slots) / n)
                    // or against no split (ceil(items / slots))
                    const double mine = (double)((items - tail + slots - 1) / slots) + best;
                    if (pl.n_splits > 1)
                        take = mine <= (double)((pl.n_splits * items + slots - 1) / slots) / pl.n_splits + 1e-9;
                    else
                        take = mine < (double)((items + slots - 1) / slots) - 1e-9;
                }
                if (take) {
                    pl.n_splits = 1;
                    pl.split_tiles = 0;
                    pl.tail_units = (int)tail_units;
                    pl.tail_k = best_k;
                    pl.tail_split_tiles = (tiles + best_k - 1) / best_k;
                    pl.part_rows = (size_t)tail_units * p.G * p.s_q;
                    pl.ws_bytes = kStatusBytes + align256(pl.part_rows * best_k * p.d * 4) +
                                  align256(pl.part_rows * best_k * 4);
                }
            }
        }
        if (pl.n_splits > 1) {
            pl.part_rows = (size_t)p.B * p.h_q * p.s_q;
            pl.ws_bytes = kStatusBytes + align256(pl.part_rows * pl.n_splits * p.d * 4) +
                          align256(pl.part_rows * pl.n_splits * 4);
        }
    } else if (p.cu_q == p.cu_k && p.d <= 128 && p.dtype != FA_DTYPE_E4M3) {
        // queries and keys packed alike: tiles run over the packed token axis
        pl.tokens = 1;
        pl.n_blocks = (p.T_q + rows_per_cta - 1) / rows_per_cta;
    } else {
        pl.n_blocks = p.T_q / rows_per_cta + p.B;
    }
    // d = 64 under a narrow band (windows on both sides, a causal mask counting as a right
    // window of 0; a query tile's allowed keys span at most 384): an item sees a few key
    // tiles and its chain of waits sets the pace, so take 64-key tiles and run two CTAs per
    // SM (twice the query tiles in flight)
    if (p.d == 64 && p.dtype != FA_DTYPE_E4M3 && pl.n_splits == 1 && p.left >= 0 && p.right >= 0 &&
        (long)p.left + p.right + p.P <= 384)
        pl.kt = 64;
#ifdef FA_TRACE
    pl.off_trace = pl.ws_bytes;
    pl.ws_bytes += align256(kTraceBytes);
#endif
    return FA_OK;
}

// ------------------------------------------------------------------------------------------
// backward plan
// ------------------------------------------------------------------------------------------
struct BwdPlan {
    bool empty = true;
    int n_qtiles = 0, n_kvblocks = 0, n_bands = 1;
    int tokens = 0;  // packed batch with cu_seqlens_q == cu_seqlens_k: token blocks and tiles
    size_t off_delta = 0, off_lse2 = 0, off_dq = 0, off_sink = 0, off_count = 0, off_trace = 0;
    size_t ws_bytes = kStatusBytes;
};

fa_status plan_bwd(const Problem& p, unsigned flags, BwdPlan& pl) {
    pl = BwdPlan();
    if (!supported_d(p.d)) return FA_ERR_UNSUPPORTED;
    if (p.block_table) return FA_ERR_UNSUPPORTED;  // paged caches: forward only
    if (p.dtype == FA_DTYPE_E4M3) return FA_ERR_UNSUPPORTED;      // e4m3: forward only
    const long rows_total = p.cu_q ? (long)p.T_q : (long)p.B * p.s_q;
    const long keys_total = p.cu_q ? (long)p.T_k : (long)p.B * p.s_kv;
    if (p.B == 0 || (rows_total == 0 && keys_total == 0)) return FA_OK;
    pl.empty = false;
    const int kvb = p.d >= 192 ? 64 : kTileRows;  // keys per CTA (d = 192 / 256: 64)
    if (p.cu_q && p.cu_q == p.cu_k && p.d <= 128 && !(flags & FA_FLAG_DETERMINISTIC)) {
        // queries and keys packed alike: key blocks and query tiles run over the packed axis
        pl.tokens = 1;
        pl.n_qtiles = (p.T_q + p.P - 1) / p.P;
        pl.n_kvblocks = (p.T_k + kvb - 1) / kvb;
    } else if (p.cu_q) {
        pl.n_qtiles = p.T_q / p.P + p.B;
        pl.n_kvblocks = p.T_k / kvb + p.B;
    } else {
        pl.n_qtiles = p.B * ((p.s_q + p.P - 1) / p.P);
        pl.n_kvblocks = (p.s_kv + kvb - 1) / kvb;
        // a (batch, key/value head) unit's CTAs all read its Q and dO tiles and add into its
        // dQ accumulator rows (16-bit Q + dO, fp32 accumulator: 8 bytes per row and column);
        // take as many units at a time as keep that within half the L2, in bands of
        // near-equal size (a small last band would start its heaviest blocks last)
        const double unit_bytes = (double)p.s_q * p.G * p.d * 8.0;
        const int hb = p.h_kv * p.B;
        int u = unit_bytes > 0 ? (int)(kBandBytes / unit_bytes) : hb;
        u = u < 1 ? 1 : (u > hb ? hb : u);
        pl.n_bands = (hb + u - 1) / u;
    }
    const size_t stat = (size_t)p.h_kv * pl.n_qtiles * 128 * 4;
    pl.off_delta = kStatusBytes;
    pl.off_lse2 = pl.off_delta + align256(stat);
    pl.off_dq = pl.off_lse2 + align256(stat);
    pl.ws_bytes = pl.off_dq + align256((size_t)p.h_kv * pl.n_qtiles * 128 * p.d * 4);
    if (p.sinks) {  // per-row sink-gradient terms, summed per head in a fixed order
        pl.off_sink = pl.ws_bytes;
        pl.ws_bytes += align256(stat);
    }
    if (flags & FA_FLAG_DETERMINISTIC) {  // one counter per (key/value head, query tile)
        pl.off_count = pl.ws_bytes;
        pl.ws_bytes += align256((size_t)p.h_kv * pl.n_qtiles * 4);
    }
#ifdef FA_TRACE
    pl.off_trace = pl.ws_bytes;
    pl.ws_bytes += align256(kTraceBytes);
#endif
    return FA_OK;
}

fa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

__global__ void validate_cu_kernel(const int32_t* cu_q, const int32_t* cu_k, int n, int Tq, int Tk, int* status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i > n) return;
    bool bad = false;
    if (i == 0) bad = cu_q[0] != 0 || cu_k[0] != 0;
    if (i == n) bad = bad || cu_q[n] != Tq || cu_k[n] != Tk;
    if (i < n) bad = bad || cu_q[i + 1] < cu_q[i] || cu_k[i + 1] < cu_k[i];
    if (bad) atomicCAS(status, 0, 6);
}

fa_status maybe_validate(const Problem& p, unsigned flags, int* status, cudaStream_t st) {
    if (!(flags & FA_FLAG_VALIDATE_CU) || !p.cu_q) return FA_OK;
    validate_cu_kernel<<<(p.B + 1 + 255) / 256, 256, 0, st>>>(p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, status);
    return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

#ifdef FA_TRACE
const char* fa_version(void) { return "fa_gb300 0.1 (sm_103a, tcgen05) trace build"; }
#else
const char* fa_version(void) { return "fa_gb300 0.1 (sm_103a, tcgen05)"; }
#endif

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARG: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported problem";
        case FA_ERR_WORKSPACE: return "workspace too small";
        case FA_ERR_CUDA: return "CUDA error";
        case FA_ERR_TIMEOUT: return "kernel pipeline timed out";
        case FA_ERR_DEVICE_CHECK: return "device-side argument check failed";
    }
    return "unknown status";
}

size_t fa_fwd_workspace_size(const fa_params* in) {
    Problem p;
    if (normalise(in, p) != FA_OK) return 0;
    FwdPlan pl;
    if (plan_fwd(p, in->flags, pl) != FA_OK) return 0;
    return pl.ws_bytes;
}

size_t fa_bwd_workspace_size(const fa_params* in) {
    Problem p;
    if (normalise(in, p) != FA_OK) return 0;
    BwdPlan pl;
    if (plan_bwd(p, in->flags, pl) != FA_OK) return 0;
    return pl.ws_bytes;
}

fa_status fa_fwd(const fa_params* in, const void* q, const void* k, const void* v, void* o, float* lse,
                 void* workspace, size_t ws_bytes, struct CUstream_st* stream) {
    Problem p;
    fa_status rc = normalise(in, p);
    if (rc != FA_OK) return rc;
    FwdPlan pl;
    if ((rc = plan_fwd(p, in->flags, pl)) != FA_OK) return rc;
    if (!workspace || !aligned16(workspace)) return FA_ERR_INVALID_ARG;
    if (ws_bytes < pl.ws_bytes) return FA_ERR_WORKSPACE;
    const long rows_total = p.cu_q ? (long)p.T_q : (long)p.B * p.s_q;
    const long keys_total = p.cu_q ? (long)p.T_k : (long)p.B * p.s_kv;
    if (rows_total > 0 && (!q || !o || !aligned16(q) || !aligned16(o))) return FA_ERR_INVALID_ARG;
    if (keys_total > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return FA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int* status = reinterpret_cast<int*>(workspace);
    if ((rc = cuda_status(cudaMemsetAsync(status, 0, sizeof(int), st))) != FA_OK) return rc;
    if ((rc = maybe_validate(p, in->flags, status, st)) != FA_OK) return rc;
    if (pl.path == FwdPath::kEmpty) return FA_OK;

    const int tokens_q = p.cu_q ? p.T_q : p.s_q;
    const int tokens_k = p.cu_q ? p.T_k : p.s_kv;
    const int bdim = p.cu_q ? 1 : p.B;
    CUtensorMap tk, tv;
    const int kv_box = (pl.path == FwdPath::kDecode || p.d >= 192) ? 64 : pl.kt;
    // a paged cache is a [num_pages][page_size][h_kv][d] pool: the map's key and outer
    // dimensions are the row within a page and the page
    const int kv_rows = p.block_table ? p.page_size : tokens_k;
    const int kv_outer = p.block_table ? in->num_pages : bdim;
    const bool f16 = p.dtype == FA_DTYPE_F16;
    if (p.dtype != FA_DTYPE_E4M3 && (!encode_bhsd(&tk, k, p.d, p.h_kv, kv_rows, kv_outer, 1, kv_box, f16) ||
                                     !encode_bhsd(&tv, v, p.d, p.h_kv, kv_rows, kv_outer, 1, kv_box, f16)))
        return FA_ERR_CUDA;
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    float* o_part = reinterpret_cast<float*>(ws + kStatusBytes);
    const int part_splits = pl.tail_k > 1 ? pl.tail_k : pl.n_splits;  // pieces per row in the partials
    float* lse_part = reinterpret_cast<float*>(ws + kStatusBytes + align256(pl.part_rows * part_splits * p.d * 4));

    if (pl.path == FwdPath::kDecode) {
        DecodeArgs a{};
        a.p = p;
        a.q = reinterpret_cast<const uint16_t*>(q);
        a.n_splits = pl.n_splits;
        a.split_keys = pl.split_tiles * kDecodeKeys;
        a.o_part = o_part;
        a.lse_part = lse_part;
        a.status = status;
        cudaError_t e = timed(kDecode, st, [&] { return launch_decode(a, tk, tv, st); });
        if (e != cudaSuccess) return FA_ERR_CUDA;
        CombineArgs c{};
        c.p = p;
        c.n_splits = pl.n_splits;
        c.o_part = o_part;
        c.lse_part = lse_part;
        c.o = reinterpret_cast<uint16_t*>(o);
        c.lse = lse;
        c.status = status;
        e = timed(kCombine, st, [&] { return launch_combine(c, st); });
        return cuda_status(e);
    }

    FwdArgs a{};
    CUtensorMap tq;
    if (p.dtype == FA_DTYPE_E4M3) {
        // Q, K, V: [b][s][h][128] bytes, [1][T][h][128] packed, or K, V a page pool
        // [num_pages][page_size][h_kv][128] (the kernel transposes each V tile in shared memory)
        const cuuint64_t dq[4] = {128, (cuuint64_t)p.h_q, (cuuint64_t)tokens_q, (cuuint64_t)bdim};
        const cuuint64_t sq[3] = {128, (cuuint64_t)p.h_q * 128, (cuuint64_t)tokens_q * p.h_q * 128};
        const cuuint32_t bq[4] = {128, (cuuint32_t)p.G, (cuuint32_t)p.P, 1};
        const cuuint64_t dk[4] = {128, (cuuint64_t)p.h_kv, (cuuint64_t)kv_rows, (cuuint64_t)kv_outer};
        const cuuint64_t sk[3] = {128, (cuuint64_t)p.h_kv * 128, (cuuint64_t)kv_rows * p.h_kv * 128};
        const cuuint32_t bk[4] = {128, 1, 128, 1};
        CUtensorMap tk8, tv8;
        if (!encode_u8_4d(&tq, q, dq, sq, bq) || !encode_u8_4d(&tk8, k, dk, sk, bk) || !encode_u8_4d(&tv8, v, dk, sk, bk))
            return FA_ERR_CUDA;
        a.q_descale = in->q_descale;
        a.k_descale = in->k_descale;
        a.v_descale = in->v_descale;
        tk = tk8;
        tv = tv8;
    } else if (!encode_bhsd(&tq, q, p.d, p.h_q, tokens_q, bdim, p.G, p.P, f16)) {
        return FA_ERR_CUDA;
    }
    a.p = p;
    a.n_blocks = pl.n_blocks;
    a.n_splits = pl.n_splits;
    a.split_tiles = pl.split_tiles;
    a.unit_major = pl.unit_major;
    a.tokens = pl.tokens;
    a.kt = pl.kt;
    a.tail_k = pl.tail_k;
    a.tail_split_tiles = pl.tail_split_tiles;
    a.tail_item0 = pl.tail_k > 1 ? (p.h_kv * p.B - pl.tail_units) * pl.n_blocks : 0;
    a.tail_row0 = pl.tail_k > 1 ? (long)(p.h_kv * p.B - pl.tail_units) * p.G * p.s_q : 0;
    {
        long items = p.cu_q ? (long)pl.n_blocks * p.h_kv : (long)pl.n_blocks * pl.n_splits * p.h_kv * p.B;
        if (pl.tail_k > 1) items = a.tail_item0 + (items - a.tail_item0) * pl.tail_k;  // the tail's pieces
        const long slots = (long)sm_count() * (pl.kt == 64 ? 2 : 1);
        a.n_items = (int)items;
        a.n_ctas = (int)(items < slots ? items : slots);
        a.snake = (!p.cu_q && p.causal && !pl.unit_major) ? 1 : 0;
    }
    a.o = reinterpret_cast<uint16_t*>(o);
    a.lse = lse;
    a.o_part = o_part;
    a.lse_part = lse_part;
    a.status = status;
#ifdef FA_TRACE
    a.trace = reinterpret_cast<unsigned long long*>(ws + pl.off_trace);
    if (cudaMemsetAsync(a.trace, 0, kTraceBytes, st) != cudaSuccess) return FA_ERR_CUDA;
#endif
    cudaError_t e = timed(kFwd, st, [&] {
        return p.dtype == FA_DTYPE_E4M3 ? launch_fwd_e4m3(a, tq, tk, tv, st) : launch_fwd(a, tq, tk, tv, st);
    });
    if (e != cudaSuccess) return FA_ERR_CUDA;
    if (pl.n_splits > 1 || pl.tail_k > 1) {
        CombineArgs c{};
        c.p = p;
        c.n_splits = pl.n_splits > 1 ? pl.n_splits : pl.tail_k;
        c.row0 = pl.tail_k > 1 ? a.tail_row0 : 0;
        c.nrows = pl.tail_k > 1 ? (long)pl.part_rows : 0;
        c.o_part = o_part;
        c.lse_part = lse_part;
        c.o = reinterpret_cast<uint16_t*>(o);
        c.lse = lse;
        c.status = status;
        e = timed(kCombine, st, [&] { return launch_combine(c, st); });
    }
    return cuda_status(e);
}

fa_status fa_bwd(const fa_params* in, const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, float* dsinks, void* workspace, size_t ws_bytes,
                 struct CUstream_st* stream) {
    Problem p;
    fa_status rc = normalise(in, p);
    if (rc != FA_OK) return rc;
    BwdPlan pl;
    if ((rc = plan_bwd(p, in->flags, pl)) != FA_OK) return rc;
    if (!workspace || !aligned16(workspace)) return FA_ERR_INVALID_ARG;
    if (ws_bytes < pl.ws_bytes) return FA_ERR_WORKSPACE;
    if (p.sinks && !dsinks) return FA_ERR_INVALID_ARG;
    const long rows_total = p.cu_q ? (long)p.T_q : (long)p.B * p.s_q;
    const long keys_total = p.cu_q ? (long)p.T_k : (long)p.B * p.s_kv;
    if (rows_total > 0 && (!q || !o || !lse || !dout || !dq || !aligned16(q) || !aligned16(o) ||
                           !aligned16(dout) || !aligned16(dq)))
        return FA_ERR_INVALID_ARG;
    if (keys_total > 0 && (!k || !v || !dk || !dv || !aligned16(k) || !aligned16(v) || !aligned16(dk) ||
                           !aligned16(dv)))
        return FA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int* status = reinterpret_cast<int*>(workspace);
    if ((rc = cuda_status(cudaMemsetAsync(status, 0, sizeof(int), st))) != FA_OK) return rc;
    if (p.sinks && (rc = cuda_status(cudaMemsetAsync(dsinks, 0, sizeof(float) * p.h_q, st))) != FA_OK) return rc;
    if ((rc = maybe_validate(p, in->flags, status, st)) != FA_OK) return rc;
    if (pl.empty) return FA_OK;

    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    BwdArgs a{};
    a.p = p;
    a.n_qtiles = pl.n_qtiles;
    a.n_kvblocks = pl.n_kvblocks;
    a.n_bands = pl.n_bands;
    a.tokens = pl.tokens;
    a.n_units = (int)((long)pl.n_kvblocks * p.h_kv * (p.cu_q ? 1 : p.B));
    a.n_ctas = a.n_units < sm_count() ? a.n_units : sm_count();
    // one CTA per unit for long causal dense problems without a left window (32 or more key
    // blocks per sequence), whose units' work varies most; persistent CTAs everywhere else
    // (measured on one box: B=2 s=8192 causal 1.367 vs 1.421 ms, s=16384 causal 2.525 vs
    // 2.687; s=512 causal 0.294 vs 0.271, s=8192 2.644 vs 2.561, packed batch 1.476 vs
    // 1.411, grouped-query window (127, 0) 0.292 vs 0.287 ms, per unit vs persistent)
    a.persist = (!p.cu_q && p.causal && p.left < 0 && pl.n_kvblocks >= 32) ? 0 : 1;
    a.o = reinterpret_cast<const uint16_t*>(o);
    a.lse = lse;
    a.dout = reinterpret_cast<const uint16_t*>(dout);
    a.delta_t = reinterpret_cast<float*>(ws + pl.off_delta);
    a.lse2_t = reinterpret_cast<float*>(ws + pl.off_lse2);
    a.dq_acc = reinterpret_cast<float*>(ws + pl.off_dq);
    a.dq = reinterpret_cast<uint16_t*>(dq);
    a.dk = reinterpret_cast<uint16_t*>(dk);
    a.dv = reinterpret_cast<uint16_t*>(dv);
    a.dsinks = p.sinks ? dsinks : nullptr;
    a.sink_t = p.sinks ? reinterpret_cast<float*>(ws + pl.off_sink) : nullptr;
    a.dq_count = (in->flags & FA_FLAG_DETERMINISTIC) ? reinterpret_cast<int*>(ws + pl.off_count) : nullptr;
    a.status = status;
#ifdef FA_TRACE
    a.trace = reinterpret_cast<unsigned long long*>(ws + pl.off_trace);
    if (cudaMemsetAsync(a.trace, 0, kTraceBytes, st) != cudaSuccess) return FA_ERR_CUDA;
#endif

    const int tokens_q = p.cu_q ? p.T_q : p.s_q;
    const int tokens_k = p.cu_q ? p.T_k : p.s_kv;
    const int bdim = p.cu_q ? 1 : p.B;
    CUtensorMap tq, tk, tv, tdo;
    const bool f16 = p.dtype == FA_DTYPE_F16;
    if (!encode_bhsd(&tq, q, p.d, p.h_q, tokens_q, bdim, p.G, p.P, f16) ||
        !encode_bhsd(&tdo, dout, p.d, p.h_q, tokens_q, bdim, p.G, p.P, f16) ||
        !encode_bhsd(&tk, k, p.d, p.h_kv, tokens_k, bdim, 1, p.d >= 192 ? 64 : 128, f16) ||
        !encode_bhsd(&tv, v, p.d, p.h_kv, tokens_k, bdim, 1, p.d >= 192 ? 64 : 128, f16))
        return FA_ERR_CUDA;
    cudaError_t e = timed(kBwdPre, st, [&] { return launch_bwd_pre(a, st); });
    if (e != cudaSuccess) return FA_ERR_CUDA;
    e = timed(kBwdMain, st, [&] { return launch_bwd_main(a, tq, tk, tv, tdo, st); });
    if (e != cudaSuccess) return FA_ERR_CUDA;
    e = timed(kBwdPost, st, [&] { return launch_bwd_post(a, st); });
    return cuda_status(e);
}

fa_status fa_read_device_status(const void* workspace, struct CUstream_st* stream) {
    if (!workspace) return FA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
    if (v == FA_ERR_TIMEOUT || v == FA_ERR_DEVICE_CHECK) return (fa_status)v;
    return v == 0 ? FA_OK : FA_ERR_DEVICE_CHECK;
}

fa_status fa_profile_enable(int on) {
    Profiler& P = prof();
    std::lock_guard<std::mutex> g(P.mu);
    if (on && !P.ev[0][0]) {
        for (int i = 0; i < kNumKernels; ++i)
            for (int j = 0; j < 2; ++j)
                if (cudaEventCreate(&P.ev[i][j]) != cudaSuccess) return FA_ERR_CUDA;
    }
    P.on = on != 0;
    for (int i = 0; i < kNumKernels; ++i) P.recorded[i] = false;
    return FA_OK;
}

fa_status fa_profile_read(const char* kernel, float* ms) {
    if (!kernel || !ms) return FA_ERR_INVALID_ARG;
    Profiler& P = prof();
    std::lock_guard<std::mutex> g(P.mu);
    for (int i = 0; i < kNumKernels; ++i) {
        if (std::strcmp(kernel, kKernelNames[i]) != 0) continue;
        if (!P.recorded[i]) return FA_ERR_INVALID_ARG;
        if (cudaEventSynchronize(P.ev[i][1]) != cudaSuccess) return FA_ERR_CUDA;
        return cudaEventElapsedTime(ms, P.ev[i][0], P.ev[i][1]) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
    return FA_ERR_INVALID_ARG;
}

}  // extern "C"
