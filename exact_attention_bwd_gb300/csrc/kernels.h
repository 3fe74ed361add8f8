// Launch-argument structures shared by the host planner (api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Problem description after host-side normalisation.
struct Problem {
    int B, s_q, s_kv, h_q, h_kv, d;
    int G;             // h_q / h_kv
    int P;             // query positions per 128-row tile: floor(128 / G)
    float scale;       // softmax scale
    float scale_log2;  // softmax scale * log2(e)
    int causal;
    int left, right;   // -1 = unbounded side; a causal call has right = 0
    const float* sinks;       // [h_q] fp32 or null
    const int32_t* cu_q;      // [B+1] or null (dense)
    const int32_t* cu_k;
    int T_q, T_k;             // packed token counts (varlen)
    const int32_t* seqused_q; // [B] queries used per sequence, or null
    const int32_t* seqused_k; // [B] keys used per sequence, or null
    const int32_t* block_table;  // [B * max_blocks] pages of a paged K/V cache, or null
    int page_size, max_blocks;
    int dtype;                // input element type (FA_DTYPE_*)
    unsigned long long wait_ns;  // bound on each pipeline wait (ns) before a CTA gives up
};

// ------------------------------------------------------------------------------------------
// forward (tensor-core path)
// ------------------------------------------------------------------------------------------
struct FwdArgs {
    Problem p;
    int n_blocks;      // CTA work units along grid.x (before splitting)
    int n_splits;      // KV splits (1 = write final outputs)
    int split_tiles;   // KV tiles per split
    int unit_major;    // grid order: blocks of one (batch, kv head) adjacent (decode-like
                       // shapes, so they share K/V through L2) instead of heaviest first
    int n_items;       // work items (query blocks x kv heads [x batch x splits])
    int n_ctas;        // persistent CTAs of the d <= 128 kernel (at most one per SM)
    int snake;         // their rounds alternate direction (items heaviest first: dense causal)
    int tokens;        // packed batch with queries and keys packed alike: query tiles run over
                       // the packed token axis and may hold several sequences (d <= 128 kernel)
    int kt;            // keys per key tile of the d <= 128 kernel: 128, or 64 (d = 64 with a
                       // narrow band: two CTAs per SM)
    // tail split (d = 192 / 256, dense, one CTA per item): items from tail_item0 on (whole
    // (batch, kv head) units, the last ones) are each cut into tail_k key ranges of
    // tail_split_tiles tiles that write partials of rows [tail_row0, B h_q s_q) for the
    // combine; the other items write final outputs.  tail_k = 0: no tail split.
    int tail_item0, tail_k, tail_split_tiles;
    long tail_row0;
    uint16_t* o;       // [tokens, h_q, d] bf16, or fp16 for fp16 inputs
    float* lse;        // [B, h_q, s_q] or [h_q, T_q]; may be null
    float* o_part;     // split mode: [n_splits, rows, d] fp32
    float* lse_part;   // split mode: [n_splits, rows] fp32 (natural log, no sink)
    int* status;
    // e4m3 inputs only: per (batch, kv head) factors that turn the stored values into the
    // true ones (x = stored * descale), [B * h_kv] fp32 or null (= 1)
    const float* q_descale;
    const float* k_descale;
    const float* v_descale;
    unsigned long long* trace;  // trace builds only: the workspace's trace region (else null)
};

// ------------------------------------------------------------------------------------------
// decode (CUDA-core path for few query rows per key/value head)
// ------------------------------------------------------------------------------------------
struct DecodeArgs {
    Problem p;
    const uint16_t* q;  // [B, s_q, h_q, d] bf16 or fp16 (as the inputs)
    int n_splits;
    int split_keys;    // keys per split (a multiple of the key tile)
    float* o_part;     // [n_splits, rows, d]
    float* lse_part;   // [n_splits, rows]
    int* status;
};

struct CombineArgs {
    Problem p;
    int n_splits;
    long row0, nrows;  // the rows merged: [row0, row0 + nrows) of B h_q s_q (nrows = 0: all);
                       // the partials hold these rows only, from index 0
    const float* o_part;
    const float* lse_part;
    uint16_t* o;       // bf16 or fp16 (as the inputs)
    float* lse;
    const int* status; // the call's status word: nonzero = an earlier kernel failed, do nothing
};

// ------------------------------------------------------------------------------------------
// backward
// ------------------------------------------------------------------------------------------
struct BwdArgs {
    Problem p;
    int n_qtiles;          // q tiles per (key/value head) in the tiled layouts below
    int n_kvblocks;        // key blocks per (batch, key/value head) unit (dense) or numbered blocks (packed)
    int n_bands;           // dense grid order: the (batch, kv head) units form this many bands of
                           // near-equal size, key block slowest within a band, so a band's
                           // query-side data stays in L2
    int tokens;            // packed batch with queries and keys packed alike: key blocks and query
                           // tiles run over the packed token axis (d <= 128 kernel)
    int n_units;           // work units (key blocks x kv heads [x batch])
    int n_ctas;            // persistent CTAs of the d <= 128 main kernel (at most one per SM)
    int persist;           // 1: n_ctas persistent CTAs walk the units; 0: one CTA per unit
    // 16-bit tensors hold bf16 or fp16 (Problem::dtype) like the inputs
    const uint16_t* o;
    const float* lse;
    const uint16_t* dout;
    float* delta_t;        // [h_kv, n_qtiles, 128]  rowsum(dO * O)
    float* lse2_t;         // [h_kv, n_qtiles, 128]  LSE * log2(e) (+inf for empty rows)
    float* dq_acc;         // [h_kv, n_qtiles, 128, d] fp32
    uint16_t* dq;          // [tokens, h_q, d]
    uint16_t* dk;          // [tokens_k, h_kv, d]
    uint16_t* dv;
    float* dsinks;         // [h_q] or null
    float* sink_t;         // [h_kv, n_qtiles, 128]  per-row sink-gradient terms (with sinks)
    int* dq_count;         // [h_kv, n_qtiles] dQ contributions landed per query tile, or null:
                           // non-null = deterministic order (key blocks in descending order)
    int* status;
    unsigned long long* trace;  // trace builds only: the workspace's trace region (else null)
};

// host-side launchers (defined next to each kernel)
cudaError_t launch_fwd(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t st);
cudaError_t launch_fwd256(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          cudaStream_t st);
cudaError_t launch_fwd_e4m3(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st);
int decode_rows_max(int d);                // query rows per key/value head the decode kernel takes
int decode_ctas_per_sm(int d, int rows);   // its CTAs resident per SM
cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t st);
cudaError_t launch_bwd_main(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, cudaStream_t st);
cudaError_t launch_bwd_post(const BwdArgs& a, cudaStream_t st);

// Number of 16-byte-aligned KV tiles etc. shared by planner and kernels.
constexpr int kTileRows = 128;

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

}  // namespace fa
