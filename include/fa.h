/*
 * fa.h — C ABI of libfa_gb300.so: exact softmax attention, forward and backward,
 * on one NVIDIA GB300 (sm_103a).
 *
 * What it computes (the plain definition; the kernels reach it with an online
 * softmax that never materialises the S x S matrix):
 *
 *   O_i   = sum_j P_ij v_j,   P_ij = exp(scale * q_i.k_j - LSE_i) over the allowed keys j
 *   LSE_i = log( sum_j exp(scale * q_i.k_j) [+ exp(sink_h)] )
 *
 * following the "Flash Attention Tutorial" README (GitHub search results page for
 * "flash attention implementation notes"), sections 1-5 for the forward and
 * section 6 "Key derivations" for the backward (dV = P^T dO; D_i = dO_i.O_i;
 * dS_ij = P_ij (dO_i.v_j - D_i); dQ = scale dS K; dK = scale dS^T Q — the scale
 * is kept in dQ and dK, which that tutorial's listing omits).
 *
 * Masks are bottom-right aligned when s_q != s_kv (vllm-project/flash-attention
 * README, flash_attn_func and flash_attn_with_kvcache docstrings, changelog 2.1):
 * with off = s_kv - s_q of the sequence, query i keeps key j iff
 *   causal      : j <= i + off
 *   window_left  >= 0 : j >= i + off - window_left
 *   window_right >= 0 : j <= i + off + window_right      (inclusive; -1 = unbounded)
 * A causal call with a window keeps the intersection.  A row with no allowed key
 * gets O = 0 and LSE = -inf (LSE = sink_h when the head has a sink).
 *
 * Grouped-query heads: h_kv divides h_q and query head h reads key/value head
 * h / (h_q / h_kv) (same README, flash_attn_func docstring: 6 query heads on 2
 * key/value heads map 0,1,2 -> 0 and 3,4,5 -> 1).
 *
 * Sinks: one fp32 logit per query head joins every row's softmax denominator and
 * carries no value (dew-flash-attn PyPI page, the sinks paragraph).  The returned
 * LSE includes the sink; fa_bwd returns the sink gradient
 *   dsink_h = - sum_rows exp(sink_h - LSE_i) D_i.
 *
 * Packed batches (dew-flash-attn PyPI page, "Packed sequences"; fa4-jax PyPI page,
 * "Varlen semantics"): with cu_seqlens_q / cu_seqlens_k given, tensors are
 * [T, H, D], sequence b owns rows cu[b] .. cu[b+1]-1, masks apply per sequence,
 * attention never crosses sequences, zero-length sequences are legal, and the
 * LSE is laid out [h_q, T_q].  The offsets are read on the device and are not
 * checked unless FA_FLAG_VALIDATE_CU is set (tokens they do not cover get
 * unspecified outputs, as on the pages).  Passing the same array as cu_seqlens_q and
 * cu_seqlens_k (queries and keys packed alike, as in self-attention over a packed batch)
 * lets the d <= 128 kernels tile the packed token axis itself: a 128-row tile then holds
 * several short sequences, each row masked to its own sequence, so a batch of short
 * sequences costs about its tokens rather than a tile per sequence.  Two arrays with equal
 * contents give the same results, with tiles per sequence.
 *
 * Conventions common to every call:
 *  - Layouts: dense tensors are contiguous [B, S, H, D] (bf16 or fp16); packed ones [T, H, D].
 *    LSE is fp32 [B, h_q, s_q] (dense) or [h_q, T_q] (packed), natural log.
 *  - Ownership: every pointer is caller-owned device memory (except the params
 *    struct itself, read on the host during the call).  The library allocates no
 *    device memory; scratch lives in the caller's workspace, sized by the
 *    fa_*_workspace_size functions.  Base pointers of q, k, v, o, dout, dq, dk, dv
 *    and the workspace must be 16-byte aligned.
 *  - Streams: work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without synchronising.
 *  - Errors: arguments are checked on the host before anything is launched; a
 *    violation returns a code and launches nothing.  No C++ exception crosses this
 *    ABI and no kernel traps: a kernel whose pipeline stalls gives up after a time
 *    limit (fa_params.wait_limit_ns) and records FA_ERR_TIMEOUT in the workspace status
 *    word, which fa_read_device_status reports.  Every kernel of a call reads the status
 *    word first and does nothing when it is set, so a failed offset check
 *    (FA_FLAG_VALIDATE_CU) or a timeout leaves the outputs of the rest of the call
 *    unwritten.
 *  - Supported: bf16 and fp16 (and e4m3 for the forward at d = 128, see below); head dim d in
 *    {64, 128, 192, 256} for the forward and the backward (FA_FLAG_DETERMINISTIC included);
 *    h_q / h_kv <= 128.  d = 192 is one of the head sizes the pages pad to (dew-flash-attn
 *    PyPI page, the FA3 head-dim padding to 64 / 128 / 192 / 256).
 *    Anything else returns FA_ERR_UNSUPPORTED.
 *  - Zero-initialise fa_params (memset or `= {0}`): every optional field then means
 *    "not used".
 *
 * Partly filled slots and paged caches:
 *  - seqused_q / seqused_k (fa4-jax PyPI page, "Varlen semantics": optional seqused_q /
 *    seqused_k limit each slot to its first seqused[b] tokens, the cache case where slots
 *    are larger than what is filled): sequence b uses only its first seqused_q[b] queries
 *    and seqused_k[b] keys of its slot (s_q / s_kv for dense tensors, the cu_seqlens
 *    difference for packed ones); the bottom-right alignment uses the used lengths, unused
 *    keys are invisible, and the outputs of unused query rows (O, LSE, dQ) and the dK, dV
 *    rows of unused keys are not written (unspecified).  Values are clamped to [0, slot].
 *    Forward and backward.
 *  - block_table (forward only; fa_bwd returns FA_ERR_UNSUPPORTED; vllm-project/flash-attention
 *    README, flash_attn_with_kvcache docstring ("Does not support backward pass"):
 *    a paged cache of shape (num_blocks, page_block_size, nheads_k, headdim) addressed
 *    through block_table (batch_size, max_num_blocks_per_seq) int32): dense q only; k and
 *    v are page pools [num_pages, page_size, h_kv, d] and key j of sequence b is row
 *    j % page_size of page block_table[b * max_blocks_per_seq + j / page_size].  s_kv is
 *    the logical cache length (at most max_blocks_per_seq * page_size); page_size must be
 *    a positive multiple of 128 (the page's builds ask for 256).  Table entries are read
 *    on the device and not checked.
 *
 * FP8 forward (vllm-project/flash-attention README, "FlashAttention-3 beta release":
 * "FP8 forward"): with dtype = FA_DTYPE_E4M3, q, k and v hold e4m3 bytes (1 byte per
 * element, same layouts) and the true inputs are q * q_descale[b * h_kv + g] (likewise k,
 * v) for batch b and key/value head g; a NULL descale means 1.  S = Q K^T and O = P V run
 * on the fp8 tensor cores with fp32 accumulation, P is rounded to e4m3 for the second
 * product, o is written as bf16 and lse (fp32) is that of the descaled problem.  d = 128
 * only, dense, packed (cu_seqlens; the descale index b is then the sequence) or with a
 * paged k / v cache; seqused_k, windows, causal and sinks are supported; anything else
 * returns FA_ERR_UNSUPPORTED, and fa_bwd rejects the type.  The workspace is the bf16 forward's for the same shape (v is transposed tile by
 * tile inside the kernel, not copied).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* a null, misaligned or inconsistent argument */
    FA_ERR_UNSUPPORTED = 2,  /* a valid problem this build does not implement */
    FA_ERR_WORKSPACE = 3,    /* workspace smaller than fa_*_workspace_size */
    FA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    FA_ERR_TIMEOUT = 5,      /* a kernel pipeline stalled and gave up (device status) */
    FA_ERR_DEVICE_CHECK = 6  /* a device-side argument check failed (device status) */
} fa_status;

/* Input element types.  bf16 and fp16 (dew-flash-attn PyPI page, usage: inputs in bf16
 * or fp16; fa4-jax PyPI page, restrictions: fp16/bf16) run every path of fa_fwd and fa_bwd
 * alike: o, dq, dk and dv have the inputs' type, accumulation and lse stay fp32.  e4m3 is
 * the FP8 forward above. */
#define FA_DTYPE_BF16 0
#define FA_DTYPE_E4M3 1
#define FA_DTYPE_F16 2

/* Flags */
#define FA_FLAG_VALIDATE_CU 1u  /* check cu_seqlens on the device; result in the status word */
#define FA_FLAG_NO_SPLIT 2u     /* forward: never split the key range across CTAs */
/* backward: bitwise-reproducible results.  dQ is summed over key blocks in a fixed order
 * (descending key block) instead of in arrival order; the workspace grows by 4 bytes per
 * (query tile, key/value head).  The deterministic backward option of the
 * vllm-project/flash-attention README (changelog 2.4).  A key block's CTA waits (bounded,
 * like every wait: FA_ERR_TIMEOUT) for the later blocks' contributions, which the launch
 * puts at lower CTA indices; slower than the default, markedly so without a causal mask.
 * The sink gradient is summed in a fixed order with or without the flag.  Every head
 * dimension (at d = 192 / 256 the key blocks are 64 keys). */
#define FA_FLAG_DETERMINISTIC 4u

typedef struct fa_params {
    int B;            /* batch (dense) or number of sequences (packed) */
    int s_q, s_kv;    /* sequence lengths (dense); total tokens T_q, T_k (packed) */
    int h_q, h_kv;    /* query heads, key/value heads (h_kv divides h_q) */
    int d;            /* head dimension */
    float softmax_scale;  /* <= 0 selects 1 / sqrt(d) */
    int causal;           /* nonzero: bottom-right aligned causal mask */
    int window_left, window_right;  /* -1 = unbounded side */
    const float *sinks;             /* device fp32 [h_q], or NULL */
    const int32_t *cu_seqlens_q;    /* device int32 [B+1], or NULL for dense tensors */
    const int32_t *cu_seqlens_k;    /* device int32 [B+1]; required iff cu_seqlens_q */
    int max_seqlen_q, max_seqlen_k; /* optional hints (0 = unknown); never needed */
    unsigned flags;                 /* FA_FLAG_* */
    /* Partly filled slots and paged caches (see above).  Zero / NULL = not used. */
    const int32_t *seqused_k;       /* device int32 [B], or NULL */
    const int32_t *block_table;     /* device int32 [B * max_blocks_per_seq], or NULL */
    int page_size;                  /* keys per page (block_table only) */
    int max_blocks_per_seq;         /* row stride of block_table */
    int num_pages;                  /* pages in each of the k and v pools */
    /* Input element type (FA_DTYPE_*; 0 = bf16).  See the FP8 forward above and the types. */
    int dtype;
    const float *q_descale;         /* FA_DTYPE_E4M3 only: device fp32 [B * h_kv] or NULL (= 1) */
    const float *k_descale;
    const float *v_descale;
    const int32_t *seqused_q;       /* device int32 [B], or NULL (see partly filled slots) */
    /* Bound, in nanoseconds, on each wait of a kernel's pipeline (a stage of copies or
     * MMAs that should have landed); 0 selects 2 s.  A wait that runs past it makes the CTA
     * give up: it records FA_ERR_TIMEOUT in the status word, lets its own copies and MMAs
     * land, frees its tensor memory and returns, and the call's later kernels do nothing.
     * A limit below the kernels' own latencies (a few microseconds) turns every call into
     * such a failure, which is how the failure path is exercised; outputs of a failed call
     * are unspecified. */
    unsigned long long wait_limit_ns;
} fa_params;

/* Bytes of workspace fa_fwd / fa_bwd need for these parameters (>= 256: the first
 * 256 bytes hold the device status word).  Returns 0 when the parameters are
 * invalid or unsupported.  The forward's plan (key splits, and the split of a last
 * partial wave of work at d = 192 / 256) follows the current device's SM count, so the
 * size is queried with the device that will run the call current. */
size_t fa_fwd_workspace_size(const fa_params *p);
size_t fa_bwd_workspace_size(const fa_params *p);

/* Forward.  q: [.., h_q, d]; k, v: [.., h_kv, d]; o: layout of q (written);
 * lse: fp32 (written; may be NULL when not wanted). */
fa_status fa_fwd(const fa_params *p, const void *q, const void *k, const void *v, void *o, float *lse,
                 void *workspace, size_t workspace_bytes, struct CUstream_st *stream);

/* Backward of L = sum(O * dout).  o and lse must be what fa_fwd returned for the
 * same inputs.  dq: layout of q; dk, dv: layout of k (all written, in the inputs' type).
 * dsinks: fp32 [h_q], written when p->sinks is given (must then be non-NULL). */
fa_status fa_bwd(const fa_params *p, const void *q, const void *k, const void *v, const void *o,
                 const float *lse, const void *dout, void *dq, void *dk, void *dv, float *dsinks,
                 void *workspace, size_t workspace_bytes, struct CUstream_st *stream);

/* Synchronises `stream` and returns the status word the kernels of the last call
 * on this workspace left (FA_OK, FA_ERR_TIMEOUT or FA_ERR_DEVICE_CHECK), or
 * FA_ERR_CUDA if the stream itself reports an error. */
fa_status fa_read_device_status(const void *workspace, struct CUstream_st *stream);

/* Static text for a status code. */
const char *fa_status_string(fa_status s);

/* Per-kernel timing: when enabled, every launch the library makes is bracketed by
 * CUDA events on its stream.  fa_profile_read synchronises on the last launch of
 * the named kernel ("fwd", "decode", "combine", "bwd_pre", "bwd_main", "bwd_post")
 * and writes its duration in milliseconds; returns FA_ERR_INVALID_ARG for an
 * unknown name or a kernel not launched since profiling was enabled. */
fa_status fa_profile_enable(int on);
fa_status fa_profile_read(const char *kernel, float *ms);

/* Forward without a caller workspace, for callers that cannot allocate device memory
 * (a host framework that owns every allocation, or a loop that must not enter the CUDA
 * allocator).  No passage on the pages has a counterpart: it is fa_fwd run on a scratch
 * array of FA_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into the library, which every GPU
 * that loads the library holds until the process exits.  Arguments, layouts and results
 * are those of fa_fwd.  Allocates nothing.  Returns FA_ERR_WORKSPACE, launching nothing,
 * when the problem needs more scratch than the array holds (fa_fwd_workspace_size(p)
 * larger than FA_NOALLOC_SCRATCH_BYTES); FA_ERR_CUDA if the array's address cannot be
 * had.  The first call on each device looks the array's address up (and again after the
 * device's context was destroyed and made anew, e.g. by cudaDeviceReset), so make the
 * first call, and the first after such a reset, before any stream capture.  All calls share the array and it keeps the last call's contents:
 * each call resets what must start at zero, but calls that overlap on the GPU race on
 * it, so serialise them (one stream, or events between streams).  The kernels' status
 * word also lives in the array and is not readable through this ABI. */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
fa_status fa_fwd_noalloc(const fa_params *p, const void *q, const void *k, const void *v, void *o, float *lse,
                         struct CUstream_st *stream);

/* Library version string. */
const char *fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
