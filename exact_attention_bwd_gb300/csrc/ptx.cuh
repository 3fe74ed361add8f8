// Inline-PTX building blocks for sm_103a: mbarriers, TMA bulk copies,
// tcgen05 (tensor memory + 5th-generation MMA) and the shared-memory
// matrix descriptors the MMA reads.  Every wait here is bounded: it gives up
// after a time limit, records why in the kernel's status word and lets the
// caller drain and return instead of hanging the GPU.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

// ------------------------------------------------------------------------------------------
// status words written by kernels (mirrors fa_status in include/fa.h)
// ------------------------------------------------------------------------------------------
enum : int { kStatusOk = 0, kStatusTimeout = 5, kStatusDeviceCheck = 6 };

// A stalled pipeline gives up after this long (the default of a call's wait limit, and the
// fixed limit of the drain at exit); one wait never legitimately takes more than a few
// microseconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared abort state of one CTA: the first wait that runs out of time sets it, every
// later wait returns at once, and the kernel's status word records the reason.
struct Abort {
    volatile int* flag;   // shared memory
    int* status;          // global memory (may be null)
    unsigned long long limit;  // ns a pipeline wait may take before the CTA gives up
    __device__ __forceinline__ bool raised() const { return *flag != 0; }
    __device__ __forceinline__ void raise(int code) const {
        *flag = 1;
        if (status) atomicCAS(status, 0, code);
    }
};

// try_wait whose suspension lasts at most about `hint_ns` (instead of the hardware's own
// limit, which can exceed a short wait limit).
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and raises
// the CTA's abort) when the limit passes or another wait of the CTA already gave up.
// The first try is the plain one (the hardware picks how long it suspends; most waits end
// there).  The retries suspend for at most about the limit each, so that a short limit is
// not outlasted by one hardware suspension.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Abort& ab) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint32_t hint = ab.limit < 0xFFFFFFFFull ? (uint32_t)ab.limit : 0xFFFFFFFFu;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait_for(bar, parity, hint)) return true;
        if (ab.raised()) return false;
        if (globaltimer() - t0 > ab.limit) {
            ab.raise(kStatusTimeout);
            return false;
        }
    }
}

// Bounded wait used while draining at exit: gives up after the fixed 2 s limit (not the
// call's limit: every copy and MMA already issued must land before the CTA exits),
// without touching the abort state (the CTA is already on its way out).
__device__ __forceinline__ bool mbar_wait_quiet(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 <= kWaitLimitNs)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ------------------------------------------------------------------------------------------
// TMA
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 4-D tiled load of one box into shared memory; completion is counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// L2 cache policies (createpolicy): keep lines (evict_last) or let them go first (evict_first).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// fp32 reduction into global memory under an L2 cache policy.
__device__ __forceinline__ void red_add_hint(float* p, float v, uint64_t pol) {
    asm volatile("red.global.add.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
// Four consecutive fp32 reductions (16-byte aligned) under an L2 cache policy.
__device__ __forceinline__ void red_add4_hint(float* p, float a, float b, float c, float d, uint64_t pol) {
    asm volatile("red.global.add.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d), "l"(pol)
                 : "memory");
}
// tma_load_4d under an L2 cache policy.
__device__ __forceinline__ void tma_load_4d_hint(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                                 int c2, int c3, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
        : "memory");
}

// Contiguous global -> shared copy (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Makes generic-proxy writes to shared memory visible to the async proxy (MMA, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05: tensor memory and MMA
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives once on `bar` when every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ------------------------------------------------------------------------------------------
// MMA bursts: one GEMM (its K-steps) issued from a single asm block.  Each takes the base
// descriptor of every operand and adds the per-step offsets (in 16-byte descriptor units,
// fixed by the tile layout) as immediates, so the issuing thread runs no dependent
// instructions between the MMAs.  The first MMA accumulates iff acc0 != 0, the rest always.
// Step patterns: K-major in 128-byte-swizzled [rows][64] chunks of 16 KB (or 8 KB):
// +32 B per step, next chunk every 4 steps; MN-major: +16 rows (2 KB) per step.
// ------------------------------------------------------------------------------------------

// A, B K-major, 16 KB chunks, 8 steps (K = 128)
__device__ __forceinline__ void mma_ss_kk16_x8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t alo = (uint32_t)a, ahi = (uint32_t)(a >> 32), blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 da, db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; mov.b64 da, {ta, %4}; add.u32 tb, %5, 0; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p0;\n"
        "add.u32 ta, %3, 2; mov.b64 da, {ta, %4}; add.u32 tb, %5, 2; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 4; mov.b64 da, {ta, %4}; add.u32 tb, %5, 4; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 6; mov.b64 da, {ta, %4}; add.u32 tb, %5, 6; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1024; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1024; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1026; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1026; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1028; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1028; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1030; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1030; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi)
        : "memory");
}

// A, B K-major, 16 KB chunks, 4 steps (K = 64)
__device__ __forceinline__ void mma_ss_kk16_x4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t alo = (uint32_t)a, ahi = (uint32_t)(a >> 32), blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 da, db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; mov.b64 da, {ta, %4}; add.u32 tb, %5, 0; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p0;\n"
        "add.u32 ta, %3, 2; mov.b64 da, {ta, %4}; add.u32 tb, %5, 2; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 4; mov.b64 da, {ta, %4}; add.u32 tb, %5, 4; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 6; mov.b64 da, {ta, %4}; add.u32 tb, %5, 6; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi)
        : "memory");
}

// e4m3 operands (kind::f8f6f4), A and B K-major with 128-byte rows (one swizzle atom per
// row: K = 128 one-byte elements), 4 steps of K = 32 (+32 B each)
__device__ __forceinline__ void mma_f8_ss_k128(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t alo = (uint32_t)a, ahi = (uint32_t)(a >> 32), blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 da, db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; mov.b64 da, {ta, %4}; add.u32 tb, %5, 0; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %1, p0;\n"
        "add.u32 ta, %3, 2; mov.b64 da, {ta, %4}; add.u32 tb, %5, 2; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 4; mov.b64 da, {ta, %4}; add.u32 tb, %5, 4; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 6; mov.b64 da, {ta, %4}; add.u32 tb, %5, 6; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi)
        : "memory");
}

// A K-major (16 KB chunks), B MN-major, 8 steps
__device__ __forceinline__ void mma_ss_kmn16_x8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t alo = (uint32_t)a, ahi = (uint32_t)(a >> 32), blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 da, db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; mov.b64 da, {ta, %4}; add.u32 tb, %5, 0; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p0;\n"
        "add.u32 ta, %3, 2; mov.b64 da, {ta, %4}; add.u32 tb, %5, 128; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 4; mov.b64 da, {ta, %4}; add.u32 tb, %5, 256; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 6; mov.b64 da, {ta, %4}; add.u32 tb, %5, 384; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1024; mov.b64 da, {ta, %4}; add.u32 tb, %5, 512; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1026; mov.b64 da, {ta, %4}; add.u32 tb, %5, 640; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1028; mov.b64 da, {ta, %4}; add.u32 tb, %5, 768; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1030; mov.b64 da, {ta, %4}; add.u32 tb, %5, 896; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi)
        : "memory");
}

// A, B MN-major, 8 steps
__device__ __forceinline__ void mma_ss_mnmn_x8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t alo = (uint32_t)a, ahi = (uint32_t)(a >> 32), blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 da, db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; mov.b64 da, {ta, %4}; add.u32 tb, %5, 0; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p0;\n"
        "add.u32 ta, %3, 128; mov.b64 da, {ta, %4}; add.u32 tb, %5, 128; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 256; mov.b64 da, {ta, %4}; add.u32 tb, %5, 256; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 384; mov.b64 da, {ta, %4}; add.u32 tb, %5, 384; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 512; mov.b64 da, {ta, %4}; add.u32 tb, %5, 512; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 640; mov.b64 da, {ta, %4}; add.u32 tb, %5, 640; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 768; mov.b64 da, {ta, %4}; add.u32 tb, %5, 768; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 896; mov.b64 da, {ta, %4}; add.u32 tb, %5, 896; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi)
        : "memory");
}

// A MN-major, B K-major (one 128-byte row of K per B row), 4 steps (K = 64)
__device__ __forceinline__ void mma_ss_mnk_x4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t alo = (uint32_t)a, ahi = (uint32_t)(a >> 32), blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 da, db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; mov.b64 da, {ta, %4}; add.u32 tb, %5, 0; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p0;\n"
        "add.u32 ta, %3, 128; mov.b64 da, {ta, %4}; add.u32 tb, %5, 2; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 256; mov.b64 da, {ta, %4}; add.u32 tb, %5, 4; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 384; mov.b64 da, {ta, %4}; add.u32 tb, %5, 6; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi)
        : "memory");
}

// A K-major 16 KB chunks, B K-major 8 KB chunks, 16 steps (K = 256)
__device__ __forceinline__ void mma_ss_k16k8_x16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t alo = (uint32_t)a, ahi = (uint32_t)(a >> 32), blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 da, db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; mov.b64 da, {ta, %4}; add.u32 tb, %5, 0; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p0;\n"
        "add.u32 ta, %3, 2; mov.b64 da, {ta, %4}; add.u32 tb, %5, 2; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 4; mov.b64 da, {ta, %4}; add.u32 tb, %5, 4; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 6; mov.b64 da, {ta, %4}; add.u32 tb, %5, 6; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1024; mov.b64 da, {ta, %4}; add.u32 tb, %5, 512; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1026; mov.b64 da, {ta, %4}; add.u32 tb, %5, 514; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1028; mov.b64 da, {ta, %4}; add.u32 tb, %5, 516; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1030; mov.b64 da, {ta, %4}; add.u32 tb, %5, 518; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 2048; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1024; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 2050; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1026; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 2052; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1028; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 2054; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1030; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 3072; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1536; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 3074; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1538; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 3076; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1540; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 3078; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1542; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi)
        : "memory");
}

// A K-major 16 KB chunks, B K-major 8 KB chunks, 12 steps (K = 192)
__device__ __forceinline__ void mma_ss_k16k8_x12(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t alo = (uint32_t)a, ahi = (uint32_t)(a >> 32), blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 da, db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; mov.b64 da, {ta, %4}; add.u32 tb, %5, 0; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p0;\n"
        "add.u32 ta, %3, 2; mov.b64 da, {ta, %4}; add.u32 tb, %5, 2; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 4; mov.b64 da, {ta, %4}; add.u32 tb, %5, 4; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 6; mov.b64 da, {ta, %4}; add.u32 tb, %5, 6; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1024; mov.b64 da, {ta, %4}; add.u32 tb, %5, 512; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1026; mov.b64 da, {ta, %4}; add.u32 tb, %5, 514; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1028; mov.b64 da, {ta, %4}; add.u32 tb, %5, 516; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 1030; mov.b64 da, {ta, %4}; add.u32 tb, %5, 518; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 2048; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1024; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 2050; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1026; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 2052; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1028; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "add.u32 ta, %3, 2054; mov.b64 da, {ta, %4}; add.u32 tb, %5, 1030; mov.b64 db, {tb, %6};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi)
        : "memory");
}

// A from TMEM at columns a + 8 k, B K-major in 8 KB chunks (+32 B per step, next chunk
// every 4 steps), 16 steps (K = 256)
__device__ __forceinline__ void mma_ts_lin_k8_x16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; add.u32 tb, %4, 0; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p0;\n"
        "add.u32 ta, %3, 8; add.u32 tb, %4, 2; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 16; add.u32 tb, %4, 4; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 24; add.u32 tb, %4, 6; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 32; add.u32 tb, %4, 512; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 40; add.u32 tb, %4, 514; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 48; add.u32 tb, %4, 516; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 56; add.u32 tb, %4, 518; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 64; add.u32 tb, %4, 1024; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 72; add.u32 tb, %4, 1026; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 80; add.u32 tb, %4, 1028; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 88; add.u32 tb, %4, 1030; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 96; add.u32 tb, %4, 1536; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 104; add.u32 tb, %4, 1538; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 112; add.u32 tb, %4, 1540; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 120; add.u32 tb, %4, 1542; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(a_tmem), "r"(blo), "r"(bhi)
        : "memory");
}

// A from TMEM at columns a + 8 k, B K-major in 8 KB chunks (+32 B per step, next chunk
// every 4 steps), 12 steps (K = 192)
__device__ __forceinline__ void mma_ts_lin_k8_x12(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; add.u32 tb, %4, 0; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p0;\n"
        "add.u32 ta, %3, 8; add.u32 tb, %4, 2; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 16; add.u32 tb, %4, 4; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 24; add.u32 tb, %4, 6; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 32; add.u32 tb, %4, 512; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 40; add.u32 tb, %4, 514; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 48; add.u32 tb, %4, 516; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 56; add.u32 tb, %4, 518; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 64; add.u32 tb, %4, 1024; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 72; add.u32 tb, %4, 1026; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 80; add.u32 tb, %4, 1028; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 88; add.u32 tb, %4, 1030; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(a_tmem), "r"(blo), "r"(bhi)
        : "memory");
}

// A from TMEM at columns a + 8 k, B MN-major, 8 steps
__device__ __forceinline__ void mma_ts_lin_mn_x8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; add.u32 tb, %4, 0; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p0;\n"
        "add.u32 ta, %3, 8; add.u32 tb, %4, 128; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 16; add.u32 tb, %4, 256; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 24; add.u32 tb, %4, 384; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 32; add.u32 tb, %4, 512; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 40; add.u32 tb, %4, 640; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 48; add.u32 tb, %4, 768; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 56; add.u32 tb, %4, 896; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(a_tmem), "r"(blo), "r"(bhi)
        : "memory");
}

// A from TMEM at columns a + 8 k, B MN-major, 4 steps
__device__ __forceinline__ void mma_ts_lin_mn_x4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; add.u32 tb, %4, 0; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p0;\n"
        "add.u32 ta, %3, 8; add.u32 tb, %4, 128; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 16; add.u32 tb, %4, 256; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 24; add.u32 tb, %4, 384; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(a_tmem), "r"(blo), "r"(bhi)
        : "memory");
}

// A from TMEM at columns a + 64 (k / 4) + 8 (k % 4), B MN-major, 8 steps
__device__ __forceinline__ void mma_ts_p_mn_x8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc0) {
    const uint32_t blo = (uint32_t)b, bhi = (uint32_t)(b >> 32);
    asm volatile(
        "{\n"
        ".reg .pred p0, p1;\n"
        ".reg .b32 ta, tb;\n"
        ".reg .b64 db;\n"
        "setp.ne.b32 p0, %2, 0;\n"
        "setp.eq.b32 p1, %1, %1;\n"
        "add.u32 ta, %3, 0; add.u32 tb, %4, 0; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p0;\n"
        "add.u32 ta, %3, 8; add.u32 tb, %4, 128; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 16; add.u32 tb, %4, 256; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 24; add.u32 tb, %4, 384; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 64; add.u32 tb, %4, 512; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 72; add.u32 tb, %4, 640; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 80; add.u32 tb, %4, 768; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "add.u32 ta, %3, 88; add.u32 tb, %4, 896; mov.b64 db, {tb, %5};\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %1, p1;\n"
        "}\n"
        :: "r"(d_tmem), "r"(idesc), "r"(acc0), "r"(a_tmem), "r"(blo), "r"(bhi)
        : "memory");
}

// Instruction descriptor of kind::f16 with fp16 (f16 = true) or bf16 A and B (always the
// same type) and an fp32 accumulator.  a_mn / b_mn: operand stored MN-major (true) or
// K-major (false).
__host__ __device__ constexpr uint32_t idesc_16(int M, int N, bool a_mn, bool b_mn, bool f16) {
    return (1u << 4)                          // D: f32
           | ((f16 ? 0u : 1u) << 7)           // A: f16 (0) or bf16 (1)
           | ((f16 ? 0u : 1u) << 10)          // B: the same type as A
           | ((a_mn ? 1u : 0u) << 15)         // A major
           | ((b_mn ? 1u : 0u) << 16)         // B major
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return idesc_16(M, N, a_mn, b_mn, false);
}
static_assert(idesc_16(128, 128, true, false, true) == (idesc_bf16(128, 128, true, false) & ~((1u << 7) | (1u << 10))),
              "the fp16 descriptor differs from the bf16 one in the two operand-type fields only");

// Instruction descriptor of kind::f8f6f4 with both operands e4m3 (format code 0), fp32
// accumulator, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4)                          // D: f32
           | (0u << 7)                        // A: e4m3
           | (0u << 10)                       // B: e4m3
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle.  The operand lives in 1024-byte
// atoms of 8 rows x 128 bytes (the layout a TMA load with SWIZZLE_128B writes).
//   K-major:  rows are M (or N) indices, 64 K-elements per row; `sbo` = bytes between
//             8-row groups (1024); `lbo` is unused.
//   MN-major: rows are K indices, 64 M (or N) elements per row; `lbo` = bytes between
//             64-element MN blocks, `sbo` = bytes between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;   // SWIZZLE_128B
    return d;
}

// Loads 32 consecutive 32-bit TMEM columns (this warp's 32 lanes) and waits for them.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr + 0u) : "memory");
}

// Loads 64 consecutive 32-bit TMEM columns (this warp's 32 lanes) and waits for them.
__device__ __forceinline__ void tmem_ld_32x32b_x64(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr + 0u), "r"(taddr + 32u) : "memory");
}

// Loads 128 consecutive 32-bit TMEM columns (this warp's 32 lanes) and waits for them.
__device__ __forceinline__ void tmem_ld_32x32b_x128(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(taddr + 64u), "r"(taddr + 96u) : "memory");
}

// Stores 32 consecutive 32-bit TMEM columns (this warp's 32 lanes) and waits for the stores.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        "tcgen05.wait::st.sync.aligned;\n"
        :: "r"(taddr + 0u), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Stores 64 consecutive 32-bit TMEM columns (this warp's 32 lanes) and waits for the stores.
__device__ __forceinline__ void tmem_st_32x32b_x64(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n"
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%1], {%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65};\n"
        "tcgen05.wait::st.sync.aligned;\n"
        :: "r"(taddr + 0u), "r"(taddr + 32u), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

// ------------------------------------------------------------------------------------------
// small numeric helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// 2^x on the FMA pipe, for x in [-125, 128): Cody-Waite style reduction x = n + f with
// n = round(x) (by adding 1.5 * 2^23, which leaves n in the low mantissa bits) and
// f in [-1/2, 1/2], then a degree-3 polynomial for 2^f whose coefficients are a minimax
// (Remez) fit of relative error on [-1/2, 1/2] (max relative error 7.5e-5), and the
// exponent n added to the result's exponent field.  Two values at a time with the
// packed fp32 instructions.  Callers clamp x below at -125 so the exponent stays normal.
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
    const float2 magic = make_float2(12582912.f, 12582912.f);  // 1.5 * 2^23
    const float2 t = __fadd2_rn(x, magic);
    const float2 n = __fadd2_rn(t, make_float2(-12582912.f, -12582912.f));
    const float2 f = __ffma2_rn(n, make_float2(-1.f, -1.f), x);
    float2 p = __ffma2_rn(make_float2(0.0551716685f, 0.0551716685f), f,
                          make_float2(0.2426111251f, 0.2426111251f));
    p = __ffma2_rn(p, f, make_float2(0.6932609677f, 0.6932609677f));
    p = __ffma2_rn(p, f, make_float2(0.9999280572f, 0.9999280572f));
    // low bits of t hold n (two's complement): shifting them into the exponent field adds n
    const uint32_t ex = __float_as_uint(t.x) << 23, ey = __float_as_uint(t.y) << 23;
    return make_float2(__uint_as_float(__float_as_uint(p.x) + ex), __uint_as_float(__float_as_uint(p.y) + ey));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Four fp32 values to e4m3 (round to nearest even, saturating at +-448), a in the lowest
// byte.  cvt...e4m3x2 puts its first source in the upper byte of the 16-bit result.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// One 32-byte global store (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The 16-bit element type of a kernel instantiation: fp16 (F16) or bf16.  Two values to
// one 32-bit word (lo in the low half, round to nearest even), and the halves back to fp32.
template <bool F16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
    if constexpr (F16) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        return pack_bf16(lo, hi);
    }
}
template <bool F16>
__device__ __forceinline__ uint16_t round16(float x) {
    return (uint16_t)(pack16<F16>(x, 0.f) & 0xFFFFu);
}
template <bool F16>
__device__ __forceinline__ float lo16(uint32_t w) {
    if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
    else return bf16_lo(w);
}
template <bool F16>
__device__ __forceinline__ float hi16(uint32_t w) {
    if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    else return bf16_hi(w);
}

}  // namespace fa
