// Per-role event trace of the tensor-core kernels.  Compiled in only with -DFA_TRACE=1,
// which the build makes as a separate library (libfa_gb300_trace.so); the product library
// has none of it: every call below is then an empty inline function.
//
// In a trace build the first kTraceCtas CTAs of a launch record: each role of such a CTA
// (the TMA producer, the MMA issuer, and up to two compute warp groups, each represented
// by lane 0 of its first warp) appends records to its own slice of the trace region that
// the planner adds to the workspace.  A record is two 64-bit words: a %globaltimer stamp,
// and (event << 32 | argument).  Events are the start of a work item, the two ends of a
// wait on a named barrier, and a few marks (an MMA burst issued, an epilogue begun or
// ended).  exact_attention_bwd_gb300/trace.py turns the records into per-role time
// budgets: how long each role spent waiting on which barrier, and per work item.
#pragma once
#include <cstddef>
#include <cstdint>

#include "ptx.cuh"

namespace fa {

constexpr int kTraceCtas = 16;     // CTAs of a launch that record
constexpr int kTraceRoles = 4;     // producer, MMA, compute group 0, compute group 1 (or dQ group)
constexpr int kTraceSlots = 8192;  // records per role and CTA
constexpr size_t kTraceBytes = size_t(kTraceCtas) * kTraceRoles * kTraceSlots * 16;

// event codes (the upper word of a record's second half)
enum TraceEvent : uint32_t {
    kEvItem = 1,       // a work item starts (argument: its index)
    kEvWait = 2,       // a wait on barrier `argument` starts
    kEvGot = 3,        // ... and ends
    kEvMark = 4,       // a mark (argument: TraceMark)
};

// barrier names (arguments of kEvWait / kEvGot)
enum TraceBarrier : uint32_t {
    kBQFull = 1, kBQEmpty, kBKFull, kBKEmpty, kBVFull, kBVEmpty, kBSFull, kBPFull, kBOFull, kBOFree,
    kBDoFull, kBDoEmpty, kBKvFull, kBDpFull, kBDsFull, kBDsFree, kBDqFull, kBDqFree, kBDkvFull, kBQTmem,
    kBPvDone, kBPdsFull, kBPdsFree, kBDkvFree,
};

// marks (arguments of kEvMark)
enum TraceMark : uint32_t {
    kMIssueS = 1, kMIssuePV, kMIssueDP, kMIssueDV, kMIssueDQ, kMIssueDK, kMSoftmaxDone, kMEpilogue,
    kMEpilogueDone, kMDqReduced, kMStepDone,
};

struct Tracer {
#ifdef FA_TRACE
    unsigned long long* rec = nullptr;  // this role's records, or null (not recording)
    int n = 0;
    // `region`: the trace region of the workspace (null: not recording); only lane 0 records
    __device__ __forceinline__ void init(unsigned long long* region, int role) {
        if (region && blockIdx.x < (unsigned)kTraceCtas && (threadIdx.x & 31) == 0)
            rec = region + ((size_t)blockIdx.x * kTraceRoles + role) * kTraceSlots * 2;
    }
    __device__ __forceinline__ void ev(uint32_t code, uint32_t arg) {
        if (rec && n < kTraceSlots) {
            rec[2 * n] = globaltimer();
            rec[2 * n + 1] = ((unsigned long long)code << 32) | arg;
            ++n;
        }
    }
#else
    __device__ __forceinline__ void init(unsigned long long*, int) {}
    __device__ __forceinline__ void ev(uint32_t, uint32_t) {}
#endif
    __device__ __forceinline__ void item(int idx) { ev(kEvItem, (uint32_t)idx); }
    __device__ __forceinline__ void mark(TraceMark m) { ev(kEvMark, m); }
};

// mbar_wait with the wait's two ends recorded
__device__ __forceinline__ bool twait(Tracer& tr, TraceBarrier b, uint64_t* bar, uint32_t parity, const Abort& ab) {
    tr.ev(kEvWait, b);
    const bool ok = mbar_wait(bar, parity, ab);
    tr.ev(kEvGot, b);
    return ok;
}

}  // namespace fa
