// fa_fwd_noalloc: the forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory of their own: code that runs under a
// host framework which owns every allocation and hands out only the tensors it manages,
// plugins and real-time loops that must not enter the CUDA allocator, or hosts that
// forbid cudaMalloc after start-up.  fa_fwd needs a workspace (the status word, and for
// decode-shaped calls the split-KV partial results), which such a caller cannot provide.
// This entry point uses a fixed scratch array compiled into the library instead.
//
// The array lives in device global memory of every GPU that loads the library, for the
// life of the process.  Its device address is looked up once per device context, on the
// first call in that context (see device_scratch), so that first call should not be made
// while a stream is being captured.  A context destroyed and made again (cudaDeviceReset
// and the next runtime call) loads the module afresh and may place the array elsewhere;
// the lookup is then repeated, keyed by the driver's context id, which is never reused.
// Every call shares the one array: calls whose work overlaps on the GPU (different
// streams, or different host threads) race on it.  The forward resets the status word at the start of each call and overwrites every partial
// result it later reads, so nothing carried over from an earlier call is used.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // FA_NOALLOC_SCRATCH_BYTES

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchSlot {
    void* ptr = nullptr;            // device address of g_scratch in context `ctx_id`
    unsigned long long ctx_id = 0;  // the driver's unique id of that context (0 = none)
};
ScratchSlot g_slot[kMaxDevices];

// Unique id of the calling thread's current CUDA context, or 0 when there is none yet or
// the driver entry points are unavailable.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_scratch on device `dev` (current): looked up with that device current
// on its first call, and again whenever the device's context has changed since.  Returns
// null when the lookup fails.
void* device_scratch(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    ScratchSlot& s = g_slot[dev];
    const unsigned long long id = current_context_id();
    if (!s.ptr || id == 0 || id != s.ctx_id) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess) return nullptr;
        s.ptr = ptr;
        s.ctx_id = current_context_id();  // the lookup has made the context current
    }
    return s.ptr;
}

}  // namespace

extern "C" fa_status fa_fwd_noalloc(const fa_params* p, const void* q, const void* k, const void* v, void* o,
                                    float* lse, struct CUstream_st* stream) {
    const size_t need = fa_fwd_workspace_size(p);
    if (need == 0) {
        // invalid or unsupported: let fa_fwd's host checks report which (nothing launches)
        const fa_status rc = fa_fwd(p, q, k, v, o, lse, nullptr, 0, stream);
        return rc == FA_OK ? FA_ERR_INVALID_ARG : rc;
    }
    if (need > kScratchBytes) return FA_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    void* ws = device_scratch(dev);
    if (!ws) return FA_ERR_CUDA;
    return fa_fwd(p, q, k, v, o, lse, ws, kScratchBytes, stream);
}

static_assert(kScratchBytes == FA_NOALLOC_SCRATCH_BYTES, "scratch size and header disagree");
