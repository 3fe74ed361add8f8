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
// life of the process.  Its device address is looked up once per device, on that
// device's first call (see device_scratch), so that first call should not be made while
// a stream is being captured.  Every call shares the one array: calls whose work
// overlaps on the GPU (different streams, or different host threads) race on it.  The
// forward resets the status word at the start of each call and overwrites every partial
// result it later reads, so nothing carried over from an earlier call is used.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // FA_NOALLOC_SCRATCH_BYTES

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device, with
// that device current).  Returns null when the lookup fails.
void* device_scratch(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
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
