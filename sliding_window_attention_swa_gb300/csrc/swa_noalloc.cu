// swa_noalloc.cu -- ring-buffer decode for callers that cannot allocate device
// memory at the call site.
//
// swa_decode needs a workspace for its split partials, which the caller normally
// allocates.  Some callers can't: a serving loop that must not allocate once it is
// running (cudaMalloc may synchronise the device and can fail under memory
// pressure), or a plugin interface that hands the kernel only its inputs and
// outputs.  swa_decode_noalloc runs the same two kernels (split-K scoring, then the
// log-sum-exp merge) with the partials in a fixed scratch array compiled into the
// library, so it allocates nothing.
#include <mutex>

#include <cuda.h>

#include "swa_internal.h"

namespace {

// The scratch array: SWA_DECODE_NOALLOC_SCRATCH_BYTES of device memory on every GPU
// that loads the library, held until the process exits.  In host code its name is
// only a host-side stand-in; kernels get the device address from scratch_address().
static __device__ __align__(256) unsigned char g_decode_scratch[SWA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchEntry {
    unsigned long long ctx_id;  // context the address belongs to (0: none yet)
    void *ptr;                  // device address of g_decode_scratch in that context
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Unique ID of the calling thread's current CUDA context, 0 if it cannot be read.  The
// library's module -- and with it the scratch array -- is loaded again, possibly at
// another address, in a context created after a device reset, so a cached address is
// only reused within the context it was looked up in.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device, looked up with that
// device current the first time a context uses it, then cached for that context.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry &c = g_scratch[dev];
    const unsigned long long id = current_context_id();
    if (id != 0 && c.ctx_id == id && c.ptr) {
        *out = c.ptr;
        return cudaSuccess;
    }
    // (this also makes the device's primary context current if nothing has yet)
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    c.ctx_id = current_context_id();  // 0 (unreadable) never matches: looked up again next call
    c.ptr = p;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" swa_status swa_decode_noalloc(const swa_decode_params *p, swa_stream_t stream) {
    const swa_status st = swa::validate_decode(p);
    if (st != SWA_OK) return st;
    const size_t need = swa::decode_workspace_bytes(p);
    if (need > SWA_DECODE_NOALLOC_SCRATCH_BYTES) return SWA_ERR_WORKSPACE;
    void *ws = nullptr;
    if (swa::record_cuda_failure(scratch_address(&ws))) return SWA_ERR_CUDA;
    // Every partial the merge reads is written by the split kernel of the same call,
    // so the scratch needs no clearing between calls.
    if (swa::record_cuda_failure(swa::run_decode(p, ws, reinterpret_cast<cudaStream_t>(stream))))
        return SWA_ERR_CUDA;
    return SWA_OK;
}
