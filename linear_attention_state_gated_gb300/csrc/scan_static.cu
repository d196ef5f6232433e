// scan_static.cu -- the fixed device scratch behind hypic_segment_scan_static.
//
// Some callers cannot allocate device memory at call time: a serving engine that
// handed all free device memory to its KV-cache pool at start-up, or a host path
// that must not enter the allocator (cudaMalloc / cudaFree can synchronise the
// device).  For them the two-pass dense scan can run out of this file-scope
// array instead of a caller workspace.  Nothing in it needs to start at zero:
// a call writes every record it later reads.  One array serves every call in
// the process, so two such calls in flight at once (other streams, other host
// threads) would overwrite each other's records: callers serialise them.
#include <mutex>

#include "internal.cuh"

namespace hypic {
namespace {

constexpr int64_t kStaticScratchBytes = (int64_t)64 << 20;   // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_scan_scratch[kStaticScratchBytes];

}  // namespace

int64_t static_scratch_bytes() { return kStaticScratchBytes; }

namespace {

// Unique id of the CUDA context current on this thread (ids are never reused
// within a process, unlike context handles after a device reset); false when
// no context is current or the driver does not offer the calls.
bool current_context_id(unsigned long long *id) {
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

// Device address of the scratch in the current context.  It is looked up
// (cudaGetSymbolAddress) on the first call in a context and cached under that
// context's id; a new context on the device (after cudaDeviceReset, or a
// caller-made context) gets its own lookup.
cudaError_t static_scratch(void **p) {
    struct Slot {
        unsigned long long ctx_id;
        void *addr;
    };
    static std::mutex mu;
    static Slot slot[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> lk(mu);
    Slot &sl = slot[dev];
    if (!have_id || !sl.addr || sl.ctx_id != id) {
        void *q = nullptr;
        e = cudaGetSymbolAddress(&q, g_scan_scratch);   // makes the device's primary context current if none is
        if (e != cudaSuccess) return e;
        if (!have_id) have_id = current_context_id(&id);
        sl.addr = have_id ? q : nullptr;   // without a context id nothing is cached: looked up every call
        sl.ctx_id = id;
        *p = q;
        return cudaSuccess;
    }
    *p = sl.addr;
    return cudaSuccess;
}

}  // namespace hypic
