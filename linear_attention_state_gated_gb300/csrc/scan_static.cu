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

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t static_scratch(void **p) {
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *q = nullptr;
        e = cudaGetSymbolAddress(&q, g_scan_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = q;
    }
    *p = addr[dev];
    return cudaSuccess;
}

}  // namespace hypic
