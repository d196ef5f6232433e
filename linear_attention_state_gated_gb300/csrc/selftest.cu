// selftest.cu -- the bounded pipeline wait that every kernel uses, on its own: one
// thread waits on a fresh shared-memory mbarrier for at most a given number of
// cycles, after arriving on it first (the wait completes) or not (the wait gives
// up), and reports HYPIC_ETIMEOUT through the status word the way the pipeline
// kernels do when a wait runs out.  Nothing faults or traps; the context stays
// usable.
#include "internal.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

__global__ void wait_selftest_kernel(long long limit, int arrive, int *d_err, long long *d_cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    sm100::mbar_init(&bar, 1);
    sm100::mbar_fence_init();
    if (arrive) sm100::mbar_arrive(&bar);
    const long long t0 = clock64();
    const bool ok = sm100::mbar_wait_limit(&bar, 0, limit);
    const long long t1 = clock64();
    if (d_cycles) *d_cycles = t1 - t0;
    if (!ok && d_err) atomicExch(d_err, (int)HYPIC_ETIMEOUT);
}

}  // namespace
}  // namespace hypic

extern "C" int hypic_selftest_wait(long long limit_cycles, int arrive, int *d_err, long long *d_cycles,
                                   void *cuda_stream) {
    if (limit_cycles < 0 || limit_cycles > hypic::sm100::kWaitCycles) return HYPIC_EINVAL;
    if ((d_err && reinterpret_cast<uintptr_t>(d_err) % 4) || (d_cycles && reinterpret_cast<uintptr_t>(d_cycles) % 8))
        return HYPIC_EALIGN;
    hypic::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(cuda_stream)>>>(limit_cycles, arrive, d_err,
                                                                                      d_cycles);
    return cudaGetLastError() == cudaSuccess ? HYPIC_OK : HYPIC_ECUDA;
}
