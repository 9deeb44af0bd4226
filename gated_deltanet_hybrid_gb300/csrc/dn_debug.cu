// Device-side failure detection, tested without a fault: one thread waits
// for a flag that nothing sets, exactly as the step's kernels wait on their
// barriers, and gives up after a bounded time (global timer), recording the
// give-up in the layer's device error word.  Used by dn_debug_expire_wait;
// the error word is what dn_get_state reports.
#include "dn_internal.cuh"

namespace dn {
namespace {

__device__ int g_never_set;  // no code writes it: the wait below always runs out

__global__ void expire_wait_kernel(int *err, unsigned long long limit_ns) {
    if (threadIdx.x != 0) return;
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    const volatile int *flag = &g_never_set;
    for (;;) {
        if (*flag != 0) return;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > limit_ns) break;
        __nanosleep(1000);
    }
    atomicOr(err, 4);  // the same word every bounded wait of the step reports to
}

}  // namespace

cudaError_t launch_expire_wait(int *err, int limit_us, cudaStream_t st) {
    expire_wait_kernel<<<1, 32, 0, st>>>(err, (unsigned long long)limit_us * 1000ull);
    return cudaGetLastError();
}

}  // namespace dn
