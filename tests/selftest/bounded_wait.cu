// Test-only kernel: runs the library's bounded mbarrier wait (the one the
// bulk-copy dispatch uses) on a barrier that expects 16 bytes no copy will
// ever deliver, so the wait must give up after its limit, raise
// EP_FLAG_TIMEOUT and return with the context intact.  Nothing here faults,
// traps or spins without a bound.
#include "ep_internal.cuh"

namespace {

__global__ void bounded_wait_kernel(uint32_t* status, unsigned long long* elapsed_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ep::mbar_init(&bar, 1);
        ep::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ep::mbar_arrive_expect_tx(&bar, 16);  // phase 0 now waits for 16 bytes
        const uint64_t t0 = ep::globaltimer_ns();
        const bool done = ep::mbar_wait_bounded(&bar, 0);
        *elapsed_ns = ep::globaltimer_ns() - t0;
        if (!done) atomicOr(status, EP_FLAG_TIMEOUT);
    }
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int selftest_bounded_wait(
    uint32_t* status, unsigned long long* elapsed_ns, void* stream) {
    bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, elapsed_ns);
    return (int)cudaGetLastError();
}
