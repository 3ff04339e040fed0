// sp_selftest.cu -- a check of the bounded-wait machinery every kernel of
// the library relies on, without faulting or hanging anything.  Mode 0: one
// warp waits on an mbarrier that nothing completes, so the wait gives up
// after a short cycle limit, raises the abort flag and the status word
// (kStatusTimeout) and the kernel returns.  Mode 1: a second warp arrives
// after a short delay, so the wait completes and the status stays clear.
// Mode 2: the meeting pattern of warps that must leave a loop together (the
// prefill's FP8 converter pair): each of two warps waits on its own
// mbarrier, one of which completes and one of which never does; they decide
// together with meet_any, both leave, and neither is left waiting at the
// named barrier that follows the work they would have done.
#include "sp_device.cuh"
#include "sp_internal.h"

namespace sp {

namespace {

__global__ void __launch_bounds__(64, 1)
k_wait_selftest(int* status, long long limit, int mode) {
    __shared__ uint64_t bar, bar2;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init(&bar2, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (mode == 2) {
        // warp 1's barrier is completed by its own lane 0; warp 0's never is
        if (warp == 1 && lane == 0) mbar_arrive(&bar2);
        __syncwarp();
        const bool got = mbar_wait(warp == 0 ? &bar : &bar2, 0, &abort_flag, status, limit);
        if (!meet_any<3>(64, !got)) {
            // both waits completed: the shared step and its closing barrier
            asm volatile("bar.sync 2, 64;" ::: "memory");
        }
    } else if (warp == 0) {
        mbar_wait(&bar, 0, &abort_flag, status, limit);
    } else if (mode == 1 && lane == 0) {
        const long long t0 = clock64();
        while (clock64() - t0 < limit / 8) { }      // bounded delay, then the arrival
        mbar_arrive(&bar);
    }
    __syncthreads();
}

}  // namespace

}  // namespace sp

extern "C" sp_status sp_selftest_bounded_wait(sp_cache* c, int64_t limit_cycles, int32_t mode,
                                              void* stream) {
    using namespace sp;
    if (!c) return fail(SP_ERR_INVALID_ARG, "null handle");
    if (mode < 0 || mode > 2) return fail(SP_ERR_INVALID_ARG, "mode must be 0, 1 or 2");
    if (limit_cycles < 1000 || limit_cycles > kWaitCycles)
        return fail(SP_ERR_INVALID_ARG, "limit_cycles must lie in [1000, 2e9]");
    k_wait_selftest<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(c->meta.status, limit_cycles, mode);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return SP_OK;
}
