// pa_selftest.cu -- exercise the bounded waits every kernel of libpa relies on.
//
// One CTA waits on an mbarrier phase that nothing completes and then on a
// shared word that nothing sets.  Each wait must give up after its time
// limit, report failure, and record PA_DEVERR_TIMEOUT in the device error
// word, leaving the context usable.  Nothing here faults or spins without a
// bound: every wait is limited by the wall clock.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void wait_timeout_selftest_kernel(unsigned int *err, int *result) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    __shared__ uint32_t word;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);   // one arrival completes phase 0; none ever comes
        abort_flag = 0;
        word = 0;
        mbar_init_fence();
    }
    __syncthreads();
    const bool barrier_ok = mbar_wait(&bar, 0, &abort_flag, err);
    __syncthreads();
    if (threadIdx.x == 0) {
        result[0] = barrier_ok ? 1 : 0;
        abort_flag = 0;       // the word wait must run out on its own clock
    }
    __syncthreads();
    const bool word_ok = wait_value(&word, 1u, &abort_flag, err);
    __syncthreads();
    if (threadIdx.x == 0) result[1] = word_ok ? 1 : 0;
    // the drain wait (used on the way out of a failed kernel) gives up too
    const bool drained = mbar_wait_drain(&bar, 0);
    if (threadIdx.x == 0) result[2] = drained ? 1 : 0;
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned int *err, int *result, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 64, 0, stream>>>(err, result);
    return cudaGetLastError();
}

}  // namespace pa
