// wait_probe.cu -- a test kernel for the library's bounded on-chip waits.
//
// One warp waits on an mbarrier through mbar_wait (ptx.cuh), the helper with
// which every kernel of the library waits on its pipeline barriers.  With
// arrive == 0 nothing ever completes the barrier's phase: each wait must give
// up once its limit has passed (or once another thread has given up), the
// first to give up setting the timeout bit of the status word, and the kernel
// must return, leaving the CUDA context usable.  With arrive == 1 thread 0
// arrives first and every wait must return at once with the status untouched.
// result[0] counts the threads whose wait completed, result[1] those that gave
// up; result[2] holds the longest wait in microseconds.
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace {

__global__ void wait_probe_kernel(unsigned *status, int *result, int arrive) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        spark::mbar_init(&bar, 1);
        spark::fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) spark::mbar_arrive(&bar);
    const unsigned long long t0 = spark::globaltimer_ns();
    const bool ok = spark::mbar_wait(&bar, 0, &abort_flag, status);
    const unsigned long long us = (spark::globaltimer_ns() - t0) / 1000ull;
    atomicAdd(&result[ok ? 0 : 1], 1);
    atomicMax(&result[2], static_cast<int>(us < 0x7fffffffull ? us : 0x7fffffffull));
}

}  // namespace

extern "C" int wait_probe(unsigned *status, int *result, int arrive, void *stream) {
    wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, result, arrive);
    return static_cast<int>(cudaGetLastError());
}
