// Self-test of the bounded waits: one CTA waits on a shared-memory barrier
// that nothing arrives at, with the same wait loop the kernels use on their
// asynchronous copies (barrier_wait of kda_async.cuh), gives up after the
// given limit and reports KDA_DEVERR_TIMEOUT.  No fault, trap or hang: the
// wait ends by its own clock and the kernel returns.
#include "kda_async.cuh"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

__global__ void selftest_wait_kernel(int32_t *err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = shared_addr(&bar);
    if (threadIdx.x == 0) barrier_init(b, 1);   // one arrival expected; none comes
    __syncthreads();
    if (threadIdx.x == 0 && !barrier_wait_for(b, 0, limit_ns)) report(err, DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t *err, int wait_us, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(err, (uint64_t)wait_us * 1000ull);
    return cudaGetLastError();
}

}  // namespace kda
