// Self-test of the bounded waits: every wait of the library's kernels on an
// mbarrier (bulk-copy and MMA completion) gives up after a bounded number of
// polls and reports it in a status word instead of hanging the GPU.  This
// kernel runs that same wait on a barrier that either receives its arrival or
// never does, so a test can make the wait run out without any fault and check
// that the expiry is reported and the context stays usable.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

__global__ void bounded_wait_kernel(int32_t *status, uint32_t polls, int32_t arrive)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (arrive != 0 && threadIdx.x == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&bar)) : "memory");
    __syncthreads();
    const bool done = mbar_wait(&bar, 0, polls);
    if (threadIdx.x == 0) *status = done ? 0 : 1;
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int32_t *status, uint32_t polls, int32_t arrive, cudaStream_t st)
{
    bounded_wait_kernel<<<1, 32, 0, st>>>(status, polls, arrive);
    return cudaGetLastError();
}

}  // namespace kda
