// diag.cu -- moe_selftest_wait: the library's bounded device wait, run on its own so that the
// failure path (a wait that runs out records MOE_ERR_TIMEOUT and the kernel returns) can be
// exercised without making any of the layer's kernels fail.
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// One thread waits on an mbarrier of count 1 for its first phase.  With arrive != 0 the thread
// arrives first and the wait succeeds at once; otherwise nothing ever arrives and the wait gives
// up after limit_ns (the same mbar_wait every pipeline of the library uses).  No copy is ever in
// flight, so returning early is safe.
__global__ void selftest_wait_kernel(int *status, uint64_t limit_ns, int arrive) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int no_abort;
    if (threadIdx.x != 0) return;
    no_abort = 0;
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    if (arrive) ptx::mbar_arrive(&bar);
    if (!ptx::mbar_wait(&bar, 0u, limit_ns, (volatile int *)&no_abort)) atomicCAS(status, 0, (int)MOE_ERR_TIMEOUT);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_selftest_wait(void *ws, size_t ws_bytes, unsigned long long limit_ns, int arrive,
                                        void *stream) {
    if (!ws || ws_bytes < 256 || limit_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    selftest_wait_kernel<<<1, 32, 0, s>>>(static_cast<int *>(ws), (uint64_t)limit_ns, arrive);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
