// selftest.cu -- the bounded-wait path of the kernels, run on its own: a
// kernel waits on an mbarrier phase that nothing completes, gives up after the
// given time, and records KVD_ERR_TIMEOUT in the status word, as every decode
// and selection wait does when its data never arrives.  The test export of
// kvd_debug_wait_timeout; no fault, trap or endless loop is involved.
#include "common.cuh"
#include "internal.h"

namespace kvd {
namespace {

__global__ void __launch_bounds__(32) wait_probe_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int never;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none comes
        never = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_limit(&bar, 0, &never, limit_ns);
    if (!ok && threadIdx.x == 0) report_status(status, KVD_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_probe(int32_t *status, uint64_t limit_ns, cudaStream_t st) {
    wait_probe_kernel<<<1, 32, 0, st>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace kvd
