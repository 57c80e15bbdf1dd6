// Self-test of the bounded waits: the failure path of every kernel, exercised
// without a fault.  One CTA initialises an mbarrier that nothing arrives on and
// waits for it through the same bounded wait the kernels use; when the limit
// runs out it records KDA_ERR_TIMEOUT in dev_status and returns, leaving the
// context usable.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

__global__ void wait_timeout_kernel(long long limit_cycles, int32_t *dev_status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort;
    const uint32_t b = sm100::smem_addr(&bar);
    if (threadIdx.x == 0) {
        sm100::mbar_init(b, 1);
        abort = 0;
        sm100::mbar_fence_init();
    }
    __syncthreads();
    // every thread waits, as the kernels' warps do; nobody arrives
    const bool ok = sm100::mbar_wait(b, 0, (volatile int *)&abort, limit_cycles);
    if (!ok && threadIdx.x == 0) dev_fail(dev_status, KDA_ERR_TIMEOUT);
}

}  // namespace
}  // namespace kda

extern "C" kda_status_t kda_selftest_wait_timeout(int32_t limit_us, int32_t *dev_status,
                                                  void *stream) {
    if (limit_us <= 0 || limit_us > 10000000 || !dev_status) return KDA_ERR_INVALID_ARG;
    // SM clocks: at most ~2.1 GHz on this part, so cycles = 2100 * microseconds
    const long long cycles = 2100ll * limit_us;
    kda::wait_timeout_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(cycles, dev_status);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
