// gdn_selftest.cu -- gdn_selftest_bounded_wait: shows, on the GPU, that the bounded
// mbarrier wait every tensor-core kernel uses gives up and reports instead of
// hanging.  The kernel waits on a barrier that nothing ever arrives on, with the
// caller's time limit, then ORs GDN_DEVICE_WAIT_TIMEOUT into the status word,
// exactly as the chunk kernels do when one of their waits runs out.  It holds no
// tensor memory and issues no copies, so giving up leaves nothing in flight.
#include "gdn_kernels.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

__global__ void k_wait_selftest(int32_t *status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        umma::mbar_init(&bar, 1);
        umma::fence_mbar_init();
    }
    __syncthreads();
    const bool got = umma::mbar_wait(&bar, 0, limit_ns);  // phase 0 never completes
    if (!__syncthreads_and(got) && threadIdx.x == 0) atomicOr(status, GDN_DEVICE_WAIT_TIMEOUT);
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_selftest_bounded_wait(int32_t *device_status, uint64_t limit_ns,
                                                gdn_stream_t stream) {
    if (!device_status || (reinterpret_cast<uintptr_t>(device_status) & 3u) != 0)
        return GDN_ERR_INVALID_ARG;
    if (limit_ns < 1000u || limit_ns > 1000000000u) return GDN_ERR_INVALID_ARG;
    gdn::k_wait_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        device_status, (unsigned long long)limit_ns);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
