// selftest.cu - the device failure path, exercised without a fault: one CTA
// waits with the library's bounded mbarrier wait for a phase that nothing
// completes, gives up after the given time, records BDLM_ERR_TIMEOUT in the
// workspace header and returns.
#include <cuda_runtime.h>

#include "bdlm.h"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace bdlm {
namespace {

__global__ void __launch_bounds__(32, 1) selftest_timeout_kernel(WsHeader* hdr, unsigned long long wait_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        hdr->error = 0;
        hdr->info = 0;
        s_abort = 0;
        tc::mbar_init(tc::smem_addr(&bar), 1);  // one arrival expected, none will come
        tc::fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        const bool got = tc::mbar_wait(tc::smem_addr(&bar), 0, &s_abort, wait_ns);
        if (!got) set_error(hdr, DEV_TIMEOUT, 0);
    }
}

}  // namespace
}  // namespace bdlm

extern "C" BDLM_API int bdlm_selftest_timeout(void* workspace, size_t workspace_bytes, uint32_t wait_ns,
                                              bdlm_stream_t stream) {
    if (!workspace || workspace_bytes < sizeof(bdlm::WsHeader) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return BDLM_ERR_WORKSPACE;
    unsigned long long ns = wait_ns;
    if (ns < 1000000ull) ns = 1000000ull;
    if (ns > 2000000000ull) ns = 2000000000ull;
    bdlm::selftest_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<bdlm::WsHeader*>(workspace), ns);
    return cudaGetLastError() == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}
