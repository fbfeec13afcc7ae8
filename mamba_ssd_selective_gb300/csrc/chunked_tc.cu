// Tensor-core (tcgen05) chunked SSD prefill for bf16 inputs, and the
// bounded-wait self-test kernel.
#include "common.cuh"
#include "launch.h"
#include "ssd_scan.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

// A shared-memory barrier that nothing ever completes, waited on with a poll
// budget: the wait must give up, record SSD_ERR_TIMEOUT and let the kernel exit.
__global__ void selftest_wait_kernel(int *status, int spin_limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t addr = tc::smem_u32(&bar);
        bool done = false;
        for (int i = 0; i < spin_limit && !done; ++i) done = tc::mbar_try_wait(addr, 0);
        if (!done) atomicCAS(status, SSD_OK, SSD_ERR_TIMEOUT);
    }
}

}  // namespace

cudaError_t launch_selftest_wait(int *status, int spin_limit, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, spin_limit);
    return cudaGetLastError();
}

bool chunked_tc_supported(const ChunkedArgs &) { return false; }

cudaError_t launch_chunked_tc(const ChunkedArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ssd
