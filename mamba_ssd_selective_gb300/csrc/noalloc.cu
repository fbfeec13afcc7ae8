// ssd_scan_chunked_noalloc: the chunked SSD prefill for callers that cannot
// allocate device memory.
//
// Some callers of this library are not allowed to call cudaMalloc at the
// point where they run the scan: plug-ins whose host framework owns all
// device memory and forbids allocation inside its enqueue call, and
// latency-critical loops that cannot afford the implicit device-wide
// synchronisation of an allocation and its release. Such
// callers still own their inputs and outputs; what they cannot provide is the
// per-chunk state workspace. This entry point takes it from a fixed scratch
// array compiled into the library instead.
//
// The scratch is a file-scope __device__ array of kScratchBytes (64 MiB).
// Every GPU that loads this part of the library holds it until the process
// exits. Its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device; make that first call before any stream capture starts. All
// calls on a device share the one array and it keeps whatever the last call
// left there: the kernels never depend on its previous contents (the status
// word is cleared by every call), but two calls whose kernels overlap on the
// GPU (different streams, no ordering between them) race on it.
#include <cstdarg>
#include <mutex>

#include "launch.h"
#include "ssd_scan.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
ssd_status scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return (ssd_status)ssd::set_error(SSD_ERR_CUDA, "ssd_scan_chunked_noalloc: cudaGetDevice: %s",
                                          cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return (ssd_status)ssd::set_error(SSD_ERR_UNSUPPORTED, "ssd_scan_chunked_noalloc: device %d out of range",
                                          dev);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p)
            return (ssd_status)ssd::set_error(SSD_ERR_CUDA,
                                              "ssd_scan_chunked_noalloc: cudaGetSymbolAddress: %s",
                                              cudaGetErrorString(e));
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SSD_OK;
}

}  // namespace

extern "C" ssd_status ssd_scan_chunked_noalloc(const ssd_dims *dims, const void *x, const void *dt, const float *A,
                                               const void *B, const void *C, const float *D,
                                               const float *init_state, int chunk_size, void *y,
                                               float *final_state, cudaStream_t stream) {
    const size_t need = ssd_workspace_size(dims, chunk_size);
    if (need == 0)  // invalid sizes: let the regular entry point describe the problem
        return ssd_scan_chunked(dims, x, dt, A, B, C, D, init_state, chunk_size, y, final_state, nullptr, 0,
                                stream);
    if (need > kScratchBytes)
        return (ssd_status)ssd::set_error(
            SSD_ERR_UNSUPPORTED,
            "ssd_scan_chunked_noalloc: these sizes need %zu bytes of scratch, the built-in scratch holds %zu "
            "(use a larger chunk size, a shorter sequence or ssd_scan_chunked with a workspace)",
            need, kScratchBytes);
    void *scratch = nullptr;
    ssd_status s = scratch_address(&scratch);
    if (s != SSD_OK) return s;
    return ssd_scan_chunked(dims, x, dt, A, B, C, D, init_state, chunk_size, y, final_state, scratch,
                            kScratchBytes, stream);
}

// The scratch begins with the status word of the workspace layout, so its
// status is read exactly as a caller workspace's is.
extern "C" ssd_status ssd_scan_chunked_noalloc_status(cudaStream_t stream, void **scratch_addr) {
    void *scratch = nullptr;
    ssd_status s = scratch_address(&scratch);
    if (s != SSD_OK) return s;
    if (scratch_addr) *scratch_addr = scratch;
    return ssd_workspace_status(scratch, stream);
}
