// Bounds predicates for debug builds (compiled with -DSSD_DEBUG_BOUNDS).
//
// The kernels put their raw global-memory accesses (those that TMA does not
// clip) behind SSD_IN_BOUNDS(first, count, extent, site): in a debug build the
// predicate checks that elements [first, first + count) lie inside [0, extent);
// when they do not, the access is skipped and the first failing site and
// element index are recorded in this translation unit's device word, which
// ssd_debug_bounds_status() reads. Nothing traps: the kernel runs to its end
// and the context stays usable. In a release build the predicate is the
// constant true and costs nothing.
#pragma once
#include <stdint.h>

namespace ssd {

// Sites (the first failing one is reported).
enum BoundsSite : int {
    kSiteDecodeState = 1,
    kSiteDecodeIO = 2,
    kSiteDiagIO = 3,
    kSiteDiagBC = 4,
    kSiteDiagState = 5,
    kSiteFusedCarry = 6,
    kSiteFusedFlags = 7,
    kSiteFusedDt = 8,
    kSiteStatePass = 9,
};

#ifdef SSD_DEBUG_BOUNDS
// bit 63 set once a check failed; site in bits 48..55; element index in bits 0..47
static __device__ unsigned long long g_bounds_word;

__device__ __forceinline__ bool ssd_in_bounds(int64_t first, int64_t count, int64_t extent, int site) {
    if (first >= 0 && count >= 0 && first + count <= extent) return true;
    const unsigned long long w = (1ull << 63) | ((unsigned long long)(site & 0xff) << 48) |
                                 ((unsigned long long)first & 0xffffffffffffull);
    atomicCAS(&g_bounds_word, 0ull, w);
    return false;
}
#define SSD_IN_BOUNDS(first, count, extent, site) ::ssd::ssd_in_bounds((first), (count), (extent), (site))
#define SSD_BOUNDS_HOST_READER(name)                                                            \
    cudaError_t name(unsigned long long *out, bool clear) {                                     \
        cudaError_t e = cudaMemcpyFromSymbol(out, g_bounds_word, sizeof(*out));                 \
        if (e != cudaSuccess || !clear) return e;                                                \
        const unsigned long long z = 0;                                                          \
        return cudaMemcpyToSymbol(g_bounds_word, &z, sizeof(z));                                 \
    }
#else
#define SSD_IN_BOUNDS(first, count, extent, site) true
#define SSD_BOUNDS_HOST_READER(name)                                                            \
    cudaError_t name(unsigned long long *out, bool) {                                           \
        *out = 0;                                                                                \
        return cudaSuccess;                                                                      \
    }
#endif

}  // namespace ssd
