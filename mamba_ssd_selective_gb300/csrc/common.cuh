// Shared device helpers of the SSD kernels: element conversion, warp
// reductions and the chunk-local inclusive cumulative sum of dt*A.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Programmatic dependent launch. A kernel launched by launch_programmatic()
// may be placed on the GPU while the work before it in the stream drains; its
// first statement is pdl_wait() (or pdl_enter()), in every thread and before
// any early return: wait until that work has completed (its writes visible).
// Because every such kernel waits before it can finish, "the previous kernel
// has completed" also covers the ones before it. pdl_trigger() lets the next
// launch be placed once every CTA has triggered or exited: early for
// memory-bound kernels, at the end of the CTA's work for issue-bound ones,
// whose throughput drops when the next grid's CTAs sit resident beside them
// (measured on the Mamba-1 scan). Without the launch attribute these
// instructions do nothing.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_trigger();
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_programmatic(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Four consecutive elements (4-element aligned) as float32.
template <typename T> __device__ __forceinline__ float4 ld4(const T *p);
template <> __device__ __forceinline__ float4 ld4<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <> __device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}

template <typename I> __host__ __device__ __forceinline__ I imin(I a, I b) { return a < b ? a : b; }
template <typename I> __host__ __device__ __forceinline__ I imax(I a, I b) { return a > b ? a : b; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Inclusive prefix sum over a[0..n) held one value per thread (threads >= n
// hold 0), for blockDim.x a multiple of 32 of at least 256 and n <= 256.
// Result written to out[0..n). Fixed association (warp shuffle scan, then a
// scan of the first 8 warp totals), so it is bitwise reproducible and the same
// for any such block size. `scratch` holds at least 8 floats. Every thread of
// the block calls it; ends with a __syncthreads().
__device__ __forceinline__ void block_inclusive_scan_256(float a, int n, float *out, float *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float v = a;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31 && warp < 8) scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float t = lane < 8 ? scratch[lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            float u = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += u;
        }
        if (lane < 8) scratch[lane] = t;  // inclusive totals
    }
    __syncthreads();
    if (warp > 0 && warp < 8) v += scratch[warp - 1];
    if ((int)threadIdx.x < n) out[threadIdx.x] = v;
    __syncthreads();
}

}  // namespace ssd
