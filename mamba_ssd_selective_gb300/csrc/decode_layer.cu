// Decode-layer neighbours of the SSD decode step: the causal depthwise
// convolution step with its rolling window, and the gated RMS norm. They are
// the two pieces that must run on the device for a token's layer body to stay
// resident and be replayed as one CUDA graph ("Mamba-2 SSD fused layer via
// VGpuWarp — design sketch", section "What has to become a device op",
// items 1 and 2).
//
// Both are HBM-streaming: the convolution reads and rewrites each channel's
// window (16 bytes at width 4) and reads one input element; the norm reads y
// and z and writes the output, with one block reduction per group.
#include "common.cuh"
#include "launch.h"

namespace ssd {
namespace {

__device__ __forceinline__ float silu_f(float v) { return v / (1.f + expf(-v)); }

// One thread per (b, c). The window is W floats at state[(b*C + c)*W], oldest
// first; the new input shifts in, then out = act(w[c,:] . window + bias[c]).
// The output of channel c goes to segment s (c in [seg_end[s-1], seg_end[s])),
// a contiguous [B, width_s] array, so that one call can write the x | B | C
// parts of a conv output into the separate arrays the decode step reads.
template <typename T, int W>
__global__ void __launch_bounds__(256) conv1d_step_kernel(const __grid_constant__ ConvArgs a) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.B * a.C) return;
    const int64_t b = i / a.C, c = i % a.C;
    const int Wn = W > 0 ? W : a.W;
    float *win = a.state + i * Wn;
    const float *wc = a.w + c * Wn;
    const float xv = to_f32(static_cast<const T *>(a.x)[i]);
    float acc = a.bias ? a.bias[c] : 0.f;
    if (W == 4) {
        const float4 s = *reinterpret_cast<const float4 *>(win);
        const float4 w4 = *reinterpret_cast<const float4 *>(wc);
        const float4 ns = make_float4(s.y, s.z, s.w, xv);
        *reinterpret_cast<float4 *>(win) = ns;
        acc = fmaf(w4.x, ns.x, acc);
        acc = fmaf(w4.y, ns.y, acc);
        acc = fmaf(w4.z, ns.z, acc);
        acc = fmaf(w4.w, ns.w, acc);
    } else {
        float prev = xv;
        // walk from the newest slot down, shifting each value one slot older
        for (int k = Wn - 1; k >= 0; --k) {
            const float old = win[k];
            win[k] = prev;
            prev = old;
        }
        for (int k = 0; k < Wn; ++k) acc = fmaf(wc[k], win[k], acc);
    }
    const float o = a.act ? silu_f(acc) : acc;
    int s = 0;
    while (s < 2 && c >= a.seg_end[s]) ++s;
    const int64_t c0 = s == 0 ? 0 : a.seg_end[s - 1];
    const int64_t width = a.seg_end[s] - c0;
    static_cast<T *>(a.out[s])[b * width + (c - c0)] = from_f32<T>(o);
}

// One CTA per (b, group of `group` channels): g = y * silu(z) (z may be
// null), sum of g^2 by a block reduction, then out = g * rsqrt(mean + eps) * w.
// The second pass recomputes g from y and z, which the first pass left in L1/L2.
constexpr int kNormThreads = 512;

template <typename T>
__global__ void __launch_bounds__(kNormThreads) gated_rmsnorm_kernel(const __grid_constant__ NormArgs a) {
    const int64_t ngrp = a.D / a.group;
    const int64_t b = blockIdx.x / ngrp, g0 = (blockIdx.x % ngrp) * a.group;
    const T *y = static_cast<const T *>(a.y) + b * a.D + g0;
    const T *z = a.z ? static_cast<const T *>(a.z) + b * a.D + g0 : nullptr;
    T *out = static_cast<T *>(a.out) + b * a.D + g0;
    float ss = 0.f;
    for (int64_t i = threadIdx.x; i < a.group; i += kNormThreads) {
        const float g = to_f32(y[i]) * (z ? silu_f(to_f32(z[i])) : 1.f);
        ss = fmaf(g, g, ss);
    }
    __shared__ float part[kNormThreads / 32];
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < kNormThreads / 32; ++k) tot += part[k];
    const float r = rsqrtf(tot / (float)a.group + a.eps);
    for (int64_t i = threadIdx.x; i < a.group; i += kNormThreads) {
        const float g = to_f32(y[i]) * (z ? silu_f(to_f32(z[i])) : 1.f);
        out[i] = from_f32<T>(g * r * a.w[g0 + i]);
    }
}

template <typename T>
cudaError_t launch_conv_t(const ConvArgs &a, cudaStream_t stream) {
    const int64_t n = a.B * a.C;
    const unsigned grid = (unsigned)((n + 255) / 256);
    if (a.W == 4)
        conv1d_step_kernel<T, 4><<<grid, 256, 0, stream>>>(a);
    else
        conv1d_step_kernel<T, 0><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv1d_step(int io, const ConvArgs &a, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    return io == IO_BF16 ? launch_conv_t<__nv_bfloat16>(a, stream) : launch_conv_t<float>(a, stream);
}

cudaError_t launch_gated_rmsnorm(int io, const NormArgs &a, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    const unsigned grid = (unsigned)(a.B * (a.D / a.group));
    if (io == IO_BF16)
        gated_rmsnorm_kernel<__nv_bfloat16><<<grid, kNormThreads, 0, stream>>>(a);
    else
        gated_rmsnorm_kernel<float><<<grid, kNormThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace ssd
