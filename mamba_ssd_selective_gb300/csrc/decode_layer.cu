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
    pdl_enter();
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
// Fast path (REG): the group is read once in 16-byte vectors and each
// thread's g values stay in registers between the reduction and the output;
// otherwise a second pass recomputes g from y and z.
constexpr int kNormThreads = 512;
constexpr int kNormRegVecs = 4;  // 16-byte vectors per thread held in registers (REG)

template <typename T>
__device__ __forceinline__ float norm_reduce(float ss, float *part) {
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < kNormThreads / 32; ++k) tot += part[k];
    return tot;
}

template <typename T, bool REG>
__global__ void __launch_bounds__(kNormThreads) gated_rmsnorm_kernel(const __grid_constant__ NormArgs a) {
    pdl_enter();
    constexpr int V = 16 / sizeof(T);  // elements per 16-byte vector
    const int64_t ngrp = a.D / a.group;
    const int64_t b = blockIdx.x / ngrp, g0 = (blockIdx.x % ngrp) * a.group;
    const T *y = static_cast<const T *>(a.y) + b * a.D + g0;
    const T *z = a.z ? static_cast<const T *>(a.z) + b * a.D + g0 : nullptr;
    T *out = static_cast<T *>(a.out) + b * a.D + g0;
    __shared__ float part[kNormThreads / 32];
    if constexpr (REG) {
        float g[kNormRegVecs][V], wv[kNormRegVecs][V];
        float ss = 0.f;
        const int64_t nv = a.group / V;
#pragma unroll
        for (int r = 0; r < kNormRegVecs; ++r) {
            const int64_t v = threadIdx.x + (int64_t)r * kNormThreads;
            if (v < nv) {
                // the weights too, before the reduction: no load after it
#pragma unroll
                for (int k = 0; k < V; k += 4) {
                    const float4 w4 = *reinterpret_cast<const float4 *>(a.w + g0 + v * V + k);
                    wv[r][k] = w4.x;
                    wv[r][k + 1] = w4.y;
                    wv[r][k + 2] = w4.z;
                    wv[r][k + 3] = w4.w;
                }
                const uint4 yv = *reinterpret_cast<const uint4 *>(y + v * V);
                const T *ye = reinterpret_cast<const T *>(&yv);
                uint4 zv = make_uint4(0, 0, 0, 0);
                if (z) zv = *reinterpret_cast<const uint4 *>(z + v * V);
                const T *ze = reinterpret_cast<const T *>(&zv);
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    g[r][k] = to_f32(ye[k]) * (z ? silu_f(to_f32(ze[k])) : 1.f);
                    ss = fmaf(g[r][k], g[r][k], ss);
                }
            }
        }
        const float rr = rsqrtf(norm_reduce<T>(ss, part) / (float)a.group + a.eps);
#pragma unroll
        for (int r = 0; r < kNormRegVecs; ++r) {
            const int64_t v = threadIdx.x + (int64_t)r * kNormThreads;
            if (v < nv) {
                uint4 ov;
                T *oe = reinterpret_cast<T *>(&ov);
#pragma unroll
                for (int k = 0; k < V; ++k) oe[k] = from_f32<T>(g[r][k] * rr * wv[r][k]);
                *reinterpret_cast<uint4 *>(out + v * V) = ov;
            }
        }
    } else {
        float ss = 0.f;
        for (int64_t i = threadIdx.x; i < a.group; i += kNormThreads) {
            const float g = to_f32(y[i]) * (z ? silu_f(to_f32(z[i])) : 1.f);
            ss = fmaf(g, g, ss);
        }
        const float rr = rsqrtf(norm_reduce<T>(ss, part) / (float)a.group + a.eps);
        for (int64_t i = threadIdx.x; i < a.group; i += kNormThreads) {
            const float g = to_f32(y[i]) * (z ? silu_f(to_f32(z[i])) : 1.f);
            out[i] = from_f32<T>(g * rr * a.w[g0 + i]);
        }
    }
}

template <typename T>
cudaError_t launch_conv_t(const ConvArgs &a, cudaStream_t stream) {
    const int64_t n = a.B * a.C;
    const unsigned grid = (unsigned)((n + 255) / 256);
    return launch_programmatic(a.W == 4 ? conv1d_step_kernel<T, 4> : conv1d_step_kernel<T, 0>, dim3(grid),
                               dim3(256), 0, stream, a);
}

}  // namespace

cudaError_t launch_conv1d_step(int io, const ConvArgs &a, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    return io == IO_BF16 ? launch_conv_t<__nv_bfloat16>(a, stream) : launch_conv_t<float>(a, stream);
}

cudaError_t launch_gated_rmsnorm(int io, const NormArgs &a, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    const unsigned grid = (unsigned)(a.B * (a.D / a.group));
    // register path: whole 16-byte vectors, aligned rows, a group that fits
    const int64_t V = io == IO_BF16 ? 8 : 4;
    const auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    const bool reg = a.group % V == 0 && a.D % V == 0 && a.group <= V * kNormThreads * kNormRegVecs && al(a.y) &&
                     al(a.out) && al(a.w) && (!a.z || al(a.z));
    void (*kern)(NormArgs);
    if (io == IO_BF16)
        kern = reg ? gated_rmsnorm_kernel<__nv_bfloat16, true> : gated_rmsnorm_kernel<__nv_bfloat16, false>;
    else
        kern = reg ? gated_rmsnorm_kernel<float, true> : gated_rmsnorm_kernel<float, false>;
    return launch_programmatic(kern, dim3(grid), dim3(kNormThreads), 0, stream, a);
}

}  // namespace ssd
