// One-token SSD decode step over a batch, state updated in place.
//
// Memory-bound: every step reads and writes the whole float32 state
// [B, H, P, N] once. Layout is N-contiguous, so one warp streams one
// (b, h, p) row: lane l owns n = 4l .. 4l+3 (float4), the 128-bit accesses of a
// warp cover 512 contiguous bytes, and y[p] = sum_n C[n] h[p,n] is a warp
// shuffle reduction. Each warp keeps RB rows in flight to cover HBM latency.
// The state is touched once, with streaming cache hints, so it does not evict
// the small per-token inputs from L2.
#include "common.cuh"
#include "debug_bounds.cuh"
#include "launch.h"

namespace ssd {
namespace {

constexpr int kRB = 4;         // rows in flight per warp

// THREADS per (b, h): 128 (four warps, eight CTAs per SM) when the batch of
// heads fills the GPU many times over, 256 (eight warps) for small batches,
// where each (b, h) needs the extra warps; both measured on GB300.
template <typename T, int VW, int THREADS>
__global__ void __launch_bounds__(THREADS, THREADS == 128 ? 8 : 4)
decode_step_kernel(float *__restrict__ state, const T *__restrict__ x, const T *__restrict__ dt,
                   const float *__restrict__ A, const T *__restrict__ Bm, const T *__restrict__ Cm,
                   const float *__restrict__ D, T *__restrict__ y, int H, int P, int N, int G) {
    pdl_enter();  // the previous step's state update is complete
    const int64_t bh = blockIdx.x;  // b * H + h
    const int h = (int)(bh % H);
    const int64_t b = bh / H;
    const int g = h / (H / G);
    // extents of the buffers (the grid is B * H): state, x / y, B / C
    const int64_t n_state = (int64_t)gridDim.x * P * N, n_io = (int64_t)gridDim.x * P;
    const int64_t n_bc = (int64_t)(gridDim.x / H) * G * N;
    (void)n_state; (void)n_io; (void)n_bc;
    const float dtv = to_f32(dt[bh]);
    const float alpha = expf(dtv * A[h]);
    const float Dh = D ? D[h] : 0.f;
    const T *Bp = Bm + (b * G + g) * N;
    const T *Cp = Cm + (b * G + g) * N;
    float *st = state + bh * (int64_t)P * N;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nwarps = THREADS / 32;

    for (int p0 = warp; p0 < P; p0 += nwarps * kRB) {
        float acc[kRB], xp[kRB];
#pragma unroll
        for (int r = 0; r < kRB; ++r) {
            const int p = p0 + r * nwarps;
            acc[r] = 0.f;
            xp[r] = (p < P && SSD_IN_BOUNDS(bh * P + p, 1, n_io, kSiteDecodeIO)) ? to_f32(x[bh * P + p]) : 0.f;
        }
        for (int n0 = lane * VW; n0 < N; n0 += 32 * VW) {
            float bv[VW], cv[VW];
#pragma unroll
            const bool bc_ok = SSD_IN_BOUNDS((b * G + g) * N + n0, VW, n_bc, kSiteDecodeIO);
#pragma unroll
            for (int k = 0; k < VW; ++k) {
                bv[k] = bc_ok ? to_f32(Bp[n0 + k]) : 0.f;
                cv[k] = bc_ok ? to_f32(Cp[n0 + k]) : 0.f;
            }
            float hv[kRB][VW];
            // issue all loads of the row batch before any arithmetic
#pragma unroll
            for (int r = 0; r < kRB; ++r) {
                const int p = p0 + r * nwarps;
                if (p < P && SSD_IN_BOUNDS(bh * P * N + (int64_t)p * N + n0, VW, n_state, kSiteDecodeState)) {
                    if constexpr (VW == 4) {
                        float4 v = __ldcs(reinterpret_cast<const float4 *>(st + (int64_t)p * N + n0));
                        hv[r][0] = v.x; hv[r][1] = v.y; hv[r][2] = v.z; hv[r][3] = v.w;
                    } else {
                        hv[r][0] = __ldcs(st + (int64_t)p * N + n0);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kRB; ++r) {
                const int p = p0 + r * nwarps;
                if (p < P && SSD_IN_BOUNDS(bh * P * N + (int64_t)p * N + n0, VW, n_state, kSiteDecodeState)) {
                    const float u = dtv * xp[r];
#pragma unroll
                    for (int k = 0; k < VW; ++k) {
                        hv[r][k] = fmaf(alpha, hv[r][k], u * bv[k]);
                        acc[r] = fmaf(cv[k], hv[r][k], acc[r]);
                    }
                    if constexpr (VW == 4) {
                        __stcs(reinterpret_cast<float4 *>(st + (int64_t)p * N + n0),
                               make_float4(hv[r][0], hv[r][1], hv[r][2], hv[r][3]));
                    } else {
                        __stcs(st + (int64_t)p * N + n0, hv[r][0]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRB; ++r) {
            const float s = warp_sum(acc[r]);
            const int p = p0 + r * nwarps;
            if (lane == 0 && p < P && SSD_IN_BOUNDS(bh * P + p, 1, n_io, kSiteDecodeIO))
                y[bh * P + p] = from_f32<T>(s + Dh * xp[r]);
        }
    }
}

template <typename T>
cudaError_t launch_t(int64_t B, int64_t H, int64_t P, int64_t N, int64_t G, float *state, const void *x,
                     const void *dt, const float *A, const void *Bm, const void *Cm, const float *D, void *y,
                     cudaStream_t stream) {
    const int64_t grid = B * H;
    if (grid == 0) return cudaSuccess;
    const bool vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(state) & 15) == 0);
    const bool wide = grid >= 8 * sm_count(1);  // many (b, h) per SM: four warps each
    auto go = [&](auto kern, int threads) {
        return launch_programmatic(kern, dim3((unsigned)grid), dim3(threads), 0, stream, state, (const T *)x,
                                   (const T *)dt, A, (const T *)Bm, (const T *)Cm, D, (T *)y, (int)H, (int)P,
                                   (int)N, (int)G);
    };
    if (vec) return wide ? go(decode_step_kernel<T, 4, 128>, 128) : go(decode_step_kernel<T, 4, 256>, 256);
    return wide ? go(decode_step_kernel<T, 1, 128>, 128) : go(decode_step_kernel<T, 1, 256>, 256);
}

}  // namespace

SSD_BOUNDS_HOST_READER(bounds_word_decode)

cudaError_t launch_decode(int io, int64_t B, int64_t H, int64_t P, int64_t N, int64_t G, float *state,
                          const void *x, const void *dt, const float *A, const void *Bm, const void *Cm,
                          const float *D, void *y, cudaStream_t stream) {
    if (io == IO_BF16)
        return launch_t<__nv_bfloat16>(B, H, P, N, G, state, x, dt, A, Bm, Cm, D, y, stream);
    return launch_t<float>(B, H, P, N, G, state, x, dt, A, Bm, Cm, D, y, stream);
}

}  // namespace ssd
