// Mamba-1 selective scan with a per-channel diagonal A[d, n].
//
// One thread owns one (b, d) channel and its dstate recurrences in registers;
// the N recurrences are independent, which gives each thread N-way
// instruction-level parallelism on the exp / FMA chain. A CTA covers 128
// consecutive channels of one sequence and walks the sequence in passes of
// `chunk` tokens; inside a pass, tiles of kTT tokens of x, dt (per channel)
// and B, C (shared by every channel) are staged through shared memory with
// coalesced loads. The state is carried exactly from pass to pass, so the
// output does not depend on the chunk size at all (runtime chunk routing is
// output preserving, "COREY ...", section 5.4).
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace ssd {
namespace {

constexpr int kCh = 128;  // channels per CTA (= threads)
constexpr int kTT = 32;   // tokens per staged tile

template <typename T, int NMAX>
__global__ void __launch_bounds__(kCh)
diag_scan_kernel(int64_t L, int64_t Dm, int N, const T *__restrict__ x, const T *__restrict__ dt,
                 const float *__restrict__ A, const T *__restrict__ Bm, const T *__restrict__ Cm,
                 const float *__restrict__ D, const float *__restrict__ init, int chunk, T *__restrict__ y,
                 float *__restrict__ final_state) {
    const int64_t b = blockIdx.y;
    const int tid = threadIdx.x;
    const int64_t d0 = (int64_t)blockIdx.x * kCh;
    const int64_t d = d0 + tid;
    const bool valid = d < Dm;

    __shared__ float sx[kTT][kCh], sdt[kTT][kCh];
    __shared__ float sB[kTT][NMAX], sC[kTT][NMAX];

    float h[NMAX], Ad[NMAX];
#pragma unroll
    for (int n = 0; n < NMAX; ++n) {
        const bool on = valid && n < N;
        h[n] = (on && init) ? init[(b * Dm + d) * N + n] : 0.f;
        Ad[n] = on ? A[d * N + n] : 0.f;
    }
    const float Dd = (valid && D) ? D[d] : 0.f;

    for (int64_t c0 = 0; c0 < L; c0 += chunk) {
        const int64_t cend = imin<int64_t>(L, c0 + chunk);
        for (int64_t t0 = c0; t0 < cend; t0 += kTT) {
            const int tn = (int)imin<int64_t>(kTT, cend - t0);
            __syncthreads();
            for (int tt = 0; tt < tn; ++tt) {
                const int64_t o = (b * L + t0 + tt) * Dm + d;
                sx[tt][tid] = valid ? to_f32(x[o]) : 0.f;
                sdt[tt][tid] = valid ? to_f32(dt[o]) : 0.f;
            }
            for (int e = tid; e < tn * NMAX; e += kCh) {
                const int tt = e / NMAX, n = e % NMAX;
                const int64_t o = (b * L + t0 + tt) * N + n;
                sB[tt][n] = n < N ? to_f32(Bm[o]) : 0.f;
                sC[tt][n] = n < N ? to_f32(Cm[o]) : 0.f;
            }
            __syncthreads();
            for (int tt = 0; tt < tn; ++tt) {
                const float dtv = sdt[tt][tid], xv = sx[tt][tid];
                const float u = dtv * xv;
                float acc = 0.f;
#pragma unroll
                for (int n = 0; n < NMAX; ++n) {
                    if (n < N) {
                        h[n] = fmaf(expf(dtv * Ad[n]), h[n], u * sB[tt][n]);
                        acc = fmaf(sC[tt][n], h[n], acc);
                    }
                }
                if (valid) y[(b * L + t0 + tt) * Dm + d] = from_f32<T>(acc + Dd * xv);
            }
        }
    }
    if (final_state && valid) {
#pragma unroll
        for (int n = 0; n < NMAX; ++n)
            if (n < N) final_state[(b * Dm + d) * N + n] = h[n];
    }
}

template <typename T, int NMAX>
cudaError_t launch_n(int64_t B, int64_t L, int64_t Dm, int64_t N, const void *x, const void *dt, const float *A,
                     const void *Bm, const void *Cm, const float *D, const float *init, int chunk, void *y,
                     float *final_state, cudaStream_t stream) {
    dim3 grid((unsigned)((Dm + kCh - 1) / kCh), (unsigned)B);
    diag_scan_kernel<T, NMAX><<<grid, kCh, 0, stream>>>(L, Dm, (int)N, (const T *)x, (const T *)dt, A,
                                                        (const T *)Bm, (const T *)Cm, D, init, chunk, (T *)y,
                                                        final_state);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(int64_t B, int64_t L, int64_t Dm, int64_t N, const void *x, const void *dt, const float *A,
                     const void *Bm, const void *Cm, const float *D, const float *init, int chunk, void *y,
                     float *final_state, cudaStream_t stream) {
    if (N <= 16) return launch_n<T, 16>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init, chunk, y, final_state, stream);
    if (N <= 32) return launch_n<T, 32>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init, chunk, y, final_state, stream);
    return launch_n<T, 64>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init, chunk, y, final_state, stream);
}

}  // namespace

cudaError_t launch_diag(int io, int64_t B, int64_t L, int64_t Dm, int64_t N, const void *x, const void *dt,
                        const float *A, const void *Bm, const void *Cm, const float *D, const float *init_state,
                        int chunk, void *y, float *final_state, cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    if (io == IO_BF16)
        return launch_t<__nv_bfloat16>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init_state, chunk, y, final_state, stream);
    return launch_t<float>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init_state, chunk, y, final_state, stream);
}

}  // namespace ssd
