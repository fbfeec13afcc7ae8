// Mamba-1 selective scan with a per-channel diagonal A[d, n].
//
// The dstate recurrences of one (b, d) channel live in registers; they are
// independent, which gives each thread several-way instruction-level
// parallelism on the exp / FMA chain (the bf16 path splits a channel's states
// over two threads and joins their y partial sums with one shuffle). The work
// per element (t, d, n) is one exponential and three FMA-pipe operations:
//     h_n = 2^(dt * A2[d,n]) * h_n + (dt * x) * B_t[n];   acc += C_t[n] * h_n
// with A2 = A * log2(e) prepared once per thread, so that each decay is a
// single SFU ex2 instruction; the exp and FMA rates, not HBM, bound this kernel
// on GB300.
//
// A CTA covers kCh consecutive channels of one sequence and walks the
// sequence in passes of `chunk` tokens, carrying the state exactly from pass
// to pass, so the output does not depend on the chunk size at all (runtime
// chunk routing is output preserving, "COREY ...", section 5.4). Inside a
// pass, tiles of kTT tokens of x and dt (per channel) and B, C (shared by all
// channels) are staged through shared memory with 16-byte cp.async copies,
// double-buffered so the next tile lands while this one is computed; y is
// staged in shared memory and written back with 16-byte stores.
#include "common.cuh"
#include "launch.h"

namespace ssd {
namespace {

constexpr int kCh = 64;   // channels per CTA of the bf16 path (2 threads each)
constexpr int kTT = 32;   // tokens per staged tile
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed float32 pairs (sm_100 family f32x2 arithmetic): two lanes of work per
// FP32-pipe instruction.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void up2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool pred) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    const int n = pred ? 16 : 0;  // zero-fill when out of range
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Vectorised bf16 path: dim % 8 == 0, N % 8 == 0, N <= 2 * NH, 16-byte aligned
// rows. Two threads share a channel, each owning NH of its states; their
// partial y sums meet in one shuffle. Partial accumulators per thread keep the
// dependent FMA chain short.
template <int NH>
__global__ void __launch_bounds__(2 * kCh)
diag_scan_bf16_kernel(int64_t L, int64_t Dm, int N, const __nv_bfloat16 *__restrict__ x,
                      const __nv_bfloat16 *__restrict__ dt, const float *__restrict__ A,
                      const __nv_bfloat16 *__restrict__ Bm, const __nv_bfloat16 *__restrict__ Cm,
                      const float *__restrict__ D, const float *__restrict__ init, int chunk,
                      __nv_bfloat16 *__restrict__ y, float *__restrict__ final_state) {
    constexpr int kThr = 2 * kCh;
    constexpr int NMAX = 2 * NH;
    const int64_t b = blockIdx.y;
    const int tid = threadIdx.x;
    const int ch = tid >> 1, half = tid & 1;   // channel in the CTA, which half of its states
    const int64_t d0 = (int64_t)blockIdx.x * kCh;
    const int64_t d = d0 + ch;
    const bool valid = d < Dm;
    const int nb = half * NH;                  // first state index of this thread

    __shared__ __align__(16) __nv_bfloat16 sx[2][kTT][kCh], sdt[2][kTT][kCh];
    __shared__ __align__(16) __nv_bfloat16 sB[2][kTT][NMAX], sC[2][kTT][NMAX];
    __shared__ __align__(16) __nv_bfloat16 sy[kTT][kCh];
    __shared__ __align__(16) float sBf[kTT][NMAX], sCf[kTT][NMAX];

    uint64_t h2[NH / 2], a2[NH / 2];  // state pairs and decay-rate pairs (base 2)
#pragma unroll
    for (int jp = 0; jp < NH / 2; ++jp) {
        float hv[2], av[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int n = nb + 2 * jp + u;
            const bool on = valid && n < N;
            hv[u] = (on && init) ? init[(b * Dm + d) * N + n] : 0.f;
            av[u] = on ? A[d * N + n] * kLog2e : 0.f;
        }
        h2[jp] = pk2(hv[0], hv[1]);
        a2[jp] = pk2(av[0], av[1]);
    }
    const float Dd = (valid && D) ? D[d] : 0.f;

    // stage tile [t0, t0 + tn) into buffer s: x, dt rows of kCh channels
    // (8 bf16 per 16-byte copy), B and C rows of N values (zero past N)
    auto stage = [&](int s, int64_t t0, int tn) {
        constexpr int kV = kCh / 8;  // 16-byte vectors per row
        for (int e = tid; e < kTT * kV; e += kThr) {
            const int tt = e / kV, v = e % kV;
            const bool in = tt < tn && d0 + v * 8 < Dm;
            const int64_t o = (b * L + t0 + (in ? tt : 0)) * Dm + d0 + (in ? v * 8 : 0);
            cp_async16(&sx[s][tt][v * 8], x + o, in);
            cp_async16(&sdt[s][tt][v * 8], dt + o, in);
        }
        constexpr int nv = NMAX / 8;
        for (int e = tid; e < kTT * nv; e += kThr) {
            const int tt = e / nv, v = e % nv;
            const bool in = tt < tn && v * 8 < N;
            const int64_t o = (b * L + t0 + (tt < tn ? tt : 0)) * N + (in ? v * 8 : 0);
            cp_async16(&sB[s][tt][v * 8], Bm + o, in);
            cp_async16(&sC[s][tt][v * 8], Cm + o, in);
        }
        cp_async_commit();
    };

    for (int64_t c0 = 0; c0 < L; c0 += chunk) {
        const int64_t cend = imin<int64_t>(L, c0 + chunk);
        int buf = 0;
        stage(0, c0, (int)imin<int64_t>(kTT, cend - c0));
        for (int64_t t0 = c0; t0 < cend; t0 += kTT) {
            const int tn = (int)imin<int64_t>(kTT, cend - t0);
            const int64_t t1 = t0 + kTT;
            if (t1 < cend) {
                stage(buf ^ 1, t1, (int)imin<int64_t>(kTT, cend - t1));
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            // B and C of the tile as float32, shared by every channel of the CTA
            for (int e = tid; e < tn * NMAX; e += kThr) {
                const int tt = e / NMAX, n = e % NMAX;
                sBf[tt][n] = __bfloat162float(sB[buf][tt][n]);
                sCf[tt][n] = __bfloat162float(sC[buf][tt][n]);
            }
            __syncthreads();
            for (int tt = 0; tt < tn; ++tt) {
                const float dtv = __bfloat162float(sdt[buf][tt][ch]);
                const float xv = __bfloat162float(sx[buf][tt][ch]);
                const uint64_t d2 = pk2(dtv, dtv), u2 = pk2(dtv * xv, dtv * xv);
                uint64_t acc2 = pk2(0.f, 0.f);
#pragma unroll
                for (int jp = 0; jp < NH / 2; ++jp) {
                    float e0, e1;
                    up2(mul2(d2, a2[jp]), e0, e1);
                    const uint64_t al = pk2(ex2f(e0), ex2f(e1));
                    const float2 bf = *reinterpret_cast<const float2 *>(&sBf[tt][nb + 2 * jp]);
                    const float2 cf = *reinterpret_cast<const float2 *>(&sCf[tt][nb + 2 * jp]);
                    h2[jp] = fma2(al, h2[jp], mul2(u2, pk2(bf.x, bf.y)));
                    acc2 = fma2(pk2(cf.x, cf.y), h2[jp], acc2);
                }
                float a0, a1;
                up2(acc2, a0, a1);
                float acc = a0 + a1;
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                if (half == 0) sy[tt][ch] = __float2bfloat16_rn(acc + Dd * xv);
            }
            __syncthreads();
            // write the tile's y rows back, 16 bytes per copy
            constexpr int kV = kCh / 8;
            for (int e = tid; e < tn * kV; e += kThr) {
                const int tt = e / kV, v = e % kV;
                if (d0 + v * 8 < Dm)
                    *reinterpret_cast<uint4 *>(y + (b * L + t0 + tt) * Dm + d0 + v * 8) =
                        *reinterpret_cast<const uint4 *>(&sy[tt][v * 8]);
            }
            buf ^= 1;
        }
    }
    if (final_state && valid) {
#pragma unroll
        for (int jp = 0; jp < NH / 2; ++jp) {
            float h0, h1;
            up2(h2[jp], h0, h1);
            if (nb + 2 * jp < N) final_state[(b * Dm + d) * N + nb + 2 * jp] = h0;
            if (nb + 2 * jp + 1 < N) final_state[(b * Dm + d) * N + nb + 2 * jp + 1] = h1;
        }
    }
}

// General path (float32 I/O, or shapes the vectorised path does not take).
template <typename T, int NMAX>
__global__ void __launch_bounds__(128)
diag_scan_kernel(int64_t L, int64_t Dm, int N, const T *__restrict__ x, const T *__restrict__ dt,
                 const float *__restrict__ A, const T *__restrict__ Bm, const T *__restrict__ Cm,
                 const float *__restrict__ D, const float *__restrict__ init, int chunk, T *__restrict__ y,
                 float *__restrict__ final_state) {
    constexpr int kC = 128;
    const int64_t b = blockIdx.y;
    const int tid = threadIdx.x;
    const int64_t d0 = (int64_t)blockIdx.x * kC;
    const int64_t d = d0 + tid;
    const bool valid = d < Dm;

    __shared__ float sx[kTT][kC], sdt[kTT][kC];
    __shared__ float sB[kTT][NMAX], sC[kTT][NMAX];

    float h[NMAX], A2[NMAX];
#pragma unroll
    for (int n = 0; n < NMAX; ++n) {
        const bool on = valid && n < N;
        h[n] = (on && init) ? init[(b * Dm + d) * N + n] : 0.f;
        A2[n] = on ? A[d * N + n] * kLog2e : 0.f;
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
            for (int e = tid; e < tn * NMAX; e += kC) {
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
                        h[n] = fmaf(ex2f(dtv * A2[n]), h[n], u * sB[tt][n]);
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
cudaError_t launch_general(int64_t B, int64_t L, int64_t Dm, int64_t N, const void *x, const void *dt,
                           const float *A, const void *Bm, const void *Cm, const float *D, const float *init,
                           int chunk, void *y, float *final_state, cudaStream_t stream) {
    dim3 grid((unsigned)((Dm + 127) / 128), (unsigned)B);
    diag_scan_kernel<T, NMAX><<<grid, 128, 0, stream>>>(L, Dm, (int)N, (const T *)x, (const T *)dt, A,
                                                       (const T *)Bm, (const T *)Cm, D, init, chunk, (T *)y,
                                                       final_state);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(int64_t B, int64_t L, int64_t Dm, int64_t N, const void *x, const void *dt, const float *A,
                     const void *Bm, const void *Cm, const float *D, const float *init, int chunk, void *y,
                     float *final_state, cudaStream_t stream) {
    if (N <= 16) return launch_general<T, 16>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init, chunk, y, final_state, stream);
    if (N <= 32) return launch_general<T, 32>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init, chunk, y, final_state, stream);
    return launch_general<T, 64>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init, chunk, y, final_state, stream);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

cudaError_t launch_diag(int io, int64_t B, int64_t L, int64_t Dm, int64_t N, const void *x, const void *dt,
                        const float *A, const void *Bm, const void *Cm, const float *D, const float *init_state,
                        int chunk, void *y, float *final_state, cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    if (io == IO_BF16) {
        const bool vec = Dm % 8 == 0 && N % 8 == 0 && N <= 32 && aligned16(x) && aligned16(dt) && aligned16(Bm) &&
                         aligned16(Cm) && aligned16(y);
        if (vec) {
            dim3 grid((unsigned)((Dm + kCh - 1) / kCh), (unsigned)B);
            if (N <= 16)
                diag_scan_bf16_kernel<8><<<grid, 2 * kCh, 0, stream>>>(
                    L, Dm, (int)N, (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)dt, A,
                    (const __nv_bfloat16 *)Bm, (const __nv_bfloat16 *)Cm, D, init_state, chunk,
                    (__nv_bfloat16 *)y, final_state);
            else
                diag_scan_bf16_kernel<16><<<grid, 2 * kCh, 0, stream>>>(
                    L, Dm, (int)N, (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)dt, A,
                    (const __nv_bfloat16 *)Bm, (const __nv_bfloat16 *)Cm, D, init_state, chunk,
                    (__nv_bfloat16 *)y, final_state);
            return cudaGetLastError();
        }
        return launch_t<__nv_bfloat16>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init_state, chunk, y, final_state, stream);
    }
    return launch_t<float>(B, L, Dm, N, x, dt, A, Bm, Cm, D, init_state, chunk, y, final_state, stream);
}

}  // namespace ssd
