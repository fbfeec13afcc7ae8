// Mamba-1 selective scan with a per-channel diagonal A[d, n].
//
// The dstate recurrences of one (b, d) channel live in registers; they are
// independent, which gives each thread several-way instruction-level
// parallelism on the exp / FMA chain (the bf16 path splits a channel's states
// over two threads, one thread at N <= 8, and joins their y partial sums with
// one shuffle). The work per element (t, d, n) is one exponential and four
// float32 operations, issued as packed pairs of states:
//     h_n = 2^(dt * A2[d,n]) * h_n + (dt * x) * B_t[n];   acc += C_t[n] * h_n
// with A2 = A * log2(e) prepared once per thread, so that each decay is a
// single SFU ex2 instruction; the exp and FMA rates and the latency of that
// chain, not HBM, bound this kernel on GB300.
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
#include "debug_bounds.cuh"
#include "launch.h"

namespace ssd {
namespace {

constexpr int kCh = 64;   // channels per CTA of the bf16 path at two threads per channel
constexpr int kCh1 = 64;  // channels per CTA of the bf16 path at one thread per channel
constexpr int kUnr1 = 2;  // token-loop unroll at one thread per channel
constexpr int kUnr2 = 8;  // token-loop unroll at two threads per channel
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

// Per-token step transform and output gate of selective_scan_fn's options:
// dt <- softplus(dt + delta_bias[d]) (softplus only when asked), and
// out <- out * silu(z). softplus(v) is v itself above 20, where log(1 + e^v)
// and v round to the same float32.
__device__ __forceinline__ float step_of(float raw, float bias, bool softplus) {
    const float v = raw + bias;
    return softplus ? (v > 20.f ? v : log1pf(expf(v))) : v;
}
__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

// Vectorised bf16 path: dim % 8 == 0, N % 8 == 0, N <= TPC * NH, 16-byte
// aligned rows. TPC threads share a channel (1 or 2), each owning NH of its
// states; with two, their partial y sums meet in one shuffle. A CTA covers CH
// channels. B and C rows are read from shared memory four floats at a time
// (one broadcast load per four states), and two partial accumulators keep the
// dependent FMA chain of y short. OPT instantiations also apply delta_bias,
// delta_softplus and the z gate; z tiles are staged beside x and dt.
//
// MODE selects the part of a time-segmented scan (blockIdx.z = segment):
//   kWhole   one segment per sequence: the state enters from init_state and
//            leaves to final_state;
//   kLocal   each segment from a zero state, y not formed: writes the
//            segment's end state and the sum of its steps to the workspace;
//   kOutput  each segment from the entering state that the segment pass left
//            in the workspace, writing y.
enum { kWhole = 0, kLocal = 1, kOutput = 2 };
template <int NH, int TPC, int CH, int UNR, bool OPT, int MODE>
__global__ void __launch_bounds__(TPC * CH) diag_scan_bf16_kernel(const __grid_constant__ DiagArgs a) {
    static_assert(TPC == 1 || TPC == 2, "one or two threads per channel");
    static_assert(NH % 4 == 0 && CH % 8 == 0, "four-state groups, 16-byte channel rows");
    pdl_wait();  // the next launch is let in at the end (issue-bound kernel)
    constexpr int kThr = TPC * CH;
    constexpr int NMAX = TPC * NH;
    const int64_t L = a.L, Dm = a.Dm;
    const int N = a.N;
    const __nv_bfloat16 *__restrict__ x = static_cast<const __nv_bfloat16 *>(a.x);
    const __nv_bfloat16 *__restrict__ dt = static_cast<const __nv_bfloat16 *>(a.dt);
    const __nv_bfloat16 *__restrict__ zg = static_cast<const __nv_bfloat16 *>(a.z);
    const __nv_bfloat16 *__restrict__ Bm = static_cast<const __nv_bfloat16 *>(a.Bm);
    const __nv_bfloat16 *__restrict__ Cm = static_cast<const __nv_bfloat16 *>(a.Cm);
    __nv_bfloat16 *__restrict__ y = static_cast<__nv_bfloat16 *>(a.y);
    const int64_t b = blockIdx.y;
    const int tid = threadIdx.x;
    const int ch = TPC == 2 ? tid >> 1 : tid;   // channel in the CTA
    const int half = TPC == 2 ? tid & 1 : 0;    // which part of its states
    const int64_t d0 = (int64_t)blockIdx.x * CH;
    const int64_t d = d0 + ch;
    const bool valid = d < Dm;
    const int nb = half * NH;                   // first state index of this thread
    const bool has_z = OPT && zg != nullptr && MODE != kLocal;
    const bool softplus = OPT && a.softplus;
    const int64_t seg = blockIdx.z;
    const int64_t t_begin = seg * a.seg_len, t_end = imin<int64_t>(L, t_begin + a.seg_len);
    // entering state: init_state, zero, or the segment pass's result
    const float *h_in = MODE == kWhole ? a.init : MODE == kLocal ? nullptr : a.ws_h + seg * a.B * Dm * N;

    __shared__ __align__(16) __nv_bfloat16 sx[2][kTT][CH], sdt[2][kTT][CH];
    __shared__ __align__(16) __nv_bfloat16 sz[2][kTT][OPT ? CH : 8];
    __shared__ __align__(16) __nv_bfloat16 sB[2][kTT][NMAX], sC[2][kTT][NMAX];
    __shared__ __align__(16) __nv_bfloat16 sy[kTT][CH];
    __shared__ __align__(16) float sBf[kTT][NMAX], sCf[kTT][NMAX];

    uint64_t h2[NH / 2], a2[NH / 2];  // state pairs and decay-rate pairs (base 2)
#pragma unroll
    for (int jp = 0; jp < NH / 2; ++jp) {
        float hv[2], av[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int n = nb + 2 * jp + u;
            const bool on = valid && n < N;
            hv[u] = (on && h_in && SSD_IN_BOUNDS((b * Dm + d) * N + n, 1, a.B * Dm * N, kSiteDiagState))
                        ? h_in[(b * Dm + d) * N + n] : 0.f;
            av[u] = on ? a.A[d * N + n] * kLog2e : 0.f;
        }
        h2[jp] = pk2(hv[0], hv[1]);
        a2[jp] = pk2(av[0], av[1]);
    }
    const float Dd = (valid && a.D) ? a.D[d] : 0.f;
    const float bias = (OPT && valid && a.delta_bias) ? a.delta_bias[d] : 0.f;
    float dt_sum = 0.f;  // kLocal: sum of the segment's steps

    // stage tile [t0, t0 + tn) into buffer s: x, dt (and z) rows of CH
    // channels (8 bf16 per 16-byte copy), B and C rows of N values (zero past N)
    auto stage = [&](int s, int64_t t0, int tn) {
        constexpr int kV = CH / 8;  // 16-byte vectors per row
        for (int e = tid; e < kTT * kV; e += kThr) {
            const int tt = e / kV, v = e % kV;
            const bool in = tt < tn && d0 + v * 8 < Dm &&
                            SSD_IN_BOUNDS((b * L + t0 + tt) * Dm + d0 + v * 8, 8, a.B * L * Dm, kSiteDiagIO);
            // a valid address when zero-filling
            const int64_t o = (b * L + t0 + (in ? tt : 0)) * Dm + d0 + (in ? v * 8 : 0);
            cp_async16(&sx[s][tt][v * 8], x + o, in);
            cp_async16(&sdt[s][tt][v * 8], dt + o, in);
            if (has_z) cp_async16(&sz[s][tt][v * 8], zg + o, in);
        }
        constexpr int nv = NMAX / 8;
        for (int e = tid; e < kTT * nv; e += kThr) {
            const int tt = e / nv, v = e % nv;
            const bool in = tt < tn && v * 8 < N &&
                            SSD_IN_BOUNDS((b * L + t0 + tt) * N + v * 8, 8, a.B * L * N, kSiteDiagBC);
            const int64_t o = (b * L + t0 + (in ? tt : 0)) * N + (in ? v * 8 : 0);
            cp_async16(&sB[s][tt][v * 8], Bm + o, in);
            cp_async16(&sC[s][tt][v * 8], Cm + o, in);
        }
        cp_async_commit();
    };

    for (int64_t c0 = t_begin; c0 < t_end; c0 += a.chunk) {
        const int64_t cend = imin<int64_t>(t_end, c0 + a.chunk);
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
            // one token of the recurrence for this thread's states; returns the
            // thread's part of sum_n C_n h_n. With `finish` the token's y is
            // completed here (the partner thread's part by a shuffle).
            auto token = [&](int tt, bool finish) -> float {
                float dtv = __bfloat162float(sdt[buf][tt][ch]);
                if (OPT) dtv = step_of(dtv, bias, softplus);
                if (MODE == kLocal) dt_sum += dtv;
                const float xv = __bfloat162float(sx[buf][tt][ch]);
                const uint64_t d2 = pk2(dtv, dtv), u2 = pk2(dtv * xv, dtv * xv);
                uint64_t acc2 = pk2(0.f, 0.f);  // packed partial sums of C_n h_n
#pragma unroll
                for (int q = 0; q < NH / 4; ++q) {
                    const float4 bq = *reinterpret_cast<const float4 *>(&sBf[tt][nb + 4 * q]);
                    const float4 cq = *reinterpret_cast<const float4 *>(&sCf[tt][nb + 4 * q]);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int jp = 2 * q + r;
                        float e0, e1;
                        up2(mul2(d2, a2[jp]), e0, e1);
                        const uint64_t al = pk2(ex2f(e0), ex2f(e1));
                        const uint64_t bb = r ? pk2(bq.z, bq.w) : pk2(bq.x, bq.y);
                        const uint64_t cc = r ? pk2(cq.z, cq.w) : pk2(cq.x, cq.y);
                        h2[jp] = fma2(al, h2[jp], mul2(u2, bb));
                        if (MODE != kLocal) acc2 = fma2(cc, h2[jp], acc2);
                    }
                }
                if (MODE == kLocal) return 0.f;
                float a0, a1;
                up2(acc2, a0, a1);
                float acc = a0 + a1;
                // without the options half 0's part carries D x (finish8 then needs no x)
                if (!finish) return OPT ? acc : fmaf(half ? 0.f : Dd, xv, acc);
                if (TPC == 2) acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                float out = acc + Dd * xv;
                if (has_z) out *= silu(__bfloat162float(sz[buf][tt][ch]));
                if (half == 0) sy[tt][ch] = __float2bfloat16_rn(out);
                return 0.f;
            };
            // y of eight tokens from both threads' parts: the pair exchanges
            // halves with four shuffles and each thread completes four tokens
            // (half 0 the first four). With the options these are the sums of
            // `finish` (a + b = b + a); without, D x is already in half 0's part.
            // Tiles start at multiples of 32 tokens whatever the chunk size, so
            // which tokens take this path does not depend on it.
            auto finish8 = [&](int tt0, const float (&pt)[8]) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float recv = __shfl_xor_sync(0xffffffffu, half ? pt[j] : pt[j + 4], 1);
                    const int tt = tt0 + (half ? j + 4 : j);
                    float out = (half ? pt[j + 4] : pt[j]) + recv;
                    if (OPT) out += Dd * __bfloat162float(sx[buf][tt][ch]);
                    if (has_z) out *= silu(__bfloat162float(sz[buf][tt][ch]));
                    sy[tt][ch] = __float2bfloat16_rn(out);
                }
            };
            // full tiles unrolled so the decays of the next tokens overlap this
            // token's dependent chain; the same arithmetic either way
            if (tn == kTT) {
                if constexpr (TPC == 2 && MODE != kLocal && !OPT) {
                    // the whole tile's four groups of eight unrolled: measured
                    // faster without the options, slower with them (z gate, softplus)
#pragma unroll 4
                    for (int tt0 = 0; tt0 < kTT; tt0 += 8) {
                        float pt[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) pt[j] = token(tt0 + j, false);
                        finish8(tt0, pt);
                    }
                } else if constexpr (TPC == 2 && MODE != kLocal) {
#pragma unroll 1
                    for (int tt0 = 0; tt0 < kTT; tt0 += 8) {
                        float pt[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) pt[j] = token(tt0 + j, false);
                        finish8(tt0, pt);
                    }
                } else {
#pragma unroll UNR
                    for (int tt = 0; tt < kTT; ++tt) token(tt, true);
                }
            } else {
                for (int tt = 0; tt < tn; ++tt) token(tt, true);
            }
            __syncthreads();
            // write the tile's y rows back, 16 bytes per copy
            constexpr int kV = CH / 8;
            if (MODE != kLocal)
                for (int e = tid; e < tn * kV; e += kThr) {
                    const int tt = e / kV, v = e % kV;
                    if (d0 + v * 8 < Dm && SSD_IN_BOUNDS((b * L + t0 + tt) * Dm + d0 + v * 8, 8, a.B * L * Dm, kSiteDiagIO))
                        *reinterpret_cast<uint4 *>(y + (b * L + t0 + tt) * Dm + d0 + v * 8) =
                            *reinterpret_cast<const uint4 *>(&sy[tt][v * 8]);
                }
            buf ^= 1;
        }
    }
    pdl_trigger();
    float *h_out = MODE == kWhole ? a.final_state : MODE == kLocal ? a.ws_h + seg * a.B * Dm * N : nullptr;
    if (h_out && valid && SSD_IN_BOUNDS((b * Dm + d) * N + nb, imax(0, imin(NH, N - nb)), a.B * Dm * N, kSiteDiagState)) {
#pragma unroll
        for (int jp = 0; jp < NH / 2; ++jp) {
            float h0, h1;
            up2(h2[jp], h0, h1);
            if (nb + 2 * jp < N) h_out[(b * Dm + d) * N + nb + 2 * jp] = h0;
            if (nb + 2 * jp + 1 < N) h_out[(b * Dm + d) * N + nb + 2 * jp + 1] = h1;
        }
    }
    if (MODE == kLocal && valid && half == 0) a.ws_s[(seg * a.B + b) * Dm + d] = dt_sum;
}

// Segment pass of the time-segmented scan: one thread per (b, d, n) walks the
// segments in order. Segment s changes the state h entering it to
//     exp(A[d,n] * sum of its steps) * h + (its end state from zero),
// the diagonal decay over a segment being the exponential of A times the sum
// of its steps. The state entering each segment replaces that segment's local
// end state in ws_h; the state after the last is the final state.
__global__ void __launch_bounds__(256) diag_segment_pass_kernel(const __grid_constant__ DiagArgs a) {
    constexpr int kPF = 16;  // segments whose values are loaded before the chain consumes them
    pdl_enter();
    const int64_t Dm = a.Dm, N = a.N, B = a.B;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (b, d, n)
    if (i >= B * Dm * N) return;
    const int64_t n = i % N, d = (i / N) % Dm, b = i / (N * Dm);
    const float a2 = a.A[d * N + n] * kLog2e;
    float h = a.init ? a.init[i] : 0.f;
    for (int s0 = 0; s0 < a.nseg; s0 += kPF) {
        float loc[kPF], sum[kPF];
#pragma unroll
        for (int u = 0; u < kPF; ++u) {
            if (s0 + u < a.nseg) {
                loc[u] = a.ws_h[(int64_t)(s0 + u) * B * Dm * N + i];
                sum[u] = a.ws_s[((int64_t)(s0 + u) * B + b) * Dm + d];
            }
        }
#pragma unroll
        for (int u = 0; u < kPF; ++u) {
            if (s0 + u < a.nseg) {
                a.ws_h[(int64_t)(s0 + u) * B * Dm * N + i] = h;
                h = fmaf(ex2f(a2 * sum[u]), h, loc[u]);
            }
        }
    }
    if (a.final_state) a.final_state[i] = h;
}

// General path (float32 I/O, or shapes the vectorised path does not take).
template <typename T, int NMAX, bool OPT>
__global__ void __launch_bounds__(128) diag_scan_kernel(const __grid_constant__ DiagArgs a) {
    pdl_wait();  // the next launch is let in at the end (issue-bound kernel)
    constexpr int kC = 128;
    const int64_t L = a.L, Dm = a.Dm;
    const int N = a.N;
    const T *__restrict__ x = static_cast<const T *>(a.x);
    const T *__restrict__ dt = static_cast<const T *>(a.dt);
    const T *__restrict__ zg = static_cast<const T *>(a.z);
    const T *__restrict__ Bm = static_cast<const T *>(a.Bm);
    const T *__restrict__ Cm = static_cast<const T *>(a.Cm);
    T *__restrict__ y = static_cast<T *>(a.y);
    const int64_t b = blockIdx.y;
    const int tid = threadIdx.x;
    const int64_t d0 = (int64_t)blockIdx.x * kC;
    const int64_t d = d0 + tid;
    const bool valid = d < Dm;
    const bool has_z = OPT && zg != nullptr;
    const bool softplus = OPT && a.softplus;

    __shared__ float sx[kTT][kC], sdt[kTT][kC], sz[kTT][OPT ? kC : 1];
    __shared__ float sB[kTT][NMAX], sC[kTT][NMAX];

    float h[NMAX], A2[NMAX];
#pragma unroll
    for (int n = 0; n < NMAX; ++n) {
        const bool on = valid && n < N;
        h[n] = (on && a.init) ? a.init[(b * Dm + d) * N + n] : 0.f;
        A2[n] = on ? a.A[d * N + n] * kLog2e : 0.f;
    }
    const float Dd = (valid && a.D) ? a.D[d] : 0.f;
    const float bias = (OPT && valid && a.delta_bias) ? a.delta_bias[d] : 0.f;

    for (int64_t c0 = 0; c0 < L; c0 += a.chunk) {
        const int64_t cend = imin<int64_t>(L, c0 + a.chunk);
        for (int64_t t0 = c0; t0 < cend; t0 += kTT) {
            const int tn = (int)imin<int64_t>(kTT, cend - t0);
            __syncthreads();
            for (int tt = 0; tt < tn; ++tt) {
                const int64_t o = (b * L + t0 + tt) * Dm + d;
                sx[tt][tid] = valid ? to_f32(x[o]) : 0.f;
                sdt[tt][tid] = valid ? to_f32(dt[o]) : 0.f;
                if (has_z) sz[tt][tid] = valid ? to_f32(zg[o]) : 0.f;
            }
            for (int e = tid; e < tn * NMAX; e += kC) {
                const int tt = e / NMAX, n = e % NMAX;
                const int64_t o = (b * L + t0 + tt) * N + n;
                sB[tt][n] = n < N ? to_f32(Bm[o]) : 0.f;
                sC[tt][n] = n < N ? to_f32(Cm[o]) : 0.f;
            }
            __syncthreads();
            for (int tt = 0; tt < tn; ++tt) {
                float dtv = sdt[tt][tid];
                if (OPT) dtv = step_of(dtv, bias, softplus);
                const float xv = sx[tt][tid];
                const float u = dtv * xv;
                float acc = 0.f;
#pragma unroll
                for (int n = 0; n < NMAX; ++n) {
                    if (n < N) {
                        h[n] = fmaf(ex2f(dtv * A2[n]), h[n], u * sB[tt][n]);
                        acc = fmaf(sC[tt][n], h[n], acc);
                    }
                }
                float out = acc + Dd * xv;
                if (has_z) out *= silu(sz[tt][tid]);
                if (valid) y[(b * L + t0 + tt) * Dm + d] = from_f32<T>(out);
            }
        }
    }
    pdl_trigger();
    if (a.final_state && valid) {
#pragma unroll
        for (int n = 0; n < NMAX; ++n)
            if (n < N) a.final_state[(b * Dm + d) * N + n] = h[n];
    }
}

template <typename T, bool OPT>
cudaError_t launch_general(const DiagArgs &a, int64_t B, cudaStream_t stream) {
    dim3 grid((unsigned)((a.Dm + 127) / 128), (unsigned)B);
    void (*kern)(DiagArgs) = a.N <= 16   ? diag_scan_kernel<T, 16, OPT>
                             : a.N <= 32 ? diag_scan_kernel<T, 32, OPT>
                                         : diag_scan_kernel<T, 64, OPT>;
    return launch_programmatic(kern, grid, dim3(128), 0, stream, a);
}

template <bool OPT, int MODE>
cudaError_t launch_bf16_vec(const DiagArgs &a, cudaStream_t stream) {
    const unsigned nz = MODE == kWhole ? 1u : (unsigned)a.nseg;
    const dim3 grid1((unsigned)((a.Dm + kCh1 - 1) / kCh1), (unsigned)a.B, nz);
    const dim3 grid2((unsigned)((a.Dm + kCh - 1) / kCh), (unsigned)a.B, nz);
    if (a.N <= 8)
        return launch_programmatic(diag_scan_bf16_kernel<8, 1, kCh1, kUnr1, OPT, MODE>, grid1, dim3(kCh1), 0,
                                   stream, a);
    if (a.N <= 16)
        return launch_programmatic(diag_scan_bf16_kernel<8, 2, kCh, kUnr2, OPT, MODE>, grid2, dim3(2 * kCh), 0,
                                   stream, a);
    return launch_programmatic(diag_scan_bf16_kernel<16, 2, kCh, kUnr2, OPT, MODE>, grid2, dim3(2 * kCh), 0,
                               stream, a);
}

template <bool OPT>
cudaError_t launch_bf16(const DiagArgs &a, cudaStream_t stream) {
    if (a.nseg <= 1) return launch_bf16_vec<OPT, kWhole>(a, stream);
    cudaError_t e = launch_bf16_vec<OPT, kLocal>(a, stream);
    if (e != cudaSuccess) return e;
    const int64_t n = a.B * a.Dm * a.N;
    e = launch_programmatic(diag_segment_pass_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream, a);
    if (e != cudaSuccess) return e;
    return launch_bf16_vec<OPT, kOutput>(a, stream);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

SSD_BOUNDS_HOST_READER(bounds_word_diag)

// Time segments: one pass per sequence keeps ~B * dim / 32 CTAs busy; when
// that leaves the GPU mostly idle (fewer than kSegEnablePerSM threads per SM)
// the sequence is cut into segments of at least 64 tokens (a multiple of 32),
// as many as bring the threads of all segments to about kSegTargetPerSM per
// SM: measured on GB300, more and shorter segments kept paying down to 64
// tokens (B1 L4096 D1024: 81 -> 75 us from 32 to 64 segments; B2 L8192
// D1536: 406 -> 312 us) even though every segment's first tile load is
// exposed. The split depends on the shape and the device's SM count (152 on
// GB300, also assumed where no device can be queried), never on chunk_size.
constexpr int64_t kSegEnablePerSM = 256;
constexpr int64_t kSegTargetPerSM = 4096;

int diag_segments(int64_t B, int64_t L, int64_t Dm, int64_t N, int io) {
    if (io != IO_BF16 || Dm % 8 != 0 || N % 8 != 0 || N > 32 || B < 1 || L < 128) return 1;
    const int64_t sms = sm_count(152);
    const int64_t thr = B * ((Dm + kCh - 1) / kCh) * (N <= 8 ? kCh1 : 2 * kCh);
    if (thr >= kSegEnablePerSM * sms) return 1;
    int64_t want = (kSegTargetPerSM * sms + thr - 1) / thr;
    want = imin<int64_t>(want, L / 64);
    if (want <= 1) return 1;
    const int64_t seg_len = ((L + want - 1) / want + 31) / 32 * 32;
    return (int)((L + seg_len - 1) / seg_len);
}

static int64_t diag_seg_len(int64_t L, int nseg) { return ((L + nseg - 1) / nseg + 31) / 32 * 32; }

size_t diag_workspace_bytes(int64_t B, int64_t L, int64_t Dm, int64_t N, int io) {
    const int nseg = diag_segments(B, L, Dm, N, io);
    if (nseg <= 1) return 0;
    const size_t h = (size_t)nseg * B * Dm * N * sizeof(float);
    return (h + 255) / 256 * 256 + (size_t)nseg * B * Dm * sizeof(float);
}

cudaError_t launch_diag(int io, const DiagArgs &a0, cudaStream_t stream) {
    if (a0.B == 0) return cudaSuccess;
    const bool opt = a0.z || a0.delta_bias || a0.softplus;
    DiagArgs a = a0;
    if (a.nseg > 1) a.seg_len = diag_seg_len(a.L, a.nseg);
    else {
        a.nseg = 1;
        a.seg_len = a.L;
    }
    if (io == IO_BF16) {
        const bool vec = a.Dm % 8 == 0 && a.N % 8 == 0 && a.N <= 32 && aligned16(a.x) && aligned16(a.dt) &&
                         aligned16(a.Bm) && aligned16(a.Cm) && aligned16(a.y) && (!a.z || aligned16(a.z));
        if (vec) return opt ? launch_bf16<true>(a, stream) : launch_bf16<false>(a, stream);
        return opt ? launch_general<__nv_bfloat16, true>(a, a.B, stream)
                   : launch_general<__nv_bfloat16, false>(a, a.B, stream);
    }
    return opt ? launch_general<float, true>(a, a.B, stream) : launch_general<float, false>(a, a.B, stream);
}

}  // namespace ssd
