// Chunked SSD prefill on the CUDA cores, float32 arithmetic.
//
// The sequence is cut into chunks of Q tokens, each chunk continuing from the
// previous chunk's state ("Recurrence Scan", first section). With
// a_t = dt_t * A_h and cs the inclusive cumulative sum of a inside a chunk,
// the recurrence re-associates exactly into three steps:
//
//   chunk state  S_c[p,n]   = sum_j exp(cs_end - cs_j) dt_j x_j[p] B_j[n]
//   state pass   h_in(c+1)  = exp(cs_end(c)) h_in(c) + S_c,  h_in(0) = h0
//   chunk scan   y_i[p]     = sum_{j<=i} (C_i . B_j) exp(cs_i - cs_j) dt_j x_j[p]
//                           + exp(cs_i) sum_n C_i[n] h_in(c)[p,n] + D x_i[p]
//
// (j, i run over the tokens of one chunk). The causal mask is a static
// predicate on (i, j) ("Compiler-First State Space Duality ...", Table 7:
// static mask). This path serves float32 inputs and every shape the
// tensor-core path does not take; its register tiles are 4x4 per thread over
// 64x64 output tiles.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "debug_bounds.cuh"
#include "launch.h"
#include "ssd_scan.h"

namespace ssd {
namespace {

constexpr int kT = 256;
constexpr int kTile = 64;

// Loads dt of one chunk (zero past the end of the sequence) into s_dt and the
// inclusive cumulative sum of dt*A into s_cs.
template <typename T>
__device__ __forceinline__ void chunk_cumsum(const T *__restrict__ dt, int64_t b, int64_t L, int64_t H, int h,
                                             int64_t t0, int Q, float Ah, float *s_dt, float *s_cs,
                                             float *scratch) {
    const int tid = threadIdx.x;
    float d = 0.f;
    if (tid < Q && t0 + tid < L) d = to_f32(dt[(b * L + t0 + tid) * H + h]);
    if (tid < Q) s_dt[tid] = d;
    block_inclusive_scan_256(d * Ah, Q, s_cs, scratch);
}

// S_c for one (b, c, h) and one 64x64 tile of (p, n).
template <typename T>
__global__ void __launch_bounds__(kT) chunk_state_simt(ChunkedArgs a, int tilesP, int tilesN) {
    // this call's status word starts clear (the first kernel of the call)
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) *a.status = SSD_OK;
    const int c = blockIdx.x;
    const int tiles = tilesP * tilesN;
    const int h = blockIdx.y / tiles, pt = (blockIdx.y % tiles) / tilesN, nt = blockIdx.y % tilesN;
    const int64_t b = blockIdx.z;
    const int64_t L = a.L, H = a.H, P = a.P, N = a.N, G = a.G;
    const int Q = a.Q;
    const int g = (int)(h / (H / G));
    const int64_t t0 = (int64_t)c * Q;
    const int Qv = (int)imin<int64_t>(Q, L - t0);
    const T *x = (const T *)a.x, *Bm = (const T *)a.Bm;

    __shared__ float s_dt[256], s_cs[256], s_w[256], scratch[8];
    __shared__ __align__(16) float Xs[32][kTile + 4], Bs[32][kTile + 4];  // 16-byte aligned rows

    chunk_cumsum<T>((const T *)a.dt, b, L, H, h, t0, Q, a.A[h], s_dt, s_cs, scratch);
    const float cs_end = s_cs[Q - 1];  // padded tokens carry a = 0
    const int tid = threadIdx.x;
    if (tid < Q) s_w[tid] = expf(cs_end - s_cs[tid]) * s_dt[tid];
    if (pt == 0 && nt == 0 && tid == 0) a.chunk_sum[(b * H + h) * a.nc + c] = expf(cs_end);  // decay over the chunk
    __syncthreads();

    const int ty = tid / 16, tx = tid % 16;
    float acc[4][4] = {};
    // with P and N multiples of 4 (16-byte aligned rows) each thread loads its
    // 16-byte vectors of a 32-token block together, then stores them
    const bool vec = P % 4 == 0 && N % 4 == 0;
    constexpr int kU = 32 * kTile / 4 / kT;
    for (int j0 = 0; j0 < Qv; j0 += 32) {
        if (vec) {
            const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            float4 xv[kU], bv[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = tid + u * kT, jj = e / (kTile / 4), q = (e % (kTile / 4)) * 4, j = j0 + jj;
                const int64_t p = (int64_t)pt * kTile + q, n = (int64_t)nt * kTile + q;
                const int64_t tok = b * L + t0 + j;
                xv[u] = (j < Qv && p < P) ? ld4(x + (tok * H + h) * P + p) : z4;
                bv[u] = (j < Qv && n < N) ? ld4(Bm + (tok * G + g) * N + n) : z4;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = tid + u * kT, jj = e / (kTile / 4), q = (e % (kTile / 4)) * 4;
                const float w = j0 + jj < Qv ? s_w[j0 + jj] : 0.f;
                *reinterpret_cast<float4 *>(&Xs[jj][q]) = make_float4(w * xv[u].x, w * xv[u].y, w * xv[u].z, w * xv[u].w);
                *reinterpret_cast<float4 *>(&Bs[jj][q]) = bv[u];
            }
        } else {
            for (int e = tid; e < 32 * kTile; e += kT) {
                const int jj = e / kTile, q = e % kTile, j = j0 + jj;
                const int64_t p = (int64_t)pt * kTile + q, n = (int64_t)nt * kTile + q;
                const int64_t tok = b * L + t0 + j;
                Xs[jj][q] = (j < Qv && p < P) ? s_w[j] * to_f32(x[(tok * H + h) * P + p]) : 0.f;
                Bs[jj][q] = (j < Qv && n < N) ? to_f32(Bm[(tok * G + g) * N + n]) : 0.f;
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int jj = 0; jj < 32; ++jj) {
            const float4 x4 = *reinterpret_cast<const float4 *>(&Xs[jj][ty * 4]);
            const float4 b4 = *reinterpret_cast<const float4 *>(&Bs[jj][tx * 4]);
            const float xa[4] = {x4.x, x4.y, x4.z, x4.w}, bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[i][k] = fmaf(xa[i], bb[k], acc[i][k]);
        }
        __syncthreads();
    }
    float *S = a.states + (((b * a.nc + c) * H + h) * P) * N;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t p = (int64_t)pt * kTile + ty * 4 + i, n = (int64_t)nt * kTile + tx * 4;
        if (p >= P) continue;
        if (vec) {
            if (n < N) *reinterpret_cast<float4 *>(S + p * N + n) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (n + k < N) S[p * N + n + k] = acc[i][k];
        }
    }
}

// Serial pass over the chunks of one (b, h): replaces S_c with the entering
// state h_in(c) (float32 in place and/or a bfloat16 copy) and writes the
// final state. The chunk states are float32 (CUDA-core path) or bfloat16
// (tensor-core path, read from and replaced in states_bf16). VW consecutive
// state elements per thread; the chunk states of kPF chunks are loaded
// before the serial update consumes them, so each thread keeps kPF
// independent loads in flight: 16 on the float32 in-place path (the CUDA-core
// prefill and the backward's recompute), 8 where more registers are live.

template <typename TIn, bool F32_INPLACE, bool BF16, int VW>
__global__ void __launch_bounds__(kT, 2) state_pass_kernel(ChunkedArgs a) {
    // with no tokens this is the call's first kernel: clear its status word
    if (a.nc == 0 && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) *a.status = SSD_OK;
    // Wait for the producer of the chunk states when launched as a programmatic
    // dependent of it; a no-op for an ordinary launch.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the chunk scan may start its independent prologue now; it waits for
    // this grid's completion before it reads the entering states
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t PN = a.P * a.N;
    const int64_t e = ((int64_t)blockIdx.x * kT + threadIdx.x) * VW;
    const int h = blockIdx.y;
    const int64_t b = blockIdx.z;
    if (e >= PN) return;
    const int64_t H = a.H, nc = a.nc;
    const TIn *src = std::is_same<TIn, float>::value ? reinterpret_cast<const TIn *>(a.states)
                                                      : reinterpret_cast<const TIn *>(a.states_bf16);
    float hv[VW];
#pragma unroll
    for (int k = 0; k < VW; ++k) hv[k] = a.init_state ? a.init_state[(b * H + h) * PN + e + k] : 0.f;
    const float *cs = a.chunk_sum + (b * H + h) * nc;
    const int64_t stride = H * PN;  // next chunk, same (b, h, element)
    const int64_t base = ((b * nc) * H + h) * PN + e;
    constexpr int kPF = std::is_same<TIn, float>::value && F32_INPLACE && !BF16 ? 16 : 8;
    for (int64_t c0 = 0; c0 < nc; c0 += kPF) {
        float s[kPF][VW], dA[kPF];
#pragma unroll
        for (int u = 0; u < kPF; ++u) {
            if (c0 + u < nc) {
                const TIn *p = src + base + (c0 + u) * stride;
                if constexpr (VW == 4 && std::is_same<TIn, float>::value) {
                    const float4 v = *reinterpret_cast<const float4 *>(p);
                    s[u][0] = v.x; s[u][1] = v.y; s[u][2] = v.z; s[u][3] = v.w;
                } else if constexpr (VW == 4) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(p);
                    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
                    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
                    s[u][0] = lo.x; s[u][1] = lo.y; s[u][2] = hi.x; s[u][3] = hi.y;
                } else {
                    s[u][0] = to_f32(*p);
                }
                dA[u] = cs[c0 + u];
            }
        }
#pragma unroll
        for (int u = 0; u < kPF; ++u) {
            if (c0 + u < nc) {
                const int64_t idx = base + (c0 + u) * stride;
                if (F32_INPLACE) {
                    if constexpr (VW == 4)
                        *reinterpret_cast<float4 *>(a.states + idx) = make_float4(hv[0], hv[1], hv[2], hv[3]);
                    else
                        a.states[idx] = hv[0];
                }
                if (BF16) {
                    if constexpr (VW == 4) {
                        __nv_bfloat162 lo = __floats2bfloat162_rn(hv[0], hv[1]);
                        __nv_bfloat162 hi = __floats2bfloat162_rn(hv[2], hv[3]);
                        uint2 pk = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
                        *reinterpret_cast<uint2 *>(a.states_bf16 + idx) = pk;
                    } else {
                        __nv_bfloat16 v = __float2bfloat16_rn(hv[0]);
                        a.states_bf16[idx] = *reinterpret_cast<uint16_t *>(&v);
                    }
                }
#pragma unroll
                for (int k = 0; k < VW; ++k) hv[k] = fmaf(dA[u], hv[k], s[u][k]);
            }
        }
    }
    if (a.final_state) {
#pragma unroll
        for (int k = 0; k < VW; ++k) a.final_state[(b * H + h) * PN + e + k] = hv[k];
    }
}

// y for 64 rows of one chunk and one 64-wide tile of p, for one (b, h).
template <typename T>
__global__ void __launch_bounds__(kT) chunk_scan_simt(ChunkedArgs a, int tilesP) {
    const int RBs = a.Q / kTile;
    const int c = blockIdx.x / RBs, rb = blockIdx.x % RBs;
    const int h = blockIdx.y / tilesP, pt = blockIdx.y % tilesP;
    const int64_t b = blockIdx.z;
    const int64_t L = a.L, H = a.H, P = a.P, N = a.N, G = a.G;
    const int Q = a.Q;
    const int g = (int)(h / (H / G));
    const int64_t t0 = (int64_t)c * Q;
    const int Qv = (int)imin<int64_t>(Q, L - t0);
    if (rb * kTile >= Qv) return;
    const T *x = (const T *)a.x, *Bm = (const T *)a.Bm, *Cm = (const T *)a.Cm;
    T *y = (T *)a.y;
    const int K = (rb + 1) * kTile;  // columns j of this row block: 0 .. K-1
    const int GS = K + 1;            // padded row stride of G_s

    extern __shared__ float smem[];
    float *s_dt = smem, *s_cs = smem + 256, *scratch = smem + 512;
    float *G_s = smem + 520;                 // [64][GS]
    float *Cs = G_s + kTile * GS;            // [64][33]
    float *Ws = Cs + kTile * 33;             // [64][33] or [32][65]

    chunk_cumsum<T>((const T *)a.dt, b, L, H, h, t0, Q, a.A[h], s_dt, s_cs, scratch);
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int i_base = rb * kTile;  // chunk-local first row

    // Phase 1: G[i, j] = (C_i . B_j) exp(cs_i - cs_j) dt_j for j <= i, else 0.
    for (int jb = 0; jb <= rb; ++jb) {
        float acc[4][4] = {};
        for (int n0 = 0; n0 < N; n0 += 32) {
            for (int e = tid; e < kTile * 32; e += kT) {
                const int r = e / 32, nn = e % 32;
                const int64_t n = n0 + nn;
                const int ic = i_base + r, jc = jb * kTile + r;
                Cs[r * 33 + nn] = (ic < Qv && n < N) ? to_f32(Cm[((b * L + t0 + ic) * G + g) * N + n]) : 0.f;
                Ws[r * 33 + nn] = (jc < Qv && n < N) ? to_f32(Bm[((b * L + t0 + jc) * G + g) * N + n]) : 0.f;
            }
            __syncthreads();
#pragma unroll 8
            for (int nn = 0; nn < 32; ++nn) {
                float ca[4], bb[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) ca[i] = Cs[(ty * 4 + i) * 33 + nn];
#pragma unroll
                for (int k = 0; k < 4; ++k) bb[k] = Ws[(tx * 4 + k) * 33 + nn];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[i][k] = fmaf(ca[i], bb[k], acc[i][k]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int il = i_base + ty * 4 + i;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int jl = jb * kTile + tx * 4 + k;
                float v = 0.f;
                if (jl <= il && jl < Qv) v = acc[i][k] * expf(s_cs[il] - s_cs[jl]) * s_dt[jl];
                G_s[(ty * 4 + i) * GS + jb * kTile + tx * 4 + k] = v;
            }
        }
    }
    __syncthreads();

    // Phase 2: intra-chunk part G . X plus the entering-state part.
    const int64_t p_base = (int64_t)pt * kTile;
    float acc[4][4] = {};
    for (int j0 = 0; j0 < K; j0 += 32) {
        for (int e = tid; e < 32 * kTile; e += kT) {
            const int jj = e / kTile, q = e % kTile, j = j0 + jj;
            const int64_t p = p_base + q;
            Ws[jj * 65 + q] = (j < Qv && p < P) ? to_f32(x[((b * L + t0 + j) * H + h) * P + p]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int jj = 0; jj < 32; ++jj) {
            float ga[4], xb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) ga[i] = G_s[(ty * 4 + i) * GS + j0 + jj];
#pragma unroll
            for (int k = 0; k < 4; ++k) xb[k] = Ws[jj * 65 + tx * 4 + k];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[i][k] = fmaf(ga[i], xb[k], acc[i][k]);
        }
        __syncthreads();
    }
    float off[4][4] = {};
    const float *hin = a.states + (((b * a.nc + c) * H + h) * P) * N;
    for (int n0 = 0; n0 < N; n0 += 32) {
        for (int e = tid; e < kTile * 32; e += kT) {
            const int r = e / 32, nn = e % 32;
            const int64_t n = n0 + nn;
            const int ic = i_base + r;
            const int64_t p = p_base + r;
            Cs[r * 33 + nn] = (ic < Qv && n < N) ? to_f32(Cm[((b * L + t0 + ic) * G + g) * N + n]) : 0.f;
            Ws[r * 33 + nn] = (p < P && n < N) ? hin[p * N + n] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int nn = 0; nn < 32; ++nn) {
            float ca[4], hb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) ca[i] = Cs[(ty * 4 + i) * 33 + nn];
#pragma unroll
            for (int k = 0; k < 4; ++k) hb[k] = Ws[(tx * 4 + k) * 33 + nn];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int k = 0; k < 4; ++k) off[i][k] = fmaf(ca[i], hb[k], off[i][k]);
        }
        __syncthreads();
    }
    const float Dh = a.D ? a.D[h] : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int il = i_base + ty * 4 + i;
        if (il >= Qv) continue;
        const float decay_in = expf(s_cs[il]);
        const int64_t tok = b * L + t0 + il;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t p = p_base + tx * 4 + k;
            if (p >= P) continue;
            const int64_t o = (tok * H + h) * P + p;
            const float xv = to_f32(x[o]);
            y[o] = from_f32<T>(acc[i][k] + decay_in * off[i][k] + Dh * xv);
        }
    }
}

size_t scan_smem_bytes(int Q) {
    const int K = Q;  // largest row block
    return sizeof(float) * (520 + (size_t)kTile * (K + 1) + kTile * 33 + std::max(kTile * 33, 32 * 65));
}

template <typename T>
cudaError_t launch_simt_t(const ChunkedArgs &a, cudaStream_t stream) {
    const int tilesP = (int)((a.P + kTile - 1) / kTile), tilesN = (int)((a.N + kTile - 1) / kTile);
    cudaError_t e0 = mark_stage(a, 0, stream);
    if (e0 != cudaSuccess) return e0;
    if (a.nc > 0 && a.B > 0) {
        chunk_state_simt<T><<<dim3((unsigned)a.nc, (unsigned)(a.H * tilesP * tilesN), (unsigned)a.B), kT, 0,
                              stream>>>(a, tilesP, tilesN);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = mark_stage(a, 1, stream);
    if (e != cudaSuccess) return e;
    e = launch_state_pass(a, true, false, stream, false);
    if (e != cudaSuccess) return e;
    e = mark_stage(a, 2, stream);
    if (e != cudaSuccess) return e;
    if (a.nc > 0 && a.B > 0) {
        const size_t smem = scan_smem_bytes(a.Q);
        static DeviceOnce configured;  // the largest chunk's size, set once per device
        int dev = 0;
        if (configured.pending(&dev, &e)) {
            e = cudaFuncSetAttribute(chunk_scan_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)scan_smem_bytes(256));
            if (e != cudaSuccess) return e;
            configured.done(dev);
        } else if (e != cudaSuccess) {
            return e;
        }
        chunk_scan_simt<T><<<dim3((unsigned)(a.nc * (a.Q / kTile)), (unsigned)(a.H * tilesP), (unsigned)a.B), kT,
                             smem, stream>>>(a, tilesP);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return mark_stage(a, 3, stream);
}

}  // namespace

SSD_BOUNDS_HOST_READER(bounds_word_simt)

// Tensor-core path: bfloat16 chunk states in states_bf16, replaced in place by
// the bfloat16 entering states; 2 elements per thread. Up to PF chunks are
// loaded before the chain runs (one register per chunk), so that one round
// trip to L2 brings in the whole chain of sequences up to PF chunks long.
// Short chains (nc <= 16) take PF = 16 at six CTAs per SM, which keeps more
// loads in flight per SM than PF = 32 at three.
template <int PF, int MINB>
__global__ void __launch_bounds__(kT, MINB) state_pass_bf16_kernel(ChunkedArgs a) {
    __shared__ float s_dA[PF];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t PN = a.P * a.N;
    const int64_t e = ((int64_t)blockIdx.x * kT + threadIdx.x) * 2;
    const int h = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t H = a.H, nc = a.nc;
    float h0 = 0.f, h1 = 0.f;
    if (a.init_state && e < PN) {
        const float2 v = *reinterpret_cast<const float2 *>(a.init_state + (b * H + h) * PN + e);
        h0 = v.x;
        h1 = v.y;
    }
    const float *cs = a.chunk_sum + (b * H + h) * nc;
    const int64_t stride = H * PN;
    __nv_bfloat16 *base = reinterpret_cast<__nv_bfloat16 *>(a.states_bf16) + ((b * nc) * H + h) * PN + e;
    const bool act = e < PN;
    for (int64_t c0 = 0; c0 < nc; c0 += PF) {
        // the chunk decays of this (b, h), shared by the CTA
        __syncthreads();
        if (threadIdx.x < PF && c0 + threadIdx.x < nc) s_dA[threadIdx.x] = cs[c0 + threadIdx.x];
        __syncthreads();
        if (!act) continue;
        uint32_t raw[PF];
        const int64_t n_states = a.B * nc * H * PN, e0 = ((b * nc) * H + h) * PN + e;
        (void)n_states; (void)e0;
#pragma unroll
        for (int u = 0; u < PF; ++u)
            if (c0 + u < nc && SSD_IN_BOUNDS(e0 + (c0 + u) * stride, 2, n_states, kSiteStatePass))
                raw[u] = *reinterpret_cast<const uint32_t *>(base + (c0 + u) * stride);
#pragma unroll
        for (int u = 0; u < PF; ++u) {
            if (c0 + u < nc && SSD_IN_BOUNDS(e0 + (c0 + u) * stride, 2, n_states, kSiteStatePass)) {
                const __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
                *reinterpret_cast<__nv_bfloat162 *>(base + (c0 + u) * stride) = hv;
                const float2 sv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw[u]));
                const float dA = s_dA[u];
                h0 = fmaf(dA, h0, sv.x);
                h1 = fmaf(dA, h1, sv.y);
            }
        }
    }
    if (!act) return;
    if (a.final_state)
        *reinterpret_cast<float2 *>(a.final_state + (b * H + h) * PN + e) = make_float2(h0, h1);
}

template <typename TIn, int VW>
void (*pick_state_pass(bool f32, bool bf16))(ChunkedArgs) {
    if (f32 && bf16) return state_pass_kernel<TIn, true, true, VW>;
    if (f32) return state_pass_kernel<TIn, true, false, VW>;
    if (bf16) return state_pass_kernel<TIn, false, true, VW>;
    return state_pass_kernel<TIn, false, false, VW>;
}

cudaError_t launch_state_pass(const ChunkedArgs &a, bool write_f32_inplace, bool write_bf16, cudaStream_t stream,
                              bool programmatic, bool bf16_in) {
    if (a.B == 0) return cudaSuccess;
    const int64_t PN = a.P * a.N;
    // 4-wide path: every (b, c, h) block of PN states starts aligned
    const bool vec = (PN % 4 == 0) && (reinterpret_cast<uintptr_t>(a.init_state) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.final_state) % 16 == 0);
    const int VW = vec ? 4 : 1;
    dim3 grid((unsigned)((PN / VW + kT - 1) / kT), (unsigned)a.H, (unsigned)a.B);
    void (*kern)(ChunkedArgs);
    if (bf16_in && vec && write_bf16 && !write_f32_inplace) {
        kern = a.nc <= 16 ? state_pass_bf16_kernel<16, 6> : state_pass_bf16_kernel<32, 3>;
        grid.x = (unsigned)((PN / 2 + kT - 1) / kT);
    }
    else if (bf16_in)
        kern = vec ? pick_state_pass<__nv_bfloat16, 4>(write_f32_inplace, write_bf16)
                   : pick_state_pass<__nv_bfloat16, 1>(write_f32_inplace, write_bf16);
    else
        kern = vec ? pick_state_pass<float, 4>(write_f32_inplace, write_bf16)
                   : pick_state_pass<float, 1>(write_f32_inplace, write_bf16);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kT);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (programmatic) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_forward_states(const ChunkedArgs &a, cudaStream_t stream) {
    if (a.nc > 0 && a.B > 0) {
        const int tilesP = (int)((a.P + kTile - 1) / kTile), tilesN = (int)((a.N + kTile - 1) / kTile);
        const dim3 grid((unsigned)a.nc, (unsigned)(a.H * tilesP * tilesN), (unsigned)a.B);
        if (a.io == IO_BF16)
            chunk_state_simt<__nv_bfloat16><<<grid, kT, 0, stream>>>(a, tilesP, tilesN);
        else
            chunk_state_simt<float><<<grid, kT, 0, stream>>>(a, tilesP, tilesN);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_state_pass(a, true, false, stream, false);
}

cudaError_t launch_chunked_simt(const ChunkedArgs &a, cudaStream_t stream) {
    if (a.io == IO_BF16) return launch_simt_t<__nv_bfloat16>(a, stream);
    return launch_simt_t<float>(a, stream);
}

}  // namespace ssd
