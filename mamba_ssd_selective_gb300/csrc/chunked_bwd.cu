// Backward of the chunked SSD scan on the CUDA cores, float32 arithmetic.
//
// The forward states are recomputed in chunks of 64 tokens (chunk state and
// state pass of the forward), then, with a_t = dt_t A, cs the inclusive
// cumulative sum of a inside a chunk, e_t = exp(cs_t), and for one (b, h):
//
//   adjoint chunk state   Sbar_c       = sum_t e_t dy_t C_t^T              (P x N)
//   reverse state pass    G_c          = Sbar_c + exp(cs_end(c)) G_{c+1},   G_nc = dfinal
//                         (G_c: cotangent of the state entering chunk c; dinit = G_0)
//
// and per chunk, with Gn = G_{c+1} the cotangent of the state leaving it,
// hin the state entering it, Ld[t,s] = exp(cs_t - cs_s) for s <= t (else 0),
// u_s = dt_s x_s and eend_s = exp(cs_end - cs_s):
//
//   M1 = Ld o (C B^T),  M2 = Ld o (dY X^T) o dt_s
//   du  = M1^T dY + eend o (B Gn^T)         dx = dt o du + D dY
//   dB  = M2^T C  + (dt eend) o (X Gn)      dC = M2 B + e o (dY hin)
//   d cs_t (from the decays): sum_{s<t} W[t,s] - sum_{t'>t} W[t',t]
//          + e_t dY_t . (hin C_t) - r_t,    W = M1 o (dY X^T) o dt_s,
//          r_s = eend_s dt_s x_s . (Gn B_s); the chunk's last token also takes
//          sum_s r_s + exp(cs_end) <Gn, hin>
//   da_k = sum_{t >= k} d cs_t,  ddt = da A + x . du,  dA = sum da dt,  dD = sum dY . x
//
// These are the reverse-mode derivatives of the token recurrence
// h_t = exp(dt_t A) h_{t-1} + dt_t x_t B_t^T, y_t = C_t h_t + D x_t, grouped
// by chunk the way the forward re-associates it ("Recurrence Scan", first
// section; the training step of "Compiler-First State Space Duality ...",
// Table 13). Every sum runs in a fixed order: no atomics, run-to-run
// bit-identical. dB and dC of a B/C group sum the heads' parts in head order.
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "ssd_scan.h"

namespace ssd {
namespace {

constexpr int kT = 256;
constexpr int kQ = BwdArgs::kChunk;  // 64 tokens per backward chunk


// Adjoint chunk state of one (b, c, h) and one 64x64 tile of (p, n), for
// chunks of Q tokens (the dt scan covers the chunk, the sum runs over
// sub-tiles of 64 tokens staged in shared memory in turn).
template <typename T, int Q>
__global__ void __launch_bounds__(kT) adj_chunk_state_kernel(const __grid_constant__ BwdArgs a, int tilesP,
                                                             int tilesN) {
    static_assert(Q % 64 == 0 && Q <= 256, "chunks of 64-token sub-tiles");
    const int c = blockIdx.x;
    const int tiles = tilesP * tilesN;
    const int h = blockIdx.y / tiles, pt = (blockIdx.y % tiles) / tilesN, nt = blockIdx.y % tilesN;
    const int64_t b = blockIdx.z;
    const int64_t L = a.L, H = a.H, P = a.P, N = a.N, G = a.G;
    const int g = (int)(h / (H / G));
    const int64_t t0 = (int64_t)c * Q;
    const int Qv = (int)imin<int64_t>(Q, L - t0);
    const T *dy = static_cast<const T *>(a.dy), *Cm = static_cast<const T *>(a.Cm);
    const T *dt = static_cast<const T *>(a.dt);
    __shared__ float s_cs[256], s_e[Q], scratch[8];
    __shared__ __align__(16) float Ys[64][68], Cs[64][68];  // 16-byte aligned rows
    const int tid = threadIdx.x;
    const bool vec = P % 4 == 0 && N % 4 == 0;
    const float d = (tid < Qv) ? to_f32(dt[(b * L + t0 + tid) * H + h]) : 0.f;
    block_inclusive_scan_256(d * a.A[h], Q, s_cs, scratch);
    if (tid < Q) s_e[tid] = expf(s_cs[tid]);
    const int ty = tid / 16, tx = tid % 16;
    float acc[4][4] = {};
    for (int j0 = 0; j0 < Qv; j0 += 64) {
        // the dy and C rows of this sub-tile: with P and N multiples of 4, four
        // 16-byte vectors of each per thread; else element by element
        if (vec) {
            constexpr int kU = 64 * 16 / kT;
            const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            float4 yv[kU], cv[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = tid + u * kT, j = e / 16, q = (e % 16) * 4;
                const int64_t p = (int64_t)pt * 64 + q, n = (int64_t)nt * 64 + q, tok = b * L + t0 + j0 + j;
                yv[u] = (j0 + j < Qv && p < P) ? ld4(dy + (tok * H + h) * P + p) : z4;
                cv[u] = (j0 + j < Qv && n < N) ? ld4(Cm + (tok * G + g) * N + n) : z4;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = tid + u * kT, j = e / 16, q = (e % 16) * 4;
                *reinterpret_cast<float4 *>(&Ys[j][q]) = yv[u];
                *reinterpret_cast<float4 *>(&Cs[j][q]) = cv[u];
            }
        } else {
            for (int e = tid; e < 64 * 64; e += kT) {
                const int j = e / 64, q = e % 64;
                const int64_t p = (int64_t)pt * 64 + q, n = (int64_t)nt * 64 + q, tok = b * L + t0 + j0 + j;
                Ys[j][q] = (j0 + j < Qv && p < P) ? to_f32(dy[(tok * H + h) * P + p]) : 0.f;
                Cs[j][q] = (j0 + j < Qv && n < N) ? to_f32(Cm[(tok * G + g) * N + n]) : 0.f;
            }
        }
        __syncthreads();
        const int jn = imin(64, Qv - j0);
        for (int j = 0; j < jn; ++j) {
            const float w = s_e[j0 + j];
            const float4 y4 = *reinterpret_cast<const float4 *>(&Ys[j][ty * 4]);
            const float4 c4 = *reinterpret_cast<const float4 *>(&Cs[j][tx * 4]);
            const float ya[4] = {w * y4.x, w * y4.y, w * y4.z, w * y4.w}, cb[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[i][k] = fmaf(ya[i], cb[k], acc[i][k]);
        }
        __syncthreads();  // the sub-tile is read before the next one replaces it
    }
    float *S = a.adj + (((b * a.nc + c) * H + h) * P) * N;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t p = (int64_t)pt * 64 + ty * 4 + i, n = (int64_t)nt * 64 + tx * 4;
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

// Reverse pass over the chunks of one (b, h), VW state elements per thread:
// replaces Sbar_c by the cotangent of the state leaving chunk c and writes
// dinit. Decays exp(cs_end(c)) come from the forward recompute. The values of
// kPFA chunks are loaded before the chain consumes them, so that each thread
// keeps kPFA independent loads in flight.
constexpr int kPFA = 16;

template <int VW>
__global__ void __launch_bounds__(kT) adj_state_pass_kernel(const __grid_constant__ BwdArgs a) {
    const int64_t PN = a.P * a.N;
    const int64_t e = ((int64_t)blockIdx.x * kT + threadIdx.x) * VW;
    const int h = blockIdx.y;
    const int64_t b = blockIdx.z;
    if (e >= PN) return;
    const int64_t H = a.H, nc = a.nc;
    float carry[VW];
#pragma unroll
    for (int k = 0; k < VW; ++k) carry[k] = a.dfinal ? a.dfinal[(b * H + h) * PN + e + k] : 0.f;
    const float *dec = a.chunk_sum + (b * H + h) * nc;
    for (int64_t c1 = nc; c1 > 0; c1 -= kPFA) {
        float v[kPFA][VW], dc[kPFA];
#pragma unroll
        for (int u = 0; u < kPFA; ++u) {
            const int64_t c = c1 - 1 - u;
            if (c >= 0) {
                const float *p = a.adj + ((b * nc + c) * H + h) * PN + e;
                if constexpr (VW == 4) {
                    const float4 q = *reinterpret_cast<const float4 *>(p);
                    v[u][0] = q.x; v[u][1] = q.y; v[u][2] = q.z; v[u][3] = q.w;
                } else {
                    v[u][0] = *p;
                }
                dc[u] = dec[c];
            }
        }
#pragma unroll
        for (int u = 0; u < kPFA; ++u) {
            const int64_t c = c1 - 1 - u;
            if (c >= 0) {
                float *p = a.adj + ((b * nc + c) * H + h) * PN + e;
                if constexpr (VW == 4)
                    *reinterpret_cast<float4 *>(p) = make_float4(carry[0], carry[1], carry[2], carry[3]);
                else
                    *p = carry[0];
#pragma unroll
                for (int k = 0; k < VW; ++k) carry[k] = fmaf(dc[u], carry[k], v[u][k]);
            }
        }
    }
    if (a.dinit) {
#pragma unroll
        for (int k = 0; k < VW; ++k) a.dinit[(b * H + h) * PN + e + k] = carry[k];
    }
}

// 64 x 64 output blocks, 4 x 4 per thread (ty = tid / 16 picks rows ty*4 + i):
//   mm_nt  acc[i][j] += sum_k A[row][k] * Bt[col][k],  col = c0 + tx + 16 j
//   mm_nn  acc[i][j] += sum_k A[row][k] * B[k][col],    col = c0 + tx*4 + j
//   mm_tn  acc[i][j] += sum_k At[k][row] * B[k][col],   col = c0 + tx*4 + j
// Every operand is read as 16-byte vectors (mm_nt and mm_nn fetch four k at a
// time along rows, then add them one k after another: the same sums in the
// same order as one k per step). K is rounded up to a multiple of 4: rows hold
// zeros past the call's sizes. Row strides of 68 and 132 floats (4 mod 32)
// keep the row reads of a warp (two rows of A, sixteen of Bt) two 128-byte
// wavefronts at most.
__device__ __forceinline__ float f4at(const float4 &v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

__device__ __forceinline__ void mm_nt(float (&acc)[4][4], int K, int c0, const float *A, int sa, const float *Bt,
                                      int sb) {
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const float *ar = A + ty * 4 * sa, *br = Bt + (c0 + tx) * sb;
    const int K4 = (K + 3) & ~3;
    // operands of the next four k are loaded while the current four are used
    float4 av[4], bv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) av[i] = *reinterpret_cast<const float4 *>(ar + i * sa);
#pragma unroll
    for (int j = 0; j < 4; ++j) bv[j] = *reinterpret_cast<const float4 *>(br + j * 16 * sb);
#pragma unroll 2
    for (int k = 0; k < K4; k += 4) {
        const int kn = k + 4 < K4 ? k + 4 : k;
        float4 an[4], bn[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) an[i] = *reinterpret_cast<const float4 *>(ar + i * sa + kn);
#pragma unroll
        for (int j = 0; j < 4; ++j) bn[j] = *reinterpret_cast<const float4 *>(br + j * 16 * sb + kn);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(f4at(av[i], kk), f4at(bv[j], kk), acc[i][j]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            av[i] = an[i];
            bv[i] = bn[i];
        }
    }
}

__device__ __forceinline__ void mm_nn(float (&acc)[4][4], int K, int c0, const float *A, int sa, const float *B,
                                      int sb) {
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const float *ar = A + ty * 4 * sa, *bc = B + c0 + tx * 4;
    const int K4 = (K + 3) & ~3;
    float4 av[4], bv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) av[i] = *reinterpret_cast<const float4 *>(ar + i * sa);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) bv[kk] = *reinterpret_cast<const float4 *>(bc + kk * sb);
#pragma unroll 2
    for (int k = 0; k < K4; k += 4) {
        const int kn = k + 4 < K4 ? k + 4 : k;
        float4 an[4], bn[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) an[i] = *reinterpret_cast<const float4 *>(ar + i * sa + kn);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) bn[kk] = *reinterpret_cast<const float4 *>(bc + (kn + kk) * sb);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(f4at(av[i], kk), f4at(bv[kk], j), acc[i][j]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            av[i] = an[i];
            bv[i] = bn[i];
        }
    }
}

// Two products in one k loop, for twice the independent FMA chains per warp
// (eight warps per SM leave little else to hide shared-memory latency):
//   mm_nt_2  acc1 += A Bt1^T, acc2 += A Bt2^T   (shared A)
//   mm_nn_2  acc1 += A1 B1,   acc2 += A2 B2     (same strides and K)
// Each sum keeps the one-k-after-another order of mm_nt / mm_nn.
__device__ __forceinline__ void mm_nt_2(float (&acc1)[4][4], float (&acc2)[4][4], int K, const float *A, int sa,
                                        const float *Bt1, const float *Bt2, int sb) {
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const float *ar = A + ty * 4 * sa, *b1 = Bt1 + tx * sb, *b2 = Bt2 + tx * sb;
    const int K4 = (K + 3) & ~3;
#pragma unroll 1
    for (int k = 0; k < K4; k += 4) {
        float4 av[4], bv1[4], bv2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = *reinterpret_cast<const float4 *>(ar + i * sa + k);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            bv1[j] = *reinterpret_cast<const float4 *>(b1 + j * 16 * sb + k);
            bv2[j] = *reinterpret_cast<const float4 *>(b2 + j * 16 * sb + k);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc1[i][j] = fmaf(f4at(av[i], kk), f4at(bv1[j], kk), acc1[i][j]);
                    acc2[i][j] = fmaf(f4at(av[i], kk), f4at(bv2[j], kk), acc2[i][j]);
                }
    }
}

__device__ __forceinline__ void mm_nn_2(float (&acc1)[4][4], float (&acc2)[4][4], int K, int c0, const float *A1,
                                        const float *A2, int sa, const float *B1, const float *B2, int sb) {
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const float *a1 = A1 + ty * 4 * sa, *a2 = A2 + ty * 4 * sa, *c1 = B1 + c0 + tx * 4, *c2 = B2 + c0 + tx * 4;
    const int K4 = (K + 3) & ~3;
#pragma unroll 1
    for (int k = 0; k < K4; k += 4) {
        float4 av1[4], av2[4], bv1[4], bv2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            av1[i] = *reinterpret_cast<const float4 *>(a1 + i * sa + k);
            av2[i] = *reinterpret_cast<const float4 *>(a2 + i * sa + k);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            bv1[kk] = *reinterpret_cast<const float4 *>(c1 + (k + kk) * sb);
            bv2[kk] = *reinterpret_cast<const float4 *>(c2 + (k + kk) * sb);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc1[i][j] = fmaf(f4at(av1[i], kk), f4at(bv1[kk], j), acc1[i][j]);
                    acc2[i][j] = fmaf(f4at(av2[i], kk), f4at(bv2[kk], j), acc2[i][j]);
                }
    }
}

__device__ __forceinline__ void mm_tn(float (&acc)[4][4], int K, int c0, const float *At, int sa, const float *B,
                                      int sb) {
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const float *ac = At + ty * 4, *bc = B + c0 + tx * 4;
    float4 a4 = *reinterpret_cast<const float4 *>(ac), b4 = *reinterpret_cast<const float4 *>(bc);
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        const int kn = k + 1 < K ? k + 1 : k;
        const float4 an = *reinterpret_cast<const float4 *>(ac + kn * sa);
        const float4 bn = *reinterpret_cast<const float4 *>(bc + kn * sb);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        a4 = an;
        b4 = bn;
    }
}

// Per-token dot products over p (or s) by four threads per token: token
// t = tid / 4, thread q = tid % 4 takes p = q, q + 4, ...; the four partial
// sums meet in a fixed-order butterfly, identical in all four threads. With row
// strides of 4 mod 32 the reads of a warp (eight tokens x four q) hit 32
// distinct banks.
__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

// Shared memory of the per-chunk gradient kernel (floats), laid out for the
// largest supported head (P 64, N 128) whatever the call's sizes: rows and
// columns past P, N and the chunk's tokens hold zeros, so every 16-byte
// vector read stays inside its array and contributes nothing.
constexpr int kSX = 68;   // row stride of X, dY  [64 tokens][64 p]
constexpr int kSN = 132;  // row stride of B, C [64 tokens][128 n] and hin, Gn [64 p][128 n]
constexpr int kSM = 68;   // row stride of M1, M2, W [64 tokens][64]
struct ChunkSmem {
    static constexpr int x = 0, y = x + kQ * kSX, bm = y + kQ * kSX, cm = bm + kQ * kSN, hin = cm + kQ * kSN,
                         gn = hin + 64 * kSN, m1 = gn + 64 * kSN, m2 = m1 + kQ * kSM, w = m2 + kQ * kSM,
                         vec = w + kQ * kSM, total = vec + 10 * kQ + kT + 8;
};

template <typename T>
__global__ void __launch_bounds__(kT) chunk_bwd_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int c = blockIdx.x, h = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t L = a.L, H = a.H, G = a.G, nc = a.nc;
    const int P = (int)a.P, N = (int)a.N;
    const int g = (int)(h / (H / G));
    const int64_t t0 = (int64_t)c * kQ;
    const int Qv = (int)imin<int64_t>(kQ, L - t0);
    const int tid = threadIdx.x;
    float *X = sm + ChunkSmem::x, *Y = sm + ChunkSmem::y, *Bs = sm + ChunkSmem::bm, *Cs = sm + ChunkSmem::cm;
    float *Hin = sm + ChunkSmem::hin, *Gn = sm + ChunkSmem::gn, *M1 = sm + ChunkSmem::m1, *M2 = sm + ChunkSmem::m2;
    float *Wb = sm + ChunkSmem::w;
    float *v_dt = sm + ChunkSmem::vec, *v_cs = v_dt + kQ, *v_e = v_cs + kQ, *v_eend = v_e + kQ, *v_dcs = v_eend + kQ;
    float *v_ddt = v_dcs + kQ, *v_r = v_ddt + kQ, *v_v = v_r + kQ, *v_dd = v_v + kQ, *v_da = v_dd + kQ;
    float *red = v_da + kQ, *scratch = red + kT;
    const T *x = static_cast<const T *>(a.x), *dy = static_cast<const T *>(a.dy);
    const T *Bm = static_cast<const T *>(a.Bm), *Cm = static_cast<const T *>(a.Cm);
    const T *dtp = static_cast<const T *>(a.dt);
    const float Ah = a.A[h], Dh = a.D ? a.D[h] : 0.f;

    // ---- loads: x, dy, B, C, entering state, leaving cotangent, dt and its
    //      cumulative sum. Rows of four consecutive elements when P and N are
    //      multiples of 4 (base pointers are 16-byte aligned), else one element
    //      at a time. Vector loads go out in two batches held in registers (x,
    //      dy, B, C before the dt scan; hin, Gn after it), so each batch costs
    //      one memory round trip.
    const bool vec = P % 4 == 0 && N % 4 == 0;
    const int64_t so = ((b * nc + c) * H + h) * (int64_t)P * N;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int kXU = kQ * 16 / kT, kBU = kQ * 32 / kT, kHU = 64 * 32 / kT;  // vectors per thread
    float4 xr[kXU], yr[kXU], br[kBU], cr[kBU];
    if (vec) {
#pragma unroll
        for (int u = 0; u < kXU; ++u) {
            const int e = tid + u * kT, j = e / 16, p = (e % 16) * 4;
            const bool in = j < Qv && p < P;
            const int64_t o = ((b * L + t0 + j) * H + h) * P + p;
            xr[u] = in ? ld4(x + o) : z4;
            yr[u] = in ? ld4(dy + o) : z4;
        }
#pragma unroll
        for (int u = 0; u < kBU; ++u) {
            const int e = tid + u * kT, j = e / 32, n = (e % 32) * 4;
            const bool in = j < Qv && n < N;
            const int64_t o = ((b * L + t0 + j) * G + g) * N + n;
            br[u] = in ? ld4(Bm + o) : z4;
            cr[u] = in ? ld4(Cm + o) : z4;
        }
    }
    const float dv = (tid < Qv) ? to_f32(dtp[(b * L + t0 + tid) * H + h]) : 0.f;
    if (tid < kQ) v_dt[tid] = dv;
    block_inclusive_scan_256(dv * Ah, kQ, v_cs, scratch);
    const float cs_end = v_cs[kQ - 1];  // padded tokens carry a = 0
    if (tid < kQ) {
        v_e[tid] = expf(v_cs[tid]);
        v_eend[tid] = expf(cs_end - v_cs[tid]);
    }
    if (vec) {
        float4 hr[kHU], gr[kHU];
#pragma unroll
        for (int u = 0; u < kHU; ++u) {
            const int e = tid + u * kT, p = e / 32, n = (e % 32) * 4;
            const bool in = p < P && n < N;
            hr[u] = in ? ld4(a.hin + so + p * N + n) : z4;
            gr[u] = in ? ld4(a.adj + so + p * N + n) : z4;
        }
#pragma unroll
        for (int u = 0; u < kXU; ++u) {
            const int e = tid + u * kT, j = e / 16, p = (e % 16) * 4;
            *reinterpret_cast<float4 *>(X + j * kSX + p) = xr[u];
            *reinterpret_cast<float4 *>(Y + j * kSX + p) = yr[u];
        }
#pragma unroll
        for (int u = 0; u < kBU; ++u) {
            const int e = tid + u * kT, j = e / 32, n = (e % 32) * 4;
            *reinterpret_cast<float4 *>(Bs + j * kSN + n) = br[u];
            *reinterpret_cast<float4 *>(Cs + j * kSN + n) = cr[u];
        }
#pragma unroll
        for (int u = 0; u < kHU; ++u) {
            const int e = tid + u * kT, p = e / 32, n = (e % 32) * 4;
            *reinterpret_cast<float4 *>(Hin + p * kSN + n) = hr[u];
            *reinterpret_cast<float4 *>(Gn + p * kSN + n) = gr[u];
        }
    } else {
        for (int e = tid; e < kQ * 64; e += kT) {
            const int j = e / 64, p = e % 64;
            const bool in = j < Qv && p < P;
            const int64_t o = ((b * L + t0 + j) * H + h) * P + p;
            X[j * kSX + p] = in ? to_f32(x[o]) : 0.f;
            Y[j * kSX + p] = in ? to_f32(dy[o]) : 0.f;
        }
        for (int e = tid; e < kQ * 128; e += kT) {
            const int j = e / 128, n = e % 128;
            const bool in = j < Qv && n < N;
            const int64_t o = ((b * L + t0 + j) * G + g) * N + n;
            Bs[j * kSN + n] = in ? to_f32(Bm[o]) : 0.f;
            Cs[j * kSN + n] = in ? to_f32(Cm[o]) : 0.f;
        }
        for (int e = tid; e < 64 * 128; e += kT) {
            const int p = e / 128, n = e % 128;
            const bool in = p < P && n < N;
            Hin[p * kSN + n] = in ? a.hin[so + p * N + n] : 0.f;
            Gn[p * kSN + n] = in ? a.adj[so + p * N + n] : 0.f;
        }
    }
    __syncthreads();

    const int ty = tid / 16, tx = tid % 16;
    const int tq = tid >> 2, tq4 = tid & 3;  // token and quarter of the four-thread dot products
    // ---- CB = C B^T and YX = dY X^T (rows t, columns s = tx + 16 j), then the
    //      masked, decayed forms
    // HC[t][p] = sum_n C[t][n] hin[p][n] (p = tx + 16 j) comes out of the same
    // loop as CB and stays in registers until its use at the end
    float hc[4][4] = {};
    {
        float cb[4][4] = {}, yx[4][4] = {};
        mm_nt_2(cb, hc, N, Cs, kSN, Bs, Hin, kSN);
        mm_nt(yx, P, 0, Y, kSX, X, kSX);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = ty * 4 + i, s = tx + 16 * j;
                const float ld = s <= t ? expf(v_cs[t] - v_cs[s]) : 0.f;
                const float m1 = ld * cb[i][j], m2 = ld * v_dt[s] * yx[i][j];
                M1[t * kSM + s] = m1;
                M2[t * kSM + s] = m2;
                Wb[t * kSM + s] = s < t ? m1 * v_dt[s] * yx[i][j] : 0.f;
            }
    }
    __syncthreads();
    // d cs from the in-chunk decays: row sum minus column sum of W
    {
        float rs = 0.f, cl = 0.f;
        for (int s = tq4; s < kQ; s += 4) {
            rs += Wb[tq * kSM + s];
            cl += Wb[s * kSM + tq];
        }
        rs = quad_sum(rs);
        cl = quad_sum(cl);
        if (tq4 == 0) v_dcs[tq] = rs - cl;
    }
    __syncthreads();
    // ---- GB[s][p] = sum_n B[s][n] Gn[p][n] into Wb (p = tx + 16 j; zero for p >= P)
    {
        float gb[4][4] = {};
        mm_nt(gb, N, 0, Bs, kSN, Gn, kSN);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) Wb[(ty * 4 + i) * kSM + tx + 16 * j] = gb[i][j];
    }
    __syncthreads();
    // r_s = eend_s dt_s x_s . GB_s
    {
        float r = 0.f;
        for (int p = tq4; p < P; p += 4) r = fmaf(X[tq * kSX + p], Wb[tq * kSM + p], r);
        r = quad_sum(r);
        if (tq4 == 0) v_r[tq] = v_eend[tq] * v_dt[tq] * r;
    }
    // ---- du = M1^T dY + eend o GB; dx = dt du + D dY; ddt (input part) = x . du
    {
        float du[4][4] = {};
        mm_tn(du, kQ, 0, M1, kSM, Y, kSX);
        __syncthreads();  // every thread has read M1 before du replaces it
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = ty * 4 + i;
            float dxv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int p = tx * 4 + j;
                const float u = du[i][j] + v_eend[s] * Wb[s * kSM + p];
                M1[s * kSM + p] = u;  // du, for the token dot products below
                dxv[j] = fmaf(v_dt[s], u, Dh * Y[s * kSX + p]);
            }
            float *dxr = a.dx + ((b * L + t0 + s) * H + h) * (int64_t)P;
            if (s < Qv) {
                if (vec) {
                    if (tx * 4 < P) *reinterpret_cast<float4 *>(dxr + tx * 4) = make_float4(dxv[0], dxv[1], dxv[2], dxv[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (tx * 4 + j < P) dxr[tx * 4 + j] = dxv[j];
                }
            }
        }
    }
    __syncthreads();
    {
        float dd = 0.f, xd = 0.f;
        for (int p = tq4; p < P; p += 4) {
            dd = fmaf(X[tq * kSX + p], M1[tq * kSM + p], dd);
            xd = fmaf(Y[tq * kSX + p], X[tq * kSX + p], xd);
        }
        dd = quad_sum(dd);
        xd = quad_sum(xd);
        if (tq4 == 0) {
            v_ddt[tq] = dd;
            v_dd[tq] = xd;
        }
    }
    // ---- dB = M2^T C + (dt eend) o (X Gn); dC = M2 B + e o (dY hin), 64 columns of n per pass
    for (int n0 = 0; n0 < N; n0 += 64) {
        float db[4][4] = {}, dc[4][4] = {};
        mm_tn(db, kQ, n0, M2, kSM, Cs, kSN);
        mm_nn(dc, kQ, n0, M2, kSM, Bs, kSN);
        {
            float xg[4][4] = {}, yh[4][4] = {};
            mm_nn_2(xg, yh, P, n0, X, Y, kSX, Gn, Hin, kSN);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    db[i][j] = fmaf(v_dt[ty * 4 + i] * v_eend[ty * 4 + i], xg[i][j], db[i][j]);
                    dc[i][j] = fmaf(v_e[ty * 4 + i], yh[i][j], dc[i][j]);
                }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = ty * 4 + i;
            if (t >= Qv) continue;
            const int n = n0 + tx * 4;
            const int64_t o = ((b * L + t0 + t) * H + h) * (int64_t)N + n;
            if (vec) {
                if (n < N) {
                    *reinterpret_cast<float4 *>(a.dB_part + o) = make_float4(db[i][0], db[i][1], db[i][2], db[i][3]);
                    *reinterpret_cast<float4 *>(a.dC_part + o) = make_float4(dc[i][0], dc[i][1], dc[i][2], dc[i][3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < N) {
                        a.dB_part[o + j] = db[i][j];
                        a.dC_part[o + j] = dc[i][j];
                    }
            }
        }
    }
    __syncthreads();
    // ---- HC (computed with CB) into Wb; v_t = e_t dY_t . HC_t
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) Wb[(ty * 4 + i) * kSM + tx + 16 * j] = hc[i][j];
    // <Gn, hin>: fixed per-thread ranges (zeros past P, N), then a fixed-order sum
    {
        float qv = 0.f;
        for (int e = tid; e < 64 * 128; e += kT) qv = fmaf(Gn[(e / 128) * kSN + e % 128], Hin[(e / 128) * kSN + e % 128], qv);
        red[tid] = qv;
    }
    __syncthreads();
    {
        float vv = 0.f;
        for (int p = tq4; p < P; p += 4) vv = fmaf(Y[tq * kSX + p], Wb[tq * kSM + p], vv);
        vv = quad_sum(vv);
        if (tq4 == 0) v_v[tq] = v_e[tq] * vv;
    }
    __syncthreads();
    // ---- d cs, da (reverse cumulative sum), ddt, dA and dD parts: the first two
    //      warps, one token per lane, fixed-order shuffle trees
    const int lane = tid & 31, w2 = tid >> 5;
    float suf = 0.f;  // in-warp suffix sum of d cs
    if (tid < kQ) {
        float q = (red[4 * tid] + red[4 * tid + 1]) + (red[4 * tid + 2] + red[4 * tid + 3]);  // kT = 4 kQ
        float rv = tid < Qv ? v_r[tid] : 0.f;
        q = warp_sum(q);
        rv = warp_sum(rv);
        if (lane == 0) {
            scratch[w2] = q;
            scratch[2 + w2] = rv;
        }
    }
    __syncthreads();
    if (tid < kQ) {
        const float q = scratch[0] + scratch[1], rsum = scratch[2] + scratch[3];
        float dcs = tid < Qv ? v_dcs[tid] + v_v[tid] - v_r[tid] : 0.f;
        if (tid == Qv - 1) dcs += rsum + expf(cs_end) * q;
        suf = dcs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_down_sync(0xffffffffu, suf, o);
            if (lane + o < 32) suf += u;
        }
        if (lane == 0) scratch[4 + w2] = suf;  // each warp's total
    }
    __syncthreads();
    if (tid < kQ) {
        const float da = suf + (w2 == 0 ? scratch[5] : 0.f);
        if (tid < Qv) v_da[tid] = da;
        float pa = tid < Qv ? da * v_dt[tid] : 0.f, pd = tid < Qv ? v_dd[tid] : 0.f;
        pa = warp_sum(pa);
        pd = warp_sum(pd);
        if (lane == 0) {
            scratch[6 + w2] = pa;
            red[w2] = pd;
        }
    }
    __syncthreads();
    if (tid == 0) {
        a.dA_part[(b * nc + c) * H + h] = scratch[6] + scratch[7];
        a.dD_part[(b * nc + c) * H + h] = red[0] + red[1];
    }
    if (tid < Qv) a.ddt[(b * L + t0 + tid) * H + h] = fmaf(v_da[tid], Ah, v_ddt[tid]);
}

// dB, dC: sum of the heads' parts of each B/C group, in head order; dA, dD:
// sum over (b, chunk) in order.
__global__ void __launch_bounds__(kT) bwd_reduce_kernel(const __grid_constant__ BwdArgs a) {
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;  // (b, t, g, n)
    const int64_t N = a.N, G = a.G, H = a.H, hpg = a.H / a.G;
    const int64_t total = a.B * a.L * G * N;
    if (i < total) {
        const int64_t n = i % N, g = (i / N) % G, bt = i / (N * G);
        float sb = 0.f, sc = 0.f;
        // eight heads' parts loaded before they are added (in head order)
        for (int64_t k0 = 0; k0 < hpg; k0 += 8) {
            float vb[8], vc[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t o = (bt * H + g * hpg + k0 + u) * N + n;
                vb[u] = k0 + u < hpg ? a.dB_part[o] : 0.f;
                vc[u] = k0 + u < hpg ? a.dC_part[o] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (k0 + u < hpg) {
                    sb += vb[u];
                    sc += vc[u];
                }
        }
        a.dB[i] = sb;
        a.dC[i] = sc;
    }
    if (i < H) {
        float sa = 0.f, sd = 0.f;
        for (int64_t bc = 0; bc < a.B * a.nc; ++bc) {
            sa += a.dA_part[bc * H + i];
            sd += a.dD_part[bc * H + i];
        }
        a.dA[i] = sa;
        if (a.dD) a.dD[i] = sd;
    }
}

// The same sums with four n per thread (N a multiple of 4): sixteen 16-byte
// loads in flight per thread, the heads still added in order.
__global__ void __launch_bounds__(kT) bwd_reduce4_kernel(const __grid_constant__ BwdArgs a) {
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;  // (b, t, g, n/4)
    const int64_t N4 = a.N / 4, G = a.G, H = a.H, hpg = a.H / a.G;
    const int64_t total = a.B * a.L * G * N4;
    if (i < total) {
        const int64_t n4 = i % N4, g = (i / N4) % G, bt = i / (N4 * G);
        const float4 *pb = reinterpret_cast<const float4 *>(a.dB_part) + (bt * H + g * hpg) * N4 + n4;
        const float4 *pc = reinterpret_cast<const float4 *>(a.dC_part) + (bt * H + g * hpg) * N4 + n4;
        float4 sb = make_float4(0.f, 0.f, 0.f, 0.f), sc = sb;
        for (int64_t k0 = 0; k0 < hpg; k0 += 8) {
            float4 vb[8], vc[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (k0 + u < hpg) {
                    vb[u] = pb[(k0 + u) * N4];
                    vc[u] = pc[(k0 + u) * N4];
                }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (k0 + u < hpg) {
                    sb.x += vb[u].x; sb.y += vb[u].y; sb.z += vb[u].z; sb.w += vb[u].w;
                    sc.x += vc[u].x; sc.y += vc[u].y; sc.z += vc[u].z; sc.w += vc[u].w;
                }
        }
        reinterpret_cast<float4 *>(a.dB)[i] = sb;
        reinterpret_cast<float4 *>(a.dC)[i] = sc;
    }
    if (i < H) {
        float sa = 0.f, sd = 0.f;
        for (int64_t bc = 0; bc < a.B * a.nc; ++bc) {
            sa += a.dA_part[bc * H + i];
            sd += a.dD_part[bc * H + i];
        }
        a.dA[i] = sa;
        if (a.dD) a.dD[i] = sd;
    }
}

template <typename T>
cudaError_t launch_bwd_t(const BwdArgs &a, cudaStream_t stream) {
    cudaError_t e;
    if (a.Q == 128) {
        // chunks of 128 tokens: chunk states, the passes over the chunks and
        // the per-chunk gradients on the tensor cores
        if ((e = launch_bwd_states_tc(a, stream)) != cudaSuccess) return e;
        if ((e = launch_chunk_bwd_tc(a, stream)) != cudaSuccess) return e;
        const int64_t n = imax<int64_t>(a.B * a.L * a.G * a.N / 4, a.H);  // N is 128 here
        bwd_reduce4_kernel<<<(unsigned)((n + kT - 1) / kT), kT, 0, stream>>>(a);
        return cudaGetLastError();
    }
    const int tilesP = (int)((a.P + 63) / 64), tilesN = (int)((a.N + 63) / 64);
    adj_chunk_state_kernel<T, 64><<<dim3((unsigned)a.nc, (unsigned)(a.H * tilesP * tilesN), (unsigned)a.B), kT, 0,
                                    stream>>>(a, tilesP, tilesN);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // float4 elements when every (b, c, h) block of P*N states and the optional
    // cotangent arrays start 16-byte aligned
    const int64_t PN = a.P * a.N;
    const bool vec = PN % 4 == 0 && reinterpret_cast<uintptr_t>(a.dfinal) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(a.dinit) % 16 == 0;
    if (vec)
        adj_state_pass_kernel<4><<<dim3((unsigned)((PN / 4 + kT - 1) / kT), (unsigned)a.H, (unsigned)a.B), kT, 0,
                                   stream>>>(a);
    else
        adj_state_pass_kernel<1><<<dim3((unsigned)((PN + kT - 1) / kT), (unsigned)a.H, (unsigned)a.B), kT, 0,
                                   stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem = (size_t)ChunkSmem::total * sizeof(float);
    static DeviceOnce configured;  // set the attribute once per device
    int dev = 0;
    if (configured.pending(&dev, &e)) {
        e = cudaFuncSetAttribute(chunk_bwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured.done(dev);
    } else if (e != cudaSuccess) {
        return e;
    }
    chunk_bwd_kernel<T><<<dim3((unsigned)a.nc, (unsigned)a.H, (unsigned)a.B), kT, smem, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t n = imax<int64_t>(a.B * a.L * a.G * a.N, a.H);
    bwd_reduce_kernel<<<(unsigned)((n + kT - 1) / kT), kT, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_chunk_smem_bytes(int64_t, int64_t) { return (size_t)ChunkSmem::total * sizeof(float); }

cudaError_t launch_ssd_bwd(const BwdArgs &a, cudaStream_t stream) {
    if (a.B == 0 || a.nc == 0) return cudaSuccess;
    return a.io == IO_BF16 ? launch_bwd_t<__nv_bfloat16>(a, stream) : launch_bwd_t<float>(a, stream);
}

}  // namespace ssd
