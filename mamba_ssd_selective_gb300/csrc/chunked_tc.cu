// Tensor-core chunked SSD prefill for bf16 inputs with headdim P = 64 and
// d_state N = 128 (the Mamba-2 layer shapes), and the bounded-wait self-test.
//
// Same three steps as the CUDA-core path (see chunked_simt.cu for the algebra:
// chunk state, state passing, chunk scan), with both chunk kernels built on
// tcgen05 MMAs: bf16 operands staged in shared memory by TMA with the 128-byte
// swizzle, float32 accumulators in tensor memory (TMEM), one elected thread
// issuing the MMAs, 4 warps moving accumulators TMEM -> registers for the
// epilogues. Decays, cumulative sums and exponentials stay float32.
//
//   chunk_state_tc  one CTA per (b, chunk c, group of hb heads sharing B):
//       S_c^T[n, (k, p)] = sum_j B_j[n] * (w_k,j x_k,j[p]),
//       w_k,j = exp(cs_end - cs_j) dt_j of head k; one MMA chain M = 128 (n),
//       N = 64 hb, K = Q (j); both operands MN-major (tokens are the outer
//       dimension in HBM). States leave as bfloat16, plus exp(cs_end).
//   state_pass      (chunked_simt.cu) updates the bf16 states in place into the
//       entering states h_in, the B operand of the output MMA.
//   chunk_scan_tc_persistent  (Q <= 128) one CTA per SM over work items
//       (b, 128-token tile, head group); warp-specialised, see its comment.
//   chunk_scan_tc   (Q = 256) one CTA per (b, 128-token tile, head h):
//       S  = C_tile B_k^T            (M = 128 rows i, N = 128 cols j, K = N)
//       S' = S o exp(cs_i - cs_j) dt_j, static causal & same-chunk mask
//       Y += S' X_k                  (M = 128, N = P, K = 128)  per K-block k
//       Yo = C_tile h_in^T           (M = 128, N = P, K = N)    per chunk
//       y  = Y + exp(cs_i - cs_chunk_start) Yo + D x  -> bf16 -> TMA store
//   The K-blocks of a tile are the 128-token blocks from the start of the
//   tile's chunk up to the tile (2 for the second half of a 256-token chunk).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "ssd_scan.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: a wait this long means something is broken
constexpr int kRows = 128;                   // token rows per tile (MMA M)
constexpr int kP = 64;                       // headdim handled here
constexpr int kN = 128;                      // d_state handled here
constexpr float kLog2e = 1.4426950408889634f;

struct TcParams {
    ChunkedArgs a;
    CUtensorMap mx;    // x  as (H*P, L, B), box (64, R, 1)
    CUtensorMap mb;    // B  as (G*N, L, B), box (64, R, 1)
    CUtensorMap mc;    // C  as (G*N, L, B), box (64, 128, 1)   (chunk scan)
    CUtensorMap my;    // y  as (H*P, L, B), box (64, 128, 1)   (chunk scan)
    CUtensorMap mh;    // bf16 entering states as (N, B*nc*H*P), box (64, 64)   (chunk scan)
    int hb;            // heads per work item of the persistent chunk scan (divides H / G)
    int nhg;           // head groups, H / hb
    int64_t n_items;   // work items of the persistent chunk scan, B * tiles * nhg
};

// ---------------------------------------------------------------- helpers

// In-place inclusive prefix sum of buf[0..n) (n <= 256) by a 128-thread CTA;
// thread t owns elements 2t and 2t+1. Fixed association. `tot` holds 4 floats.
__device__ __forceinline__ void cta128_inclusive_scan(float *buf, int n, float *tot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int e0 = 2 * tid, e1 = e0 + 1;
    const float v0 = e0 < n ? buf[e0] : 0.f, v1 = e1 < n ? buf[e1] : 0.f;
    const float s = v0 + v1;
    float incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) tot[warp] = incl;
    __syncthreads();
    float base = 0.f;
    for (int w = 0; w < warp; ++w) base += tot[w];
    const float excl = base + incl - s;
    if (e0 < n) buf[e0] = excl + v0;
    if (e1 < n) buf[e1] = excl + v0 + v1;
    __syncthreads();
}

__device__ __forceinline__ void record_failure(int *status) { atomicCAS(status, SSD_OK, SSD_ERR_TIMEOUT); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// --------------------------------------------------------- chunk state

// bytes of the operand space of chunk_state_tc: B^T and x
__host__ __device__ constexpr int state_region(int Q, int hb) { return Q * 256 + hb * Q * 128; }
constexpr int kStateHBMax = 8;  // heads per chunk-state CTA (TMEM: 64 columns each)
//
// One CTA per (b, chunk c, group of hb heads sharing a B/C group). All heads
// of the group share the A operand B^T, so their chunk states come out of one
// MMA chain with N = 64 hb (the tensor core's cost per instruction is nearly
// flat in N up to 256): S^T[n, (k, p)] = sum_j B_j[n] (w_k,j x_k,j[p]) with
// w_k,j = exp(cs_end - cs_j) dt_j of head k. The states go out as bfloat16.

__global__ void __launch_bounds__(256) chunk_state_tc(const __grid_constant__ TcParams prm) {
    const ChunkedArgs &a = prm.a;
    const int c = blockIdx.x, hg = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int HB = prm.hb;
    const int h0 = hg * HB;
    const int Q = a.Q, R = Q < kRows ? Q : kRows;
    const int g = (int)(h0 / (a.H / a.G));
    const int64_t t0 = (int64_t)c * Q;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sB = smem;                    // B^T operand: 2 panels (n 0-63, 64-127) x Q rows x 128 B
    uint8_t *sX = smem + Q * 256;          // x operands of the hb heads: hb panels of Q rows x 128 B
    float *s_w = reinterpret_cast<float *>(smem + state_region(Q, HB));  // [hb][256]
    uint64_t *bar_ld = reinterpret_cast<uint64_t *>(s_w + kStateHBMax * 256);
    uint64_t *bar_mma = bar_ld + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_mma + 1);
    int *s_fail = reinterpret_cast<int *>(tmem_slot + 1);
    const uint32_t ncols = HB > 4 ? 512u : HB > 2 ? 256u : HB == 2 ? 128u : 64u;  // power of 2 >= 64 hb

    // TMEM first: until a CTA has given up its allocation permit, no other
    // CTA is placed on its SM
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, ncols);
        tc::tmem_relinquish();
    }
    // Launched as a programmatic dependent of whatever kernel precedes it in the
    // stream: no global memory is touched before that grid has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // this call's status word starts clear (the first kernel of the call)
    if (tid == 32 && c == 0 && hg == 0 && b == 0) *a.status = SSD_OK;
    // B^T and x by TMA; the cumulative sums and the CTA barrier overlap the loads
    if (tid == 0) {
        tc::mbar_init(bar_ld, 1);
        tc::mbar_init(bar_mma, 1);
        tc::fence_mbar_init();
        *s_fail = 0;
        tc::mbar_arrive_expect_tx(bar_ld, (uint32_t)Q * 256u + (uint32_t)HB * Q * 128u);
        for (int half = 0; half < 2; ++half)
            for (int r0 = 0; r0 < Q; r0 += R)
                tc::tma_load_3d(sB + half * Q * 128 + r0 * 128, &prm.mb, bar_ld, g * kN + half * 64,
                                (int)(t0 + r0), (int)b);
        for (int k = 0; k < HB; ++k)
            for (int r0 = 0; r0 < Q; r0 += R)
                tc::tma_load_3d(sX + k * Q * 128 + r0 * 128, &prm.mx, bar_ld, (h0 + k) * kP, (int)(t0 + r0),
                                (int)b);
    }
    // warps < hb: dt of head h0 + warp, lane l owning Q/32 consecutive tokens
    float dv[8];
    if (warp < HB) {
        const __nv_bfloat16 *dt = static_cast<const __nv_bfloat16 *>(a.dt);
        const int per = Q / 32;  // 2, 4 or 8
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int j = lane * per + q;
            dv[q] = (q < per && t0 + j < a.L) ? __bfloat162float(dt[(b * a.L + t0 + j) * a.H + h0 + warp]) : 0.f;
        }
    }

    // warp k: in-chunk cumulative sum of dt*A (base 2) of head k and its
    // weights w_j; lane l owns Q/32 consecutive tokens
    if (warp < HB) {
        const int h = h0 + warp;
        const float A2 = a.A[h] * kLog2e;
        const int per = Q / 32;
        float cs[8];
        float run = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            run += dv[q] * A2;
            cs[q] = run;
        }
        float incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        const float excl = incl - run;
        const float cs_end = __shfl_sync(0xffffffffu, incl, 31);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (q < per) s_w[warp * 256 + lane * per + q] = tc::ex2(cs_end - (excl + cs[q])) * dv[q];
        if (lane == 0) a.chunk_sum[(b * a.H + h) * a.nc + c] = tc::ex2(cs_end);  // decay over the chunk
    }

    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (!tc::mbar_wait(bar_ld, 0, kWaitNs)) *s_fail = 1;
    __syncthreads();
    if (!*s_fail) {
        // x_k,j <- w_k,j x_k,j in place (packed bf16 multiplies). Thread t
        // takes 16-byte piece t & 7 of rows r = t / 8 + 32 i (row r = k Q + j
        // holds all 64 p of token j of head k); the swizzle only permutes the
        // pieces within a row.
        const int lq = Q == 64 ? 6 : Q == 128 ? 7 : 8;
        const int rows = HB * Q;
        for (int r = tid >> 3; r < rows; r += 32) {
            uint4 *ptr = reinterpret_cast<uint4 *>(sX + r * 128 + (tid & 7) * 16);
            uint4 v = *ptr;
            const __nv_bfloat162 w2 = __float2bfloat162_rn(s_w[(r >> lq) * 256 + (r & (Q - 1))]);
            __nv_bfloat162 *u = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
            for (int q = 0; q < 4; ++q) u[q] = __hmul2(u[q], w2);
            *ptr = v;
        }
        tc::fence_proxy_async_smem();
    }
    __syncthreads();
    if (*s_fail) {
        if (tid == 0) record_failure(a.status);
    } else {
        if (tid == 0) {
            tc::tc_fence_after();
            // chains of at most 4 heads (N <= 256): heads h0c .. h0c + nh - 1
            const uint32_t b0 = tc::smem_u32(sB), x0 = tc::smem_u32(sX);
            for (int h0c = 0; h0c < HB; h0c += 4) {
                const int nh = HB - h0c < 4 ? HB - h0c : 4;
                const uint32_t idesc = tc::idesc_bf16(128, kP * nh, true, true);
                const uint32_t xc = x0 + (uint32_t)(h0c * Q * 128);
                for (int k = 0; k < Q; k += 16) {
                    const uint64_t da = tc::sdesc_sw128(b0 + k * 128, Q * 128, 1024);
                    const uint64_t db = tc::sdesc_sw128(xc + k * 128, Q * 128, 1024);
                    tc::mma_bf16(tmem + (uint32_t)(h0c * kP), da, db, idesc, k > 0 ? 1u : 0u);
                }
            }
            tc::mma_commit(bar_mma);
        }
        __syncwarp();
        if (!tc::mbar_wait(bar_mma, 0, kWaitNs)) *s_fail = 1;
        __syncthreads();
        if (*s_fail) {
            if (tid == 0) record_failure(a.status);
        } else {
            tc::tc_fence_after();
            // lane 32*(warp%4) + l of TMEM holds n; column 64 k + p. Warps w and
            // w + 4 share a lane quarter and split the heads.
            const int n = (warp & 3) * 32 + lane;
            __nv_bfloat16 *S = reinterpret_cast<__nv_bfloat16 *>(a.states_bf16);
            for (int k = warp >> 2; k < HB; k += 2) {
                __nv_bfloat16 *Sk = S + (((b * a.nc + c) * a.H + h0 + k) * kP) * kN + n;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float v[32];
                    tc::tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + k * 64 + half * 32, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 32; ++q) Sk[(half * 32 + q) * kN] = __float2bfloat16_rn(v[q]);
                }
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, ncols);
    // let the state pass start its launch while this grid drains
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------- chunk scan

__global__ void __launch_bounds__(128) chunk_scan_tc(const __grid_constant__ TcParams prm) {
    const ChunkedArgs &a = prm.a;
    const int tile = blockIdx.x, h = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int Q = a.Q;
    const int g = (int)(h / (a.H / a.G));
    const int64_t t0 = (int64_t)tile * kRows;
    // K-range: from the start of the tile's chunk (Q >= 128) or the tile itself
    const int64_t ks = Q > kRows ? (t0 / Q) * Q : t0;
    const int nk = (int)((t0 - ks) / kRows) + 1;  // K-blocks of 128 tokens
    const int kl = nk * kRows;
    const int roff = (int)(t0 - ks);              // K-range index of tile row 0
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i = tid;                            // tile row = TMEM lane

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sC = smem;                   // C tile, K-major: 2 panels x 128 rows x 128 B (later: y staging)
    uint8_t *sB = smem + 32768;           // B block, K-major: 2 panels x 128 rows (later: S', then h_in)
    uint8_t *sX = smem + 65536;           // x block, MN-major: 128 rows x 128 B
    float *s_dt = reinterpret_cast<float *>(smem + 81920);
    float *s_cs = s_dt + 256;
    float *s_colf = s_cs + 256;  // exp(cs_r - cs_j) dt_j, r = last column of j's 32-block
    float *s_tot = s_colf + 256;
    uint64_t *bar_ld = reinterpret_cast<uint64_t *>(s_tot + 8);
    uint64_t *bar_mma = bar_ld + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_mma + 1);
    int *s_fail = reinterpret_cast<int *>(tmem_slot + 1);

    if (tid == 0) {
        tc::mbar_init(bar_ld, 1);
        tc::mbar_init(bar_mma, 1);
        tc::fence_mbar_init();
        *s_fail = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, 256);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's lane quarter
    uint32_t ph_ld = 0, ph_mma = 0;

    auto load_block = [&](int kb) {  // B and x rows of K-block kb
        const int64_t r = ks + (int64_t)kb * kRows;
        tc::mbar_arrive_expect_tx(bar_ld, kb == 0 ? 32768u + 32768u + 16384u : 32768u + 16384u);
        if (kb == 0) {
            tc::tma_load_3d(sC, &prm.mc, bar_ld, g * kN, (int)t0, (int)b);
            tc::tma_load_3d(sC + 16384, &prm.mc, bar_ld, g * kN + 64, (int)t0, (int)b);
        }
        tc::tma_load_3d(sB, &prm.mb, bar_ld, g * kN, (int)r, (int)b);
        tc::tma_load_3d(sB + 16384, &prm.mb, bar_ld, g * kN + 64, (int)r, (int)b);
        tc::tma_load_3d(sX, &prm.mx, bar_ld, h * kP, (int)r, (int)b);
    };
    if (tid == 0) load_block(0);

    // cumulative sum of dt*A over the K-range
    const __nv_bfloat16 *dt = static_cast<const __nv_bfloat16 *>(a.dt);
    const float Ah = a.A[h];
    for (int j = tid; j < kl; j += 128) {
        const float d = (ks + j < a.L) ? __bfloat162float(dt[(b * a.L + ks + j) * a.H + h]) : 0.f;
        s_dt[j] = d;
        s_cs[j] = d * Ah;
    }
    __syncthreads();
    cta128_inclusive_scan(s_cs, kl, s_tot);
    for (int j = tid; j < kl; j += 128) s_colf[j] = __expf(s_cs[j | 31] - s_cs[j]) * s_dt[j];
    __syncthreads();

    const int ir = roff + i;  // K-range index of this thread's row
    const float cs_i = s_cs[ir];
    const uint32_t idesc_s = tc::idesc_bf16(128, 128, false, false);
    const uint32_t idesc_y = tc::idesc_bf16(128, kP, false, true);
    const uint32_t idesc_o = tc::idesc_bf16(128, kP, false, false);
    const uint32_t c0 = tc::smem_u32(sC), b0 = tc::smem_u32(sB), x0 = tc::smem_u32(sX);
    bool ok = true;

    for (int kb = 0; kb < nk && ok; ++kb) {
        if (!tc::mbar_wait(bar_ld, ph_ld, kWaitNs)) *s_fail = 1;
        ph_ld ^= 1;
        __syncthreads();
        if (*s_fail) { ok = false; break; }
        // S = C B_kb^T into TMEM columns [0, 128)
        if (tid == 0) {
            tc::tc_fence_after();
            for (int k = 0; k < kN; k += 16) {
                const uint64_t da = tc::sdesc_sw128(c0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                const uint64_t db = tc::sdesc_sw128(b0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                tc::mma_bf16(tmem, da, db, idesc_s, k > 0 ? 1u : 0u);
            }
            tc::mma_commit(bar_mma);
        }
        __syncwarp();
        if (!tc::mbar_wait(bar_mma, ph_mma, kWaitNs)) *s_fail = 1;
        ph_mma ^= 1;
        __syncthreads();
        if (*s_fail) { ok = false; break; }
        tc::tc_fence_after();
        // S' = S o decay o dt_j under the causal same-chunk mask, bf16, K-major,
        // into the B block's space (B is no longer needed). Columns come in
        // 32-wide blocks J of the K-range; this warp's rows all lie in block
        // Jd. Blocks after Jd are zero; blocks before it use the factorised
        // decay exp(cs_i - cs_r) exp(cs_r - cs_j) with r the last column of
        // the block (both factors <= 1 for a decaying head); block Jd takes
        // exp(cs_i - cs_j) directly.
        const int Jd = (roff >> 5) + warp;
        for (int cc = 0; cc < 4; ++cc) {
            const int J = kb * 4 + cc;
            float v[32];
            if (J <= Jd) {
                tc::tmem_ld32(tl + cc * 32, v);
                tc::tmem_ld_wait();
                if (J < Jd) {
                    const bool same = Q >= kRows || (J >> 1) == (Jd >> 1);
                    const float rf = same ? __expf(cs_i - s_cs[J * 32 + 31]) : 0.f;
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] = v[q] * rf * s_colf[J * 32 + q];
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int jr = J * 32 + q;
                        v[q] = jr <= ir ? v[q] * __expf(cs_i - s_cs[jr]) * s_dt[jr] : 0.f;
                    }
                }
            } else {
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = 0.f;
            }
#pragma unroll
            for (int q = 0; q < 32; q += 8) {
                const uint4 pk = make_uint4(pack_bf16x2(v[q], v[q + 1]), pack_bf16x2(v[q + 2], v[q + 3]),
                                            pack_bf16x2(v[q + 4], v[q + 5]), pack_bf16x2(v[q + 6], v[q + 7]));
                *reinterpret_cast<uint4 *>(sB + tc::sw128_offset(i, cc * 32 + q, kRows)) = pk;
            }
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        // Y (+)= S' X_kb into TMEM columns [128, 192)
        if (tid == 0) {
            tc::tc_fence_after();
            for (int k = 0; k < kRows; k += 16) {
                const uint64_t da = tc::sdesc_sw128(b0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                const uint64_t db = tc::sdesc_sw128(x0 + k * 128, 16384, 1024);
                tc::mma_bf16(tmem + 128, da, db, idesc_y, (kb > 0 || k > 0) ? 1u : 0u);
            }
            tc::mma_commit(bar_mma);
        }
        __syncwarp();
        if (!tc::mbar_wait(bar_mma, ph_mma, kWaitNs)) *s_fail = 1;
        ph_mma ^= 1;
        __syncthreads();
        if (*s_fail) { ok = false; break; }
        if (kb + 1 < nk && tid == 0) load_block(kb + 1);
    }

    // entering states of the tile's chunk(s): written by the state pass
    const int nsub = Q < kRows ? kRows / Q : 1;  // chunks in this tile (2 for Q = 64)
    if (ok) {
        if (tid == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            tc::mbar_arrive_expect_tx(bar_ld, (uint32_t)nsub * 16384u);
            for (int s = 0; s < nsub; ++s) {
                const int64_t cidx = (t0 + (int64_t)s * Q) / Q;
                const int row0 = (int)(((b * a.nc + cidx) * a.H + h) * kP);
                tc::tma_load_2d(sB + s * 16384, &prm.mh, bar_ld, 0, row0);
                tc::tma_load_2d(sB + s * 16384 + 8192, &prm.mh, bar_ld, 64, row0);
            }
        }
        if (!tc::mbar_wait(bar_ld, ph_ld, kWaitNs)) *s_fail = 1;
        ph_ld ^= 1;
        __syncthreads();
        ok = !*s_fail;
    }
    if (ok) {
        // Yo_s = C h_in(s)^T into TMEM columns [64 s, 64 s + 64)
        if (tid == 0) {
            tc::tc_fence_after();
            for (int s = 0; s < nsub; ++s) {
                const uint32_t h0 = b0 + s * 16384;
                for (int k = 0; k < kN; k += 16) {
                    const uint64_t da = tc::sdesc_sw128(c0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                    const uint64_t db = tc::sdesc_sw128(h0 + (k >> 6) * 8192 + (k & 63) * 2, 16, 1024);
                    tc::mma_bf16(tmem + s * 64, da, db, idesc_o, k > 0 ? 1u : 0u);
                }
            }
            tc::mma_commit(bar_mma);
        }
        __syncwarp();
        if (!tc::mbar_wait(bar_mma, ph_mma, kWaitNs)) *s_fail = 1;
        ph_mma ^= 1;
        __syncthreads();
        ok = !*s_fail;
    }
    if (ok) {
        tc::tc_fence_after();
        // epilogue: y = Y + exp(cs_i - cs at the chunk start) Yo + D x
        const int sub = Q < kRows ? (i / Q) : 0;  // warp-uniform (Q = 64: warps 0-1 / 2-3)
        const float base = sub > 0 ? s_cs[roff + sub * Q - 1] : 0.f;
        const float sc = __expf(cs_i - base);
        const float Dh = a.D ? a.D[h] : 0.f;
        for (int half = 0; half < 2; ++half) {
            float yv[32], ov[32];
            tc::tmem_ld32(tl + 128 + half * 32, yv);
            tc::tmem_ld32(tl + sub * 64 + half * 32, ov);
            tc::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; q += 8) {
                const int p0 = half * 32 + q;
                const uint4 xr = *reinterpret_cast<const uint4 *>(sX + tc::sw128_offset(i, p0, kRows));
                const uint32_t *xu = reinterpret_cast<const uint32_t *>(&xr);
                uint32_t pk[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xu[m]));
                    const float y0 = yv[q + 2 * m] + sc * ov[q + 2 * m] + Dh * xf.x;
                    const float y1 = yv[q + 2 * m + 1] + sc * ov[q + 2 * m + 1] + Dh * xf.y;
                    pk[m] = pack_bf16x2(y0, y1);
                }
                *reinterpret_cast<uint4 *>(sC + tc::sw128_offset(i, p0, kRows)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
        tc::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc::tma_store_3d(&prm.my, sC, h * kP, (int)t0, (int)b);
            tc::bulk_commit();
            tc::bulk_wait_all();
        }
    } else if (tid == 0) {
        record_failure(a.status);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
    (void)lane;
}

// ------------------------------------------- persistent chunk scan (Q <= 128)
//
// One CTA per SM walks work items (b, 128-token tile, group of hb heads that
// share a B/C group). Per item, in tensor memory (TMEM, 512 columns):
//   S       = C B^T                      columns [0, 128)          (MMA1)
//   Yo(s,k) = C h_in(s, k)^T             128 + 64 (s hb + k)       (MMA3, one
//             chain per chunk s of the tile with N = 64 hb: the C operand is
//             read once for all heads of the item)
//   S'(k)   = S o decay_k (+ D_k on the diagonal), bf16     384 / 448 (two buffers)
//   Y(k)    = Yo'(k) + S'(k) X_k, accumulated by MMA2 onto Yo'(k) = the
//             row-scaled entering-state term, which the epilogue writes back
//             into the columns of Yo(0, k) before MMA2 (A operand of MMA2
//             read from TMEM: S' never touches shared memory)
// so y(k) = Y(k) leaves TMEM in one read. Warp roles:
//   warp 0       TMA producer: C, B (per item), x (per head, 4-deep ring)
//   warp 1       MMA issuer (one lane)
//   warp 2       TMA producer of the entering states (waits for the state
//                pass) and TMA store of each head's y tile staged in shared memory
//   warp 3       per-item scalars one item ahead: cumulative sums of dt A,
//                decays and rescale factors of every head
//   warps 4..19  epilogue, one warp per (TMEM lane quarter, 32-column group):
//                per head S', the entering-state rescale and the staging of
//                its 16 columns of y
// All waits are bounded: a timeout raises a CTA-wide flag, every role then
// runs to the end of its loop without waiting and the status word records
// SSD_ERR_TIMEOUT.

constexpr int kHBMax = 4;
constexpr int kEpiWarp0 = 4;                        // first epilogue warp
constexpr int kEpiThreads = 512;                    // 16 epilogue warps
constexpr int kScanPThreads = 32 * kEpiWarp0 + kEpiThreads;  // 20 warps (5 per SMSP: 96 registers each)
constexpr int kXStages = 4;

__device__ __forceinline__ bool pwait(uint64_t *bar, uint32_t parity, volatile int *fail) {
    const uint32_t addr = tc::smem_u32(bar);
    if (tc::mbar_try_wait(addr, parity)) return true;
    if (*fail) return false;
    const uint64_t t0 = tc::global_ns();
    for (;;) {
        if (tc::mbar_try_wait(addr, parity)) return true;
        if (*fail) return false;
        if (tc::global_ns() - t0 > kWaitNs) {
            *fail = 1;
            return false;
        }
    }
}


__global__ void __launch_bounds__(kScanPThreads, 1) chunk_scan_tc_persistent(const __grid_constant__ TcParams prm) {
    const ChunkedArgs &a = prm.a;
    const int Q = a.Q;               // 64 or 128
    const int nsub = kRows / Q;      // chunks per tile
    const int HB = prm.hb, nhg = prm.nhg;
    const int64_t ntiles = (a.L + kRows - 1) / kRows;
    const int64_t n_items = prm.n_items;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t HT = (uint32_t)HB * 16384u;  // entering-state tiles of one chunk (HB heads)

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sC = smem;                  // C tile, K-major, 2 panels
    uint8_t *sB = smem + 32768;          // B tile, K-major, 2 panels
    uint8_t *sX = smem + 65536;          // x ring: kXStages x 16 KB, MN-major
    uint8_t *sH = sX + kXStages * 16384; // entering states: per chunk s, 2 panels of 64 hb rows (K-major, N = (k, p))
    // per-item scalars of every row and head, double-buffered by item:
    // [2][kScal] floats = cs | dt | colf | sc, each [kHBMax][128], then D [kHBMax]
    constexpr int kScal = 4 * kHBMax * 128 + kHBMax;
    uint8_t *sY = sH + 65536;            // y of one head (128 rows x 128 B, 128-byte swizzle) for the TMA store
    float *s_scal = reinterpret_cast<float *>(sY + 16384);
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_scal + 2 * kScal + 4);
    uint64_t *tile_full = bars + 0, *tile_empty = bars + 1;
    uint64_t *h_full = bars + 2, *h_empty = bars + 3;
    uint64_t *s_full = bars + 4, *s_empty = bars + 5;
    uint64_t *yo_full = bars + 6, *acc_empty = bars + 7;
    uint64_t *y_full = bars + 8;                                        // [2]
    uint64_t *p_full = bars + 10, *p_empty = bars + 12;                 // [2] each
    uint64_t *x_full = bars + 14, *x_empty = bars + 14 + kXStages;      // [kXStages] each
    uint64_t *c_full = bars + 14 + 2 * kXStages, *c_empty = c_full + 2;  // [2] each
    uint64_t *ys_full = bars + 18 + 2 * kXStages, *ys_empty = ys_full + 1;
    constexpr int kBars = 20 + 2 * kXStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBars);
    volatile int *s_fail = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int hpg = (int)(a.H / a.G);  // heads per B/C group
    auto decode = [&](int64_t u, int64_t &b, int64_t &tile, int &hg) {
        hg = (int)(u % nhg);
        const int64_t t = u / nhg;
        tile = t % ntiles;
        b = t / ntiles;
    };
    // C and B of item u; returns the x column of its first head, the tile's
    // first token and the sequence, for load_x
    auto issue_tile = [&](int64_t u, int &xcol, int &t0, int &bb) {
        int64_t b, tile;
        int hg;
        decode(u, b, tile, hg);
        t0 = (int)(tile * kRows);
        bb = (int)b;
        xcol = hg * HB * kP;
        const int g = hg * HB / hpg;
        tc::mbar_arrive_expect_tx(tile_full, 65536u);
        tc::tma_load_3d(sC, &prm.mc, tile_full, g * kN, t0, bb);
        tc::tma_load_3d(sC + 16384, &prm.mc, tile_full, g * kN + 64, t0, bb);
        tc::tma_load_3d(sB, &prm.mb, tile_full, g * kN, t0, bb);
        tc::tma_load_3d(sB + 16384, &prm.mb, tile_full, g * kN + 64, t0, bb);
    };
    auto load_x = [&](int xcol, int t0, int bb, uint32_t x) {
        tc::mbar_arrive_expect_tx(&x_full[x], 16384u);
        tc::tma_load_3d(sX + x * 16384, &prm.mx, &x_full[x], xcol, t0, bb);
    };

    if (tid == 0) {
        for (int k = 0; k < kBars; ++k) tc::mbar_init(bars + k, 1);
        tc::mbar_init(s_empty, kEpiThreads);
        tc::mbar_init(acc_empty, kEpiThreads);
        tc::mbar_init(p_full + 0, kEpiThreads);
        tc::mbar_init(p_full + 1, kEpiThreads);
        tc::mbar_init(c_empty + 0, kEpiThreads);
        tc::mbar_init(c_empty + 1, kEpiThreads);
        tc::mbar_init(ys_full, kEpiThreads);
        tc::fence_mbar_init();
        *s_fail = 0;
        // the first item's operands (the x ring starts empty and holds every
        // head of an item) go out before the TMEM allocation and the CTA barrier
        if (blockIdx.x < n_items) {
            int xcol, t0, bb;
            issue_tile(blockIdx.x, xcol, t0, bb);
            for (int k = 0; k < HB; ++k) load_x(xcol + k * kP, t0, bb, (uint32_t)k);
        }
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tAcc = tmem + 128, tP = tmem + 384;
    // the next call's chunk state may start its launch now; it waits for this
    // grid's completion before it touches memory
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            // the first item went out before the CTA barrier
            uint32_t tcnt = 1, xi = (uint32_t)HB % kXStages, xph = HB == kXStages ? 1u : 0u;
            for (int64_t u = blockIdx.x + gridDim.x; u < n_items && !*s_fail; u += gridDim.x) {
                if (!pwait(tile_empty, (tcnt & 1) ^ 1, s_fail)) break;
                ++tcnt;
                int xcol, t0, bb;
                issue_tile(u, xcol, t0, bb);
                for (int k = 0; k < HB; ++k) {
                    if (!pwait(&x_empty[xi], xph ^ 1, s_fail)) break;
                    load_x(xcol + k * kP, t0, bb, xi);
                    if (++xi == kXStages) { xi = 0; xph ^= 1; }
                }
            }
        }
    } else if (warp == 2) {
        // ---------- TMA producer of entering states, and TMA store of y: one
        // head at a time the epilogue stages y(k) in sY, this warp writes it with
        // one tensor store (full 128-byte lines, instead of each thread's 16-byte
        // pieces of rows 3 KB apart). Item u's entering states are loaded as soon
        // as item u - 1's entering-state MMA has read the previous ones, then
        // item u - 1's heads are stored as the epilogue produces them.
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            uint32_t hcnt = 0, ny = 0;
            int64_t pb = -1, ptile = 0;
            int phg = 0;
            auto store_item = [&](int64_t sb_, int64_t stile, int shg) {
                for (int k = 0; k < HB; ++k, ++ny) {
                    if (!pwait(ys_full, ny & 1, s_fail)) return;
                    tc::tma_store_3d(&prm.my, sY, (shg * HB + k) * kP, (int)(stile * kRows), (int)sb_);
                    tc::bulk_commit();
                    tc::bulk_wait_read_all();  // sY may be written again
                    tc::mbar_arrive(ys_empty);
                }
            };
            for (int64_t u = blockIdx.x; u < n_items && !*s_fail; u += gridDim.x) {
                int64_t b, tile;
                int hg;
                decode(u, b, tile, hg);
                const int64_t t0 = tile * kRows;
                if (!pwait(h_empty, (hcnt & 1) ^ 1, s_fail)) break;
                ++hcnt;
                tc::mbar_arrive_expect_tx(h_full, (uint32_t)nsub * HT);
                for (int sb = 0; sb < nsub; ++sb) {
                    const int64_t cidx = (t0 + (int64_t)sb * Q) / Q;
                    for (int k = 0; k < HB; ++k) {
                        const int row0 = (int)(((b * a.nc + cidx) * a.H + hg * HB + k) * kP);
                        uint8_t *dst = sH + sb * HT + k * 8192;
                        tc::tma_load_2d(dst, &prm.mh, h_full, 0, row0);
                        tc::tma_load_2d(dst + HB * 8192, &prm.mh, h_full, 64, row0);
                    }
                }
                if (pb >= 0) store_item(pb, ptile, phg);
                pb = b;
                ptile = tile;
                phg = hg;
            }
            if (pb >= 0 && !*s_fail) store_item(pb, ptile, phg);
            tc::bulk_wait_all();  // every store of this CTA is complete
        }
    } else if (warp == 3) {
        // ------------------ per-item scalars, one item ahead of the epilogue
        // For every head k of the item and tile row i (base-2 units):
        //   cs   inclusive cumulative sum of dt*A over the tile's rows
        //   colf exp(cs at the end of row i's 32-row block - cs_i) * dt_i
        //   sc   exp(cs_i - cs at the start of row i's chunk)
        // Lane l owns rows 4l .. 4l + 3.
        const __nv_bfloat16 *dtp = static_cast<const __nv_bfloat16 *>(a.dt);
        uint32_t ci = 0;
        for (int64_t u = blockIdx.x; u < n_items && !*s_fail; u += gridDim.x, ++ci) {
            int64_t b, tile;
            int hg;
            decode(u, b, tile, hg);
            const int64_t t0 = tile * kRows;
            float dv[kHBMax][4];
#pragma unroll
            for (int k = 0; k < kHBMax; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t t = t0 + 4 * lane + q;
                    dv[k][q] = (k < HB && t < a.L) ? __bfloat162float(dtp[(b * a.L + t) * a.H + hg * HB + k]) : 0.f;
                }
            const uint32_t buf = ci & 1;
            if (!pwait(&c_empty[buf], ((ci >> 1) & 1) ^ 1, s_fail)) break;
            float *cs_ = s_scal + buf * kScal, *dt_ = cs_ + kHBMax * 128, *cf_ = dt_ + kHBMax * 128;
            float *sc_ = cf_ + kHBMax * 128, *D_ = sc_ + kHBMax * 128;
#pragma unroll
            for (int k = 0; k < kHBMax; ++k) {
                if (k < HB) {
                    const int h = hg * HB + k;
                    const float A2 = a.A[h] * kLog2e;
                    float c[4], run = 0.f;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        run += dv[k][q] * A2;
                        c[q] = run;
                    }
                    float incl = run;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float w = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += w;
                    }
                    const float excl = incl - run;
#pragma unroll
                    for (int q = 0; q < 4; ++q) c[q] += excl;
                    const float blk_end = __shfl_sync(0xffffffffu, c[3], lane | 7);
                    const float mid = __shfl_sync(0xffffffffu, c[3], 15);  // end of the first 64 rows
                    const float c0 = (Q < kRows && lane >= 16) ? mid : 0.f;
                    float4 vcs, vdt, vcf, vsc;
                    vcs = make_float4(c[0], c[1], c[2], c[3]);
                    vdt = make_float4(dv[k][0], dv[k][1], dv[k][2], dv[k][3]);
                    vcf = make_float4(tc::ex2(blk_end - c[0]) * dv[k][0], tc::ex2(blk_end - c[1]) * dv[k][1],
                                      tc::ex2(blk_end - c[2]) * dv[k][2], tc::ex2(blk_end - c[3]) * dv[k][3]);
                    vsc = make_float4(tc::ex2(c[0] - c0), tc::ex2(c[1] - c0), tc::ex2(c[2] - c0), tc::ex2(c[3] - c0));
                    reinterpret_cast<float4 *>(cs_ + k * 128)[lane] = vcs;
                    reinterpret_cast<float4 *>(dt_ + k * 128)[lane] = vdt;
                    reinterpret_cast<float4 *>(cf_ + k * 128)[lane] = vcf;
                    reinterpret_cast<float4 *>(sc_ + k * 128)[lane] = vsc;
                    if (lane == 0) D_[k] = a.D ? a.D[h] : 0.f;
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&c_full[buf]);
        }
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idS = tc::idesc_bf16(128, 128, false, false);
            const uint32_t idY = tc::idesc_bf16(128, kP, false, true);
            const uint32_t idO = tc::idesc_bf16(128, kP * HB, false, false);
            const uint32_t c0 = tc::smem_u32(sC), b0 = tc::smem_u32(sB), h0 = tc::smem_u32(sH);
            uint32_t tph = 0, sph = 0, hph = 0, aph = 0, xi = 0, xph = 0, nh = 0;
            for (int64_t u = blockIdx.x; u < n_items && !*s_fail; u += gridDim.x) {
                if (!pwait(tile_full, tph, s_fail)) break;
                tph ^= 1;
                // S = C B^T (the previous item's S has been read)
                if (!pwait(s_empty, sph ^ 1, s_fail)) break;
                sph ^= 1;
                tc::tc_fence_after();
                for (int k = 0; k < kN; k += 16) {
                    const uint64_t da = tc::sdesc_sw128(c0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                    const uint64_t db = tc::sdesc_sw128(b0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                    tc::mma_bf16(tS, da, db, idS, k > 0 ? 1u : 0u);
                }
                tc::mma_commit(s_full);
                // Yo(s, .) = C h_in(s, .)^T for all heads at once (the previous
                // item's accumulators have been read)
                if (!pwait(h_full, hph, s_fail)) break;
                hph ^= 1;
                if (!pwait(acc_empty, aph ^ 1, s_fail)) break;
                aph ^= 1;
                tc::tc_fence_after();
                for (int sb = 0; sb < nsub; ++sb)
                    for (int k = 0; k < kN; k += 16) {
                        const uint64_t da = tc::sdesc_sw128(c0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                        const uint64_t db =
                            tc::sdesc_sw128(h0 + sb * HT + (k >> 6) * (HT / 2) + (k & 63) * 2, 16, 1024);
                        tc::mma_bf16(tAcc + sb * HB * 64, da, db, idO, k > 0 ? 1u : 0u);
                    }
                tc::mma_commit(yo_full);
                tc::mma_commit(h_empty);
                tc::mma_commit(tile_empty);  // C and B are not read after this point
                // Y(k) = Yo'(k) + S'(k) X_k
                for (int kh = 0; kh < HB; ++kh, ++nh) {
                    const uint32_t pb = nh & 1, pph = (nh >> 1) & 1;
                    if (!pwait(&x_full[xi], xph, s_fail)) break;
                    if (!pwait(&p_full[pb], pph, s_fail)) break;
                    tc::tc_fence_after();
                    const uint32_t x0 = tc::smem_u32(sX + xi * 16384);
                    for (int k = 0; k < kRows; k += 16) {
                        const uint64_t db = tc::sdesc_sw128(x0 + k * 128, 16384, 1024);
                        tc::mma_bf16_ts(tAcc + kh * 64, tP + pb * 64 + k / 2, db, idY, 1u);
                    }
                    tc::mma_commit(&p_empty[pb]);
                    tc::mma_commit(&x_empty[xi]);
                    tc::mma_commit(&y_full[pb]);
                    if (++xi == kXStages) { xi = 0; xph ^= 1; }
                }
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        // 16 warps: TMEM lane quarter qd = warp % 4 (rows 32 qd .. 32 qd + 31)
        // and column group grp. Per head, warp (qd, grp) owns block J = grp
        // (32 columns j) of S' for its rows when that block lies before the
        // diagonal, columns [8 grp, 8 grp + 8) of the diagonal block J = qd
        // (the costly one, shared by the four warps of the quarter), and the
        // 16 columns p in [16 grp, 16 grp + 16) of the entering-state term and of y.
        const int grp = (warp - kEpiWarp0) >> 2;
        const int qd = warp & 3;
        const int i = qd * 32 + lane;       // tile row
        const uint32_t lq = (uint32_t)(qd * 32) << 16;
        const int J = grp;
        const int sub = (Q < kRows && i >= Q) ? 1 : 0;  // chunk of this row inside the tile
        // blocks of S' that are zero for every head (after this warp's rows, or
        // in the other 64-token chunk of the tile) are written once, here
        const bool zero_blk = J > qd || (Q < kRows && (J >> 1) != (qd >> 1));
        const bool fact_blk = J < qd && !zero_blk;  // before the diagonal, same chunk
        if (zero_blk) {
            uint32_t z[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) z[q] = 0u;
            tc::tmem_st16(tP + lq + J * 16, z);
            tc::tmem_st16(tP + lq + 64 + J * 16, z);
            tc::tmem_st_wait();
        }
        uint32_t sph = 0, yoph = 0, nh = 0, ci = 0;

        for (int64_t u = blockIdx.x; u < n_items; u += gridDim.x, ++ci) {
            int64_t b, tile;
            int hg;
            decode(u, b, tile, hg);
            // the item's cumulative sums and decays, from the scalar warp
            const uint32_t buf = ci & 1;
            pwait(&c_full[buf], (ci >> 1) & 1, s_fail);
            const float *s_cs = s_scal + buf * kScal, *s_dt = s_cs + kHBMax * 128, *s_colf = s_dt + kHBMax * 128;
            const float *s_sc = s_colf + kHBMax * 128, *s_D = s_sc + kHBMax * 128;
            pwait(s_full, sph, s_fail);
            sph ^= 1;
            pwait(yo_full, yoph, s_fail);
            yoph ^= 1;
            tc::tc_fence_after();

            // S'(k) block J into TMEM buffer n & 1, and the rescaled entering-state
            // term Yo'(k) = exp(cs_i - cs_chunk_start) Yo(sub(i), k) into the
            // columns of Yo(0, k), where MMA2 accumulates S'(k) X_k onto it
            auto prepare = [&](int k, uint32_t n) {
                const float *cs_ = s_cs + k * 128, *dt_ = s_dt + k * 128, *cf_ = s_colf + k * 128;
                const float cs_i = cs_[i], Dh = s_D[k], sc = s_sc[k * 128 + i];
                pwait(&p_empty[n & 1], ((n >> 1) & 1) ^ 1, s_fail);
                tc::tc_fence_after();
                {
                    float vd[8];
                    tc::tmem_ld8(tS + lq + qd * 32 + 8 * grp, vd);
                    tc::tmem_ld_wait();
                    // this warp's 8 columns of the diagonal block: exact decay,
                    // causal mask, D on the diagonal
                    uint32_t pk4[4];
#pragma unroll
                    for (int q = 0; q < 8; q += 2) {
                        float f[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int cc = 8 * grp + q + u, jr = qd * 32 + cc;
                            const float e = tc::ex2(fminf(cs_i - cs_[jr], 0.f)) * dt_[jr];
                            f[u] = cc <= lane ? vd[q + u] * e : 0.f;
                            f[u] += cc == lane ? Dh : 0.f;
                        }
                        pk4[q / 2] = pack_bf16x2(f[0], f[1]);
                    }
                    tc::tmem_st4(tP + lq + (n & 1) * 64 + qd * 16 + 4 * grp, pk4);
                }
                if (fact_blk) {
                    // block before this warp's rows: factorised decay
                    float v[32];
                    tc::tmem_ld32(tS + lq + J * 32, v);
                    tc::tmem_ld_wait();
                    const float rf = tc::ex2(cs_i - cs_[J * 32 + 31]);
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] = v[q] * rf * cf_[J * 32 + q];
                    uint32_t pkd[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) pkd[q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
                    tc::tmem_st16(tP + lq + (n & 1) * 64 + J * 16, pkd);
                }
                float ov[16];
                tc::tmem_ld16(tAcc + lq + (sub * HB + k) * 64 + 16 * grp, ov);
                tc::tmem_ld_wait();
                uint32_t r[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) r[q] = __float_as_uint(sc * ov[q]);
                tc::tmem_st16(tAcc + lq + k * 64 + 16 * grp, r);
                tc::tmem_st_wait();
                tc::tc_fence_before();
                if (k == HB - 1) tc::mbar_arrive(s_empty);  // S fully read for this item
                tc::mbar_arrive(&p_full[n & 1]);
            };
            // y(k) = Y(k): this warp's 32 rows x the 16 columns p in [16 grp, 16 grp + 16).
            // Head n completes y_full[n & 1]; the MMA of head n + 2 needs
            // prepare(n + 2), which every thread runs after yout(n), so a
            // barrier is never two phases ahead of its waiter.
            // (warp 2 writes the staged head to y; rows past L are clipped by the TMA store)
            auto yout = [&](int k, uint32_t n) {
                pwait(&y_full[n & 1], (n >> 1) & 1, s_fail);
                tc::tc_fence_after();
                float yv[16];
                tc::tmem_ld16(tAcc + lq + k * 64 + 16 * grp, yv);
                tc::tmem_ld_wait();
                pwait(ys_empty, (n & 1) ^ 1, s_fail);  // the previous head has left sY
                uint8_t *yrow = sY + i * 128;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int q = c * 8;
                    const uint4 pk = make_uint4(pack_bf16x2(yv[q], yv[q + 1]), pack_bf16x2(yv[q + 2], yv[q + 3]),
                                                pack_bf16x2(yv[q + 4], yv[q + 5]), pack_bf16x2(yv[q + 6], yv[q + 7]));
                    *reinterpret_cast<uint4 *>(yrow + (((2 * grp + c) ^ (i & 7)) << 4)) = pk;
                }
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(ys_full);
            };
            // prepare(k) runs one head ahead of yout(k - 1); one call site each
#pragma unroll 1
            for (int k = 0; k <= HB; ++k) {
                if (k < HB) prepare(k, nh + k);
                if (k >= 1) yout(k - 1, nh + k - 1);
            }
            tc::tc_fence_before();
            tc::mbar_arrive(acc_empty);     // every accumulator of this item has been read
            tc::mbar_arrive(&c_empty[buf]);  // and every scalar
            nh += HB;
        }
        tc::tc_fence_before();
    }
    __syncthreads();
    if (tid == 0 && *s_fail) record_failure(a.status);
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// A shared-memory barrier that nothing ever completes, waited on with a poll
// budget: the wait must give up, record SSD_ERR_TIMEOUT and let the kernel exit.
__global__ void selftest_wait_kernel(int *status, int spin_limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t addr = tc::smem_u32(&bar);
        bool done = false;
        for (int k = 0; k < spin_limit && !done; ++k) done = tc::mbar_try_wait(addr, 0);
        if (!done) atomicCAS(status, SSD_OK, SSD_ERR_TIMEOUT);
    }
}

// ------------------------------------------------------- host helpers

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// bf16 tensor map, 128-byte swizzle for 64-column boxes and 64-byte swizzle
// for 32-column boxes; dims/strides innermost first, strides in bytes for
// dims 1..rank-1.
struct MapKey {
    const void *base;
    int rank;
    int f32;  // float32 elements (else bf16)
    uint64_t dims[3], strides[2];
    uint32_t box[3];
    bool operator==(const MapKey &o) const {
        if (base != o.base || rank != o.rank || f32 != o.f32) return false;
        for (int k = 0; k < rank; ++k)
            if (dims[k] != o.dims[k] || box[k] != o.box[k]) return false;
        for (int k = 0; k + 1 < rank; ++k)
            if (strides[k] != o.strides[k]) return false;
        return true;
    }
};

constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapKey g_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_next = 0, g_map_count = 0;

bool make_map(CUtensorMap *out, const MapKey &k) {
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        for (int e = 0; e < g_map_count; ++e)
            if (g_keys[e] == k) {
                *out = g_maps[e];
                return true;
            }
    }
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    for (int e = 0; e < k.rank; ++e) {
        dims[e] = k.dims[e];
        box[e] = k.box[e];
    }
    for (int e = 0; e + 1 < k.rank; ++e) strides[e] = k.strides[e];
    CUtensorMap m;
    const uint32_t row_bytes = k.box[0] * (k.f32 ? 4u : 2u);
    CUresult r = enc(&m, k.f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)k.rank,
                     const_cast<void *>(k.base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     row_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lock(g_map_mu);
    g_keys[g_map_next] = k;
    g_maps[g_map_next] = m;
    g_map_next = (g_map_next + 1) % kMapCache;
    if (g_map_count < kMapCache) ++g_map_count;
    *out = m;
    return true;
}

// (inner, rows, batch) view of a [B, L, inner] bf16 (or float32) tensor, box
// (box_cols, box_rows, 1); the 128-byte swizzle for boxes of 128-byte rows,
// else the 64-byte swizzle
bool map_tokens(CUtensorMap *out, const void *base, int64_t inner, int64_t L, int64_t B, int box_rows,
                int box_cols = 64, bool f32 = false) {
    MapKey k{};
    k.base = base;
    k.rank = 3;
    k.f32 = f32 ? 1 : 0;
    const uint64_t es = f32 ? 4 : 2;
    k.dims[0] = (uint64_t)inner;
    k.dims[1] = (uint64_t)L;
    k.dims[2] = (uint64_t)B;
    k.strides[0] = (uint64_t)inner * es;
    k.strides[1] = (uint64_t)inner * L * es;
    k.box[0] = (uint32_t)box_cols;
    k.box[1] = (uint32_t)box_rows;
    k.box[2] = 1;
    return make_map(out, k);
}

// An integer attribute of the current device, kept per device ordinal (below
// 64; others are queried on every call). Returns `fallback` when the query fails.
int device_attr(cudaDeviceAttr attr, std::atomic<int> (&cache)[64], int fallback) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fallback;
    const bool keep = dev >= 0 && dev < 64;
    if (keep && (v = cache[dev].load(std::memory_order_relaxed)) > 0) return v;
    if (cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess || v <= 0) return fallback;
    if (keep) cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

int device_cc_major() {
    static std::atomic<int> cache[64];
    return device_attr(cudaDevAttrComputeCapabilityMajor, cache, -1);
}

constexpr size_t kSmemPerSM = 233472;  // shared memory of one SM with the maximum carveout (228 KB)
size_t state_smem(int Q, int hb) { return (size_t)state_region(Q, hb) + kStateHBMax * 1024 + 64 + 1024; }
constexpr size_t kScanSmem = 81920 + 5120 + 1024;

size_t scanp_smem(int) { return 65536 + 4 * 16384 + 65536 + 16384 + 2 * (4 * kHBMax * 128 + kHBMax) * 4 + 16 + 512 + 1024; }

int num_sms() { return sm_count(1); }

cudaError_t launch_ex(void (*kern)(TcParams), dim3 grid, size_t smem, cudaStream_t stream, bool pdl,
                      const TcParams &p, int threads = 128) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

bool tma_map_tokens(CUtensorMap *out, const void *base, int64_t inner, int64_t L, int64_t B, int box_rows,
                    int box_cols) {
    return map_tokens(out, base, inner, L, B, box_rows, box_cols);
}

bool tma_map_tokens_f32(CUtensorMap *out, const void *base, int64_t inner, int64_t L, int64_t B, int box_rows,
                        int box_cols) {
    return map_tokens(out, base, inner, L, B, box_rows, box_cols, true);
}

int device_cc_major_cached() { return device_cc_major(); }

int sm_count(int fallback) {
    static std::atomic<int> cache[64];
    return device_attr(cudaDevAttrMultiProcessorCount, cache, fallback);
}

cudaError_t launch_selftest_wait(int *status, int spin_limit, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, spin_limit);
    return cudaGetLastError();
}

bool chunked_tc_supported(const ChunkedArgs &a) {
    if (a.io != IO_BF16 || a.P != kP || a.N != kN) return false;
    if (!(a.Q == 64 || a.Q == 128 || a.Q == 256)) return false;
    if (a.L <= 0 || a.L > 0x7fffffffLL || a.B > 0x7fffffffLL) return false;
    if (a.B * a.nc * a.H * a.P > 0x7fffffffLL) return false;
    if (((a.H * a.P * 2) % 16) != 0 || ((a.G * a.N * 2) % 16) != 0) return false;
    return device_cc_major() == 10;
}

cudaError_t launch_chunked_tc(const ChunkedArgs &a, cudaStream_t stream) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    p.a = a;
    const int R = a.Q < kRows ? a.Q : kRows;
    const int64_t ntiles = (a.L + kRows - 1) / kRows;
    bool ok = true;
    ok &= map_tokens(&p.mx, a.x, a.H * a.P, a.L, a.B, kRows);
    ok &= map_tokens(&p.mb, a.Bm, a.G * a.N, a.L, a.B, kRows);
    ok &= map_tokens(&p.mc, a.Cm, a.G * a.N, a.L, a.B, kRows);
    ok &= map_tokens(&p.my, a.y, a.H * a.P, a.L, a.B, kRows);
    {
        MapKey k{};
        k.base = a.states_bf16;
        k.rank = 2;
        k.dims[0] = kN;
        k.dims[1] = (uint64_t)(a.B * a.nc * a.H * kP);
        k.strides[0] = kN * 2;
        k.box[0] = 64;
        k.box[1] = 64;
        ok &= make_map(&p.mh, k);
    }
    if (!ok) return cudaErrorInvalidValue;
    TcParams ps = p;  // the chunk-state kernel reads Q-row boxes for Q = 64
    if (R != kRows) {
        ok &= map_tokens(&ps.mx, a.x, a.H * a.P, a.L, a.B, R);
        ok &= map_tokens(&ps.mb, a.Bm, a.G * a.N, a.L, a.B, R);
        if (!ok) return cudaErrorInvalidValue;
    }

    static DeviceOnce configured;
    int dev = 0;
    cudaError_t de = cudaSuccess;
    if (configured.pending(&dev, &de)) {
        cudaError_t e = cudaFuncSetAttribute(chunk_state_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)state_smem(256, 4));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chunk_scan_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chunk_scan_tc_persistent, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)scanp_smem(64));
        if (e != cudaSuccess) return e;
        // all of the unified L1 / shared memory as shared memory, so that two
        // chunk-state CTAs fit on an SM from the start
        for (const void *f : {(const void *)chunk_state_tc, (const void *)chunk_scan_tc,
                              (const void *)chunk_scan_tc_persistent}) {
            e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
        }
        configured.done(dev);
    } else if (de != cudaSuccess) {
        return de;
    }
    // persistent chunk scan for Q <= 128: head groups of hb heads sharing a B/C
    // group, at most 4 / (chunks per tile) so that their accumulators fit TMEM.
    // An item costs about one head's epilogue of fixed work plus one per head,
    // and the busiest SM runs ceil(items / SMs) of them: take the hb that
    // minimises that product (ties to the larger hb).
    const int hpg = (int)(a.H / a.G);
    const int hbmax = a.Q >= kRows ? 4 : 2;
    {
        int64_t best = INT64_MAX;
        for (int hb = hbmax; hb >= 1; --hb) {
            if (hpg % hb) continue;
            const int64_t items = a.B * ntiles * (a.H / hb);
            const int64_t cost = (items + num_sms() - 1) / num_sms() * (1 + hb);
            if (cost < best) { best = cost; p.hb = hb; }
        }
    }
    p.nhg = (int)(a.H / p.hb);
    p.n_items = a.B * ntiles * p.nhg;
    const bool staged = a.stage_ev[0] != nullptr;  // per-stage timing: no programmatic overlap
    cudaError_t e = mark_stage(a, 0, stream);
    if (e != cudaSuccess) return e;
    // chunk state: groups of hb <= 8 heads (64 TMEM columns and Q x 128 bytes of
    // x each, at most 4 for 256-token chunks). The busiest SM does
    // ceil(CTAs / SMs) * hb heads' work plus about two heads' worth of load
    // latency per round of co-resident CTAs; `res` CTAs fit on an SM at once
    // (shared memory and TMEM columns), and co-resident CTAs overlap one's
    // loads with another's MMA and stores. Take the hb that minimises that
    // (ties to the larger hb).
    {
        int64_t best = INT64_MAX;
        for (int hb = kStateHBMax; hb >= 1; --hb) {
            if (hpg % hb || (a.Q > 128 && hb > 4)) continue;
            const int64_t ctas = a.B * a.nc * (a.H / hb);
            const int ncol = hb > 4 ? 512 : hb > 2 ? 256 : hb == 2 ? 128 : 64;
            int res = (int)(kSmemPerSM / state_smem(a.Q, hb));
            res = res < 512 / ncol ? res : 512 / ncol;
            res = res < 1 ? 1 : res;
            const int64_t cost = (ctas + num_sms() - 1) / num_sms() * hb +
                                 (ctas + num_sms() * res - 1) / (num_sms() * res) * 2;
            if (cost < best) { best = cost; ps.hb = hb; }
        }
    }
    e = launch_ex(chunk_state_tc, dim3((unsigned)a.nc, (unsigned)(a.H / ps.hb), (unsigned)a.B),
                  state_smem(a.Q, ps.hb), stream, !staged, ps, 256);
    if (e != cudaSuccess) return e;
    if ((e = mark_stage(a, 1, stream)) != cudaSuccess) return e;
    e = launch_state_pass(a, false, true, stream, !staged, /*bf16_in=*/true);
    if (e != cudaSuccess) return e;
    if ((e = mark_stage(a, 2, stream)) != cudaSuccess) return e;
    if (a.Q <= kRows) {
        const int64_t grid = p.n_items < num_sms() ? p.n_items : num_sms();
        e = launch_ex(chunk_scan_tc_persistent, dim3((unsigned)grid), scanp_smem(a.Q), stream, !staged, p,
                      kScanPThreads);
    } else {
        e = launch_ex(chunk_scan_tc, dim3((unsigned)ntiles, (unsigned)a.H, (unsigned)a.B), kScanSmem, stream,
                      !staged, p);
    }
    if (e != cudaSuccess) return e;
    return mark_stage(a, 3, stream);
}

}  // namespace ssd
