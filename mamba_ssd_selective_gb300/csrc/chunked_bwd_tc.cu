// Per-chunk gradients of the chunked SSD scan on the tensor cores: bf16
// inputs, headdim P = 64, d_state N = 128, chunks of Q = 128 tokens.
//
// The algebra is that of chunk_bwd_kernel (chunked_bwd.cu, where it is
// written out): for one (b, chunk, head), with cs the inclusive cumulative
// sum of dt A in the chunk, e = exp(cs), eend = exp(cs_end - cs),
// Ld[t,s] = exp(cs_t - cs_s) for s <= t (else 0), h_in the state entering the
// chunk and Gn the cotangent of the state leaving it,
//
//   M1 = Ld o (C B^T),  M2 = Ld o (dY X^T) o dt_s,  W = M1 o (dY X^T) o dt_s
//   du = M1^T dY + eend o (B Gn^T)          dx  = dt o du + D dY
//   dB = M2^T C + (dt eend) o (X Gn)        dC  = M2 B + e o (dY h_in)
//   d cs_t = sum_{s<t} W[t,s] - sum_{t'>t} W[t',t] + e_t dY_t . (h_in C_t) - r_t,
//   r_s = eend_s dt_s x_s . (Gn B_s), the last token also taking
//   sum_s r_s + exp(cs_end) <Gn, h_in>; da = suffix sums of d cs,
//   ddt = da A + x . du, dA = sum da dt, dD = sum dY . x.
//
// Nine tcgen05 MMA groups in two phases, float32 accumulators in TMEM (512
// columns), operands bf16 in shared memory with the 128-byte swizzle (rows of
// 64 elements; the same tile serves as a K-major or an MN-major operand
// depending on the product):
//   phase 1  BC = B C^T, XY = X dY^T (rows s: the transposed scores),
//            HC = C h_in^T (rows t), GB = B Gn^T (rows s)
//   phase 2  du = M1^T dY, dB = M2^T C + Xs Gn (Xs = x scaled by dt eend per
//            row), dC^T = B^T M2^T and (dY h_in)^T (rows n)
// The epilogues run on the CUDA cores in float32, a thread per TMEM lane and
// column quarter: after phase 1, M1^T and M2^T (bf16, the phase-2 A operands),
// the sums of W along each row of the transposed scores (W's column sums) and
// across the lanes of each warp (its row sums), the per-token dot products;
// after phase 2, the gradients. h_in and Gn enter the products rounded to bf16
// (as do M1 and M2); <Gn, h_in> and every elementwise step stay float32. Sums
// run in a fixed order (no atomics).
#include <cuda.h>

#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "launch.h"
#include "ssd_scan.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

constexpr int kQ = 128, kP = 64, kN = 128, kThreads = 256;
// the per-chunk gradient kernel: 16 warps, warp w on TMEM lane quarter w % 4
// and column quarter w / 4 of every product it reads back
constexpr int kBT = 512;
constexpr uint64_t kWaitNs = 2000000000ull;

struct BwdTcParams {
    BwdArgs a;
    CUtensorMap mx, mdy, mb, mc;  // bf16 inputs, boxes 64 x 128
    CUtensorMap mdx;              // float32 dx, boxes 16 x 32 (64-byte swizzle)
    CUtensorMap mdb, mdc;         // float32 dB and dC parts, boxes 32 x 32 (128-byte swizzle)
    int64_t prefetch_ahead;       // items between a CTA and the one whose tiles it prefetches (0: none)
};

// shared memory (bytes from the 1024-aligned base)
constexpr uint32_t kOffC = 0;        // C  [128 t][128 n]: 2 panels of n (16 KB each)
constexpr uint32_t kOffB = 32768;    // B  [128 s][128 n]
constexpr uint32_t kOffX = 65536;    // x  [128 t][64 p]
constexpr uint32_t kOffY = 81920;    // dy [128 t][64 p]
constexpr uint32_t kOffHin = 98304;  // h_in [64 p][128 n]: 2 panels of n (8 KB each)
constexpr uint32_t kOffGn = 114688;  // Gn   [64 p][128 n]
constexpr uint32_t kOffM1 = 131072;  // M1^T [128 s][128 t]: 2 panels of t
constexpr uint32_t kOffM2 = 163840;  // M2^T [128 s][128 t]
constexpr uint32_t kOffXs = 196608;  // x scaled by dt_s eend_s [128 s][64 p]
constexpr uint32_t kOffV = 212992;   // float32 vectors of kQ values
enum {
    V_CS = 0, V_E, V_EEND, V_DT,
    V_ROW, V_COL = V_ROW + 4, V_HC = V_COL + 4, V_R = V_HC + 4, V_XDU = V_R + 4, V_DD = V_XDU + 4,  // [4] quarters
    kNV = V_DD + 4
};
constexpr uint32_t kOffRed = kOffV + kNV * kQ * 4;               // kBT partial sums + 16 scratch
constexpr uint32_t kOffBar = kOffRed + (kBT + 16) * 4;
constexpr uint32_t kSmemBytes = kOffBar + 8 * 8 + 16 + 1024;
static_assert(kSmemBytes <= 232448, "one CTA per SM with the maximum opt-in shared memory");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
// 16-byte piece `piece` (0..7) of row `row` of a 128-byte-swizzled tile of 128-byte rows
__device__ __forceinline__ uint32_t swz(int row, int piece) { return (uint32_t)(row * 128 + ((piece ^ (row & 7)) << 4)); }

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

__global__ void __launch_bounds__(kBT, 1) chunk_bwd_tc_kernel(const __grid_constant__ BwdTcParams prm) {
    const BwdArgs &a = prm.a;
    const int c = blockIdx.x, h = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t L = a.L, H = a.H, G = a.G, nc = a.nc;
    const int g = (int)(h / (H / G));
    const int64_t t0 = (int64_t)c * kQ;
    const int Qv = (int)imin<int64_t>(kQ, L - t0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, cq = warp >> 2;  // TMEM lane quarter, column quarter
    const uint32_t lq = (uint32_t)(qd * 32) << 16;
    const int row = qd * 32 + lane;  // this thread's TMEM lane (t, s or n)

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *V = reinterpret_cast<float *>(sm + kOffV);
    float *red = reinterpret_cast<float *>(sm + kOffRed), *scratch = red + kBT;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 8);
    volatile int *s_fail = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *v_cs = V + V_CS * kQ, *v_e = V + V_E * kQ, *v_eend = V + V_EEND * kQ, *v_dt = V + V_DT * kQ;
    // sum of the four column quarters' partials of vector k at index i, in a fixed order
    auto q4sum = [&](int k, int i) {
        return (V[k * kQ + i] + V[(k + 1) * kQ + i]) + (V[(k + 2) * kQ + i] + V[(k + 3) * kQ + i]);
    };

    if (tid == 0) {
        for (int k = 0; k < 7; ++k) tc::mbar_init(bars + k, 1);
        tc::fence_mbar_init();
        *s_fail = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t T0 = tmem, T1 = tmem + 128, T2 = tmem + 256, T3 = tmem + 320, T4 = tmem + 384;

    // x, dy, B, C of the chunk by TMA (rows past L read as zero) on one
    // barrier; h_in and Gn (float32 [p][n], contiguous per (b, chunk, head)) by
    // bulk copies into the M1^T / M2^T regions, which epilogue 1 fills later, on
    // another. The call's inputs are read before the wait for the state passes
    // (this kernel is their programmatic dependent), the states after it; only
    // the thread that issues the copies waits.
    const int64_t so = ((b * nc + c) * H + h) * (int64_t)kP * kN;
    if (tid == 0) {
        tc::mbar_arrive_expect_tx(&bars[0], 6u * 16384u);
        tc::tma_load_3d(sm + kOffX, &prm.mx, &bars[0], h * kP, (int)t0, (int)b);
        tc::tma_load_3d(sm + kOffY, &prm.mdy, &bars[0], h * kP, (int)t0, (int)b);
        tc::tma_load_3d(sm + kOffB, &prm.mb, &bars[0], g * kN, (int)t0, (int)b);
        tc::tma_load_3d(sm + kOffB + 16384, &prm.mb, &bars[0], g * kN + 64, (int)t0, (int)b);
        tc::tma_load_3d(sm + kOffC, &prm.mc, &bars[0], g * kN, (int)t0, (int)b);
        tc::tma_load_3d(sm + kOffC + 16384, &prm.mc, &bars[0], g * kN + 64, (int)t0, (int)b);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        tc::mbar_arrive_expect_tx(&bars[6], 2u * 32768u);
        tc::bulk_load(sm + kOffM1, a.hin + so, (uint32_t)(kP * kN * 4), &bars[6]);
        tc::bulk_load(sm + kOffM2, a.adj + so, (uint32_t)(kP * kN * 4), &bars[6]);
        // into L2 ahead of time: the per-head tiles of the item one CTA per SM
        // later in launch order, which starts about when this one ends
        const int64_t nxt = ((b * H + h) * nc + c) + prm.prefetch_ahead;
        if (prm.prefetch_ahead > 0 && nxt < nc * H * a.B) {
            const int c_ = (int)(nxt % nc), h_ = (int)((nxt / nc) % H);
            const int64_t b_ = nxt / (nc * H);
            const int64_t so_ = ((b_ * nc + c_) * H + h_) * (int64_t)kP * kN;
            tc::prefetch_l2_3d(&prm.mx, h_ * kP, c_ * kQ, (int)b_);
            tc::prefetch_l2_3d(&prm.mdy, h_ * kP, c_ * kQ, (int)b_);
            tc::prefetch_l2(a.hin + so_, (uint32_t)(kP * kN * 4));
            tc::prefetch_l2(a.adj + so_, (uint32_t)(kP * kN * 4));
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // dt and its cumulative sum over the chunk (padded tokens carry dt = 0)
    const __nv_bfloat16 *dtp = static_cast<const __nv_bfloat16 *>(a.dt);
    const float dv = tid < Qv ? __bfloat162float(dtp[(b * L + t0 + tid) * H + h]) : 0.f;
    block_inclusive_scan_256(dv * a.A[h], kQ, v_cs, scratch);
    const float cs_end = v_cs[kQ - 1];
    if (tid < kQ) {
        v_dt[tid] = dv;
        v_e[tid] = expf(v_cs[tid]);
        v_eend[tid] = expf(cs_end - v_cs[tid]);
    }

    const uint32_t c0 = tc::smem_u32(sm + kOffC), b0 = tc::smem_u32(sm + kOffB);
    const uint32_t x0 = tc::smem_u32(sm + kOffX), y0 = tc::smem_u32(sm + kOffY);
    const uint32_t hn0 = tc::smem_u32(sm + kOffHin), gn0 = tc::smem_u32(sm + kOffGn);
    const uint32_t m10 = tc::smem_u32(sm + kOffM1), m20 = tc::smem_u32(sm + kOffM2), xs0 = tc::smem_u32(sm + kOffXs);
    // K-major tile with panels of 64 along K (panel bytes `pb`), K offset k
    auto kmaj = [](uint32_t base, int k, uint32_t pb) {
        return tc::sdesc_sw128(base + (k >> 6) * pb + (k & 63) * 2, 16, 1024);
    };
    // MN-major tile: K offset k in rows of 128 bytes, panels of 64 along M/N `pb` apart
    auto mnmaj = [](uint32_t base, int k, uint32_t pb) { return tc::sdesc_sw128(base + k * 128, pb, 1024); };
    const uint32_t id128 = tc::idesc_bf16(128, 128, false, false), id64 = tc::idesc_bf16(128, 64, false, false);

    // ---- phase 1a: BC = B C^T, XY = X dY^T (rows s: the transposed scores), as
    // soon as the tiles are in, while the states are rounded below
    pwait(&bars[0], 0, s_fail);
    if (tid == 0 && !*s_fail) {
        tc::tc_fence_after();
        for (int k = 0; k < kN; k += 16) tc::mma_bf16(T0, kmaj(b0, k, 16384), kmaj(c0, k, 16384), id128, k > 0);
        for (int k = 0; k < kP; k += 16) tc::mma_bf16(T1, kmaj(x0, k, 0), kmaj(y0, k, 0), id128, k > 0);
        tc::mma_commit(&bars[1]);
    }
    pwait(&bars[6], 0, s_fail);
    __syncthreads();
    // h_in and Gn into bf16 tiles (rows p, panels of 64 n), 8 n per 16-byte
    // piece; <Gn, h_in> in float32 on the way
    {
        float q = 0.f;
        for (int e = tid; e < kP * kN / 8; e += kBT) {
            const int p = e >> 4, n8 = e & 15;
            const float4 *hp = reinterpret_cast<const float4 *>(sm + kOffM1 + e * 32);
            const float4 *gp = reinterpret_cast<const float4 *>(sm + kOffM2 + e * 32);
            const float4 h0 = hp[0], h1 = hp[1], g0 = gp[0], g1 = gp[1];
            q = fmaf(g0.x, h0.x, q); q = fmaf(g0.y, h0.y, q); q = fmaf(g0.z, h0.z, q); q = fmaf(g0.w, h0.w, q);
            q = fmaf(g1.x, h1.x, q); q = fmaf(g1.y, h1.y, q); q = fmaf(g1.z, h1.z, q); q = fmaf(g1.w, h1.w, q);
            const uint32_t off = (uint32_t)(n8 >> 3) * 8192u + swz(p, n8 & 7);
            *reinterpret_cast<uint4 *>(sm + kOffHin + off) = make_uint4(
                pack_bf16x2(h0.x, h0.y), pack_bf16x2(h0.z, h0.w), pack_bf16x2(h1.x, h1.y), pack_bf16x2(h1.z, h1.w));
            *reinterpret_cast<uint4 *>(sm + kOffGn + off) = make_uint4(
                pack_bf16x2(g0.x, g0.y), pack_bf16x2(g0.z, g0.w), pack_bf16x2(g1.x, g1.y), pack_bf16x2(g1.z, g1.w));
        }
        red[tid] = q;
    }
    // Xs: x scaled by dt_s eend_s (a 16-byte piece per step; the swizzle only
    // permutes pieces inside a row, so the row of piece e is e / 8)
    for (int e = tid; e < kQ * 8; e += kBT) {
        const int s = e >> 3;
        const float f = v_dt[s] * v_eend[s];
        float xv[8];
        unpack8(*reinterpret_cast<const uint4 *>(sm + kOffX + e * 16), xv);
        *reinterpret_cast<uint4 *>(sm + kOffXs + e * 16) =
            make_uint4(pack_bf16x2(f * xv[0], f * xv[1]), pack_bf16x2(f * xv[2], f * xv[3]),
                       pack_bf16x2(f * xv[4], f * xv[5]), pack_bf16x2(f * xv[6], f * xv[7]));
    }
    tc::fence_proxy_async_smem();  // h_in, Gn, Xs written here are read by the MMAs
    tc::tc_fence_before();
    __syncthreads();

    // ---- phase 1b: HC = C h_in^T (rows t), GB = B Gn^T (rows s)
    if (tid == 0 && !*s_fail) {
        tc::tc_fence_after();
        for (int k = 0; k < kN; k += 16) tc::mma_bf16(T2, kmaj(c0, k, 16384), kmaj(hn0, k, 8192), id64, k > 0);
        for (int k = 0; k < kN; k += 16) tc::mma_bf16(T3, kmaj(b0, k, 16384), kmaj(gn0, k, 8192), id64, k > 0);
        tc::mma_commit(&bars[3]);
    }
    pwait(&bars[1], 0, s_fail);
    tc::tc_fence_after();
    // epilogue B (lanes s, this quarter's 32 t): M1^T and M2^T rows (bf16), W
    // (t > s) summed along the row (its column sums) and across the warp's 32
    // lanes (its row sums, a partial per lane quarter), x_s . GB_s over this
    // quarter's 16 p; and, for the token t of this thread's TMEM lane, dY_t . HC_t
    // over the same 16 p
    {
        const int s = row, tb = 32 * cq;
        const float cs_s = v_cs[s], dts = v_dt[s];
        float bc[32], xy[32];
        tc::tmem_ld32(T0 + lq + tb, bc);
        tc::tmem_ld32(T1 + lq + tb, xy);
        tc::tmem_ld_wait();
        float cl = 0.f;
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
            uint32_t m1p[4], m2p[4];
#pragma unroll
            for (int u = 0; u < 8; u += 2) {
                float m1v[2], m2v[2];
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int j = 8 * pc + u + e2, t = tb + j;
                    const float ld = s <= t ? expf(v_cs[t] - cs_s) : 0.f;
                    const float m1 = ld * bc[j];
                    const float w = t > s ? m1 * dts * xy[j] : 0.f;
                    cl += w;
                    m1v[e2] = m1;
                    m2v[e2] = ld * dts * xy[j];
                    bc[j] = w;  // W[t, s], summed across the lanes below
                }
                m1p[u / 2] = pack_bf16x2(m1v[0], m1v[1]);
                m2p[u / 2] = pack_bf16x2(m2v[0], m2v[1]);
            }
            const uint32_t off = (uint32_t)(tb >> 6) * 16384u + swz(s, ((tb & 63) >> 3) + pc);
            *reinterpret_cast<uint4 *>(sm + kOffM1 + off) = make_uint4(m1p[0], m1p[1], m1p[2], m1p[3]);
            *reinterpret_cast<uint4 *>(sm + kOffM2 + off) = make_uint4(m2p[0], m2p[1], m2p[2], m2p[3]);
        }
        V[(V_COL + cq) * kQ + s] = cl;
        // reduce-scatter over the 32 lanes: halve the live columns each step,
        // keeping the half this lane's bit selects; lane j ends with the sum
        // of column j over the warp's lanes
#pragma unroll
        for (int k = 16; k >= 1; k >>= 1) {
            const bool up = (lane & k) != 0;
#pragma unroll
            for (int i = 0; i < k; ++i) {
                const float send = up ? bc[i] : bc[i + k];
                const float keep = up ? bc[i + k] : bc[i];
                bc[i] = keep + __shfl_xor_sync(0xffffffffu, send, k);
            }
        }
        V[(V_ROW + qd) * kQ + tb + lane] = bc[0];
        pwait(&bars[3], 0, s_fail);
        tc::tc_fence_after();
        float gb[16], hc[16];
        tc::tmem_ld16(T3 + lq + 16 * cq, gb);
        tc::tmem_ld16(T2 + lq + 16 * cq, hc);
        tc::tmem_ld_wait();
        float rr = 0.f, acc = 0.f;
#pragma unroll
        for (int pc = 0; pc < 2; ++pc) {
            float xv[8], dy[8];
            unpack8(*reinterpret_cast<const uint4 *>(sm + kOffX + swz(s, 2 * cq + pc)), xv);
            unpack8(*reinterpret_cast<const uint4 *>(sm + kOffY + swz(s, 2 * cq + pc)), dy);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                rr = fmaf(xv[i], gb[8 * pc + i], rr);
                acc = fmaf(dy[i], hc[8 * pc + i], acc);
            }
        }
        V[(V_R + cq) * kQ + s] = rr;
        V[(V_HC + cq) * kQ + s] = acc;
    }
    tc::fence_proxy_async_smem();  // M1^T, M2^T are read by the phase-2 MMAs
    tc::tc_fence_before();
    __syncthreads();

    // ---- phase 2: du, dB, dC^T, (dY h_in)^T
    if (tid == 0 && !*s_fail) {
        tc::tc_fence_after();
        // du = M1^T dY: A rows s (K = t), B = dy as MN-major (N = p, K = t)
        const uint32_t idu = tc::idesc_bf16(128, 64, false, true);
        for (int k = 0; k < kQ; k += 16) tc::mma_bf16(T2, kmaj(m10, k, 16384), mnmaj(y0, k, 16384), idu, k > 0);
        tc::mma_commit(&bars[4]);  // du: dx is formed while the rest run
        // dB = M2^T C + Xs Gn: B operands MN-major (N = n)
        const uint32_t idb = tc::idesc_bf16(128, 128, false, true);
        for (int k = 0; k < kQ; k += 16) tc::mma_bf16(T0, kmaj(m20, k, 16384), mnmaj(c0, k, 16384), idb, k > 0);
        for (int k = 0; k < kP; k += 16) tc::mma_bf16(T0, kmaj(xs0, k, 0), mnmaj(gn0, k, 8192), idb, 1u);
        tc::mma_commit(&bars[5]);  // dB: C, Gn, Xs and M1 are free from here
        // dC1^T = B^T M2^T: rows n (A = B as MN-major, M = n), N = t (M2^T as MN-major)
        const uint32_t idc = tc::idesc_bf16(128, 128, true, true);
        for (int k = 0; k < kQ; k += 16) tc::mma_bf16(T4, mnmaj(b0, k, 16384), mnmaj(m20, k, 16384), idc, k > 0);
        // (dY h_in)^T = h_in^T dY^T: rows n (A = h_in as MN-major), N = t (dy K-major, K = p)
        const uint32_t idy = tc::idesc_bf16(128, 128, true, false);
        for (int k = 0; k < kP; k += 16) tc::mma_bf16(T1, mnmaj(hn0, k, 8192), kmaj(y0, k, 0), idy, k > 0);
        tc::mma_commit(&bars[2]);
    }
    pwait(&bars[4], 0, s_fail);
    tc::tc_fence_after();
    const float Dh = a.D ? a.D[h] : 0.f;
    // epilogue after phase 2: du, dx and x . du (lanes s, this quarter's 16 p); dB (lanes
    // s, this quarter's 32 n); dC (lanes n, this quarter's 32 t); dY . x. Each
    // warp stages its three float32 boxes (dx 32 x 16 with the 64-byte swizzle,
    // dB and dC 32 x 32 with the 128-byte swizzle) in shared memory that the
    // phase-2 MMAs still running no longer read -- dx in Gn / Xs and dB in C / M1
    // once du and dB are done, dC in B / M2 once every product is -- and
    // stores them by TMA; rows past L are clipped by the tensor maps.
    uint8_t *stg_dx = sm + (warp < 8 ? kOffGn + warp * 2048 : kOffXs + (warp - 8) * 2048);
    uint8_t *stg_db = sm + (warp < 8 ? kOffC + warp * 4096 : kOffM1 + (warp - 8) * 4096);
    uint8_t *stg_dc = sm + (warp < 8 ? kOffB + warp * 4096 : kOffM2 + (warp - 8) * 4096);
    {
        const int s = row;
        float du[16], gb[16];
        tc::tmem_ld16(T2 + lq + 16 * cq, du);
        tc::tmem_ld16(T3 + lq + 16 * cq, gb);
        tc::tmem_ld_wait();
        const float ee = v_eend[s], dts = v_dt[s];
        float xd = 0.f, yxd = 0.f, dxv[16];
#pragma unroll
        for (int pc = 0; pc < 2; ++pc) {
            float xv[8], yv[8];
            unpack8(*reinterpret_cast<const uint4 *>(sm + kOffX + swz(s, 2 * cq + pc)), xv);
            unpack8(*reinterpret_cast<const uint4 *>(sm + kOffY + swz(s, 2 * cq + pc)), yv);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float u = fmaf(ee, gb[8 * pc + i], du[8 * pc + i]);
                xd = fmaf(xv[i], u, xd);
                yxd = fmaf(yv[i], xv[i], yxd);
                dxv[8 * pc + i] = fmaf(dts, u, Dh * yv[i]);
            }
        }
        V[(V_XDU + cq) * kQ + s] = xd;
        V[(V_DD + cq) * kQ + s] = yxd;
        pwait(&bars[5], 0, s_fail);
        tc::tc_fence_after();
        // dx box: rows of 64 bytes, 16-byte piece k of row r at k ^ ((r >> 1) & 3)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<float4 *>(stg_dx + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                make_float4(dxv[4 * k], dxv[4 * k + 1], dxv[4 * k + 2], dxv[4 * k + 3]);
        {
            float v[32];
            tc::tmem_ld32(T0 + lq + 32 * cq, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 8; ++k)
                *reinterpret_cast<float4 *>(stg_db + swz(lane, k)) =
                    make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && qd * 32 < Qv) {
            const int rs = (int)t0 + qd * 32;
            tc::tma_store_3d(&prm.mdx, stg_dx, h * kP + 16 * cq, rs, (int)b);
            tc::tma_store_3d(&prm.mdb, stg_db, h * kN + 32 * cq, rs, (int)b);
            tc::bulk_commit();
        }
        pwait(&bars[2], 0, s_fail);
        tc::tc_fence_after();
        {
            const int tb = 32 * cq;
            float d1[32], yh[32];
            tc::tmem_ld32(T4 + lq + tb, d1);
            tc::tmem_ld32(T1 + lq + tb, yh);
            tc::tmem_ld_wait();
            uint8_t *box = stg_dc + (lane & 3) * 4;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                *reinterpret_cast<float *>(box + u * 128 + (((lane >> 2) ^ (u & 7)) << 4)) =
                    fmaf(v_e[tb + u], yh[u], d1[u]);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (32 * cq < Qv) tc::tma_store_3d(&prm.mdc, stg_dc, h * kN + 32 * qd, (int)t0 + 32 * cq, (int)b);
            tc::bulk_commit();
        }
    }
    tc::tc_fence_before();
    __syncthreads();

    // ---- d cs, da (suffix sums), ddt, dA and dD parts: tokens on warps 0-3
    float suf = 0.f;
    if (tid < kQ) {
        const int t = tid;
        const float q = (red[4 * t] + red[4 * t + 1]) + (red[4 * t + 2] + red[4 * t + 3]);
        const float rv = t < Qv ? v_eend[t] * v_dt[t] * q4sum(V_R, t) : 0.f;
        const float qs = warp_sum(q), rs = warp_sum(rv);
        if (lane == 0) {
            scratch[warp] = qs;
            scratch[4 + warp] = rs;
        }
        V[V_R * kQ + t] = rv;  // r_t replaces this thread's own partials, read just above
    }
    __syncthreads();
    if (tid < kQ) {
        const int t = tid;
        const float q = (scratch[0] + scratch[1]) + (scratch[2] + scratch[3]);
        const float rsum = (scratch[4] + scratch[5]) + (scratch[6] + scratch[7]);
        float dcs = 0.f;
        if (t < Qv) dcs = q4sum(V_ROW, t) - q4sum(V_COL, t) + v_e[t] * q4sum(V_HC, t) - V[V_R * kQ + t];
        if (t == Qv - 1) dcs += rsum + expf(cs_end) * q;
        suf = dcs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_down_sync(0xffffffffu, suf, o);
            if (lane + o < 32) suf += u;
        }
        if (lane == 0) scratch[8 + warp] = suf;  // each warp's total
    }
    __syncthreads();
    if (tid < kQ) {
        const int t = tid;
        float later = 0.f;
        for (int w = warp + 1; w < 4; ++w) later += scratch[8 + w];
        const float da = suf + later;
        const float xdu = q4sum(V_XDU, t);
        if (t < Qv) a.ddt[(b * L + t0 + t) * H + h] = fmaf(da, a.A[h], xdu);
        float pa = t < Qv ? da * v_dt[t] : 0.f, pd = t < Qv ? q4sum(V_DD, t) : 0.f;
        pa = warp_sum(pa);
        pd = warp_sum(pd);
        if (lane == 0) {
            red[kBT - 8 + warp] = pa;
            red[kBT - 4 + warp] = pd;
        }
    }
    __syncthreads();
    if (tid == 0) {
        a.dA_part[(b * nc + c) * H + h] = (red[kBT - 8] + red[kBT - 7]) + (red[kBT - 6] + red[kBT - 5]);
        a.dD_part[(b * nc + c) * H + h] = (red[kBT - 4] + red[kBT - 3]) + (red[kBT - 2] + red[kBT - 1]);
        if (*s_fail && a.status) atomicCAS(a.status, SSD_OK, SSD_ERR_TIMEOUT);
    }
    if (lane == 0) tc::bulk_wait_read_all();  // this warp's staged boxes have been read
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// Float32 chunk states on the tensor cores, for the backward's chunks of 128
// tokens (bf16, P 64, N 128), one CTA per (b, chunk, one or two heads) and
// direction (blockIdx.z < B: forward, else adjoint for batch z - B):
//   forward  S_c[p,n]    = sum_t exp(cs_end - cs_t) dt_t x[t,p] B[t,n]
//            (and the chunk decay exp(cs_end); block (0, 0, 0) also clears
//            the status word, this being the call's first kernel)
//   adjoint  Sbar_c[p,n] = sum_t exp(cs_t) dy[t,p] C[t,n]
// as one MMA chain: rows n (B or C as the MN-major A operand), columns p (x
// or dy, its rows scaled in place by the weights, the MN-major B operand),
// K = t; the weights and the scaled operand are rounded to bf16 for the MMA.
struct StateTcParams {
    CUtensorMap mb, mx;   // forward: B as (G*N, L, B), x as (H*P, L, B); boxes 64 x 128
    CUtensorMap mc, mdy;  // adjoint: C, dy
    const __nv_bfloat16 *dt;
    const float *A;
    float *states, *adj;  // [B, nc, H, P, N]
    float *chunk_sum;     // [B, H, nc]
    int *status;
    int64_t B, L, H, G, nc;
};
// Shared memory of the chunk-state kernel for HB heads per CTA: the B or C
// tile, HB x / dy tiles, per head the cumulative sums and the weights.
template <int HB> struct StSmem {
    static constexpr uint32_t A = 0, X = 32768, V = X + HB * 16384;
    static constexpr uint32_t Bar = V + (HB * 2 * kQ + 16) * 4;
    static constexpr uint32_t total = Bar + 2 * 8 + 16 + 1024;
};

// HB heads per CTA (2 when a group's heads pair up): they share the B or C
// tile, and one MMA chain of N = 64 HB covers both.
template <int HB>
__global__ void __launch_bounds__(kThreads) chunk_states_tc(const __grid_constant__ StateTcParams p) {
    using SM = StSmem<HB>;
    const bool adj = blockIdx.z >= p.B;
    const int c = blockIdx.x, h0 = blockIdx.y * HB;
    const int64_t b = adj ? blockIdx.z - p.B : blockIdx.z;
    const int64_t L = p.L, H = p.H;
    const int g = (int)(h0 / (H / p.G));
    const int64_t t0 = (int64_t)c * kQ;
    const int Qv = (int)imin<int64_t>(kQ, L - t0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *vec = reinterpret_cast<float *>(sm + SM::V), *scratch = vec + HB * 2 * kQ;  // head k: cs, then w
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM::Bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
    volatile int *s_fail = reinterpret_cast<volatile int *>(tmem_slot + 1);
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && p.status) *p.status = SSD_OK;
    if (tid == 0) {
        tc::mbar_init(bars, 1);
        tc::mbar_init(bars + 1, 1);
        tc::fence_mbar_init();
        *s_fail = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, 64 * HB);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) {
        const CUtensorMap *ma = adj ? &p.mc : &p.mb, *mx = adj ? &p.mdy : &p.mx;
        tc::mbar_arrive_expect_tx(&bars[0], (2u + HB) * 16384u);
        tc::tma_load_3d(sm + SM::A, ma, &bars[0], g * kN, (int)t0, (int)b);
        tc::tma_load_3d(sm + SM::A + 16384, ma, &bars[0], g * kN + 64, (int)t0, (int)b);
#pragma unroll
        for (int k = 0; k < HB; ++k)
            tc::tma_load_3d(sm + SM::X + k * 16384, mx, &bars[0], (h0 + k) * kP, (int)t0, (int)b);
    }
#pragma unroll
    for (int k = 0; k < HB; ++k) {
        float *v_cs = vec + k * 2 * kQ, *v_w = v_cs + kQ;
        const float dv = tid < Qv ? __bfloat162float(p.dt[(b * L + t0 + tid) * H + h0 + k]) : 0.f;
        block_inclusive_scan_256(dv * p.A[h0 + k], kQ, v_cs, scratch);
        const float cs_end = v_cs[kQ - 1];
        if (tid < kQ) v_w[tid] = adj ? expf(v_cs[tid]) : expf(cs_end - v_cs[tid]) * dv;
        if (!adj && tid == 0) p.chunk_sum[(b * H + h0 + k) * p.nc + c] = expf(cs_end);
    }
    pwait(&bars[0], 0, s_fail);
    __syncthreads();
    for (int e = tid; e < HB * kQ * 8; e += kThreads) {  // rows of x / dy scaled by their head's weights
        const int k = e / (kQ * 8);
        const float f = vec[k * 2 * kQ + kQ + ((e % (kQ * 8)) >> 3)];
        float xv[8];
        unpack8(*reinterpret_cast<const uint4 *>(sm + SM::X + e * 16), xv);
        *reinterpret_cast<uint4 *>(sm + SM::X + e * 16) =
            make_uint4(pack_bf16x2(f * xv[0], f * xv[1]), pack_bf16x2(f * xv[2], f * xv[3]),
                       pack_bf16x2(f * xv[4], f * xv[5]), pack_bf16x2(f * xv[6], f * xv[7]));
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0 && !*s_fail) {
        tc::tc_fence_after();
        const uint32_t a0 = tc::smem_u32(sm + SM::A), x0 = tc::smem_u32(sm + SM::X);
        const uint32_t id = tc::idesc_bf16(128, 64 * HB, true, true);
        for (int k = 0; k < kQ; k += 16)
            tc::mma_bf16(tmem, tc::sdesc_sw128(a0 + k * 128, 16384, 1024), tc::sdesc_sw128(x0 + k * 128, 16384, 1024),
                         id, k > 0);
        tc::mma_commit(&bars[1]);
    }
    pwait(&bars[1], 0, s_fail);
    tc::tc_fence_after();
    {
        // lanes n, columns (head, p): for each column the warp's 32 lanes store 32 consecutive n
        const int qd = warp & 3, hf = warp >> 2, n = qd * 32 + lane;
#pragma unroll 1
        for (int j = 0; j < HB; ++j) {
            const int col0 = 32 * HB * hf + 32 * j, k = col0 / kP, p0 = col0 % kP;
            float v[32];
            tc::tmem_ld32(tmem + ((uint32_t)(qd * 32) << 16) + col0, v);
            tc::tmem_ld_wait();
            float *o = (adj ? p.adj : p.states) + ((b * p.nc + c) * H + h0 + k) * (int64_t)kP * kN + n;
#pragma unroll
            for (int q = 0; q < 32; ++q) o[(int64_t)(p0 + q) * kN] = v[q];
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0 && *s_fail && p.status) atomicCAS(p.status, SSD_OK, SSD_ERR_TIMEOUT);
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 64 * HB);
    }
}

// Both passes over the chunks of one (b, h), four state elements per thread
// (blockIdx.z < B: forward, else adjoint for batch z - B):
//   forward  states[c] <- h entering chunk c (init, or zero, before chunk 0),
//            h <- exp(cs_end(c)) h + S_c
//   adjoint  adj[c] <- cotangent of the state leaving chunk c (dfinal, or
//            zero, after the last), g <- exp(cs_end(c)) g + Sbar_c; dinit = g
// The values of kPF chunks are loaded before the chain consumes them.
struct PassParams {
    float *states, *adj, *dinit;
    const float *init, *dfinal, *chunk_sum;
    int64_t B, H, PN, nc;
};
constexpr int kPF = 16;

constexpr int kPassThreads = 128;  // smaller blocks: the passes' grid fills the GPU in one wave at small sizes

__global__ void __launch_bounds__(kPassThreads) bwd_state_passes(const __grid_constant__ PassParams p) {
    // the gradient kernel (a programmatic dependent of this one) may be
    // scheduled now; it waits for this grid before it reads the states
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const bool adj = blockIdx.z >= p.B;
    const int64_t b = adj ? blockIdx.z - p.B : blockIdx.z;
    const int64_t PN = p.PN, H = p.H, nc = p.nc;
    const int64_t e = ((int64_t)blockIdx.x * kPassThreads + threadIdx.x) * 4;
    const int h = blockIdx.y;
    if (e >= PN) return;
    const float *src0 = adj ? p.dfinal : p.init;
    float4 carry = src0 ? *reinterpret_cast<const float4 *>(src0 + (b * H + h) * PN + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    float *buf = adj ? p.adj : p.states;
    const float *dec = p.chunk_sum + (b * H + h) * nc;
    for (int64_t k0 = 0; k0 < nc; k0 += kPF) {
        float4 v[kPF];
        float dc[kPF];
#pragma unroll
        for (int u = 0; u < kPF; ++u)
            if (k0 + u < nc) {
                const int64_t c = adj ? nc - 1 - (k0 + u) : k0 + u;
                v[u] = *reinterpret_cast<const float4 *>(buf + ((b * nc + c) * H + h) * PN + e);
                dc[u] = dec[c];
            }
#pragma unroll
        for (int u = 0; u < kPF; ++u)
            if (k0 + u < nc) {
                const int64_t c = adj ? nc - 1 - (k0 + u) : k0 + u;
                *reinterpret_cast<float4 *>(buf + ((b * nc + c) * H + h) * PN + e) = carry;
                carry.x = fmaf(dc[u], carry.x, v[u].x);
                carry.y = fmaf(dc[u], carry.y, v[u].y);
                carry.z = fmaf(dc[u], carry.z, v[u].z);
                carry.w = fmaf(dc[u], carry.w, v[u].w);
            }
    }
    if (adj && p.dinit) *reinterpret_cast<float4 *>(p.dinit + (b * H + h) * PN + e) = carry;
}

}  // namespace

bool chunk_bwd_tc_supported(int io, int64_t P, int64_t N) {
    return io == IO_BF16 && P == kP && N == kN && device_cc_major_cached() == 10;
}

cudaError_t launch_chunk_bwd_tc(const BwdArgs &a, cudaStream_t stream) {
    if (a.Q != kQ || a.P != kP || a.N != kN || a.io != IO_BF16) return cudaErrorInvalidValue;
    BwdTcParams p;
    memset(&p, 0, sizeof(p));
    p.a = a;
    bool ok = true;
    ok &= tma_map_tokens(&p.mx, a.x, a.H * a.P, a.L, a.B, kQ);
    ok &= tma_map_tokens(&p.mdy, a.dy, a.H * a.P, a.L, a.B, kQ);
    ok &= tma_map_tokens(&p.mb, a.Bm, a.G * a.N, a.L, a.B, kQ);
    ok &= tma_map_tokens(&p.mc, a.Cm, a.G * a.N, a.L, a.B, kQ);
    ok &= tma_map_tokens_f32(&p.mdx, a.dx, a.H * a.P, a.L, a.B, 32, 16);
    ok &= tma_map_tokens_f32(&p.mdb, a.dB_part, a.H * a.N, a.L, a.B, 32);
    ok &= tma_map_tokens_f32(&p.mdc, a.dC_part, a.H * a.N, a.L, a.B, 32);
    if (!ok) return cudaErrorInvalidValue;
    // one CTA per SM: prefetch one SM count ahead, on grids of four waves or
    // more (measured: B4 L2048 H80 734 -> 725 us; at 2.5 waves, B1 L2048 H24,
    // it cost ~1 us)
    const int64_t sms = sm_count(152);
    p.prefetch_ahead = a.nc * a.H * a.B >= 4 * sms ? sms : 0;
    static DeviceOnce configured;
    int dev = 0;
    cudaError_t e = cudaSuccess;
    if (configured.pending(&dev, &e)) {
        e = cudaFuncSetAttribute(chunk_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.done(dev);
    } else if (e != cudaSuccess) {
        return e;
    }
    // a programmatic dependent of the state passes (measured: 85 -> 81 us at
    // B1 L2048 H24, unchanged at B4 L2048 H80; programmatic launches of the
    // passes or of the reduce were slower on large grids)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.nc, (unsigned)a.H, (unsigned)a.B);
    cfg.blockDim = dim3(kBT);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chunk_bwd_tc_kernel, p);
}

}  // namespace ssd

namespace ssd {

cudaError_t launch_bwd_states_tc(const BwdArgs &a, cudaStream_t stream) {
    if (a.Q != kQ || a.P != kP || a.N != kN || a.io != IO_BF16) return cudaErrorInvalidValue;
    StateTcParams p;
    memset(&p, 0, sizeof(p));
    bool ok = true;
    ok &= tma_map_tokens(&p.mb, a.Bm, a.G * a.N, a.L, a.B, kQ);
    ok &= tma_map_tokens(&p.mx, a.x, a.H * a.P, a.L, a.B, kQ);
    ok &= tma_map_tokens(&p.mc, a.Cm, a.G * a.N, a.L, a.B, kQ);
    ok &= tma_map_tokens(&p.mdy, a.dy, a.H * a.P, a.L, a.B, kQ);
    if (!ok) return cudaErrorInvalidValue;
    p.dt = static_cast<const __nv_bfloat16 *>(a.dt);
    p.A = a.A;
    p.states = a.hin;
    p.adj = a.adj;
    p.chunk_sum = const_cast<float *>(a.chunk_sum);
    p.status = a.status;
    p.B = a.B;
    p.L = a.L;
    p.H = a.H;
    p.G = a.G;
    p.nc = a.nc;
    // two heads per CTA when the heads of a group pair up
    const int hb = (a.H / a.G) % 2 == 0 ? 2 : 1;
    static DeviceOnce configured[2];
    int dev = 0;
    cudaError_t e = cudaSuccess;
    auto kern = hb == 2 ? chunk_states_tc<2> : chunk_states_tc<1>;
    const uint32_t smem = hb == 2 ? StSmem<2>::total : StSmem<1>::total;
    if (configured[hb - 1].pending(&dev, &e)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured[hb - 1].done(dev);
    } else if (e != cudaSuccess) {
        return e;
    }
    kern<<<dim3((unsigned)a.nc, (unsigned)(a.H / hb), (unsigned)(2 * a.B)), kThreads, smem, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    PassParams q;
    q.states = a.hin;
    q.adj = a.adj;
    q.dinit = a.dinit;
    q.init = a.init;
    q.dfinal = a.dfinal;
    q.chunk_sum = a.chunk_sum;
    q.B = a.B;
    q.H = a.H;
    q.PN = (int64_t)kP * kN;
    q.nc = a.nc;
    bwd_state_passes<<<dim3((unsigned)(q.PN / 4 / kPassThreads), (unsigned)a.H, (unsigned)(2 * a.B)), kPassThreads, 0,
                       stream>>>(q);
    return cudaGetLastError();
}

}  // namespace ssd
