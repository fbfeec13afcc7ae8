// Single-pass tensor-core chunked SSD prefill: bf16 inputs, headdim P = 64,
// d_state N = 128, chunks of Q = 128 tokens.
//
// The three-step decomposition (chunk state, state passing, chunk scan; see
// chunked_simt.cu for the algebra) runs as ONE persistent kernel. Its unit of
// work is (b, chunk c, pair of heads k = 0, 1 sharing a B/C group); per unit:
//
//   S      = C B^T                      (M = 128 rows i, N = 128 cols j, K = N)
//   h_in   = the state entering chunk c: h_next of chunk c - 1 of the same
//            (b, heads), kept in TMEM, or carried in float32 through global
//            memory (L2) where the chain passes from one CTA to the next;
//            h_in(0) = init_state (or 0)
//   h_next = alpha h_in + B^T (w o x)   (M = n, N = (k, p) of both heads, K = j):
//            the chunk-state MMA accumulates onto alpha h_in, alpha =
//            exp(cs_end), w_j = exp(cs_end - cs_j) dt_j; h_next = h_in(c+1)
//   Yo_k   = C h_in,k^T                 (M = 128, N = 64 per head, K = n)
//   Y_k    = exp(cs_i) Yo_k + S'_k X_k, S'_k = S o decay_k o dt_j (+ D_k on the diagonal)
//
// so x, B, C and dt are read once, y is written once and the chunk states
// never leave the chip except as the float32 carry of the recurrence ("each
// chunk continuing from the previous chunk's state", "Recurrence Scan", first
// section). The carry of the last chunk is the final state.
//
// Work is balanced by chunks: the chains (b, head pair), each of nc chunks,
// are laid end to end (chain j = b nhg + hg, then its chunks in order) and
// CTA i takes the i-th of gridDim.x equal segments of that sequence (to one
// chunk). A segment splits into work items at chain boundaries: the tail of
// the chain it begins in (a continuation, when the segment starts inside a
// chain), whole chains, and the head of the chain it ends in (a prefix, when
// it ends inside one). Inside an item the state stays in TMEM from chunk to
// chunk; between items it is carried in float32 through global memory (L2).
// A CTA runs its prefix first, then its whole chains, then its continuation,
// which waits (bounded) on a flag that the previous CTA's prefix of the same
// chain sets once its carry is written. With the grid at most one CTA per
// SM and at most one per chain, a segment is at least one chain long, so a
// chain spans at most two CTAs, every prefix starts at chunk 0 and waits on
// nothing, and every wait ends; the previous CTA runs that prefix first, so
// the wait is normally already satisfied when it is reached.
//
// TMEM (512 columns): S [0,128), Y [128,256) (64 per head), the carried state
// [256,384) (lanes = n, columns = (k, p): a warp's 32 lanes are 32
// consecutive n, so each load or store of the float32 carry, [.., p, n] with
// n contiguous, is one 128-byte line), S'_0 [384,448), S'_1 [448,512).
//
// Warp roles (20 warps, one CTA per SM):
//   warp 0       TMA producer: x (two chunks x two heads), C (two chunks), B;
//                each x tile is loaded twice: for the chunk-state MMA, which
//                reads it after the chain group has scaled it in place by w,
//                and again (from L2, microseconds later) for S' X
//   warp 1       MMA issuer (one lane)
//   warp 2       idle
//   warp 3       per-item scalars: cumulative sums of dt A (base 2), decays
//   warps 4-11   chain group, one item ahead of the output group: w o x, the
//                carried state in (alpha h_in into TMEM, h_in as bf16 for Yo),
//                the next state out
//   warps 12-19  output group: S', the Yo rescale and y (each warp stores its
//                32 x 32 part of a head's y tile with its own TMA store)
//   warp 20      chain flags: waits for the flag of the item's predecessor
//                (ahead of the chain group), and sets the item's own flag once
//                every chain-group store of its last state is done, so that
//                neither wait stalls the chain group
// Every wait is bounded (2 s): a timeout raises a CTA-wide flag, every role
// then runs to the end of its loop without waiting, and the status word
// records SSD_ERR_TIMEOUT.
#include <cuda.h>

#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "debug_bounds.cuh"
#include "launch.h"
#include "ssd_scan.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kQ = 128, kP = 64, kN = 128, kHB = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kChainWarp0 = 4, kOutWarp0 = 12, kGroupThreads = 256;
constexpr int kFlagWarp = 20;
constexpr int kThreads = 32 * kOutWarp0 + kGroupThreads + 32;  // 21 warps, 80 registers each

struct FusedParams {
    ChunkedArgs a;
    CUtensorMap mx, mb, mc, my;  // my: y in boxes of 32 rows x 32 columns (one output warp's part)
    int nhg;          // head pairs, H / 2
    int *flags;       // [B][nhg][nc]: 1 once the state leaving chunk c is in `carry`
    float *carry;     // [B][H][P][N] float32 carried state (the final state at the end)
};

// shared memory carve (bytes from the 1024-aligned base)
constexpr uint32_t kOffC = 0;          // 2 x 32 KB: C tiles (chunk & 1), K-major, 2 panels of n
constexpr uint32_t kOffB = 65536;      // 32 KB: B tile (K-major for S, MN-major for the chunk state)
constexpr uint32_t kOffX = 98304;      // 4 x 16 KB: x tiles, slot 2 (chunk & 1) + k; the two slots of a
                                       // chunk are the N = (k, p) panels of the chunk-state B operand
constexpr uint32_t kOffH = 163840;     // 32 KB: h_in bf16, rows n, 2 panels (k) of 64 p
constexpr uint32_t kOffY = 196608;     // 8 x 2 KB: y staging of each output warp, 64-byte swizzle
constexpr uint32_t kOffS = 212992;     // scalars, two item buffers
constexpr int kScal = 5 * kHB * kQ + 2 * kHB;  // cs | dt | colf | sc | w, then D, alpha
constexpr uint32_t kOffBar = kOffS + 2 * kScal * 4;
enum {
    BAR_C_FULL = 0,     // [2]
    BAR_C_EMPTY = 2,    // [2]
    BAR_B_FULL = 4,
    BAR_B_EMPTY = 5,    // S and the chunk-state MMA have read B and the scaled x
    BAR_X_FULL = 6,     // [4] first load of x (scaled in place for the chunk state)
    BAR_X2_FULL = 10,   // [4] second load of x (for S' X)
    BAR_X_EMPTY = 14,   // [4]
    BAR_S_FULL = 18,
    BAR_S_EMPTY = 19,
    BAR_WX_FULL = 20,
    BAR_HIN_FULL = 21,
    BAR_SC_FULL = 22,
    BAR_H_EMPTY = 23,
    BAR_YO_FULL = 24,
    BAR_P_FULL = 25,    // [2]
    BAR_P_EMPTY = 27,   // [2]
    BAR_Y_FULL = 29,    // [2]
    BAR_ACC_EMPTY = 31,
    BAR_SCAL_FULL = 32,   // [2]
    BAR_SCAL_EMPTY = 34,  // [2]
    BAR_CARRY_DONE = 36,
    BAR_FLAG_OK = 37,
    kBars = 38
};
constexpr uint32_t kSmemBytes = kOffBar + kBars * 8 + 16 + 1024;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

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

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Zeroes the chain flags and the status word of this call.
__global__ void fused_init(int *status, int *flags, int64_t nflags) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nflags; i += stride) flags[i] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) *status = SSD_OK;
}

__global__ void __launch_bounds__(kThreads, 1) chunk_fused_tc(const __grid_constant__ FusedParams prm) {
    const ChunkedArgs &a = prm.a;
    const int nhg = prm.nhg;
    const int64_t nc = a.nc, Bsz = a.B;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sC = smem + kOffC, *sB = smem + kOffB, *sX = smem + kOffX;
    uint8_t *sH = smem + kOffH, *sY = smem + kOffY;
    float *s_scal = reinterpret_cast<float *>(smem + kOffS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBars);
    volatile int *s_fail = reinterpret_cast<volatile int *>(tmem_slot + 1);

    // This CTA's work items, set up once by thread 0 (below) in static shared
    // memory: s_seg = {prefix chain, prefix end, first whole chain,
    // continuation chain, continuation start, continuation end} and s_nseg =
    // {prefixes (0 or 1), whole chains, continuations (0 or 1)}.
    __shared__ int s_seg[6];
    __shared__ int s_nseg[3];
    // item k of this CTA, in the order it runs them: the prefix, the whole
    // chains, the continuation
    auto item_at = [&](int k, int &j, int &c0, int &c1) {
        if (k < s_nseg[0]) {
            j = s_seg[0], c0 = 0, c1 = s_seg[1];
        } else if (k < s_nseg[0] + s_nseg[1]) {
            j = s_seg[2] + (k - s_nseg[0]), c0 = 0, c1 = (int)nc;
        } else {
            j = s_seg[3], c0 = s_seg[4], c1 = s_seg[5];
        }
    };
    // item(j, c0, c1) for each work item of this CTA; stops when item returns false
    auto for_items = [&](auto &&item) {
        const int n = s_nseg[0] + s_nseg[1] + s_nseg[2];
        for (int k = 0; k < n; ++k) {
            int j, c0, c1;
            item_at(k, j, c0, c1);
            if (!item(j, c0, c1)) return;
        }
    };
    // body(b, c, hg, it, first, last) for each chunk of this CTA's items, in
    // order (it counts them); stops when body returns false
    auto for_chunks = [&](auto &&body) {
        uint32_t it = 0;
        for_items([&](int j, int c0, int c1) -> bool {
            const int bi = j / nhg, hg = j - bi * nhg;
            for (int c = c0; c < c1; ++c, ++it)
                if (!body((int64_t)bi, (int64_t)c, hg, it, c == c0, c + 1 == c1)) return false;
            return true;
        });
    };

    if (tid == 0) {
        // the chunks [start, end) of the chains laid end to end, split at chain boundaries
        const int64_t total = Bsz * nhg * nc, G = gridDim.x;
        const int64_t start = (int64_t)blockIdx.x * total / G, end = ((int64_t)blockIdx.x + 1) * total / G;
        s_nseg[0] = s_nseg[1] = s_nseg[2] = 0;
        if (start < end) {
            const int64_t j0 = start / nc, j1 = (end - 1) / nc, cs = start % nc, ce = (end - 1) % nc + 1;
            if (j0 == j1 && (cs > 0 || ce < nc)) {
                s_seg[3] = (int)j0, s_seg[4] = (int)cs, s_seg[5] = (int)ce;  // a part of one chain
                s_nseg[2] = 1;
            } else {
                if (ce < nc) s_seg[0] = (int)j1, s_seg[1] = (int)ce, s_nseg[0] = 1;
                const int64_t jf0 = cs > 0 ? j0 + 1 : j0, jf1 = ce < nc ? j1 - 1 : j1;
                s_seg[2] = (int)jf0;
                s_nseg[1] = jf1 >= jf0 ? (int)(jf1 - jf0 + 1) : 0;
                if (cs > 0) s_seg[3] = (int)j0, s_seg[4] = (int)cs, s_seg[5] = (int)nc, s_nseg[2] = 1;
            }
        }
        for (int k = 0; k < kBars; ++k) tc::mbar_init(bars + k, 1);
        const int group_counted[] = {BAR_S_EMPTY,    BAR_WX_FULL,   BAR_HIN_FULL,  BAR_P_FULL,
                                     BAR_P_FULL + 1, BAR_ACC_EMPTY, BAR_CARRY_DONE};
        for (int k : group_counted) tc::mbar_init(bars + k, kGroupThreads);
        tc::mbar_init(bars + BAR_SCAL_EMPTY, 2 * kGroupThreads);
        tc::mbar_init(bars + BAR_SCAL_EMPTY + 1, 2 * kGroupThreads);
        tc::fence_mbar_init();
        *s_fail = 0;
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tY = tmem + 128, tH = tmem + 256, tP = tmem + 384;
    // the flags were zeroed and the inputs written by the work before this
    // grid in the stream; nothing global is touched before it has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            // the unscaled x of chunk `rit` back into its slots, for S' X
            auto reload_x = [&](int rb, int64_t rc, int rhg, uint32_t rit) {
                for (int k = 0; k < kHB; ++k) {
                    const int slot = 2 * (int)(rit & 1) + k;
                    tc::mbar_arrive_expect_tx(&bars[BAR_X2_FULL + slot], 16384u);
                    tc::tma_load_3d(sX + slot * 16384, &prm.mx, &bars[BAR_X2_FULL + slot], (rhg * kHB + k) * kP,
                                    (int)(rc * kQ), rb);
                }
            };
            int pb = 0, phg = 0;
            int64_t pc = 0;
            uint32_t n_done = 0;
            for_chunks([&](int64_t b, int64_t c, int hg, uint32_t it, bool, bool) -> bool {
                if (*s_fail) return false;
                n_done = it + 1;
                const uint32_t par = it & 1, ph = it & 1, ph2 = (it >> 1) & 1;
                const int t0 = (int)(c * kQ), bb = (int)b;
                const int g = (int)((int64_t)hg * kHB / (a.H / a.G));
                for (int k = 0; k < kHB; ++k) {
                    const int slot = 2 * par + k;
                    if (!pwait(&bars[BAR_X_EMPTY + slot], ph2 ^ 1, s_fail)) return false;
                    tc::mbar_arrive_expect_tx(&bars[BAR_X_FULL + slot], 16384u);
                    tc::tma_load_3d(sX + slot * 16384, &prm.mx, &bars[BAR_X_FULL + slot], (hg * kHB + k) * kP, t0,
                                    bb);
                }
                if (!pwait(&bars[BAR_C_EMPTY + par], ph2 ^ 1, s_fail)) return false;  // Yo of chunk it - 2 is done
                tc::mbar_arrive_expect_tx(&bars[BAR_C_FULL + par], 32768u);
                tc::tma_load_3d(sC + par * 32768, &prm.mc, &bars[BAR_C_FULL + par], g * kN, t0, bb);
                tc::tma_load_3d(sC + par * 32768 + 16384, &prm.mc, &bars[BAR_C_FULL + par], g * kN + 64, t0, bb);
                if (!pwait(&bars[BAR_B_EMPTY], ph ^ 1, s_fail)) return false;  // chunk it - 1's MMAs read B, w o x
                tc::mbar_arrive_expect_tx(&bars[BAR_B_FULL], 32768u);
                tc::tma_load_3d(sB, &prm.mb, &bars[BAR_B_FULL], g * kN, t0, bb);
                tc::tma_load_3d(sB + 16384, &prm.mb, &bars[BAR_B_FULL], g * kN + 64, t0, bb);
                if (it > 0) reload_x(pb, pc, phg, it - 1);  // chunk it - 1's slots are free again
                pb = bb;
                pc = c;
                phg = hg;
                return true;
            });
            // the last chunk's reload, once its MMAs have read the scaled x
            if (n_done > 0 && !*s_fail && pwait(&bars[BAR_B_EMPTY], (n_done - 1) & 1, s_fail))
                reload_x(pb, pc, phg, n_done - 1);
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idS = tc::idesc_bf16(128, 128, false, false);
            const uint32_t idH = tc::idesc_bf16(128, 128, true, true);
            const uint32_t idO = tc::idesc_bf16(128, 128, false, true);
            const uint32_t idY = tc::idesc_bf16(128, kP, false, true);
            const uint32_t b0 = tc::smem_u32(sB);
            const uint32_t h0 = tc::smem_u32(sH);
            for_chunks([&](int64_t, int64_t, int, uint32_t it, bool, bool) -> bool {
                if (*s_fail) return false;
                const uint32_t par = it & 1, ph = it & 1, ph2 = (it >> 1) & 1;
                const uint32_t c0 = tc::smem_u32(sC + par * 32768), w0 = tc::smem_u32(sX + 2 * par * 16384);
                if (!pwait(&bars[BAR_C_FULL + par], ph2, s_fail)) return false;
                if (!pwait(&bars[BAR_B_FULL], ph, s_fail)) return false;
                // S = C B^T (the previous chunk's S has been read)
                if (!pwait(&bars[BAR_S_EMPTY], ph ^ 1, s_fail)) return false;
                tc::tc_fence_after();
                for (int k = 0; k < kN; k += 16) {
                    const uint64_t da = tc::sdesc_sw128(c0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                    const uint64_t db = tc::sdesc_sw128(b0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                    tc::mma_bf16(tS, da, db, idS, k > 0 ? 1u : 0u);
                }
                tc::mma_commit(&bars[BAR_S_FULL]);
                // h_next = alpha h_in + B^T (w o x), accumulated onto alpha h_in
                if (!pwait(&bars[BAR_WX_FULL], ph, s_fail)) return false;
                if (!pwait(&bars[BAR_HIN_FULL], ph, s_fail)) return false;
                tc::tc_fence_after();
                for (int k = 0; k < kQ; k += 16) {
                    const uint64_t da = tc::sdesc_sw128(b0 + k * 128, 16384, 1024);
                    const uint64_t db = tc::sdesc_sw128(w0 + k * 128, 16384, 1024);
                    tc::mma_bf16(tH, da, db, idH, 1u);
                }
                tc::mma_commit(&bars[BAR_SC_FULL]);
                tc::mma_commit(&bars[BAR_B_EMPTY]);
                // Yo = C h_in^T for both heads into Y (the previous chunk's y has been read)
                if (!pwait(&bars[BAR_ACC_EMPTY], ph ^ 1, s_fail)) return false;
                tc::tc_fence_after();
                for (int k = 0; k < kN; k += 16) {
                    const uint64_t da = tc::sdesc_sw128(c0 + (k >> 6) * 16384 + (k & 63) * 2, 16, 1024);
                    const uint64_t db = tc::sdesc_sw128(h0 + k * 128, 16384, 1024);
                    tc::mma_bf16(tY, da, db, idO, k > 0 ? 1u : 0u);
                }
                tc::mma_commit(&bars[BAR_YO_FULL]);
                tc::mma_commit(&bars[BAR_H_EMPTY]);
                tc::mma_commit(&bars[BAR_C_EMPTY + par]);
                // Y_k += S'_k X_k onto the rescaled Yo_k
                for (int kh = 0; kh < kHB; ++kh) {
                    const int slot = 2 * par + kh;
                    if (!pwait(&bars[BAR_X2_FULL + slot], ph2, s_fail)) return false;  // the unscaled x again
                    if (!pwait(&bars[BAR_P_FULL + kh], ph, s_fail)) return false;
                    tc::tc_fence_after();
                    const uint32_t x0 = tc::smem_u32(sX + slot * 16384);
                    for (int k = 0; k < kQ; k += 16)
                        tc::mma_bf16_ts(tY + kh * 64, tP + kh * 64 + k / 2,
                                        tc::sdesc_sw128(x0 + k * 128, 16384, 1024), idY, 1u);
                    tc::mma_commit(&bars[BAR_P_EMPTY + kh]);
                    tc::mma_commit(&bars[BAR_X_EMPTY + slot]);
                    tc::mma_commit(&bars[BAR_Y_FULL + kh]);
                }
                return true;
            });
        }
    } else if (warp == 2) {
        // idle (every other branch below is taken by its own warps only)
    } else if (warp == 3) {
        // ---------------------------------------------------- per-item scalars
        // For both heads k and chunk rows i (base-2 units; lane l owns rows 4l..4l+3):
        //   cs    inclusive cumulative sum of dt A over the chunk
        //   colf  exp(cs at the end of row i's 32-row block - cs_i) dt_i
        //   sc    exp(cs_i)                 (decay of the entering state to row i)
        //   w     exp(cs_end - cs_i) dt_i   (weight of row i in the chunk state)
        //   alpha exp(cs_end)               (decay over the chunk)
        const __nv_bfloat16 *dtp = static_cast<const __nv_bfloat16 *>(a.dt);
        for_chunks([&](int64_t b, int64_t c, int hg, uint32_t it, bool, bool) -> bool {
            if (*s_fail) return false;
            const int64_t t0 = c * kQ;
            float dv[kHB][4];
#pragma unroll
            for (int k = 0; k < kHB; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t t = t0 + 4 * lane + q;
                    const int64_t o = (b * a.L + t) * a.H + hg * kHB + k;
                    dv[k][q] = (t < a.L && SSD_IN_BOUNDS(o, 1, a.B * a.L * a.H, kSiteFusedDt)) ? __bfloat162float(dtp[o])
                                                                                               : 0.f;
                }
            const uint32_t par = it & 1;
            if (!pwait(&bars[BAR_SCAL_EMPTY + par], ((it >> 1) & 1) ^ 1, s_fail)) return false;
            float *base = s_scal + par * kScal;
#pragma unroll
            for (int k = 0; k < kHB; ++k) {
                const int h = hg * kHB + k;
                const float A2 = a.A[h] * kLog2e;
                float cv[4], run = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    run += dv[k][q] * A2;
                    cv[q] = run;
                }
                float incl = run;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float w = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += w;
                }
                const float excl = incl - run;
#pragma unroll
                for (int q = 0; q < 4; ++q) cv[q] += excl;
                const float blk_end = __shfl_sync(0xffffffffu, cv[3], lane | 7);
                const float cs_end = __shfl_sync(0xffffffffu, cv[3], 31);
                float *cs_ = base + k * kQ, *dt_ = base + kHB * kQ + k * kQ, *cf_ = base + 2 * kHB * kQ + k * kQ;
                float *sc_ = base + 3 * kHB * kQ + k * kQ, *w_ = base + 4 * kHB * kQ + k * kQ;
                reinterpret_cast<float4 *>(cs_)[lane] = make_float4(cv[0], cv[1], cv[2], cv[3]);
                reinterpret_cast<float4 *>(dt_)[lane] = make_float4(dv[k][0], dv[k][1], dv[k][2], dv[k][3]);
                reinterpret_cast<float4 *>(cf_)[lane] =
                    make_float4(tc::ex2(blk_end - cv[0]) * dv[k][0], tc::ex2(blk_end - cv[1]) * dv[k][1],
                                tc::ex2(blk_end - cv[2]) * dv[k][2], tc::ex2(blk_end - cv[3]) * dv[k][3]);
                reinterpret_cast<float4 *>(sc_)[lane] =
                    make_float4(tc::ex2(cv[0]), tc::ex2(cv[1]), tc::ex2(cv[2]), tc::ex2(cv[3]));
                reinterpret_cast<float4 *>(w_)[lane] =
                    make_float4(tc::ex2(cs_end - cv[0]) * dv[k][0], tc::ex2(cs_end - cv[1]) * dv[k][1],
                                tc::ex2(cs_end - cv[2]) * dv[k][2], tc::ex2(cs_end - cv[3]) * dv[k][3]);
                if (lane == 0) {
                    base[5 * kHB * kQ + k] = a.D ? a.D[h] : 0.f;
                    base[5 * kHB * kQ + kHB + k] = tc::ex2(cs_end);
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BAR_SCAL_FULL + par]);
            return true;
        });
    } else if (warp < kOutWarp0) {
        // ---------------------------------------------------- chain group
        // Warp (qd, hf): TMEM lanes 32 qd .. 32 qd + 31 = state columns n;
        // head hf, all 64 p (TMEM columns 64 hf + p).
        const int qd = warp & 3, hf = (warp - kChainWarp0) >> 2;
        const int ctid = tid - 32 * kChainWarp0;
        const uint32_t lq = (uint32_t)(qd * 32) << 16;
        const int nn = qd * 32 + lane;
        uint32_t nfirst = 0;  // work items begun (parity of FLAG_OK)
        for_chunks([&](int64_t b, int64_t c, int hg, uint32_t it, bool first, bool last) -> bool {
            const uint32_t par = it & 1, ph = it & 1, ph2 = (it >> 1) & 1;
            pwait(&bars[BAR_SCAL_FULL + par], ph2, s_fail);
            const float *base = s_scal + par * kScal;
            const float *s_w = base + 4 * kHB * kQ, *s_alpha = base + 5 * kHB * kQ + kHB;

            // (1) w o x of both heads in place, row j of head k scaled by w_k,j
            // (the 128-byte swizzle only permutes 16-byte pieces inside a row)
            pwait(&bars[BAR_X_FULL + 2 * par], ph2, s_fail);
            pwait(&bars[BAR_X_FULL + 2 * par + 1], ph2, s_fail);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int v = ctid + kGroupThreads * r;  // 16-byte piece of the two 16 KB tiles
                const int k = v >> 10, j = (v >> 3) & 127;
                const uint4 xr = *reinterpret_cast<const uint4 *>(sX + (2 * par + k) * 16384 + (v & 1023) * 16);
                const float w = s_w[k * kQ + j];
                const uint32_t *xu = reinterpret_cast<const uint32_t *>(&xr);
                uint32_t o[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xu[m]));
                    o[m] = pack_bf16x2(f.x * w, f.y * w);
                }
                *reinterpret_cast<uint4 *>(sX + (2 * par + k) * 16384 + (v & 1023) * 16) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            }
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(&bars[BAR_WX_FULL]);

            // (2) the state entering chunk c: for the item's first chunk from
            // global memory (warp 20 has seen the predecessor item's flag), or
            // init_state / zero; otherwise the previous chunk's h_next in TMEM
            // this thread's state elements: [b, h0 + hf, p, nn] for p = 0 .. 63
            const int64_t st0 = ((b * a.H + hg * kHB + hf) * kP) * kN + nn;
            const float al = s_alpha[hf];
            pwait(&bars[BAR_H_EMPTY], ph ^ 1, s_fail);  // the previous chunk's Yo has read sH
            const float *src = nullptr;
            if (first) {
                pwait(&bars[BAR_FLAG_OK], nfirst & 1, s_fail);
                ++nfirst;
                src = c > 0 ? prm.carry + st0 : (a.init_state ? a.init_state + st0 : nullptr);
                if (*s_fail || !SSD_IN_BOUNDS(st0, (kP - 1) * kN + 1, a.B * a.H * kP * kN, kSiteFusedCarry))
                    src = nullptr;
            } else {
                tc::tc_fence_after();  // the previous chunk's MMA is complete (SC_FULL was waited for)
            }
            // in two halves of 32 p: h_in as bf16 into the B operand of Yo
            // (row n, columns (k, p), 16-byte stores) and alpha h_in into
            // TMEM, where the chunk-state MMA accumulates
#pragma unroll 1
            for (int s2 = 0; s2 < 2; ++s2) {
                float hv[32];
                if (!first) {
                    tc::tmem_ld32(tH + lq + hf * kP + 32 * s2, hv);
                    tc::tmem_ld_wait();
                } else if (src) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) hv[q] = __ldcg(src + (32 * s2 + q) * kN);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) hv[q] = 0.f;
                }
                // row n of head hf's panel (p contiguous, 128-byte swizzle): four
                // 16-byte pieces of eight p each
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int piece = 4 * s2 + u;
                    *reinterpret_cast<uint4 *>(sH + hf * 16384 + nn * 128 + ((piece ^ (nn & 7)) << 4)) =
                        make_uint4(pack_bf16x2(hv[8 * u], hv[8 * u + 1]), pack_bf16x2(hv[8 * u + 2], hv[8 * u + 3]),
                                   pack_bf16x2(hv[8 * u + 4], hv[8 * u + 5]), pack_bf16x2(hv[8 * u + 6], hv[8 * u + 7]));
                }
                uint32_t r[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(al * hv[q]);
                tc::tmem_st32(tH + lq + hf * kP + 32 * s2, r);
            }
            tc::tmem_st_wait();
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::mbar_arrive(&bars[BAR_HIN_FULL]);

            // (3) h_in(c + 1) is complete in TMEM; after the item's last chunk
            // it goes out to the carry (warp 20 then sets the item's flag)
            pwait(&bars[BAR_SC_FULL], ph, s_fail);
            if (last) {
                tc::tc_fence_after();
#pragma unroll 1
                for (int s = 0; s < 2; ++s) {
                    float hv2[32];
                    tc::tmem_ld32(tH + lq + hf * kP + 32 * s, hv2);
                    tc::tmem_ld_wait();
                    if (!*s_fail && SSD_IN_BOUNDS(st0 + (int64_t)(32 * s) * kN, 31 * kN + 1, a.B * a.H * kP * kN,
                                                  kSiteFusedCarry)) {
                        float *dst = prm.carry + st0 + (int64_t)(32 * s) * kN;
#pragma unroll
                        for (int q = 0; q < 32; ++q) __stcg(dst + q * kN, hv2[q]);
                    }
                }
                tc::tc_fence_before();
                tc::mbar_arrive(&bars[BAR_CARRY_DONE]);
            }
            tc::mbar_arrive(&bars[BAR_SCAL_EMPTY + par]);
            return true;
        });
        tc::tc_fence_before();
    } else if (warp == kFlagWarp) {
        // ------------------------------------------------------ chain flags
        // Per work item: a continuation waits (acquire, bounded) for the flag
        // of the chunk before it, which the previous CTA's prefix sets, and
        // tells the chain group (mbarrier); then, once every chain-group thread
        // has stored its part of the item's last state (the mbarrier orders
        // their stores before this thread), a prefix publishes it with one
        // release store.
        if (lane == 0) {
            uint32_t it = 0;
            const int64_t n_flags = Bsz * nhg * nc;
            (void)n_flags;
            for_items([&](int j, int c0, int c1) -> bool {
                if (c0 > 0 && !*s_fail && SSD_IN_BOUNDS(j * nc + (c0 - 1), 1, n_flags, kSiteFusedFlags)) {
                    const int *fp = prm.flags + (j * nc + (c0 - 1));
                    if (ld_acquire(fp) == 0) {
                        const uint64_t t0 = tc::global_ns();
                        while (ld_acquire(fp) == 0) {
                            if (*s_fail) break;
                            if (tc::global_ns() - t0 > kWaitNs) {
                                *s_fail = 1;
                                break;
                            }
                        }
                    }
                }
                tc::mbar_arrive(&bars[BAR_FLAG_OK]);
                if (!pwait(&bars[BAR_CARRY_DONE], it & 1, s_fail)) return false;
                ++it;
                if (c1 < nc && !*s_fail && SSD_IN_BOUNDS(j * nc + (c1 - 1), 1, n_flags, kSiteFusedFlags))
                    st_release(prm.flags + (j * nc + (c1 - 1)), 1);
                return true;
            });
        }
    } else {
        // ---------------------------------------------------- output group
        // Warp (qd, ho): TMEM lanes = chunk rows i = 32 qd + lane. S' blocks
        // J in {2 ho, 2 ho + 1} off the diagonal, columns [16 ho, 16 ho + 16)
        // of the diagonal block J = qd; Yo / y columns p in [32 ho, 32 ho + 32).
        const int qd = warp & 3, ho = (warp - kOutWarp0) >> 2;
        const uint32_t lq = (uint32_t)(qd * 32) << 16;
        const int i = qd * 32 + lane;
        // blocks of S' after this warp's rows are zero for every head: written once
        {
            uint32_t z[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) z[q] = 0u;
            for (int J = 2 * ho; J < 2 * ho + 2; ++J)
                if (J > qd) {
                    tc::tmem_st16(tP + lq + J * 16, z);
                    tc::tmem_st16(tP + lq + 64 + J * 16, z);
                }
            tc::tmem_st_wait();
        }
        uint8_t *ybuf = sY + (warp - kOutWarp0) * 2048;
        for_chunks([&](int64_t b, int64_t c, int hg, uint32_t it, bool, bool) -> bool {
            const uint32_t par = it & 1, ph = it & 1, ph2 = (it >> 1) & 1;
            pwait(&bars[BAR_SCAL_FULL + par], ph2, s_fail);
            const float *base = s_scal + par * kScal;
            const float *s_cs = base, *s_dt = base + kHB * kQ, *s_colf = base + 2 * kHB * kQ;
            const float *s_sc = base + 3 * kHB * kQ, *s_D = base + 5 * kHB * kQ;
            pwait(&bars[BAR_S_FULL], ph, s_fail);
            // S'_k for both heads (needs S only)
#pragma unroll 1
            for (int k = 0; k < kHB; ++k) {
                const float *cs_ = s_cs + k * kQ, *dt_ = s_dt + k * kQ, *cf_ = s_colf + k * kQ;
                const float cs_i = cs_[i], Dh = s_D[k];
                pwait(&bars[BAR_P_EMPTY + k], ph ^ 1, s_fail);  // the previous item's S'_k X_k is done
                tc::tc_fence_after();
                {
                    float vd[16];
                    tc::tmem_ld16(tS + lq + qd * 32 + 16 * ho, vd);
                    float csv[16], dtv[16];  // columns of the diagonal block, four at a time
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 a4 = reinterpret_cast<const float4 *>(cs_ + qd * 32 + 16 * ho)[u];
                        const float4 d4 = reinterpret_cast<const float4 *>(dt_ + qd * 32 + 16 * ho)[u];
                        csv[4 * u] = a4.x, csv[4 * u + 1] = a4.y, csv[4 * u + 2] = a4.z, csv[4 * u + 3] = a4.w;
                        dtv[4 * u] = d4.x, dtv[4 * u + 1] = d4.y, dtv[4 * u + 2] = d4.z, dtv[4 * u + 3] = d4.w;
                    }
                    tc::tmem_ld_wait();
                    uint32_t pk[8];
#pragma unroll
                    for (int q = 0; q < 16; q += 2) {
                        float f[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int cc = 16 * ho + q + e;
                            const float d = tc::ex2(fminf(cs_i - csv[q + e], 0.f)) * dtv[q + e];
                            f[e] = cc <= lane ? vd[q + e] * d : 0.f;
                            f[e] += cc == lane ? Dh : 0.f;
                        }
                        pk[q / 2] = pack_bf16x2(f[0], f[1]);
                    }
                    uint32_t (&pk8)[8] = pk;
                    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                                     tP + lq + k * 64 + qd * 16 + 8 * ho),
                                 "r"(pk8[0]), "r"(pk8[1]), "r"(pk8[2]), "r"(pk8[3]), "r"(pk8[4]), "r"(pk8[5]),
                                 "r"(pk8[6]), "r"(pk8[7])
                                 : "memory");
                }
#pragma unroll 1
                for (int J = 2 * ho; J < 2 * ho + 2; ++J) {
                    if (J >= qd) continue;
                    float v[32];
                    tc::tmem_ld32(tS + lq + J * 32, v);
                    const float rf = tc::ex2(cs_i - cs_[J * 32 + 31]);
                    tc::tmem_ld_wait();
                    uint32_t pkd[16];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 c4 = reinterpret_cast<const float4 *>(cf_ + J * 32)[q];
                        pkd[2 * q] = pack_bf16x2(v[4 * q] * (rf * c4.x), v[4 * q + 1] * (rf * c4.y));
                        pkd[2 * q + 1] = pack_bf16x2(v[4 * q + 2] * (rf * c4.z), v[4 * q + 3] * (rf * c4.w));
                    }
                    tc::tmem_st16(tP + lq + k * 64 + J * 16, pkd);
                }
                tc::tmem_st_wait();
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&bars[BAR_S_EMPTY]);  // S has been read for this item
            // Yo_k rescaled by exp(cs_i) in place; then S'_k X_k may accumulate
            pwait(&bars[BAR_YO_FULL], ph, s_fail);
            tc::tc_fence_after();
#pragma unroll 1
            for (int k = 0; k < kHB; ++k) {
                const float sc = s_sc[k * kQ + i];
                float ov[32];
                tc::tmem_ld32(tY + lq + k * 64 + 32 * ho, ov);
                tc::tmem_ld_wait();
                uint32_t r[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(sc * ov[q]);
                tc::tmem_st32(tY + lq + k * 64 + 32 * ho, r);
                tc::tmem_st_wait();
                tc::tc_fence_before();
                tc::mbar_arrive(&bars[BAR_P_FULL + k]);
            }
            // y_k: 32 rows x 32 columns of this warp, staged in the warp's own
            // 2 KB (64-byte swizzle: 16-byte piece h of row r at h ^ (r / 2 % 4))
            // and written by the warp's own TMA store
#pragma unroll 1
            for (int k = 0; k < kHB; ++k) {
                pwait(&bars[BAR_Y_FULL + k], ph, s_fail);
                tc::tc_fence_after();
                float yv[32];
                tc::tmem_ld32(tY + lq + k * 64 + 32 * ho, yv);
                tc::tmem_ld_wait();
                if (lane == 0) tc::bulk_wait_read_all();  // the warp's previous store has read ybuf
                __syncwarp();
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int q = h * 8;
                    const uint4 pk = make_uint4(pack_bf16x2(yv[q], yv[q + 1]), pack_bf16x2(yv[q + 2], yv[q + 3]),
                                                pack_bf16x2(yv[q + 4], yv[q + 5]), pack_bf16x2(yv[q + 6], yv[q + 7]));
                    *reinterpret_cast<uint4 *>(ybuf + lane * 64 + ((h ^ ((lane >> 1) & 3)) << 4)) = pk;
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::tma_store_3d(&prm.my, ybuf, (hg * kHB + k) * kP + 32 * ho, (int)(c * kQ) + 32 * qd, (int)b);
                    tc::bulk_commit();
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&bars[BAR_ACC_EMPTY]);
            tc::mbar_arrive(&bars[BAR_SCAL_EMPTY + par]);
            return true;
        });
        tc::tc_fence_before();
        if (lane == 0) tc::bulk_wait_all();  // the warp's last store is complete
    }
    __syncthreads();
    if (tid == 0 && *s_fail) atomicCAS(a.status, SSD_OK, SSD_ERR_TIMEOUT);
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

SSD_BOUNDS_HOST_READER(bounds_word_fused)

bool chunked_fused_supported(const ChunkedArgs &a) {
    if (a.io != IO_BF16 || a.P != kP || a.N != kN || a.Q != kQ) return false;
    if ((a.H / a.G) % kHB != 0) return false;
    if (a.L <= 0 || a.L > 0x7fffffffLL || a.B > 0x7fffffffLL) return false;
    if (((a.H * a.P * 2) % 16) != 0 || ((a.G * a.N * 2) % 16) != 0) return false;
    return device_cc_major_cached() == 10;
}

// The single pass runs one chain (b, head pair) per CTA at least: with C
// chains and nc chunks each it takes about max(nc, C nc / SMs) chunk times,
// while the three-kernel path spreads all C nc chunk-pairs over every SM. So
// the single pass wins from ~0.6 SM count chains up. Measured on GB300 (graph
// of back-to-back calls, inputs past L2; single pass against three kernels):
// 96 chains (B8 L2048 H24, B4 L2048 H48) 80.3 / 80.7 against 83.0 / 84.4 us;
// 80 chains (B2 L2048 H80, B2 L4096 H80) 79.1 / 150.6 against 73.2 / 131.1 us;
// 192 chains (B16 L1024 H24) 63.7 against 92.5 us; 320 chains (B8 L2048 H80)
// 174 against 251 us.
bool chunked_fused_preferred(const ChunkedArgs &a) {
    return 5 * a.B * (a.H / kHB) >= 3 * (int64_t)sm_count(152);
}

cudaError_t launch_chunked_fused(const ChunkedArgs &a, cudaStream_t stream) {
    FusedParams p;
    memset(&p, 0, sizeof(p));
    p.a = a;
    bool ok = true;
    ok &= tma_map_tokens(&p.mx, a.x, a.H * a.P, a.L, a.B, kQ);
    ok &= tma_map_tokens(&p.mb, a.Bm, a.G * a.N, a.L, a.B, kQ);
    ok &= tma_map_tokens(&p.mc, a.Cm, a.G * a.N, a.L, a.B, kQ);
    ok &= tma_map_tokens(&p.my, a.y, a.H * a.P, a.L, a.B, 32, 32);
    if (!ok) return cudaErrorInvalidValue;
    p.nhg = (int)(a.H / kHB);
    // the chain flags reuse the per-chunk decay area ([B, H, nc] floats >= [B, H/2, nc] ints);
    // the carry is the caller's final state, else the per-chunk state area
    p.flags = reinterpret_cast<int *>(a.chunk_sum);
    p.carry = a.final_state ? a.final_state : a.states;

    static DeviceOnce configured;
    int dev = 0;
    cudaError_t de = cudaSuccess;
    if (configured.pending(&dev, &de)) {
        cudaError_t e = cudaFuncSetAttribute(chunk_fused_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chunk_fused_tc, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured.done(dev);
    } else if (de != cudaSuccess) {
        return de;
    }
    const bool staged = a.stage_ev[0] != nullptr;
    cudaError_t e = mark_stage(a, 0, stream);
    if (e != cudaSuccess) return e;
    const int64_t nflags = a.B * p.nhg * a.nc;
    const unsigned init_blocks = (unsigned)imin<int64_t>((nflags + 255) / 256, 64);
    if (staged) {
        fused_init<<<init_blocks, 256, 0, stream>>>(a.status, p.flags, nflags);
        e = cudaGetLastError();
    } else {
        e = launch_programmatic(fused_init, dim3(init_blocks), dim3(256), 0, stream, a.status, p.flags, nflags);
    }
    if (e != cudaSuccess) return e;
    if ((e = mark_stage(a, 1, stream)) != cudaSuccess) return e;
    if ((e = mark_stage(a, 2, stream)) != cudaSuccess) return e;
    // one CTA per SM, and no more CTAs than chains, so that a segment holds at
    // least one chain's worth of chunks
    const int64_t grid = imin<int64_t>(a.B * p.nhg, sm_count(1));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (!staged) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, chunk_fused_tc, p);
    if (e != cudaSuccess) return e;
    return mark_stage(a, 3, stream);
}

}  // namespace ssd
