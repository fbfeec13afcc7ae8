// Test-only library: one tcgen05 MMA tile (M = 128, bf16 operands, float32
// accumulator in tensor memory) for each shared-memory operand layout the
// tensor-core SSD kernels use, so that the descriptor encodings, the SW128
// swizzle and the TMEM lane layout are checked against a plain matrix product.
//
//   variant 0: A K-major [M][K], B K-major [N][K] written by threads   D = A B^T
//   variant 1: A K-major [M][K], B MN-major [K][N] written by threads  D = A B
//   variant 2: A MN-major [K][M], B MN-major [K][N] written by threads D = A^T B
//   variant 3: as variant 0 but both operands loaded by TMA (SWIZZLE_128B)
//   variant 4: as variant 2 but both operands loaded by TMA
//   variant 5: A [M][K] in tensor memory (written with tcgen05.st, two bf16
//              per 32-bit column, lane = row), B K-major [N][K] in smem
//
// Sizes: M = 128; N in {64, 128}; K in {64, 128, 256}. All shared-memory
// addresses a descriptor can reach stay inside the dynamic allocation.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc_ptx.cuh"

using namespace ssd::tc;

namespace {

constexpr int kM = 128;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct Maps {
    CUtensorMap a, b;
};

__global__ void __launch_bounds__(128)
probe_kernel(int variant, const __nv_bfloat16 *__restrict__ A, const __nv_bfloat16 *__restrict__ B,
             float *__restrict__ D, int N, int K, int *status, const __grid_constant__ Maps maps) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                       // up to 128 x 256 bf16 = 64 KB
    uint8_t *sB = smem + 65536;               // up to 256 x 128 bf16 = 64 KB
    uint64_t *bar_mma = reinterpret_cast<uint64_t *>(smem + 131072);
    uint64_t *bar_tma = bar_mma + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_mma + 2);

    const int tid = threadIdx.x, warp = tid >> 5;
    const bool a_mn = (variant == 2 || variant == 4);
    const bool b_mn = (variant == 1 || variant == 2 || variant == 4);
    const bool use_tma = variant == 3 || variant == 4;
    const bool a_tmem = variant == 5;

    if (tid == 0) {
        mbar_init(bar_mma, 1);
        mbar_init(bar_tma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    if (!use_tma && !a_tmem) {
        // A: K-major rows = m (K contiguous), or MN-major rows = k (M contiguous)
        for (int e = tid; e < kM * K; e += blockDim.x) {
            const int m = e / K, k = e % K;
            const __nv_bfloat16 v = A[e];  // A given as [M][K] for K-major, [K][M] for MN-major
            uint32_t off;
            if (!a_mn) off = sw128_offset(m, k, kM);
            else { const int kk = e / kM, mm = e % kM; off = sw128_offset(kk, mm, K); }
            *reinterpret_cast<__nv_bfloat16 *>(sA + off) = v;
        }
    }
    if (!use_tma) {
        for (int e = tid; e < N * K; e += blockDim.x) {
            const __nv_bfloat16 v = B[e];  // [N][K] for K-major, [K][N] for MN-major
            uint32_t off;
            if (!b_mn) off = sw128_offset(e / K, e % K, N);
            else off = sw128_offset(e / N, e % N, K);
            *reinterpret_cast<__nv_bfloat16 *>(sB + off) = v;
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tA = tmem + 128;  // A operand columns (variant 5): K/2 <= 128
    if (a_tmem) {
        // row m = TMEM lane; column c holds A[m][2c] (low half) and A[m][2c+1]
        const int m = warp * 32 + (tid & 31);
        for (int c0 = 0; c0 < K / 2; c0 += 32) {
            uint32_t r[32];
            for (int j = 0; j < 32; ++j) {
                const int c = c0 + j;
                uint32_t lo = 0, hi = 0;
                if (c < K / 2) {
                    lo = __bfloat16_as_ushort(A[m * K + 2 * c]);
                    hi = __bfloat16_as_ushort(A[m * K + 2 * c + 1]);
                }
                r[j] = lo | (hi << 16);
            }
            tmem_st32(tA + ((uint32_t)(warp * 32) << 16) + c0, r);
        }
        tmem_st_wait();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();

    bool ok = true;
    if (tid == 0) {
        if (use_tma) {
            const uint32_t bytes = (uint32_t)(kM * K + N * K) * 2;
            mbar_arrive_expect_tx(bar_tma, bytes);
            if (!a_mn) {
                for (int p = 0; p < K / 64; ++p) tma_load_2d(sA + p * kM * 128, &maps.a, bar_tma, p * 64, 0);
            } else {
                for (int p = 0; p < kM / 64; ++p) tma_load_2d(sA + p * K * 128, &maps.a, bar_tma, p * 64, 0);
            }
            if (!b_mn) {
                for (int p = 0; p < K / 64; ++p) tma_load_2d(sB + p * N * 128, &maps.b, bar_tma, p * 64, 0);
            } else {
                for (int p = 0; p < N / 64; ++p) tma_load_2d(sB + p * K * 128, &maps.b, bar_tma, p * 64, 0);
            }
            ok = mbar_wait(bar_tma, 0, kTimeoutNs);
        }
        if (ok) {
            const uint32_t idesc = idesc_bf16(kM, N, a_mn, b_mn);
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
            for (int k = 0; k < K; k += 16) {
                uint64_t da, db;
                if (!a_mn) da = sdesc_sw128(a0 + (k >> 6) * kM * 128 + (k & 63) * 2, 16, 1024);
                else da = sdesc_sw128(a0 + k * 128, K * 128, 1024);
                if (!b_mn) db = sdesc_sw128(b0 + (k >> 6) * N * 128 + (k & 63) * 2, 16, 1024);
                else db = sdesc_sw128(b0 + k * 128, K * 128, 1024);
                if (a_tmem) mma_bf16_ts(tmem, tA + k / 2, db, idesc, k > 0 ? 1u : 0u);
                else mma_bf16(tmem, da, db, idesc, k > 0 ? 1u : 0u);
            }
            mma_commit(bar_mma);
        } else {
            atomicExch(status, 4);
        }
    }
    __syncthreads();
    if (*(volatile int *)status == 0) {
        if (!mbar_wait(bar_mma, 0, kTimeoutNs)) atomicExch(status, 4);
    }
    tc_fence_after();
    if (*(volatile int *)status == 0) {
        const int row = warp * 32 + (tid & 31);
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) D[row * N + c0 + j] = v[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 tensor [rows][cols], box = 64 columns x box_rows rows, 128-byte swizzle.
int make_map(CUtensorMap *m, const void *base, int rows, int cols, int box_rows) {
    auto enc = get_encode();
    if (!enc) return -1;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -2;
}

}  // namespace

extern "C" int tc_probe(int variant, const void *A, const void *B, float *D, int N, int K, int *status,
                        cudaStream_t stream) {
    if (variant < 0 || variant > 5) return -10;
    if (!(N == 64 || N == 128) || !(K == 64 || K == 128 || K == 256)) return -11;
    Maps maps;
    memset(&maps, 0, sizeof(maps));
    const bool a_mn = (variant == 2 || variant == 4), b_mn = (variant == 1 || variant == 2 || variant == 4);
    if (variant == 3 || variant == 4) {
        int r = a_mn ? make_map(&maps.a, A, K, kM, K) : make_map(&maps.a, A, kM, K, kM);
        if (r) return r;
        r = b_mn ? make_map(&maps.b, B, K, N, K) : make_map(&maps.b, B, N, K, N);
        if (r) return r;
    }
    const int smem = 200 * 1024;  // slack: no descriptor can reach past it
    cudaError_t e = cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return -20;
    probe_kernel<<<1, 128, smem, stream>>>(variant, (const __nv_bfloat16 *)A, (const __nv_bfloat16 *)B, D, N, K,
                                           status, maps);
    return cudaGetLastError() == cudaSuccess ? 0 : -21;
}
