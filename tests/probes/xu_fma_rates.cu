// Throughput probe of the two pipes the Mamba-1 scan leans on: the SFU
// exponential (ex2.approx.ftz.f32, with one FADD to keep each chain bounded)
// and the packed float32 FMA (fma.rn.f32x2), alone and interleaved. Each
// thread runs 16 independent chains; every thread writes one float of a
// buffer sized for the largest grid, so every access is in bounds. Prints
// chain steps per SM per clock (the clock being the device's reported
// maximum) at 8 to 64 resident warps per SM.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

__device__ __forceinline__ float ex2f(float x) { float y; asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x)); return y; }
__device__ __forceinline__ uint64_t pk2(float a, float b) { uint64_t r; asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b)); return r; }
__device__ __forceinline__ void up2(uint64_t v, float &a, float &b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v)); }
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) { uint64_t d; asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c)); return d; }

constexpr int kChains = 16;
template <int MODE>  // 0: ex2 only, 1: fma2 only, 2: one ex2 pair + one fma2 per step per chain
__global__ void probe(float *out, int iters, float seed) {
    float v[kChains];
    uint64_t w[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) { v[i] = -0.001f * (threadIdx.x + i) * seed; w[i] = pk2(v[i], v[i] + 1.f); }
    const uint64_t m = pk2(0.999f, 0.998f), c = pk2(1e-7f, 2e-7f);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) {
            if (MODE == 0) v[i] = ex2f(v[i]) - 1.0f;
            if (MODE == 1) w[i] = fma2(w[i], m, c);
            if (MODE == 2) { v[i] = ex2f(v[i]) - 1.0f; w[i] = fma2(w[i], m, c); }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) { float a, b; up2(w[i], a, b); s += v[i] + a + b; }
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

int main() {
    int dev = 0, sms = 0, clk = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev);
    const int threads = 256;
    float *out = nullptr;
    const int maxblocks = sms * 8;
    cudaMalloc(&out, sizeof(float) * maxblocks * threads);
    const int iters = 4096;
    for (int bps : {1, 2, 4, 8}) {
        const int blocks = sms * bps;
        for (int mode = 0; mode < 3; ++mode) {
            auto k = mode == 0 ? probe<0> : mode == 1 ? probe<1> : probe<2>;
            k<<<blocks, threads>>>(out, 16, 1.f);
            cudaDeviceSynchronize();
            cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
            cudaEventRecord(e0);
            k<<<blocks, threads>>>(out, iters, 1.f);
            cudaEventRecord(e1);
            cudaEventSynchronize(e1);
            float ms = 0; cudaEventElapsedTime(&ms, e0, e1);
            const double ops = (double)blocks * threads * iters * kChains;  // chain steps
            const double cycles = ms * 1e-3 * clk * 1e3;  // clock rate in kHz
            printf("warps/SM %2d mode %d (%s): %.3f ms, %.1f chain steps per SM per clock\n", bps * threads / 32, mode,
                   mode == 0 ? "ex2 + fadd" : mode == 1 ? "fma.f32x2" : "both", ms, ops / sms / cycles);
        }
    }
    cudaError_t err = cudaGetLastError();
    printf("status %s, SM clock attribute %d kHz, %d SMs\n", cudaGetErrorString(err), clk, sms);
    cudaFree(out);
    return err == cudaSuccess ? 0 : 1;
}
