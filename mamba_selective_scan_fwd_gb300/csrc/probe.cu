// ss_measure_ex2_rate / ss_measure_fma_rate: the MUFU ex2 and FP32-pipe
// throughputs of the current GPU, the denominators of the scan's exponential
// roofline (one 2^x per (t, d, n) and direction) and of its FP32 roofline
// (the multiplies and fused multiply-adds of every state update).
//
// One 1024-thread block per SM (its dynamic shared memory keeps a second
// block off the SM) runs eight independent chains per thread -- of
// ex2.approx.ftz.f32, or of packed fma.rn.f32x2 (the form the scan kernels
// issue) -- so that the unit, not the chain latency, limits the issue.  Each
// block times its own loop with the SM's cycle counter; the rate is the
// block's results over its cycles, independent of the clock frequency.  The
// result is the median over the blocks.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "ss.h"
#include "simd.cuh"

namespace {

constexpr int kThreads = 1024, kChains = 8;

__global__ void __launch_bounds__(kThreads, 1) k_ex2_rate(int iters, unsigned long long* cycles, float* sink) {
    extern __shared__ float occupy[];
    float v[kChains];
#pragma unroll
    for (int j = 0; j < kChains; j++) v[j] = 0.03125f * (float)((threadIdx.x + 5 * j) % 31 + 1);  // in (0, 1]
    __syncthreads();
    const unsigned long long t0 = clock64();
    for (int i = 0; i < iters; i++) {
#pragma unroll
        for (int j = 0; j < kChains; j++) v[j] = ss::ex2a(-v[j]);  // stays in [1/2, 1)
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; j++) s += v[j];
    if (s < 0.f) sink[0] = s + occupy[threadIdx.x];  // never taken: keeps the chains live
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// Eight chains of v <- v / 2 + 1/4 per thread, two f32 lanes each (a packed
// f32x2 FMA is two f32 results); the values stay in [1/4, 1].
__global__ void __launch_bounds__(kThreads, 1) k_fma_rate(int iters, unsigned long long* cycles, float* sink) {
    extern __shared__ float occupy[];
    float2 v[kChains];
#pragma unroll
    for (int j = 0; j < kChains; j++)
        v[j] = make_float2(0.03125f * (float)((threadIdx.x + 5 * j) % 31 + 1), 0.03125f * (float)((threadIdx.x + 3 * j) % 29 + 2));
    __syncthreads();
    const unsigned long long t0 = clock64();
    for (int i = 0; i < iters; i++) {
#pragma unroll
        for (int j = 0; j < kChains; j++) v[j] = ss::fma2(v[j], make_float2(0.5f, 0.5f), make_float2(0.25f, 0.25f));
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; j++) s += v[j].x + v[j].y;
    if (s < 0.f) sink[0] = s + occupy[threadIdx.x];  // never taken: keeps the chains live
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// Median over the SMs of `per_thread` results per iteration per thread of one
// kernel launch of one block per SM, per SM clock cycle.
int measure_rate(void (*kernel)(int, unsigned long long*, float*), int iters, double per_thread, double* out) {
    if (iters <= 0 || iters > (1 << 20) || out == nullptr) return SS_ERR_INVALID_PROBLEM;
    int dev = 0, sms = 0, smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return SS_ERR_CUDA;
    // more than half of an SM's shared memory: one block per SM
    const int dyn = smem / 2 + 1024 < smem ? smem / 2 + 1024 : smem;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
        return SS_ERR_CUDA;
    unsigned long long* cycles = nullptr;
    float* sink = nullptr;
    if (cudaMalloc(&cycles, sizeof(unsigned long long) * sms) != cudaSuccess) return SS_ERR_CUDA;
    if (cudaMalloc(&sink, sizeof(float)) != cudaSuccess) {
        cudaFree(cycles);
        return SS_ERR_CUDA;
    }
    std::vector<unsigned long long> host(sms);
    kernel<<<sms, kThreads, dyn>>>(iters, cycles, sink);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpy(host.data(), cycles, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost);
    cudaFree(cycles);
    cudaFree(sink);
    if (e != cudaSuccess) return SS_ERR_CUDA;
    std::vector<double> rate(sms);
    for (int i = 0; i < sms; i++)
        rate[i] = host[i] ? (double)kThreads * per_thread * (double)iters / (double)host[i] : 0.0;
    std::nth_element(rate.begin(), rate.begin() + sms / 2, rate.end());
    *out = rate[sms / 2];
    return SS_OK;
}

}  // namespace

extern "C" int ss_measure_ex2_rate(int iters, double* per_clk_per_sm) {
    return measure_rate(k_ex2_rate, iters, (double)kChains, per_clk_per_sm);
}

extern "C" int ss_measure_fma_rate(int iters, double* per_clk_per_sm) {
    return measure_rate(k_fma_rate, iters, 2.0 * kChains, per_clk_per_sm);
}
