// pipe_peaks.cu -- throughput microbenchmarks for the MUFU ex2 pipe and the
// FP32 FMA pipe (scalar and packed f32x2) on the running GPU.  Each thread
// advances 8 independent chains, so the measured rate is the pipe's issue
// throughput, not its latency.  Measurement support only.
#include <cuda_runtime.h>
#include <cstdio>

#include "pipe_peaks.h"

namespace {

constexpr int kIters = 4096;
constexpr int kChains = 8;

__global__ void __launch_bounds__(256) ex2_loop(float* out, float seed) {
    float x[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = seed + 0.01f * (threadIdx.x + i);
    for (int k = 0; k < kIters; ++k) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) {
            // x <- 2^(-x) keeps x in [0.5, 1]; the negation is a source modifier.
            asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(x[i]) : "f"(-x[i]));
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += x[i];
    if (s == 12345.f) out[threadIdx.x] = s;  // keep the chains alive
}

__global__ void __launch_bounds__(256) fma_loop(float* out, float seed) {
    float x[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = seed + 0.01f * (threadIdx.x + i);
    const float a = 0.999f, b = 0.001f;
    for (int k = 0; k < kIters; ++k) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x[i]) : "f"(a), "f"(b));
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += x[i];
    if (s == 12345.f) out[threadIdx.x] = s;
}

__global__ void __launch_bounds__(256) fma2_loop(float* out, float seed) {
    float2 x[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = make_float2(seed + 0.01f * i, seed - 0.01f * i);
    const float2 a = make_float2(0.999f, 0.998f), b = make_float2(0.001f, 0.002f);
    for (int k = 0; k < kIters; ++k) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) x[i] = __ffma2_rn(x[i], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += x[i].x + x[i].y;
    if (s == 12345.f) out[threadIdx.x] = s;
}

template <typename K>
double time_kernel(K kern, int blocks, float* out, cudaStream_t stream, int* err) {
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    kern<<<blocks, 256, 0, stream>>>(out, 0.5f);  // warm-up
    cudaEventRecord(e0, stream);
    kern<<<blocks, 256, 0, stream>>>(out, 0.5f);
    cudaEventRecord(e1, stream);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) *err = int(e);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return ms * 1e-3;
}

}  // namespace

extern "C" int ssm_pipe_peaks(double out[4], cudaStream_t stream) {
    int dev = 0, sms = 0, err = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    float* buf = nullptr;
    if (cudaMalloc(&buf, 256 * sizeof(float)) != cudaSuccess) return 2;
    const int blocks = sms * 8;  // 8 blocks x 256 threads = 64 warps per SM
    const double lanes = double(blocks) * 256.0 * kIters * kChains;
    const double t_ex2 = time_kernel(ex2_loop, blocks, buf, stream, &err);
    const double t_fma = time_kernel(fma_loop, blocks, buf, stream, &err);
    const double t_fma2 = time_kernel(fma2_loop, blocks, buf, stream, &err);
    cudaFree(buf);
    out[0] = lanes / t_ex2;
    out[1] = lanes / t_fma;
    out[2] = 2.0 * lanes / t_fma2;
    out[3] = sms;
    return err;
}
