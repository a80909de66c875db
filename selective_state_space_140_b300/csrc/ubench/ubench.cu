// Throughput micro-benchmarks: SFU ex2, SFU sin/cos, fp32 FMA and packed f32x2 FMA.
// Each thread keeps 8 independent chains so that latency is hidden and the
// pipe's issue rate is what the launch time measures.
#include <cuda_runtime.h>

#include "../../../include/mamba_ubench.h"

namespace {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void ex2_kernel(float* out, int iters) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = -0.001f * float(threadIdx.x + i);
    for (int k = 0; k < iters; ++k) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = -ex2(v[i]);  // stays in [-1, -0.5]
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void ffma_kernel(float* out, int iters) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.001f * float(threadIdx.x + i);
    const float a = 0.999f, c = 0.0001f;
    for (int k = 0; k < iters; ++k) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = fmaf(v[i], a, c);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void ffma2_kernel(float* out, int iters) {
    unsigned long long v[8];
    const float x0 = 0.001f * float(threadIdx.x);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        asm("mov.b64 %0, {%1, %2};" : "=l"(v[i]) : "f"(x0 + i), "f"(x0 - i));
    unsigned long long a, c;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(0.999f), "f"(0.998f));
    asm("mov.b64 %0, {%1, %2};" : "=l"(c) : "f"(0.0001f), "f"(0.0002f));
    for (int k = 0; k < iters; ++k) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(v[i]) : "l"(a), "l"(c));
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v[i]));
        s += lo + hi;
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// SFU sine and cosine: 8 chains of each per thread (16 operations per step).
__global__ void sincos_kernel(float* out, int iters) {
    float v[8], w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = w[i] = 0.001f * float(threadIdx.x + i);
    for (int k = 0; k < iters; ++k) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            asm volatile("sin.approx.ftz.f32 %0, %0;" : "+f"(v[i]));  // stays in [-1, 1]
            asm volatile("cos.approx.ftz.f32 %0, %0;" : "+f"(w[i]));
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i] + w[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

template <typename K>
int launch(K kern, float* out, int blocks, int threads, int iters, cudaStream_t s) {
    if (!out || blocks <= 0 || threads <= 0 || iters <= 0) return 2;
    kern<<<blocks, threads, 0, s>>>(out, iters);
    return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

}  // namespace

extern "C" {
int mamba_ubench_ex2(float* out, int blocks, int threads, int iters, CUstream_st* s) {
    return launch(ex2_kernel, out, blocks, threads, iters, s);
}
int mamba_ubench_ffma(float* out, int blocks, int threads, int iters, CUstream_st* s) {
    return launch(ffma_kernel, out, blocks, threads, iters, s);
}
int mamba_ubench_ffma2(float* out, int blocks, int threads, int iters, CUstream_st* s) {
    return launch(ffma2_kernel, out, blocks, threads, iters, s);
}
int mamba_ubench_sincos(float* out, int blocks, int threads, int iters, CUstream_st* s) {
    return launch(sincos_kernel, out, blocks, threads, iters, s);
}
}
