// Throughput of the special-function unit on the GPU at hand: ex2.approx and
// rcp.approx results per SM clock, from independent chains in every thread of a
// full grid (8 chains per thread, 8 CTAs of 256 threads per SM).  The bench's
// special-function floor of the GroupNorm chain is built on these two rates.
#include <cstdio>
#include <cuda_runtime.h>

__device__ __forceinline__ float ex2f(float t) {
    float r;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

__device__ __forceinline__ float rcpf(float t) {
    float r;
    asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

template <int KIND>
__global__ void chains(float* out, int iters, float seed) {
    float v[8];
    for (int k = 0; k < 8; ++k) v[k] = seed * (threadIdx.x + k) * 1e-6f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = KIND == 0 ? ex2f(v[k]) - 1.0f : rcpf(v[k] + 1.5f);
    }
    float s = 0.f;
    for (int k = 0; k < 8; ++k) s += v[k];
    if (s == 12345.f) out[0] = s;  // keeps the chains live; never true for these inputs
}

int main() {
    int sms = 0, khz = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, 0);
    float* out = nullptr;
    if (cudaMalloc(&out, 4) != cudaSuccess) return 1;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    const int iters = 4096, blocks = sms * 8, threads = 256;
    const char* names[2] = {"ex2", "rcp"};
    for (int kind = 0; kind < 2; ++kind) {
        auto k = kind == 0 ? chains<0> : chains<1>;
        k<<<blocks, threads>>>(out, 16, 1.f);
        cudaEventRecord(e0);
        k<<<blocks, threads>>>(out, iters, 1.f);
        cudaEventRecord(e1);
        cudaEventSynchronize(e1);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        const double ops = (double)blocks * threads * iters * 8;
        printf("%s %.3f\n", names[kind], ops / (ms * 1e-3) / sms / (khz * 1e3));
    }
    const cudaError_t err = cudaGetLastError();
    printf("sms %d clock_khz %d status %s\n", sms, khz, cudaGetErrorString(err));
    return err == cudaSuccess ? 0 : 1;
}
