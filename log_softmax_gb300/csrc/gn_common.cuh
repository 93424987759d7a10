// Shared pieces of the GroupNorm kernels: Welford statistics and the
// tanh / hardswish / residual step (GroupNorm -> Tanh -> HardSwish -> residual
// add of the POPCORNBENCH page "Kimi-K2.6 / l2_p92").
#pragma once

#include "common.cuh"

namespace lse {

struct Welford {
    float n;
    float mean;
    float m2;  // sum of squared deviations from mean
};

// Chan et al.'s pairwise update of (count, mean, M2).
__device__ __forceinline__ Welford wf_merge(Welford a, Welford b) {
    const float n = a.n + b.n;
    if (n == 0.f) return a;
    const float d = b.mean - a.mean;
    const float wb = __fdividef(b.n, n);
    return Welford{n, fmaf(d, wb, a.mean), a.m2 + b.m2 + d * d * a.n * wb};
}

template <int K>
__device__ __forceinline__ Welford wf_batch(const float (&v)[K]) {
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) s += v[k];
    const float mean = s * (1.f / K);
    float m2 = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const float d = v[k] - mean;
        m2 = fmaf(d, d, m2);
    }
    return Welford{(float)K, mean, m2};
}

__device__ __forceinline__ Welford wf_shfl_xor(Welford w, int o) {
    return Welford{__shfl_xor_sync(0xffffffffu, w.n, o), __shfl_xor_sync(0xffffffffu, w.mean, o),
                   __shfl_xor_sync(0xffffffffu, w.m2, o)};
}

// tanh from u = 2 z log2(e):  tanh(z) = sign(z) * (1 - 2 / (2^|u| + 1)), with the
// hardware base-2 exponential and approximate reciprocal; absolute error ~2e-7,
// which is what the residual r = y + hardswish(tanh(z)) needs
// (|d hardswish / dt| <= 5/6 on [-1, 1]).  The result lies in [-1, 1] (or NaN).
__device__ __forceinline__ float tanh_from_u(float u) {
    const float e = ex2(fabsf(u));
    float q;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(q) : "f"(e + 1.f));
    return copysignf(fmaf(-2.f, q, 1.f), u);
}

// r = y + hardswish(tanh(z)) with z = (v - mean) * rstd * gamma + beta, from the
// table entry e = {mean, rstd * gamma * 2 log2(e), beta * 2 log2(e), 0}.
// HardSwish is t * min(max(t + 3, 0), 6) / 6; for t in [-1, 1] the clamp never
// binds (t + 3 lies in [2, 4]), so it equals t * (t / 6 + 1/2), and a NaN t
// gives NaN either way.
__device__ __forceinline__ float act_residual(float v, float4 e) {
    const float u = fmaf(v - e.x, e.y, e.z);
    const float t = tanh_from_u(u);
    return fmaf(t, fmaf(t, 1.f / 6.f, 0.5f), v);
}

}  // namespace lse
