// Form 3: GroupNorm -> tanh -> hardswish -> residual add -> logsumexp over C.
//
// POPCORNBENCH page "Kimi-K2.6 / l2_p92" (the chain after its Conv2d):
//   mean, var per (n, g): population statistics over the C/G channels of the
//   group and all HW positions; z = (y - mean)/sqrt(var + eps)*gamma_c + beta_c;
//   t = tanh(z); h = t*min(max(t+3, 0), 6)/6; r = y + h; out[n, p] = lse_c r.
// The page splits the work into a statistics kernel and a fused kernel that
// gives every pixel a 64-thread block (one thread per channel), whose loads are
// a plane (HW floats) apart across a warp.  Here:
//   gn_stats_kernel  one block per (n, g) group: a contiguous span of
//                    (C/G)*HW floats, read with 128-bit loads; per-thread
//                    batches merged by Chan's pairwise mean/M2 update
//                    (exact two-pass inside each 16-value batch), so no
//                    E[x^2] - E[x]^2 cancellation.
//   gn_apply_kernel  one thread per 4 adjacent pixels, looping over the C
//                    channels, so every load is a coalesced 128-bit read of a
//                    channel plane; the channel lse is kept online as a
//                    (max, sum) pair per pixel, one rescale per 8 channels.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace lse {

// ------------------------------------------------------------------ statistics

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

// stats[2*(n*G+g)] = mean, stats[2*(n*G+g)+1] = 1/sqrt(var + eps).
template <int VEC>
__global__ void __launch_bounds__(512) gn_stats_kernel(const float* __restrict__ y,
                                                       float* __restrict__ stats, int64_t N,
                                                       int64_t C, int64_t HW, int64_t G, float eps) {
    __shared__ Welford red[32];
    constexpr int T = 512;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t cpg = C / G;
    const int64_t count = cpg * HW;
    for (int64_t grp = blockIdx.x; grp < N * G; grp += gridDim.x) {
        const int64_t n = grp / G, g = grp - n * G;
        const float* base = y + (n * C + g * cpg) * HW;
        Welford w{0.f, 0.f, 0.f};
        const int64_t nv = count / VEC;  // VEC == 4 implies count % 4 == 0
        int64_t i = tid;
        for (; i + 3 * T < nv; i += 4 * T) {
            float v[4 * VEC];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if constexpr (VEC == 4) {
                    float4 a = ld_stream_f4(base + (i + k * T) * 4);
                    v[4 * k + 0] = a.x; v[4 * k + 1] = a.y; v[4 * k + 2] = a.z; v[4 * k + 3] = a.w;
                } else {
                    v[k] = ld_stream_f1(base + i + k * T);
                }
            }
            w = wf_merge(w, wf_batch<4 * VEC>(v));
        }
        for (; i < nv; i += T) {
            float v[VEC];
            if constexpr (VEC == 4) {
                float4 a = ld_stream_f4(base + i * 4);
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            } else {
                v[0] = ld_stream_f1(base + i);
            }
            w = wf_merge(w, wf_batch<VEC>(v));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w = wf_merge(w, wf_shfl_xor(w, o));
        __syncthreads();
        if (lane == 0) red[warp] = w;
        __syncthreads();
        if (warp == 0) {
            Welford r = (lane < T / 32) ? red[lane] : Welford{0.f, 0.f, 0.f};
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) r = wf_merge(r, wf_shfl_xor(r, o));
            if (lane == 0) {
                const float var = r.m2 / (float)count;
                stats[2 * grp] = r.mean;
                stats[2 * grp + 1] = 1.f / sqrtf(var + eps);
            }
        }
    }
}

// ------------------------------------------------------------------ fused apply + channel lse

// tanh(z) = sign(z) * (1 - 2 / (e^(2|z|) + 1)); absolute error ~2e-7, which is
// what the residual r = y + hardswish(tanh(z)) needs (|d hardswish / dt| <= 5/6).
__device__ __forceinline__ float tanh_ex2(float z) {
    const float e = ex2(fabsf(z) * (2.f * kLog2e));
    return copysignf(1.f - __fdividef(2.f, e + 1.f), z);
}

__device__ __forceinline__ float act_residual(float v, float mean, float scale, float shift) {
    const float z = fmaf(v - mean, scale, shift);
    const float t = tanh_ex2(z);
    const float h = t * fminf(fmaxf(t + 3.f, 0.f), 6.f) * (1.f / 6.f);
    return v + h;
}

template <int VEC>
__global__ void __launch_bounds__(128) gn_apply_kernel(const float* __restrict__ y,
                                                       const float* __restrict__ gamma,
                                                       const float* __restrict__ beta,
                                                       const float* __restrict__ stats,
                                                       float* __restrict__ out, int64_t N, int C,
                                                       int64_t HW, int G, int64_t tiles) {
    extern __shared__ float tab[];  // [C] mean, [C] rstd*gamma, [C] beta for the current sample
    constexpr int T = 128;
    constexpr int CH = 8;
    const int tid = threadIdx.x;
    const int cpg = C / G;
    int64_t cur_n = -1;
    for (int64_t b = blockIdx.x; b < N * tiles; b += gridDim.x) {
        const int64_t n = b / tiles;
        const int64_t tile = b - n * tiles;
        if (n != cur_n) {  // uniform across the block
            __syncthreads();
            for (int c = tid; c < C; c += T) {
                const int g = c / cpg;
                const float mean = stats[2 * (n * G + g)];
                const float rstd = stats[2 * (n * G + g) + 1];
                tab[c] = mean;
                tab[C + c] = rstd * gamma[c];
                tab[2 * C + c] = beta[c];
            }
            __syncthreads();
            cur_n = n;
        }
        const int64_t p0 = (tile * T + tid) * VEC;
        if (p0 >= HW) continue;
        const float* yp = y + n * (int64_t)C * HW + p0;
        MS st[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) st[j] = ms_empty();
        int c = 0;
        for (; c + CH <= C; c += CH) {
            float r[VEC][CH];
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const float* p = yp + (int64_t)(c + k) * HW;
                if constexpr (VEC == 4) {
                    float4 a = ld_stream_f4(p);
                    r[0][k] = a.x; r[1][k] = a.y; r[2][k] = a.z; r[3][k] = a.w;
                } else {
                    r[0][k] = ld_stream_f1(p);
                }
            }
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const float mean = tab[c + k], sc = tab[C + c + k], sh = tab[2 * C + c + k];
#pragma unroll
                for (int j = 0; j < VEC; ++j) r[j][k] = act_residual(r[j][k], mean, sc, sh);
            }
#pragma unroll
            for (int j = 0; j < VEC; ++j) ms_fold<CH>(st[j], r[j]);
        }
        for (; c < C; ++c) {
            const float* p = yp + (int64_t)c * HW;
            float r[VEC][1];
            if constexpr (VEC == 4) {
                float4 a = ld_stream_f4(p);
                r[0][0] = a.x; r[1][0] = a.y; r[2][0] = a.z; r[3][0] = a.w;
            } else {
                r[0][0] = ld_stream_f1(p);
            }
            const float mean = tab[c], sc = tab[C + c], sh = tab[2 * C + c];
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                r[j][0] = act_residual(r[j][0], mean, sc, sh);
                ms_fold<1>(st[j], r[j]);
            }
        }
        float* dst = out + n * HW + p0;
        if constexpr (VEC == 4) {
            *reinterpret_cast<float4*>(dst) =
                make_float4(ms_lse(st[0]), ms_lse(st[1]), ms_lse(st[2]), ms_lse(st[3]));
        } else {
            dst[0] = ms_lse(st[0]);
        }
    }
}

cudaError_t launch_gn_act_lse(const DeviceInfo& dev, const float* y, const float* gamma,
                              const float* beta, float* out, int64_t N, int64_t C, int64_t HW,
                              int64_t G, float eps, float* stats, cudaStream_t stream) {
    const bool y16 = (reinterpret_cast<uintptr_t>(y) & 15) == 0;
    const bool o16 = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    const bool vec_stats = (HW % 4 == 0) && y16;
    const bool vec_apply = (HW % 4 == 0) && y16 && o16;
    {
        const int64_t ngrp = N * G;
        const int64_t cap = (int64_t)dev.sm_count * 4 * 16;
        const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(ngrp, cap));
        if (vec_stats)
            gn_stats_kernel<4><<<grid, 512, 0, stream>>>(y, stats, N, C, HW, G, eps);
        else
            gn_stats_kernel<1><<<grid, 512, 0, stream>>>(y, stats, N, C, HW, G, eps);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const int VEC = vec_apply ? 4 : 1;
        const int64_t tiles = ((HW + VEC - 1) / VEC + 127) / 128;
        const int64_t nblk = N * tiles;
        const int64_t cap = (int64_t)dev.sm_count * 16 * 16;
        const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(nblk, cap));
        const size_t smem = (size_t)3 * C * sizeof(float);
        cudaError_t e;
        if (vec_apply) {
            if (smem > 48 * 1024) {
                e = cudaFuncSetAttribute(gn_apply_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
                if (e != cudaSuccess) return e;
            }
            gn_apply_kernel<4><<<grid, 128, smem, stream>>>(y, gamma, beta, stats, out, N, (int)C, HW,
                                                            (int)G, tiles);
        } else {
            if (smem > 48 * 1024) {
                e = cudaFuncSetAttribute(gn_apply_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
                if (e != cudaSuccess) return e;
            }
            gn_apply_kernel<1><<<grid, 128, smem, stream>>>(y, gamma, beta, stats, out, N, (int)C, HW,
                                                            (int)G, tiles);
        }
        return cudaGetLastError();
    }
}

}  // namespace lse
