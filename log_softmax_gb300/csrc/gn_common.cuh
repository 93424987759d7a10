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

// ---------------------------------------------------------------- packed pairs

// Two fp32 lanes in one 64-bit register pair, for the packed f32x2 arithmetic of
// sm_100 and later: one instruction does two IEEE single-precision operations
// (same rounding as the scalar ones), which halves the issue slots of the
// element-wise work when two pixels share their per-channel constants.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(f32x2 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Per-lane base-2 exponential and approximate reciprocal (the special-function unit
// has no packed form).
__device__ __forceinline__ f32x2 f2_ex2(f32x2 a) {
    float lo, hi;
    f2_unpack(a, lo, hi);
    return f2_pack(ex2(lo), ex2(hi));
}

__device__ __forceinline__ float rcp_approx(float a) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

__device__ __forceinline__ f32x2 f2_rcp(f32x2 a) {
    float lo, hi;
    f2_unpack(a, lo, hi);
    return f2_pack(rcp_approx(lo), rcp_approx(hi));
}

// max of three values, NaN if any is NaN.
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Two pairs (four adjacent floats, 16-byte aligned) with one 128-bit load; with HINT
// the load carries the L2 eviction `policy`.
template <bool HINT>
__device__ __forceinline__ void ld_pairs(const float* p, f32x2& a, f32x2& b, uint64_t policy) {
    if constexpr (HINT)
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.b64 {%0, %1}, [%2], %3;"
                     : "=l"(a), "=l"(b)
                     : "l"(p), "l"(policy));
    else
        asm volatile("ld.global.nc.L1::no_allocate.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}

// ---------------------------------------------------------------- the chain in pair form

// The residual after the activations, less its constant 2/3, from q = 1 / (2^u + 1):
// with t = tanh(z) = 1 - 2q (u = 2 z log2 e) and the HardSwish clamp inactive on
// [-1, 1], hardswish(t) = t (t + 3) / 6 = 2/3 + q (2q/3 - 5/3), so
//     r - 2/3 = y + q (2q/3 - 5/3).
// The lse over channels of r is that of r - 2/3, plus 2/3.  q lies in [0, 1] (or is
// NaN), so the quadratic is well conditioned: absolute error ~1e-7 from q's
// approximate reciprocal.  Large |u| needs no clamp: 2^u = +inf gives q = 0 (t = 1),
// 2^u = 0 gives q = 1 (t = -1).
__device__ __forceinline__ f32x2 f2_residual_less_2_3(f32x2 y, f32x2 mean, f32x2 sc, f32x2 sh) {
    const f32x2 one = f2_pack(1.f, 1.f);
    const f32x2 k23 = f2_pack(2.f / 3.f, 2.f / 3.f);
    const f32x2 k53 = f2_pack(-5.f / 3.f, -5.f / 3.f);
    const f32x2 u = f2_fma(f2_sub(y, mean), sc, sh);
    const f32x2 q = f2_rcp(f2_add(f2_ex2(u), one));
    return f2_fma(q, f2_fma(q, k23, k53), y);
}

// Table entry of one channel for the pair form: a = {mean, mean, sc, sc},
// b = {sh, sh} with sc = rstd * gamma * 2 log2 e and sh = beta * 2 log2 e.
__device__ __forceinline__ void gn_pair_entry(float mean, float sc, float sh, float4* tab_a, float2* tab_b,
                                              int c) {
    tab_a[c] = make_float4(mean, mean, sc, sc);
    tab_b[c] = make_float2(sh, sh);
}

// Running channel lse of four pixels held as two pairs: m the largest r seen per pixel
// (natural units) and s the sum of e^(r - m) over the values seen; (-inf, 0) is the
// empty set.  r is finite or NaN (a non-finite y makes its group's statistics, hence
// every r of its sample, NaN).
struct Lse4 {
    f32x2 ma, mb;  // (m0, m1), (m2, m3)
    f32x2 sa, sb;
};

__device__ __forceinline__ Lse4 lse4_empty() {
    const f32x2 ninf = f2_pack(-CUDART_INF_F, -CUDART_INF_F), zero = f2_pack(0.f, 0.f);
    return Lse4{ninf, ninf, zero, zero};
}

// Folds K channels (ra[k]: pixels 0, 1; rb[k]: pixels 2, 3): one max per pixel over
// the batch (a 3-input max tree), one rescale of the running sums by
// e^(m_old - m_new), then one exponential per value.  Each exponent is the
// difference r - m taken first, then scaled by log2 e: exact near the max, and never
// an overflow, whatever the magnitude of r (folding -m log2 e into an fma instead
// would carry the rounding of m log2 e, ~8e6 at |m| = 1e14, into the exponential).
template <int K>
__device__ __forceinline__ void lse4_fold(Lse4& st, const f32x2 (&ra)[K], const f32x2 (&rb)[K]) {
    float a0[K], a1[K], b0[K], b1[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        f2_unpack(ra[k], a0[k], a1[k]);
        f2_unpack(rb[k], b0[k], b1[k]);
    }
    float m[4];
    f2_unpack(st.ma, m[0], m[1]);
    f2_unpack(st.mb, m[2], m[3]);
    auto batch_max = [&](const float (&v)[K], float old) {
        if constexpr (K == 8)
            return max3_nan(max3_nan(v[0], v[1], v[2]), max3_nan(v[3], v[4], v[5]), max3_nan(v[6], v[7], old));
        float r = old;
#pragma unroll
        for (int k = 0; k < K; ++k) r = max_nan(r, v[k]);
        return r;
    };
    const f32x2 na = f2_pack(batch_max(a0, m[0]), batch_max(a1, m[1]));
    const f32x2 nb = f2_pack(batch_max(b0, m[2]), batch_max(b1, m[3]));
    const f32x2 lg = f2_pack(kLog2e, kLog2e);
    // e^(m_old - m_new): 1 when the max is unchanged, 0 from the empty start
    st.sa = f2_mul(st.sa, f2_ex2(f2_mul(f2_sub(st.ma, na), lg)));
    st.sb = f2_mul(st.sb, f2_ex2(f2_mul(f2_sub(st.mb, nb), lg)));
    st.ma = na;
    st.mb = nb;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        st.sa = f2_add(st.sa, f2_ex2(f2_mul(f2_sub(ra[k], na), lg)));
        st.sb = f2_add(st.sb, f2_ex2(f2_mul(f2_sub(rb[k], nb), lg)));
    }
}

__device__ __forceinline__ void lse4_unpack(const Lse4& st, float (&m)[4], float (&s)[4]) {
    f2_unpack(st.ma, m[0], m[1]);
    f2_unpack(st.mb, m[2], m[3]);
    f2_unpack(st.sa, s[0], s[1]);
    f2_unpack(st.sb, s[2], s[3]);
}

// The channel lse of one thread's four adjacent pixels of one sample (two pairs),
// from the C channel planes at stride HW (yp 16-byte aligned), written as a float4 at
// dst: batches of 8 channels, all loads in flight, then the residual of each element
// and the fold.  The result adds back the 2/3 that f2_residual_less_2_3 leaves out.
template <bool HINT>
__device__ __forceinline__ void apply_lse_pairs(const float* __restrict__ yp, const float4* tab_a,
                                                const float2* tab_b, int C, int64_t HW, float* __restrict__ dst,
                                                uint64_t policy) {
    constexpr int CH = 8;
    Lse4 st = lse4_empty();
    int c = 0;
    for (; c + CH <= C; c += CH) {
        f32x2 ra[CH], rb[CH];
#pragma unroll
        for (int k = 0; k < CH; ++k) ld_pairs<HINT>(yp + (int64_t)(c + k) * HW, ra[k], rb[k], policy);
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const float4 ta = tab_a[c + k];
            const float2 tb = tab_b[c + k];
            const f32x2 mean = f2_pack(ta.x, ta.y), sc = f2_pack(ta.z, ta.w), sh = f2_pack(tb.x, tb.y);
            ra[k] = f2_residual_less_2_3(ra[k], mean, sc, sh);
            rb[k] = f2_residual_less_2_3(rb[k], mean, sc, sh);
        }
        lse4_fold<CH>(st, ra, rb);
    }
    for (; c < C; ++c) {  // channels past the last full batch, one at a time
        f32x2 ra[1], rb[1];
        ld_pairs<HINT>(yp + (int64_t)c * HW, ra[0], rb[0], policy);
        const float4 ta = tab_a[c];
        const float2 tb = tab_b[c];
        const f32x2 mean = f2_pack(ta.x, ta.y), sc = f2_pack(ta.z, ta.w), sh = f2_pack(tb.x, tb.y);
        ra[0] = f2_residual_less_2_3(ra[0], mean, sc, sh);
        rb[0] = f2_residual_less_2_3(rb[0], mean, sc, sh);
        lse4_fold<1>(st, ra, rb);
    }
    float m[4], s[4];
    lse4_unpack(st, m, s);
    *reinterpret_cast<float4*>(dst) = make_float4(m[0] + logf(s[0]) + 2.f / 3.f, m[1] + logf(s[1]) + 2.f / 3.f,
                                                  m[2] + logf(s[2]) + 2.f / 3.f, m[3] + logf(s[3]) + 2.f / 3.f);
}

}  // namespace lse
