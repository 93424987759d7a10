// GroupNorm as rows: the slab of sample n's channel group g, y[n, g C/G .. (g + 1) C/G,
// all HW] (contiguous in NCHW, C / G x HW floats), is a row whose statistic is its mean
// and M2 and whose output is element-wise with per-channel constants (POPCORNBENCH page
// "Kimi-K2.6 / l2_p92", GroupNorm discussion):
//   group_norm        z = (y - mean) * rstd * gamma_c + beta_c,
//   gn_act_residual   y + hardswish(tanh(z)),
// rstd = 1 / sqrt(M2 / count + eps).  The rows run through the tensor-memory row kernel
// (row_tmem.cuh): each slab is read once from HBM and written once, the group of CTAs
// merging its (mean, M2) partials (Chan's pairwise update, counts from the slice
// lengths) through tagged slots.  The subtraction of the mean comes first in both
// outputs, so a mean far from the spread keeps z accurate; the chain's activation is
// the pair form of gn_common.cuh (two special-function operations per element).
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "gn_common.cuh"
#include "launch.h"
#include "row_tmem.cuh"

namespace lse {

struct GnRowParams {
    const float* gamma;
    const float* beta;
    int64_t HW;
    int G, cpg;
    float eps;
};

// OUT 1: the GroupNorm output z; 2: y + hardswish(tanh(z)).
template <int OUT>
struct GnRowOp {
    using Params = GnRowParams;
    using S = Welford;
    struct R {
        float mean, rstd;
    };
    // A thread's columns increase from call to call: the channel of the current column
    // and its constants are kept, and advanced at each multiple of HW.
    struct Cursor {
        float mean, rstd;
        const float* gamma;
        const float* beta;
        int64_t HW, next;  // first column of the channel after the current one
        int c;             // current channel
        float sc, sh;
    };
    __device__ static S empty() { return Welford{0.f, 0.f, 0.f}; }
    template <int K>
    __device__ static void fold(S& st, const float (&v)[K]) {
        st = wf_merge(st, wf_batch<K>(v));
    }
    __device__ static S warp_allreduce(S st) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) st = wf_merge(st, wf_shfl_xor(st, o));
        return st;
    }
    __device__ static S merge(S x, S y) { return wf_merge(x, y); }
    // (mean, M2) in one 64-bit word, the tag in M2's lowest bit (relative change <= 2^-23;
    // a non-finite M2 stays non-finite, and its group's output is NaN anyway).
    __device__ static unsigned long long pack(S st, uint32_t tag) {
        const uint32_t m2b = (__float_as_uint(st.m2) & ~1u) | (tag & 1u);
        return ((unsigned long long)m2b << 32) | __float_as_uint(st.mean);
    }
    __device__ static S unpack(unsigned long long w, int64_t count) {
        return Welford{(float)count, __uint_as_float((uint32_t)w), __uint_as_float((uint32_t)(w >> 32) & ~1u)};
    }
    __device__ static R finish(S st, const Params& p) { return R{st.mean, 1.f / sqrtf(st.m2 / st.n + p.eps)}; }
    __device__ static Cursor cursor(R r, const Params& p, int64_t row) {
        const int g = (int)(row % p.G);
        return Cursor{r.mean, r.rstd, p.gamma, p.beta, p.HW, 0, g * p.cpg - 1, 0.f, 0.f};
    }
    __device__ static float4 out4(Cursor& cu, float4 x, int64_t col) {
        while (col >= cu.next) {  // into the channel of col (HW % 4 == 0: four columns share it)
            ++cu.c;
            cu.next += cu.HW;
            const float k = OUT == 1 ? 1.f : 2.f * kLog2e;
            cu.sc = cu.rstd * __ldg(cu.gamma + cu.c) * k;
            cu.sh = __ldg(cu.beta + cu.c) * k;
        }
        if constexpr (OUT == 1) {
            return make_float4(fmaf(x.x - cu.mean, cu.sc, cu.sh), fmaf(x.y - cu.mean, cu.sc, cu.sh),
                               fmaf(x.z - cu.mean, cu.sc, cu.sh), fmaf(x.w - cu.mean, cu.sc, cu.sh));
        } else {
            // y + hardswish(tanh(z)) in pair form, plus the 2/3 it leaves out
            const f32x2 mean = f2_pack(cu.mean, cu.mean), sc = f2_pack(cu.sc, cu.sc), sh = f2_pack(cu.sh, cu.sh);
            const f32x2 k23 = f2_pack(2.f / 3.f, 2.f / 3.f);
            const f32x2 ra = f2_add(f2_residual_less_2_3(f2_pack(x.x, x.y), mean, sc, sh), k23);
            const f32x2 rb = f2_add(f2_residual_less_2_3(f2_pack(x.z, x.w), mean, sc, sh), k23);
            float4 o;
            f2_unpack(ra, o.x, o.y);
            f2_unpack(rb, o.z, o.w);
            return o;
        }
    }
};

// Rows = N x G slabs of C / G x HW floats (HW % 4 == 0: a float4 never straddles two
// channels).  LSE_GNR_GROUP forces the CTAs per slab, LSE_GNR_CHUNK bounds the landing
// chunks.  Defaults, measured on GB300 at y[128, 64, 126, 126] (slabs of 63,504 floats):
// GroupNorm with slices of at least 16,384 floats and chunks of at most 8,192 (3 CTAs per
// slab); the chain, whose stores are the slower side, with slices down to 12,288 floats
// and chunks up to 16,384 (4 CTAs per slab: one more row in flight per CTA).
cudaError_t plan_gn_rows(const DeviceInfo& dev, const float* y, const float* out, int64_t N, int64_t C, int64_t HW,
                         int64_t G, int out_kind, GroupPlan* plan) {
    if (HW % 4 != 0 || N < 1 || HW < 4) return cudaErrorNotSupported;
    const bool chain = out_kind == 2;
    return plan_row_tmem(dev, y, out, N * G, (C / G) * HW, env_int("LSE_GNR_GROUP", 0),
                         env_int("LSE_GNR_CHUNK", chain ? 16384 : 8192), chain ? 12288 : 16384, plan);
}

cudaError_t launch_gn_rows(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                           int64_t N, int64_t C, int64_t HW, int64_t G, float eps, const GroupPlan& plan,
                           void* scratch, cudaStream_t stream, int out_kind) {
    const GnRowParams p{gamma, beta, HW, (int)G, (int)(C / G), eps};
    // store warps: 4 for GroupNorm, 8 for the chain, whose stores carry two special-function
    // operations per element (LSE_GNR_SW = 4 or 8 sets both)
    const bool sw8 = env_int("LSE_GNR_SW", out_kind == 2 ? 8 : 4) == 8;
    if (out_kind == 1 && sw8)
        return launch_row_tmem<GnRowOp<1>, 8>(dev, y, out, N * G, (C / G) * HW, plan, scratch, stream, p,
                                              "row_tmem (group_norm)");
    if (out_kind == 1)
        return launch_row_tmem<GnRowOp<1>, 4>(dev, y, out, N * G, (C / G) * HW, plan, scratch, stream, p,
                                              "row_tmem (group_norm)");
    if (sw8)
        return launch_row_tmem<GnRowOp<2>, 8>(dev, y, out, N * G, (C / G) * HW, plan, scratch, stream, p,
                                              "row_tmem (gn_act_residual)");
    return launch_row_tmem<GnRowOp<2>, 4>(dev, y, out, N * G, (C / G) * HW, plan, scratch, stream, p,
                                          "row_tmem (gn_act_residual)");
}

}  // namespace lse
