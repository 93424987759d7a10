// Form 3 with y read once from HBM: each sample is split by pixels over a group of
// GS CTAs of a cooperative grid, and every CTA keeps its slice of the sample (all C
// channel rows of P pixels) in shared memory from the load to the last use.
//
// GroupNorm -> tanh -> hardswish -> residual -> logsumexp over C (POPCORNBENCH page
// "Kimi-K2.6 / l2_p92"): a pixel's output needs the statistics of every group of its
// sample, and a group's statistics need every pixel of the sample.  The work-queue
// kernel (gn_act_lse.cu) reads each sample twice and relies on L2 for the second
// read; here the second read is from shared memory:
//
//   gn_slab_kernel   persistent, one CTA per SM.  Group gi of GS CTAs takes samples
//                    gi, gi + groups, ...; CTA `rank` owns pixels
//                    [rank * P, rank * P + P) of each.  NB slice buffers per CTA,
//                    each filled by one 2-D tensor copy (TMA) of the box
//                    [C channel rows] x [P pixels] of y viewed as an (N*C) x HW
//                    matrix (one copy per channel row keeps too few bytes in
//                    flight per SM: ~6 GB/s per SM measured with 848-byte rows).
//                    Warp-specialised:
//                      fold warps   as a slice lands, the exact two-pass mean and
//                                   M2 of each channel group over the slice,
//                                   published to the group through tagged 64-bit
//                                   slots; they never wait for the group.
//                      apply warps  merge the GS partials of every group (Chan's
//                                   pairwise update), build the per-channel table,
//                                   run the chain on the slice from shared memory
//                                   (four lanes per pixel quad, each on every
//                                   fourth channel, merged by shuffles), write the
//                                   channel lse, and refill the buffer with the
//                                   slice of the sample NB steps ahead.
//
// A fold warp publishing step j implies every CTA of the group has finished reading
// the slots of step j - 2 NB (step j's buffer was refilled after this CTA's apply of
// step j - NB, which needed every CTA's partials of j - NB, each published after that
// CTA's refill following its apply of j - 2 NB, which read the slots of j - 2 NB); so
// 2 NB slot sets, tagged by the parity of j / (2 NB), never hold a value a reader
// still needs.  The grid is cooperative (every CTA resident), so every wait ends;
// each is bounded (about 1 s) all the same and records a timeout in the device
// status word.
#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "gn_common.cuh"
#include "launch.h"
#include "tmem.cuh"

namespace lse {

constexpr int kSlabFoldWarps = 4;
constexpr int kSlabApplyWarps = 16;
constexpr int kSlabThreads = 32 * (kSlabFoldWarps + kSlabApplyWarps);
constexpr int kSlabMaxNB = 8;
constexpr int kSlabMaxC = 256;
constexpr int kSlabMaxG = 64;
constexpr int kSlabFoldQuads = 8;  // float4 of a group held per fold lane per round
constexpr int kSlabReadsMax = 4;   // 16-byte partial reads per merging thread and step

struct GnSlabArgs {
    CUtensorMap ymap;  // y as an (N*C) x HW fp32 matrix, box P x C, no swizzle, zero fill past HW
    const float* y;
    const float* gamma;
    const float* beta;
    float* out;
    int64_t N, HW;
    int C, G, GS, P, NB;
    float eps;
    unsigned long long* slots;  // [groups][2 NB][GS][G rounded up to even] tagged (mean, M2)
    int* status;
};

// (mean, M2) of a partial in one 64-bit word, with a 1-bit tag in the lowest bit of
// the mean (a change of at most one ulp).  A NaN mean is first made the quiet NaN
// 0x7fc00000, so that the tag bit cannot turn it into an infinity.
__device__ __forceinline__ unsigned long long slab_pack(float mean, float m2, uint32_t tag) {
    uint32_t mb = __float_as_uint(mean);
    if (isnan(mean)) mb = 0x7fc00000u;
    mb = (mb & ~1u) | (tag & 1u);
    return ((unsigned long long)__float_as_uint(m2) << 32) | mb;
}

__device__ __forceinline__ uint32_t slab_tag(unsigned long long w) { return (uint32_t)w & 1u; }

// Polls a slot until it carries `tag`, for at most ~1 s (2^26 polls).
__device__ __forceinline__ unsigned long long slab_poll(const unsigned long long* p, uint32_t tag, bool& aborted,
                                                        int* status) {
    unsigned long long w = ld_relaxed_gpu_u64(p);
    if (slab_tag(w) == tag || aborted) return w;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        __nanosleep(32);
        w = ld_relaxed_gpu_u64(p);
        if (slab_tag(w) == tag) return w;
        if ((it & 255u) == 255u && globaltimer_ns() - t0 > 1000000000ull) break;
    }
    aborted = true;
    atomicExch(status, kStatusTimeout);
    return w;
}

// Two adjacent slots (16 bytes) read from L2 without ordering.  Strong (relaxed,
// gpu-scope) accesses wait for each other within a thread (~250 ns each measured),
// so the next step's partials are fetched early with these plain L2 loads and used
// only once their tags match; a stale one is polled again with strong loads.
__device__ __forceinline__ void ld_cg_pair(const unsigned long long* p, unsigned long long& a,
                                           unsigned long long& b) {
    asm volatile("ld.global.cg.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}

__device__ __forceinline__ void wf_to_slot_parts(unsigned long long w, float n, Welford& acc) {
    acc = wf_merge(acc, Welford{n, __uint_as_float((uint32_t)w), __uint_as_float((uint32_t)(w >> 32))});
}

// (m, s) pair merge for the channel lse across lanes: m finite or NaN, or -inf for a
// lane that had no channel.
__device__ __forceinline__ void ms_merge_xor(float& m, float& s, int mask) {
    const float om = __shfl_xor_sync(0xffffffffu, m, mask);
    const float os = __shfl_xor_sync(0xffffffffu, s, mask);
    const MS r = ms_merge(MS{m, s}, MS{om, os});
    m = r.m;
    s = r.s;
}

// Buffer stride in bytes: a slice rounded up to 128 bytes (tensor copies land on
// 128-byte aligned shared memory).
__host__ __device__ inline size_t slab_buf_bytes(int C, int P) { return ((size_t)C * P * 4 + 127) / 128 * 128; }

// Threads that read one CTA's row of partial slots (16 bytes = two groups each): the
// pair count rounded up to a power of two, at most 32.
__host__ __device__ inline int slab_row_readers(int G) {
    const int pairs = (G + 1) / 2;
    int t = 1;
    while (t < pairs) t <<= 1;
    return t < 32 ? t : 32;
}

template <int NBMAX>
__global__ void __launch_bounds__(kSlabThreads, 1) gn_slab_kernel(const __grid_constant__ GnSlabArgs a) {
    constexpr int NF = 32 * kSlabFoldWarps, NA = 32 * kSlabApplyWarps;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int C = a.C, G = a.G, GS = a.GS, P = a.P, NB = a.NB;
    const int cpg = C / G;
    const int Ge = (G + 1) & ~1;  // slot row stride (even: rows stay 16-byte aligned)
    const int64_t N = a.N, HW = a.HW;
    const size_t bstride = slab_buf_bytes(C, P) / 4;                                     // floats per buffer
    float* const buf0 = reinterpret_cast<float*>(smem_raw);                              // [NB][C][P] (+ pad)
    float4* const tab_a = reinterpret_cast<float4*>(buf0 + (size_t)NB * bstride);        // [C]
    float2* const tab_b = reinterpret_cast<float2*>(tab_a + C);                          // [C]
    float2* const gb = tab_b + C;                                                        // [C] gamma, beta * 2log2e
    float2* const gstat = gb + C;                                                        // [G] mean, rstd
    float4* const red = reinterpret_cast<float4*>(gstat + kSlabMaxG);                    // [AW][G] (n, mean, M2)
    uint64_t* const full = reinterpret_cast<uint64_t*>(red + kSlabApplyWarps * G);       // [NB]

    const int groups = gridDim.x / GS;
    const int gi = blockIdx.x / GS, rank = blockIdx.x % GS;
    const int64_t p_begin = (int64_t)rank * P;
    const int len = (int)std::max<int64_t>(0, std::min<int64_t>(P, HW - p_begin));  // a multiple of 4
    const int64_t nsteps = gi < N ? (N - gi + groups - 1) / groups : 0;
    const int S = 2 * NB;
    unsigned long long* const slots = a.slots + (size_t)gi * S * GS * Ge;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    bool aborted = false;

    if (tid == 0) {
        for (int b = 0; b < NB; ++b) mbar_init(&full[b], 1);
        fence_mbar_init();
    }
    for (int c = tid; c < C; c += kSlabThreads)
        gb[c] = make_float2(a.gamma[c] * (2.f * kLog2e), a.beta[c] * (2.f * kLog2e));
    __syncthreads();

    // Copies step j's slice into buffer j % NB with one tensor copy (the box past HW,
    // on the last CTA of a group, arrives zero-filled), issued by lane 0 of one warp.
    uint32_t filled[NBMAX];
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) filled[b] = 0;
    const uint64_t drop = l2_policy_evict_first();
    auto issue = [&](int64_t j) {
        // every lane of the issuing warp takes the same decision
        if (j >= nsteps || __any_sync(0xffffffffu, aborted)) return;
        const int b = (int)(j % NB);
        const int64_t n = gi + j * groups;
        if (lane == 0) {
            fence_proxy_async_smem();  // earlier generic reads of the buffer come first
            mbar_arrive_expect_tx(&full[b], (uint32_t)C * (uint32_t)P * 4u);
            tma_load_2d(buf0 + (size_t)b * bstride, &a.ymap, (int)p_begin, (int)(n * C), &full[b], drop);
        }
        ++filled[b];
    };
    if (warp == kSlabFoldWarps)
        for (int j = 0; j < NB; ++j) issue(j);

    if (warp < kSlabFoldWarps) {
        // ---------------- fold warps: per-group mean and M2 of the slice, published
        // A group's rows are cpg * P contiguous floats of the buffer (Q float4), of which
        // the columns past len (last CTA of a group: zero-filled) are not the group's.
        const int Q = cpg * P / 4, P4 = P / 4, L4 = len / 4;
        // a group starts on a row, so whether quad q0 + lane + 32u lies inside the slice's
        // len columns depends on the round start q0 only; the first round's answer is kept
        uint32_t ok0 = 0;
#pragma unroll
        for (int u = 0; u < kSlabFoldQuads; ++u) {
            const int i = lane + 32 * u;
            if (i < Q && (i % P4) < L4) ok0 |= 1u << u;
        }
        for (int64_t j = 0; j < nsteps; ++j) {
            const int b = (int)(j % NB);
            mbar_wait_bounded(&full[b], (uint32_t)((j / NB) & 1), aborted, a.status);
            const float* sl = buf0 + (size_t)b * bstride;
            const uint32_t tag = (uint32_t)(j / S) & 1u;
            unsigned long long mine = 0;  // lane k holds the k-th group of this warp
            int slot_g = -1;
            int k = 0;
            for (int g = warp; g < G; g += kSlabFoldWarps, ++k) {
                const float4* grp = reinterpret_cast<const float4*>(sl + (size_t)g * cpg * P);
                Welford acc{0.f, 0.f, 0.f};
                for (int q0 = 0; q0 < Q; q0 += 32 * kSlabFoldQuads) {
                    // one round: up to kSlabFoldQuads float4 per lane, exact two passes
                    float4 v[kSlabFoldQuads];
                    uint32_t ok = ok0;
                    if (q0 > 0) {
                        ok = 0;
#pragma unroll
                        for (int u = 0; u < kSlabFoldQuads; ++u) {
                            const int i = q0 + lane + 32 * u;
                            if (i < Q && (i % P4) < L4) ok |= 1u << u;
                        }
                    }
                    int nv = 0;  // valid float4 of the round, over the warp
#pragma unroll
                    for (int u = 0; u < kSlabFoldQuads; ++u) {
                        const int i = q0 + lane + 32 * u;
                        v[u] = i < Q ? grp[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                        nv += __popc(__ballot_sync(0xffffffffu, (ok >> u) & 1u));
                    }
                    f32x2 s2 = f2_pack(0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < kSlabFoldQuads; ++u)
                        if ((ok >> u) & 1u) s2 = f2_add(s2, f2_add(f2_pack(v[u].x, v[u].y), f2_pack(v[u].z, v[u].w)));
                    float lo, hi;
                    f2_unpack(s2, lo, hi);
                    const float cnt = 4.f * (float)nv;
                    const float mean = nv > 0 ? warp_allsum(lo + hi) / cnt : 0.f;
                    const f32x2 mm = f2_pack(mean, mean);
                    f32x2 m2 = f2_pack(0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < kSlabFoldQuads; ++u) {
                        if ((ok >> u) & 1u) {
                            const f32x2 d0 = f2_sub(f2_pack(v[u].x, v[u].y), mm), d1 = f2_sub(f2_pack(v[u].z, v[u].w), mm);
                            m2 = f2_fma(d0, d0, f2_fma(d1, d1, m2));
                        }
                    }
                    f2_unpack(m2, lo, hi);
                    const float M2 = warp_allsum(lo + hi);
                    if (nv > 0) acc = wf_merge(acc, Welford{cnt, mean, M2});
                }
                if (lane == k) {
                    mine = slab_pack(acc.mean, acc.m2, tag);
                    slot_g = g;
                }
            }
            // one store per lane holding a group, all in one instruction
            if (slot_g >= 0) st_relaxed_gpu_u64(slots + ((size_t)(j % S) * GS + rank) * Ge + slot_g, mine);
        }
    } else {
        // ---------------- apply warps
        const int at = tid - NF;             // 0 .. NA - 1
        const int aw = at >> 5;              // apply warp
        const int h = lane & 7;              // channels h, h + 8, h + 16, ...
        const int q = aw * 4 + (lane >> 3);  // pixel quad of the slice
        const int px = 4 * q;
        const bool active = px < len;
        // Partial reads: TPR threads per CTA row of slots, each 16 bytes (groups 2p, 2p + 1)
        // of rows r = at / TPR + k * (NA / TPR).
        const int tpr = slab_row_readers(G);
        const int pp = at % tpr, rr = at / tpr, rstep = NA / tpr;
        const bool reader = 2 * pp < G;
        unsigned long long w0[kSlabReadsMax], w1[kSlabReadsMax];
        auto prefetch = [&](int64_t jj) {
#pragma unroll
            for (int k = 0; k < kSlabReadsMax; ++k) {
                const int r = rr + k * rstep;
                if (reader && r < GS) ld_cg_pair(slots + ((size_t)(jj % S) * GS + r) * Ge + 2 * pp, w0[k], w1[k]);
            }
        };
        if (nsteps > 0) prefetch(0);
        for (int64_t j = 0; j < nsteps; ++j) {
            const int b = (int)(j % NB);
            const int64_t n = gi + j * groups;
            const uint32_t tag = (uint32_t)(j / S) & 1u;
            // 1. this thread's partials of groups 2pp, 2pp + 1 (polled again if stale)
            Welford acc0{0.f, 0.f, 0.f}, acc1{0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < kSlabReadsMax; ++k) {
                const int r = rr + k * rstep;
                if (reader && r < GS) {
                    const unsigned long long* p = slots + ((size_t)(j % S) * GS + r) * Ge + 2 * pp;
                    const float nr = (float)(cpg * (int)std::max<int64_t>(0, std::min<int64_t>(P, HW - (int64_t)r * P)));
                    if (slab_tag(w0[k]) != tag) w0[k] = slab_poll(p, tag, aborted, a.status);
                    wf_to_slot_parts(w0[k], nr, acc0);
                    if (2 * pp + 1 < G) {
                        if (slab_tag(w1[k]) != tag) w1[k] = slab_poll(p + 1, tag, aborted, a.status);
                        wf_to_slot_parts(w1[k], nr, acc1);
                    }
                }
            }
            // merge the readers of one pair within the warp, then the warps in shared memory
            for (int o = tpr; o < 32; o <<= 1) {
                acc0 = wf_merge(acc0, wf_shfl_xor(acc0, o));
                acc1 = wf_merge(acc1, wf_shfl_xor(acc1, o));
            }
            if (reader && lane < tpr) {
                red[aw * G + 2 * pp] = make_float4(acc0.n, acc0.mean, acc0.m2, 0.f);
                if (2 * pp + 1 < G) red[aw * G + 2 * pp + 1] = make_float4(acc1.n, acc1.mean, acc1.m2, 0.f);
            }
            named_bar_sync(1, NA);  // red complete
            if (at < G) {
                Welford t{0.f, 0.f, 0.f};
                for (int wv = 0; wv < kSlabApplyWarps; ++wv) {
                    const float4 e = red[wv * G + at];
                    t = wf_merge(t, Welford{e.x, e.y, e.z});
                }
                gstat[at] = make_float2(t.mean, 1.f / sqrtf(t.m2 / t.n + a.eps));
            }
            named_bar_sync(1, NA);  // gstat complete
            for (int c = at; c < C; c += NA) {
                const float2 st = gstat[c / cpg];
                const float2 e = gb[c];
                gn_pair_entry(st.x, st.y * e.x, e.y, tab_a, tab_b, c);
            }
            mbar_wait_bounded(&full[b], (uint32_t)((j / NB) & 1), aborted, a.status);
            named_bar_sync(1, NA);  // table complete
            if (j + 1 < nsteps) prefetch(j + 1);  // the next step's partials, in flight meanwhile
            // 2. the chain on the slice: this lane's channels of its four pixels
            const float* sl = buf0 + (size_t)b * bstride + px;
            Lse4 st = lse4_empty();
            if (active) {
                constexpr int CB = 8;
                int c = h;
                for (; c + 8 * (CB - 1) < C; c += 8 * CB) {
                    f32x2 ra[CB], rb[CB];
#pragma unroll
                    for (int k = 0; k < CB; ++k) {
                        const int cc = c + 8 * k;
                        const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(sl + (size_t)cc * P);
                        const float4 ta = tab_a[cc];
                        const float2 tb = tab_b[cc];
                        const f32x2 mean = f2_pack(ta.x, ta.y), sc = f2_pack(ta.z, ta.w), sh = f2_pack(tb.x, tb.y);
                        ra[k] = f2_residual_less_2_3(v.x, mean, sc, sh);
                        rb[k] = f2_residual_less_2_3(v.y, mean, sc, sh);
                    }
                    lse4_fold<CB>(st, ra, rb);
                }
                for (; c < C; c += 8) {  // this lane's channels past its last full batch
                    const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(sl + (size_t)c * P);
                    const float4 ta = tab_a[c];
                    const float2 tb = tab_b[c];
                    const f32x2 mean = f2_pack(ta.x, ta.y), sc = f2_pack(ta.z, ta.w), sh = f2_pack(tb.x, tb.y);
                    const f32x2 ra[1] = {f2_residual_less_2_3(v.x, mean, sc, sh)};
                    const f32x2 rb[1] = {f2_residual_less_2_3(v.y, mean, sc, sh)};
                    lse4_fold<1>(st, ra, rb);
                }
            }
            // 3. merge the eight lanes of each quad (lanes 8q' + h) and write; a lane with
            // no channel (or no pixel) holds (-inf, 0)
            float m[4], s[4];
            lse4_unpack(st, m, s);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                ms_merge_xor(m[k], s[k], 1);
                ms_merge_xor(m[k], s[k], 2);
                ms_merge_xor(m[k], s[k], 4);
            }
            if (active && h == 0) {
                float4 o;
                o.x = m[0] + logf(s[0]) + 2.f / 3.f;
                o.y = m[1] + logf(s[1]) + 2.f / 3.f;
                o.z = m[2] + logf(s[2]) + 2.f / 3.f;
                o.w = m[3] + logf(s[3]) + 2.f / 3.f;
                *reinterpret_cast<float4*>(a.out + n * HW + p_begin + px) = o;
            }
            named_bar_sync(1, NA);  // every apply warp is done with buffer b and the table
            if (aw == 0) issue(j + NB);
        }
    }
    __syncthreads();
    if (warp == kSlabFoldWarps && lane == 0 && atomicAdd(a.status, 0) != 0) {
        // After a timeout anywhere, give each buffer's last issued fill one more
        // bounded wait before the shared memory is released.
        bool again = false;
        for (int b = 0; b < NB; ++b)
            if (filled[b] > 0) mbar_wait_bounded(&full[b], (filled[b] - 1) & 1u, again, a.status);
    }
}

static size_t gn_slab_smem(int C, int G, int P, int NB) {
    return (size_t)NB * slab_buf_bytes(C, P) + (size_t)C * (sizeof(float4) + 2 * sizeof(float2)) +
           kSlabMaxG * sizeof(float2) + (size_t)kSlabApplyWarps * G * sizeof(float4) + kSlabMaxNB * sizeof(uint64_t);
}

// cuTensorMapEncodeTiled from the driver, found once through the runtime (the library
// does not link the driver library itself); null if unavailable.
EncodeTiledFn encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

bool gn_slab_plan(const DeviceInfo& dev, const float* y, const float* out, int64_t N, int64_t C, int64_t HW,
                  int64_t G, GnSlabPlan* plan) {
    // (the tensor copy's coordinates are 32-bit: rows N*C and pixels HW below 2^31)
    if (HW % 4 != 0 || C > kSlabMaxC || G > kSlabMaxG || N < 1 || HW < 4 || N * C >= (1ll << 31) ||
        HW >= (1ll << 31) || (reinterpret_cast<uintptr_t>(y) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(out) & 15) != 0 || encode_tiled() == nullptr)
        return false;
    const int rows_per_pass = 32 * kSlabApplyWarps / slab_row_readers((int)G);  // as in the kernel
    const int forced = env_int("LSE_SLAB_GROUP", 0);
    const int nb_env = env_int("LSE_SLAB_NB", 0);
    const size_t budget = (size_t)dev.max_smem_optin;
    double best = -1.0;
    for (int GS = 1; GS <= dev.sm_count; ++GS) {
        if (forced && GS != forced) continue;
        const int64_t P = ((HW + GS - 1) / GS + 3) / 4 * 4;
        // at most 4 pixel quads per apply warp, no CTA of the group without pixels, and
        // at most kSlabReadsMax partial reads per merging thread
        if (P > 16 * kSlabApplyWarps || P * (GS - 1) >= HW || GS > kSlabReadsMax * rows_per_pass) continue;
        int NB = 0;
        for (int nb = kSlabMaxNB; nb >= 2; --nb)
            if (gn_slab_smem((int)C, (int)G, (int)P, nb) <= budget) {
                NB = nb;
                break;
            }
        if (nb_env) NB = (gn_slab_smem((int)C, (int)G, (int)P, nb_env) <= budget) ? nb_env : 0;
        if (NB < 2) continue;
        const int64_t groups = std::min<int64_t>(N, dev.sm_count / GS);
        if (groups < 1) continue;
        // coverage of the SMs, deeper buffering (hides the exchange), and a cost per
        // CTA of the group (each reads GS partials of every channel group)
        const double score = (double)(groups * GS) / dev.sm_count + 0.04 * std::min(NB, 4) - 0.0005 * GS;
        if (score > best) {
            best = score;
            plan->GS = GS;
            plan->P = (int)P;
            plan->NB = NB;
            plan->groups = (int)groups;
            plan->smem = gn_slab_smem((int)C, (int)G, (int)P, NB);
            plan->scratch_bytes = (size_t)groups * 2 * NB * GS * ((G + 1) & ~1) * sizeof(unsigned long long);
        }
    }
    return best >= 0.0;
}

cudaError_t launch_gn_slab(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                           int64_t N, int64_t C, int64_t HW, int64_t G, float eps, const GnSlabPlan& p, void* scratch,
                           cudaStream_t stream) {
    // every slot starts with tag 1, which no step's first use expects
    cudaError_t e = cudaMemsetAsync(scratch, 0xFF, p.scratch_bytes, stream);
    if (e != cudaSuccess) return e;
    GnSlabArgs args;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)HW, (cuuint64_t)(N * C)};
        const cuuint64_t strides[1] = {(cuuint64_t)HW * 4};
        const cuuint32_t box[2] = {(cuuint32_t)p.P, (cuuint32_t)C};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = encode_tiled()(&args.ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(y), dims,
                                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    args.y = y;
    args.gamma = gamma;
    args.beta = beta;
    args.out = out;
    args.N = N;
    args.HW = HW;
    args.C = (int)C;
    args.G = (int)G;
    args.GS = p.GS;
    args.P = p.P;
    args.NB = p.NB;
    args.eps = eps;
    args.slots = static_cast<unsigned long long*>(scratch);
    args.status = dev.status;
    auto kern = gn_slab_kernel<kSlabMaxNB>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the group waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kSlabThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)(p.groups * p.GS));
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] gn_slab: GS=%d groups=%d P=%d NB=%d smem=%zu\n", p.GS, p.groups, p.P, p.NB, p.smem);
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace lse
