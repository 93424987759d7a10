// Form 3 with y read once from HBM, every CTA on every sample: the samples are swept in
// order by the whole grid, each CTA holding one pixel slice of all C channels.
//
// GroupNorm -> tanh -> hardswish -> residual -> logsumexp over C (POPCORNBENCH page
// "Kimi-K2.6 / l2_p92"): a pixel's output needs the statistics of every group of its
// sample, and a group's statistics need every pixel of the sample.  Here CTA j of the
// grid owns pixels [p0_j, p0_j + np_j) of every sample (about HW / grid of them, a
// multiple of 4), so a sample's statistics are one grid-wide sum per group, and a pixel's
// channel lse never leaves its thread.
//
//   gn_sweep_kernel   persistent, one CTA per SM, cooperative grid.  Roles:
//     load warp     sample s into landing slot s mod R once the slot is free: one 2-D
//                   tensor copy of the box [C rows] x [PB pixels] of y (viewed as an
//                   (N*C) x HW matrix; zero fill past HW), and one of the shifts, the
//                   first four values of each channel group (y viewed as an (N*G) x
//                   (C/G * HW) matrix), both on the slot's barrier.
//     fold warps    four: per channel group (8 lanes each, 16 groups at once) the sums
//                   S1 = sum (y - K) and S2 = sum (y - K)^2 over the slice's pixels, K
//                   the group's first value, added to the sample's fp64 accumulators;
//                   once all four warps have added, one release add counts this CTA in.
//     table warp    once every CTA of the grid is counted in for the sample, its
//                   channel table from the accumulators (mean = K + S1 / N,
//                   var = S2 / N - (S1 / N)^2 in fp64, N = C / G x HW) into one of two
//                   shared-memory tables.
//     apply warps   eight: warp a takes pixels 32 (a mod 4) .. + 31 of each 128-pixel
//                   block of the slice and half of the channels (a / 4); each thread
//                   runs the chain over its
//                   pixel's channels (channel pairs packed) and folds their lse; the
//                   two halves of a pixel meet in shared memory, and the first half's
//                   thread writes the output.  Then the slot and the table are free.
//
// K is a value of the group, so |mean - K| is of the order of the group's spread and the
// variance does not cancel.  A non-finite y makes S1 or S2 non-finite, hence a NaN
// variance, and its sample's outputs are NaN.  (The fp64 additions land in any order: the
// statistics may differ from run to run in the last bits of fp64, far below fp32.)
//
// Progress: a CTA folds its slice of sample s once the slot is free, which needs its own
// apply of sample s - R, which needs every CTA's fold of sample s - R.  Every CTA folds
// in sample order, so by induction on s every fold and every apply ends (the first R
// samples need no free slot).  Every wait is bounded (about 1 s) and records a timeout in
// the device status word.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "gn_common.cuh"
#include "launch.h"
#include "tmem.cuh"

namespace lse {

constexpr int kGsMaxSlots = 8;
constexpr int kGsMaxC = 64;        // channels (table warp: two groups per lane; apply: C / 2 per thread)
constexpr int kGsMaxBox = 256;     // pixels per slice: the tensor copy's box width
constexpr int kGsFoldWarps = 4;
constexpr int kGsApplyWarps = 8;
constexpr int kGsFold0 = 1, kGsTableWarp = kGsFold0 + kGsFoldWarps, kGsApply0 = kGsTableWarp + 1;
constexpr int kGsThreads = 32 * (kGsApply0 + kGsApplyWarps);
constexpr int kGsSegLanes = 8;     // lanes of a fold segment: one channel group at a time
constexpr int kGsSegments = kGsFoldWarps * 32 / kGsSegLanes;
constexpr int kGsApplyBar = 1, kGsFoldBar = 2;  // named barriers

struct GnSweepArgs {
    CUtensorMap ymap;  // y as an (N*C) x HW fp32 matrix, box PB x C
    CUtensorMap kmap;  // y as an (N*G) x (C/G*HW) fp32 matrix, box 4 x G (the shifts)
    const float* gamma;
    const float* beta;
    float* out;
    int64_t N, HW;
    int C, G, PB, R;
    float eps;
    unsigned* cnt;  // [N] CTAs counted in, one 128-byte line each, zero at launch
    double2* acc;   // [N][G] (S1, S2), one 128-byte line each, zero at launch
    int* status;
};

// A slot: y [C][PB], then at a 128-byte boundary the shifts [G][4].
__host__ __device__ static inline size_t gs_koff(int C, int PB) { return ((size_t)C * PB * 4 + 127) / 128 * 128; }
__host__ __device__ static inline size_t gs_slot_bytes(int C, int PB, int G) {
    return (gs_koff(C, PB) + (size_t)G * 16 + 127) / 128 * 128;
}
__host__ __device__ static inline size_t gs_smem(int C, int PB, int G, int R) {
    return (size_t)R * gs_slot_bytes(C, PB, G) + (size_t)2 * C * sizeof(float4) + (size_t)2 * 256 * sizeof(float2) +
           (size_t)2 * kGsMaxC * sizeof(float) + (size_t)(3 * kGsMaxSlots + 4) * 8;
}

__global__ void __launch_bounds__(kGsThreads, 1) gn_sweep_kernel(const __grid_constant__ GnSweepArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int C = a.C, G = a.G, PB = a.PB, R = a.R;
    const int cpg = C / G;
    const int64_t N = a.N, HW = a.HW;
    const size_t slot_bytes = gs_slot_bytes(C, PB, G);
    unsigned char* const slots = smem_raw;                                                // [R] slot: [C][PB] y, [G][4] K
    float4* const tab = reinterpret_cast<float4*>(smem_raw + (size_t)R * slot_bytes);    // [2][C]
    float2* const xbuf = reinterpret_cast<float2*>(tab + 2 * C);                          // [2][256]
    float* const gamma_s = reinterpret_cast<float*>(xbuf + 2 * 256);                      // [kGsMaxC]
    float* const beta_s = gamma_s + kGsMaxC;                                              // [kGsMaxC]
    uint64_t* const full = reinterpret_cast<uint64_t*>(beta_s + kGsMaxC);                 // [kGsMaxSlots]
    uint64_t* const sfree = full + kGsMaxSlots;                                           // [kGsMaxSlots]
    uint64_t* const folded = sfree + kGsMaxSlots;                                         // [kGsMaxSlots]
    uint64_t* const tfull = folded + kGsMaxSlots;                                         // [2]
    uint64_t* const tfree = tfull + 2;                                                    // [2]
    auto ydata = [&](int sl) { return reinterpret_cast<float*>(slots + (size_t)sl * slot_bytes); };
    auto kdata = [&](int sl) { return reinterpret_cast<float*>(slots + (size_t)sl * slot_bytes + gs_koff(C, PB)); };

    // the counter of sample s and the sums of (s, g), each alone in its 128-byte line:
    // 152 CTAs poll and add there every sample
    auto cnt_of = [&](int64_t s) { return a.cnt + (size_t)s * 32; };
    auto acc_of = [&](int64_t s, int g) { return a.acc + ((size_t)s * G + g) * 8; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's pixel slice: quads [Q j / grid, Q (j + 1) / grid)
    const int64_t Q = HW / 4;
    const int64_t q0 = Q * blockIdx.x / gridDim.x, q1 = Q * (blockIdx.x + 1) / gridDim.x;
    const int p0 = (int)(4 * q0), np = (int)(4 * (q1 - q0));
    bool aborted = false;
    int64_t issued = 0;  // load warp: samples whose copies have been issued

    if (tid == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&full[r], 1);
            mbar_init(&sfree[r], 1);
            mbar_init(&folded[r], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&tfull[k], 1);
            mbar_init(&tfree[k], 1);
        }
        fence_mbar_init();
    }
    for (int c = tid; c < C; c += kGsThreads) {
        gamma_s[c] = a.gamma[c];
        beta_s[c] = a.beta[c];
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------- load warp
        if (lane == 0) {
            const uint64_t drop = l2_policy_evict_first();
            const uint32_t bytes = (uint32_t)((size_t)C * PB * 4 + (size_t)G * 16);
            for (int64_t s = 0; s < N; ++s) {
                const int sl = (int)(s % R);
                if (s >= R) mbar_wait_bounded(&sfree[sl], (uint32_t)((s / R - 1) & 1), aborted, a.status);
                if (aborted) break;
                mbar_arrive_expect_tx(&full[sl], bytes);
                tma_load_2d(ydata(sl), &a.ymap, p0, (int)(s * C), &full[sl], drop);
                tma_load_2d(kdata(sl), &a.kmap, 0, (int)(s * G), &full[sl], drop);
                issued = s + 1;
            }
        }
    } else if (warp < kGsTableWarp) {
        // ---------------- fold warps: the slice's shifted sums per group, into the accumulators
        const int sg = (warp - kGsFold0) * (32 / kGsSegLanes) + (lane >> 3), j = lane & 7;
        const int nq = np / 4;
        // (after a timeout the loop still runs to the end, without work, so that every fold
        // warp meets the named barrier the same number of times)
        for (int64_t s = 0; s < N; ++s) {
            const int sl = (int)(s % R);
            mbar_wait_bounded(&full[sl], (uint32_t)((s / R) & 1), aborted, a.status);
            const bool skip = __any_sync(0xffffffffu, aborted);
            const float* y = ydata(sl);
            for (int g0 = 0; g0 < (skip ? 0 : G); g0 += kGsSegments) {
                const int gg = g0 + sg;
                f32x2 s1a = f2_pack(0.f, 0.f), s1b = s1a, s2a = s1a, s2b = s1a;
                if (gg < G) {
                    const float K = kdata(sl)[4 * gg];
                    const f32x2 k2v = f2_pack(K, K);
                    for (int r = 0; r < cpg; ++r) {
                        const float4* row = reinterpret_cast<const float4*>(y + (size_t)(gg * cpg + r) * PB);
                        // a row has at most kGsMaxBox / 4 quads: at most 8 per lane, loaded together
#pragma unroll
                        for (int i = 0; i < kGsMaxBox / 4 / kGsSegLanes; ++i) {
                            const int k = j + i * kGsSegLanes;
                            if (k < nq) {
                                const float4 u = row[k];
                                const f32x2 da = f2_sub(f2_pack(u.x, u.y), k2v), db = f2_sub(f2_pack(u.z, u.w), k2v);
                                s1a = f2_add(s1a, da);
                                s1b = f2_add(s1b, db);
                                s2a = f2_fma(da, da, s2a);
                                s2b = f2_fma(db, db, s2b);
                            }
                        }
                    }
                }
                float x0, x1, x2, x3, w0, w1, w2, w3;
                f2_unpack(s1a, x0, x1);
                f2_unpack(s1b, x2, x3);
                f2_unpack(s2a, w0, w1);
                f2_unpack(s2b, w2, w3);
                float s1 = (x0 + x1) + (x2 + x3), s2 = (w0 + w1) + (w2 + w3);
                for (int o = kGsSegLanes / 2; o > 0; o >>= 1) {
                    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
                    s2 += __shfl_xor_sync(0xffffffffu, s2, o);
                }
                if (j == 0 && gg < G) {
                    double* dst = reinterpret_cast<double*>(acc_of(s, gg));
                    asm volatile("red.global.add.f64 [%0], %1;" ::"l"(dst), "d"((double)s1) : "memory");
                    asm volatile("red.global.add.f64 [%0], %1;" ::"l"(dst + 1), "d"((double)s2) : "memory");
                }
            }
            // every fold warp's additions for sample s are made: count this CTA in (release,
            // cumulative over the additions ordered before it by the barrier)
            named_bar_sync(kGsFoldBar, 32 * kGsFoldWarps);
            if (warp == kGsFold0 && lane == 0) {
                if (!skip) red_release_gpu_add(cnt_of(s), 1u);
                mbar_arrive(&folded[sl]);  // the table warp polls only once this CTA is counted in
            }
        }
    } else if (warp == kGsTableWarp) {
        // ---------------- table warp: lane l takes groups l and l + 32
        const float k2 = 2.f * kLog2e;
        const double inv_n = 1.0 / ((double)cpg * (double)HW);
        const unsigned ctas = gridDim.x;
        for (int64_t s = 0; s < N; ++s) {
            const int sl = (int)(s % R), b = (int)(s & 1);
            mbar_wait_bounded(&full[sl], (uint32_t)((s / R) & 1), aborted, a.status);
            const float kA = lane < G ? kdata(sl)[4 * lane] : 0.f;
            const float kB = lane + 32 < G ? kdata(sl)[4 * (lane + 32)] : 0.f;
            mbar_wait_bounded(&folded[sl], (uint32_t)((s / R) & 1), aborted, a.status);
            if (lane == 0 && !aborted && ld_acquire_gpu_u32(cnt_of(s)) < ctas) {
                const uint64_t t0 = globaltimer_ns();
                bool ok = false;
                for (uint32_t it = 0; it < (1u << 26); ++it) {
                    __nanosleep(128);
                    if (ld_acquire_gpu_u32(cnt_of(s)) >= ctas) {
                        ok = true;
                        break;
                    }
                    if ((it & 255u) == 255u && globaltimer_ns() - t0 > 1000000000ull) break;
                }
                if (!ok) {
                    aborted = true;
                    atomicExch(a.status, kStatusTimeout);
                }
            }
            if (__any_sync(0xffffffffu, aborted)) break;  // lane 0's acquire orders the reads below
            auto stats = [&](int gg, float k, float& mean, float& rstd) {
                mean = 0.f;
                rstd = 0.f;
                if (gg >= G) return;
                const double2 sa = __ldcg(acc_of(s, gg));
                const double m1 = sa.x * inv_n;
                const double v = sa.y * inv_n - m1 * m1;        // NaN when a value is not finite
                const float var = (float)(v < 0.0 ? 0.0 : v);  // rounding below 0 only; NaN kept
                mean = (float)((double)k + m1);
                rstd = 1.f / sqrtf(var + a.eps);
            };
            float mA, rA, mB, rB;
            stats(lane, kA, mA, rA);
            stats(lane + 32, kB, mB, rB);
            if (s >= 2) mbar_wait_bounded(&tfree[b], (uint32_t)((s / 2 - 1) & 1), aborted, a.status);
            for (int c0 = 0; c0 < C; c0 += 32) {
                const int c = c0 + lane;
                const int gg = (c < C ? c : C - 1) / cpg;
                const float m0 = __shfl_sync(0xffffffffu, mA, gg & 31), m1 = __shfl_sync(0xffffffffu, mB, gg & 31);
                const float r0 = __shfl_sync(0xffffffffu, rA, gg & 31), r1 = __shfl_sync(0xffffffffu, rB, gg & 31);
                if (c < C) {
                    const float mean = gg < 32 ? m0 : m1, rstd = gg < 32 ? r0 : r1;
                    tab[(size_t)b * C + c] = make_float4(mean, rstd * gamma_s[c] * k2, beta_s[c] * k2, 0.f);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&tfull[b]);
        }
    } else {
        // ---------------- apply warps: one pixel per thread, half of the channels (after a
        // timeout the loop runs on without work, meeting the named barrier every time)
        const int aw = warp - kGsApply0;
        const int h = aw >> 2;
        const int ch = C / 2, c_lo = h * ch;
        for (int64_t s = 0; s < N; ++s) {
            const int sl = (int)(s % R), b = (int)(s & 1);
            mbar_wait_bounded(&tfull[b], (uint32_t)((s / 2) & 1), aborted, a.status);
            mbar_wait_bounded(&full[sl], (uint32_t)((s / R) & 1), aborted, a.status);
            const float4* tb = tab + (size_t)b * C;
            // pixel blocks of 128 (a slice has at most 256 pixels)
            for (int pb = 0; pb < PB; pb += 128) {
                const int p = pb + 32 * (aw & 3) + lane;
                const bool active = p < np && !aborted;
                MS st = ms_empty();
                if (active) {
                    const float* y = ydata(sl) + p;
                    // channel pairs packed: r - 2/3 of channels c, c + 1 in one pair
                    auto pair = [&](int c) {
                        const float4 e0 = tb[c], e1 = tb[c + 1];
                        return f2_residual_less_2_3(f2_pack(y[(size_t)c * PB], y[(size_t)(c + 1) * PB]),
                                                    f2_pack(e0.x, e1.x), f2_pack(e0.y, e1.y), f2_pack(e0.z, e1.z));
                    };
                    int c = c_lo;
                    for (; c + 8 <= c_lo + ch; c += 8) {
                        float r[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) f2_unpack(pair(c + 2 * k), r[2 * k], r[2 * k + 1]);
                        ms_fold<8>(st, r);
                    }
                    for (; c < c_lo + ch; c += 2) {
                        float r[2];
                        f2_unpack(pair(c), r[0], r[1]);
                        ms_fold<2>(st, r);
                    }
                }
                float2* const xb = xbuf + (size_t)b * 256 + pb;
                if (h == 1 && active) xb[p - pb] = make_float2(st.m, st.s);
                named_bar_sync(kGsApplyBar, 32 * kGsApplyWarps);  // the second halves are in xb
                if (h == 0 && active) {
                    const float2 o = xb[p - pb];
                    a.out[(size_t)s * HW + p0 + p] = ms_lse(ms_merge(st, MS{o.x, o.y})) + 2.f / 3.f;
                }
            }
            // every read of slot sl and of tab[b] is behind the last barrier
            if (aw == 0 && lane == 0) {
                mbar_arrive(&sfree[sl]);
                mbar_arrive(&tfree[b]);
            }
        }
    }
    __syncthreads();
    if (warp == 0 && lane == 0 && atomicAdd(a.status, 0) != 0) {
        // After a timeout anywhere: one more bounded wait for the copies still in flight
        // before the shared memory is released.
        bool again = false;
        for (int64_t s = std::max<int64_t>(0, issued - R); s < issued; ++s)
            mbar_wait_bounded(&full[s % R], (uint32_t)((s / R) & 1), again, a.status);
    }
}

// Scratch, zeroed at launch: the counters [N], then the accumulators [N][G] (S1, S2) in
// fp64, each in a 128-byte line of its own.
static size_t gs_acc_offset(int64_t N) { return (size_t)N * 128; }
static size_t gs_scratch_bytes(int64_t N, int64_t G) { return gs_acc_offset(N) + (size_t)N * G * 128; }

bool gn_sweep_plan(const DeviceInfo& dev, const float* y, int64_t N, int64_t C, int64_t HW, int64_t G,
                   GnSweepPlan* plan) {
    // (the tensor copies' coordinates are 32-bit: rows N*C and columns below 2^31)
    if (HW % 4 != 0 || HW < 4 || C % 4 != 0 || C < 4 || C > kGsMaxC || G < 1 || G > 64 || C % G != 0 || N < 1 ||
        N * C >= (1ll << 31) || (C / G) * HW >= (1ll << 31) || (reinterpret_cast<uintptr_t>(y) & 15) != 0 ||
        encode_tiled() == nullptr)
        return false;
    const int64_t Q = HW / 4;
    const int grid = (int)std::min<int64_t>(dev.sm_count, Q);
    const int PB = (int)(4 * ((Q + grid - 1) / grid));
    if (PB > kGsMaxBox) return false;
    const size_t budget = (size_t)dev.max_smem_optin;
    int R = 0;
    for (int r = kGsMaxSlots; r >= 3; --r)
        if (gs_smem((int)C, PB, (int)G, r) <= budget) {
            R = r;
            break;
        }
    const int slots_env = env_int("LSE_GNS_SLOTS", 0);
    if (slots_env >= 3 && slots_env < R) R = slots_env;
    if (R < 3) return false;
    plan->grid = grid;
    plan->PB = PB;
    plan->R = R;
    plan->threads = kGsThreads;
    plan->smem = std::max(gs_smem((int)C, PB, (int)G, R), budget / 2 + 1024);  // one CTA per SM
    plan->scratch_bytes = gs_scratch_bytes(N, G);
    return plan->smem <= budget;
}

cudaError_t launch_gn_sweep(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                            int64_t N, int64_t C, int64_t HW, int64_t G, float eps, const GnSweepPlan& p,
                            void* scratch, cudaStream_t stream) {
    unsigned char* base = static_cast<unsigned char*>(scratch);
    cudaError_t e = cudaMemsetAsync(base, 0, gs_scratch_bytes(N, G), stream);
    if (e != cudaSuccess) return e;
    GnSweepArgs args;
    const cuuint32_t estr[2] = {1, 1};
    {
        const cuuint64_t dims[2] = {(cuuint64_t)HW, (cuuint64_t)(N * C)};
        const cuuint64_t strides[1] = {(cuuint64_t)HW * 4};
        const cuuint32_t box[2] = {(cuuint32_t)p.PB, (cuuint32_t)C};
        const CUresult r = encode_tiled()(&args.ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(y), dims,
                                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const int64_t cpg = C / G;
        const cuuint64_t dims[2] = {(cuuint64_t)(cpg * HW), (cuuint64_t)(N * G)};
        const cuuint64_t strides[1] = {(cuuint64_t)(cpg * HW) * 4};
        const cuuint32_t box[2] = {4, (cuuint32_t)G};
        const CUresult r = encode_tiled()(&args.kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(y), dims,
                                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    args.gamma = gamma;
    args.beta = beta;
    args.out = out;
    args.N = N;
    args.HW = HW;
    args.C = (int)C;
    args.G = (int)G;
    args.PB = p.PB;
    args.R = p.R;
    args.eps = eps;
    args.cnt = reinterpret_cast<unsigned*>(base);
    args.acc = reinterpret_cast<double2*>(base + gs_acc_offset(N));
    args.status = dev.status;
    e = cudaFuncSetAttribute(gn_sweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gn_sweep_kernel, p.threads, p.smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: every sample needs every CTA
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)p.grid);
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] gn_sweep: grid=%d slice=%d R=%d smem=%zu\n", p.grid, p.PB, p.R, p.smem);
    e = cudaLaunchKernelEx(&cfg, gn_sweep_kernel, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace lse
