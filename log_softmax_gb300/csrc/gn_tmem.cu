// Form 3 with y read once from HBM and each tile parked in tensor memory between its
// statistics and its use.
//
// GroupNorm -> tanh -> hardswish -> residual -> logsumexp over C (POPCORNBENCH page
// "Kimi-K2.6 / l2_p92"): a pixel's output needs the statistics of every group of its
// sample, and a group's statistics need every pixel of the sample.  The work-queue
// kernel (gn_act_lse.cu) reads each sample twice and relies on L2 for the second
// read; here the second read is from tensor memory (256 KB per SM, unused by this
// path's arithmetic):
//
//   gn_tmem_kernel   persistent, one CTA per SM, cooperative grid.  Work items are
//                    tiles of 256 pixels x all C channels of one sample, claimed from
//                    one counter in sample order.  Roles:
//                      load warp    claims a tile once a landing slot is free,
//                                   announces it to the other roles, and copies the
//                                   box [C rows] x [256 pixels] of y (viewed as an
//                                   (N*C) x HW matrix) into the slot with one 2-D
//                                   tensor copy (zero fill past HW).
//                      fold warps   the sums of d = y - K and d^2 over each channel
//                                   group's valid pixels of the tile (8 lanes per group,
//                                   16 groups at once; K, the shift, is one element of
//                                   the group), added to the sample's fp64 accumulators
//                                   S1 = sum d, S2 = sum d^2.
//                      publish warp counts the tile in (a release add per tile, after
//                                   its fold warps' additions).
//                      copy warp    copies the folded tile into tensor memory
//                                   (tcgen05.cp, 4 KB blocks of four channel rows)
//                                   once one of the TR tile buffers is free; the
//                                   landing slot is free when the copy completes.
//                      table warp   once every tile of the tile's sample is counted
//                                   in, its channel table from the accumulators
//                                   (mean = K + S1 / N, var = S2 / N - (S1 / N)^2 in
//                                   fp64, N = C / G x HW) into shared memory.
//                      apply warps  eight: a warp reads its quarter of the lanes
//                                   (lane l holds pixels 4 (l mod 64) .. + 3 of the
//                                   even channels for l < 64 and of the odd ones
//                                   above) for half of the channel blocks, runs the
//                                   chain and folds the channel lse of its four
//                                   pixels; the four partial lse of a pixel quad meet
//                                   in shared memory, and each of the quad's four warps
//                                   merges and writes one of its pixels.
//
// K is a value of the group, so |mean - K| is of the order of the group's spread and
// var = S2 / N - (S1 / N)^2 does not cancel: the variance keeps fp32 accuracy even where
// the mean is many times the spread.  A non-finite y gives S1 or S2 infinite or NaN,
// hence a NaN variance, and its sample's outputs are NaN, as the definition has them.
// (The fp64 additions land in any order: the statistics may differ from run to run in
// the last bits of fp64, far below fp32 rounding.)
//
// y is read from HBM exactly once, but the kernel is bound by latency: a tile waits for
// the last tile of its sample and for the tiles ahead of it in its CTA, with one warp
// or eight per role and four tiles per SM in flight; on GB300 it is slower than the
// work queue, which keeps 32 warps per SM busy (the selectable LSE_GN_VARIANT=5).
//
// Claimed tiles are folded and counted in whatever the state of the other roles, so
// every sample whose tiles are all claimed becomes complete.  A CTA stops claiming
// only when all its tile buffers hold tiles of samples not yet complete; if every CTA
// stopped so, the grid would hold TR x grid tiles of the sample being claimed and
// later ones, which is impossible while TR x grid >= T (tiles per sample), the plan's
// condition.  Every wait is bounded (about 1 s) and records a timeout in the device
// status word.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "gn_common.cuh"
#include "launch.h"
#include "tmem.cuh"

namespace lse {

constexpr int kGtPix = 256;        // pixels per tile: the tensor copy's box width
constexpr int kGtMaxC = 64;        // 2 C tensor-memory columns per tile, at least 4 tiles in 512
constexpr int kGtMaxSlots = 8;     // landing slots in shared memory
constexpr int kGtMaxTiles = 8;     // tile buffers in tensor memory
constexpr int kGtRing = 32;        // announced tiles (more than slots + buffers in flight)
constexpr int kGtFoldWarps = 4;
constexpr int kGtApplyWarps = 8;
constexpr int kGtApply0 = kGtFoldWarps;
constexpr int kGtLoadWarp = kGtFoldWarps + kGtApplyWarps;
constexpr int kGtCopyWarp = kGtLoadWarp + 1;
constexpr int kGtTableWarp = kGtLoadWarp + 2;
constexpr int kGtPublishWarp = kGtLoadWarp + 3;
constexpr int kGtThreads = 32 * (kGtPublishWarp + 1);
constexpr int kGtSegLanes = 8;     // lanes of a fold segment: one channel group at a time
constexpr int kGtSegments = kGtFoldWarps * 32 / kGtSegLanes;
constexpr uint32_t kGtTmemCols = 512;

struct GnTmemArgs {
    CUtensorMap ymap;  // y as an (N*C) x HW fp32 matrix, box 256 x C, no swizzle, zero fill past HW
    const float* y;
    const float* gamma;
    const float* beta;
    float* out;
    int64_t N, HW;
    int C, G, T, TR, R;
    float eps;
    unsigned long long* next;  // tile counter, zero at launch
    unsigned* cnt;             // [N] tiles counted in, zero at launch
    double2* acc;              // [N][G] (S1, S2), zero at launch
    int* status;
};

// Valid pixels of tile t (a multiple of 4: HW is).
__device__ __forceinline__ int gt_valid(int64_t HW, int t) {
    return (int)std::min<int64_t>(kGtPix, HW - (int64_t)t * kGtPix);
}

// The shift of group g of sample n: the group's first element.
__device__ __forceinline__ float gt_shift(const GnTmemArgs& a, int64_t n, int g) {
    return __ldg(a.y + ((size_t)n * a.C + (size_t)g * (a.C / a.G)) * a.HW);
}

__global__ void __launch_bounds__(kGtThreads, 1) gn_tmem_kernel(const __grid_constant__ GnTmemArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const int C = a.C, G = a.G, T = a.T, TR = a.TR, R = a.R;
    const int cpg = C / G;
    const int64_t HW = a.HW;
    const int64_t total = a.N * T;
    const size_t slot_floats = (size_t)C * kGtPix;
    float* const slots = reinterpret_cast<float*>(smem_raw);                            // [R][C][256]
    float4* const tab = reinterpret_cast<float4*>(slots + (size_t)R * slot_floats);     // [TR][C]
    float* const xbuf = reinterpret_cast<float*>(tab + (size_t)TR * C);                 // [2][kGtApplyWarps][32][8]
    uint64_t* const full = reinterpret_cast<uint64_t*>(xbuf + 2 * kGtApplyWarps * 32 * 8);  // [kGtMaxSlots]
    uint64_t* const freed = full + kGtMaxSlots;                                         // [kGtMaxSlots]
    uint64_t* const folded = freed + kGtMaxSlots;                                       // [kGtMaxSlots]
    uint64_t* const tfree = folded + kGtMaxSlots;                                       // [kGtMaxTiles]
    uint64_t* const tready = tfree + kGtMaxTiles;                                       // [kGtMaxTiles]
    uint64_t* const tabready = tready + kGtMaxTiles;                                    // [kGtMaxTiles]
    uint64_t* const xfull = tabready + kGtMaxTiles;                                     // [2]
    uint64_t* const xfree = xfull + 2;                                                  // [2]
    uint64_t* const claimed = xfree + 2;                                                // [kGtRing]
    uint64_t* const written = claimed + kGtRing;                                        // [kGtRing]
    long long* const gid_s = reinterpret_cast<long long*>(written + kGtRing);           // [kGtRing]
    long long* const copied_s = gid_s + kGtRing;                                        // [1]
    float* const gamma_s = reinterpret_cast<float*>(copied_s + 1);                      // [kGtMaxC]
    float* const beta_s = gamma_s + kGtMaxC;                                            // [kGtMaxC]
    uint32_t* const tslot = reinterpret_cast<uint32_t*>(beta_s + kGtMaxC);              // [1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    bool aborted = false;
    int64_t issued = 0;  // load warp: tiles whose tensor copy has been issued

    if (warp == 0) tmem_alloc_warp(tslot, kGtTmemCols);
    if (tid == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&full[r], 1);
            mbar_init(&freed[r], 1);
            mbar_init(&folded[r], kGtFoldWarps);
        }
        for (int b = 0; b < TR; ++b) {
            mbar_init(&tfree[b], kGtApplyWarps);
            mbar_init(&tready[b], 1);
            mbar_init(&tabready[b], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&xfull[k], kGtApplyWarps);
            mbar_init(&xfree[k], kGtApplyWarps);
        }
        for (int k = 0; k < kGtRing; ++k) {
            mbar_init(&claimed[k], 1);
            mbar_init(&written[k], kGtFoldWarps);
        }
        *copied_s = 0;
        fence_mbar_init();
    }
    for (int c = tid; c < C; c += kGtThreads) {  // the tables' per-channel affine
        gamma_s[c] = a.gamma[c];
        beta_s[c] = a.beta[c];
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tcols = 2u * (uint32_t)C;  // tensor-memory columns of one tile

    // Item i of this CTA (its i-th claimed tile), or -1 once the work is out (or after
    // a timeout); the same value in every lane of the warp.
    auto item = [&](int64_t i) -> long long {
        mbar_wait_bounded(&claimed[i % kGtRing], (uint32_t)((i / kGtRing) & 1), aborted, a.status);
        aborted = __any_sync(0xffffffffu, aborted);
        const long long g = *reinterpret_cast<volatile long long*>(gid_s + i % kGtRing);
        return aborted ? -1ll : __shfl_sync(0xffffffffu, g, 0);
    };

    if (warp == kGtLoadWarp) {
        // ---------------- load warp: claim, announce, copy the box into a landing slot
        if (lane == 0) {
            const uint64_t drop = l2_policy_evict_first();
            for (int64_t i = 0;; ++i) {
                const int sl = (int)(i % R);
                if (i >= R) mbar_wait_bounded(&freed[sl], (uint32_t)(((i - R) / R) & 1), aborted, a.status);
                long long g = aborted ? -1ll : (long long)atomicAdd(a.next, 1ull);
                if (g >= total) g = -1;
                gid_s[i % kGtRing] = g;
                mbar_arrive(&claimed[i % kGtRing]);  // release: the announcement is visible to the waiters
                if (g < 0) break;
                const long long n = g / T;
                const int t = (int)(g - n * T);
                mbar_arrive_expect_tx(&full[sl], (uint32_t)(slot_floats * 4));
                tma_load_2d(slots + (size_t)sl * slot_floats, &a.ymap, t * kGtPix, (int)(n * C), &full[sl], drop);
                issued = i + 1;
            }
        }
    } else if (warp < kGtFoldWarps) {
        // ---------------- fold warps: per-group moments of the tile, written to global memory
        for (int64_t i = 0;; ++i) {
            const long long g = item(i);
            if (g < 0) break;
            const long long n = g / T;
            const int t = (int)(g - n * T);
            const int nv = gt_valid(HW, t);
            const int sl = (int)(i % R);
            mbar_wait_bounded(&full[sl], (uint32_t)((i / R) & 1), aborted, a.status);
            const float* slot = slots + (size_t)sl * slot_floats;
            // segment sg (8 lanes) takes groups sg, sg + 16, ...; lane j of it the float4
            // j, j + 8, ..., j + 56 of each of the group's rows (a warp load: 4 rows x 128 B).
            // Per lane, the sums of d = y - K and d^2 over its valid values (packed pairs,
            // two independent accumulators each); then the segment's sums (fixed order).
            const int sg = warp * (32 / kGtSegLanes) + (lane >> 3), j = lane & 7;
            for (int g0 = 0; g0 < G; g0 += kGtSegments) {
                const int gg = g0 + sg;
                const float K = gg < G ? gt_shift(a, n, gg) : 0.f;  // issued before the loads below
                const f32x2 k2v = f2_pack(K, K);
                f32x2 s1a = f2_pack(0.f, 0.f), s1b = s1a, s2a = s1a, s2b = s1a;
                if (gg < G) {
                    for (int r = 0; r < cpg; ++r) {
                        const float4* row = reinterpret_cast<const float4*>(slot + (size_t)(gg * cpg + r) * kGtPix);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            if (nv == kGtPix || 4 * (8 * k + j) < nv) {
                                const float4 u = row[8 * k + j];
                                const f32x2 da = f2_sub(f2_pack(u.x, u.y), k2v), db = f2_sub(f2_pack(u.z, u.w), k2v);
                                s1a = f2_add(s1a, da);
                                s1b = f2_add(s1b, db);
                                s2a = f2_fma(da, da, s2a);
                                s2b = f2_fma(db, db, s2b);
                            }
                        }
                    }
                }
                float x0, x1, x2, x3, q0, q1, q2, q3;
                f2_unpack(s1a, x0, x1);
                f2_unpack(s1b, x2, x3);
                f2_unpack(s2a, q0, q1);
                f2_unpack(s2b, q2, q3);
                float s1 = (x0 + x1) + (x2 + x3), s2 = (q0 + q1) + (q2 + q3);
                for (int o = kGtSegLanes / 2; o > 0; o >>= 1) {
                    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
                    s2 += __shfl_xor_sync(0xffffffffu, s2, o);
                }
                if (j == 0 && gg < G) {
                    double* dst = reinterpret_cast<double*>(a.acc + (size_t)n * G + gg);
                    atomicAdd(dst, (double)s1);
                    atomicAdd(dst + 1, (double)s2);
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&folded[sl]);               // this warp is done reading slot sl
                mbar_arrive(&written[i % kGtRing]);     // and its additions for item i are made
            }
        }
    } else if (warp == kGtPublishWarp) {
        // ---------------- publish warp: count each tile in once its fold warps' additions are made
        if (lane == 0) {
            for (int64_t i = 0;; ++i) {
                mbar_wait_bounded(&claimed[i % kGtRing], (uint32_t)((i / kGtRing) & 1), aborted, a.status);
                const long long g = aborted ? -1ll : *reinterpret_cast<volatile long long*>(gid_s + i % kGtRing);
                if (g < 0) break;
                mbar_wait_bounded(&written[i % kGtRing], (uint32_t)((i / kGtRing) & 1), aborted, a.status);
                // release (cumulative): the fold warps' additions, seen through the mbarrier above
                red_release_gpu_add(a.cnt + g / T, 1u);
            }
        }
    } else if (warp == kGtCopyWarp) {
        // ---------------- copy warp: folded tiles into tensor memory
        if (lane == 0) {
            long long copied = 0;
            for (int64_t i = 0;; ++i) {
                mbar_wait_bounded(&claimed[i % kGtRing], (uint32_t)((i / kGtRing) & 1), aborted, a.status);
                const long long g = aborted ? -1ll : *reinterpret_cast<volatile long long*>(gid_s + i % kGtRing);
                if (g < 0) break;
                const int sl = (int)(i % R), b = (int)(i % TR);
                mbar_wait_bounded(&folded[sl], (uint32_t)((i / R) & 1), aborted, a.status);
                if (i >= TR)  // the apply warps have released buffer b's previous tile
                    mbar_wait_bounded(&tfree[b], (uint32_t)(((i - TR) / TR) & 1), aborted, a.status);
                tmem_fence_after();
                if (aborted) break;
                const float* slot = slots + (size_t)sl * slot_floats;
                for (int k = 0; k < C / 4; ++k) tmem_cp_block(tbase + (uint32_t)b * tcols + 8u * k, slot + 1024 * k);
                tmem_commit(&freed[sl]);
                tmem_commit(&tready[b]);
                copied = i + 1;
            }
            *copied_s = copied;
        }
    } else if (warp == kGtTableWarp) {
        // ---------------- table warp: the tile's channel table, once its sample is complete.
        // Lane l holds groups l and l + 32: shifts loaded first, the counter polled, the
        // group statistics computed, and only then the wait for tab[b] to be free.
        const float k2 = 2.f * kLog2e;
        const double inv_n = 1.0 / ((double)cpg * (double)HW);
        for (int64_t i = 0;; ++i) {
            const long long g = item(i);
            if (g < 0) break;
            const long long n = g / T;
            const int b = (int)(i % TR);
            float kA = 0.f, kB = 0.f;
            if (lane < G) kA = gt_shift(a, n, lane);
            if (lane + 32 < G) kB = gt_shift(a, n, lane + 32);
            if (lane == 0 && !aborted && ld_acquire_gpu_u32(a.cnt + n) < (unsigned)T) {
                const uint64_t t0 = globaltimer_ns();
                bool ok = false;
                for (uint32_t it = 0; it < (1u << 26); ++it) {
                    __nanosleep(32);
                    if (ld_acquire_gpu_u32(a.cnt + n) >= (unsigned)T) {
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
            __syncwarp();  // lane 0's acquire orders the accumulator reads below
            // mean = K + S1 / N, var = S2 / N - (S1 / N)^2 (fp64, S1 / N of the order of the spread)
            auto stats = [&](int gg, float k, float& mean, float& rstd) {
                mean = 0.f;
                rstd = 0.f;
                if (gg >= G) return;
                const double2 sa = __ldcg(a.acc + (size_t)n * G + gg);
                const double m1 = sa.x * inv_n;
                const double v = sa.y * inv_n - m1 * m1;  // NaN when a value is not finite
                const float var = (float)(v < 0.0 ? 0.0 : v);  // rounding below 0 only; NaN kept
                mean = (float)((double)k + m1);
                rstd = 1.f / sqrtf(var + a.eps);
            };
            float mA, rA, mB, rB;
            stats(lane, kA, mA, rA);
            stats(lane + 32, kB, mB, rB);
            if (i >= TR)  // the apply warps are done with tab[b]'s previous table
                mbar_wait_bounded(&tfree[b], (uint32_t)(((i - TR) / TR) & 1), aborted, a.status);
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
            if (lane == 0) mbar_arrive(&tabready[b]);
        }
    } else {
        // ---------------- apply warps: the chain and the channel lse from tensor memory
        const int aw = warp - kGtApply0;            // 0..7
        const uint32_t quarter = (uint32_t)(warp & 3);
        const int e = (int)(quarter >> 1);          // channel parity of these lanes
        const int ph = (int)(quarter & 1);          // pixel half of the tile
        const int h = aw >> 2;                      // channel-block half
        const int nkb = C / 4;
        const int kb0 = h ? nkb / 2 : 0, kb1 = h ? nkb : nkb / 2;

        // Software pipeline: tile i's chain and partial lse, then the merge and output of
        // tile i - 1, whose partials every warp has published by then.
        const int jq = aw >> 1;
        long long pn = 0;  // sample and tile of the previous item
        int pt = 0;
        for (int64_t i = 0;; ++i) {
            const long long g = item(i);
            if (g >= 0) {
                const long long n = g / T;
                const int t = (int)(g - n * T);
                const int b = (int)(i % TR);
                mbar_wait_bounded(&tabready[b], (uint32_t)((i / TR) & 1), aborted, a.status);
                mbar_wait_bounded(&tready[b], (uint32_t)((i / TR) & 1), aborted, a.status);
                tmem_fence_after();
                __syncwarp();
                const float4* tb = tab + (size_t)b * C;
                const uint32_t taddr = tbase + (quarter << 21) + (uint32_t)b * tcols;  // lane field: 32 q << 16
                Lse4 st = lse4_empty();
                // block kb: columns 8 kb .. 8 kb + 7 = channels 4 kb + e (pixels 0-3), 4 kb + 2 + e
                auto residuals = [&](const uint32_t* r, int kb, f32x2* ra, f32x2* rb) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float4 te = tb[4 * kb + e + 2 * hh];
                        const f32x2 mean = f2_pack(te.x, te.x), sc = f2_pack(te.y, te.y), sh = f2_pack(te.z, te.z);
                        ra[hh] = f2_residual_less_2_3(
                            f2_pack(__uint_as_float(r[4 * hh]), __uint_as_float(r[4 * hh + 1])), mean, sc, sh);
                        rb[hh] = f2_residual_less_2_3(
                            f2_pack(__uint_as_float(r[4 * hh + 2]), __uint_as_float(r[4 * hh + 3])), mean, sc, sh);
                    }
                };
                int kb = kb0;
                for (; kb + 4 <= kb1; kb += 4) {
                    uint32_t r[32];
                    tmem_ld32(taddr + 8u * kb, r);
                    tmem_wait_ld_all();
                    f32x2 ra[8], rb[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) residuals(r + 8 * k, kb + k, ra + 2 * k, rb + 2 * k);
                    lse4_fold<8>(st, ra, rb);
                }
                for (; kb < kb1; ++kb) {
                    uint32_t r[8];
                    tmem_ld8(taddr + 8u * kb, r);
                    tmem_wait_ld_all();
                    f32x2 ra[2], rb[2];
                    residuals(r, kb, ra, rb);
                    lse4_fold<2>(st, ra, rb);
                }
                tmem_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tfree[b]);  // done with the tile and its table
                // the partial lse of this warp's four pixels into xbuf[i & 1] (free once every
                // warp has merged tile i - 2)
                float m[4], s[4];
                lse4_unpack(st, m, s);
                float* xb = xbuf + (size_t)(i & 1) * kGtApplyWarps * 32 * 8;
                if (i >= 2) mbar_wait_bounded(&xfree[i & 1], (uint32_t)(((i - 2) / 2) & 1), aborted, a.status);
                float4* d = reinterpret_cast<float4*>(xb + ((size_t)aw * 32 + lane) * 8);
                d[0] = make_float4(m[0], m[1], m[2], m[3]);
                d[1] = make_float4(s[0], s[1], s[2], s[3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&xfull[i & 1]);
            }
            if (i >= 1) {
                // tile i - 1: the four partial lse of each pixel quad (warps ph, ph + 2, ph + 4,
                // ph + 6, in that order); warp ph + 2 jq merges and writes pixel jq of the quad
                const int64_t ip = i - 1;
                float* xb = xbuf + (size_t)(ip & 1) * kGtApplyWarps * 32 * 8;
                mbar_wait_bounded(&xfull[ip & 1], (uint32_t)((ip / 2) & 1), aborted, a.status);
                float mp[4], sp[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float* q = xb + ((size_t)(ph + 2 * p) * 32 + lane) * 8;
                    mp[p] = q[jq];
                    sp[p] = q[4 + jq];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&xfree[ip & 1]);
                // every quad pixel has channels in some partial, so the max is finite or NaN
                const float mx = max_nan(max_nan(mp[0], mp[1]), max_nan(mp[2], mp[3]));
                float sum = 0.f;
#pragma unroll
                for (int p = 0; p < 4; ++p) sum = fmaf(sp[p], ex2((mp[p] - mx) * kLog2e), sum);
                const int px = 128 * ph + 4 * lane;
                if (px < gt_valid(HW, pt))
                    a.out[(size_t)pn * HW + (size_t)pt * kGtPix + px + jq] = mx + logf(sum) + 2.f / 3.f;
            }
            if (g < 0) break;
            pn = g / T;
            pt = (int)(g - pn * T);
        }
    }
    __syncthreads();
    if (warp == kGtLoadWarp && lane == 0 && atomicAdd(a.status, 0) != 0) {
        // After a timeout anywhere: one more bounded wait for every tensor copy and the
        // last tensor-memory copy still in flight before shared and tensor memory are
        // released (a commit completes after every earlier copy of its thread).
        bool again = false;
        for (int64_t i = std::max<int64_t>(0, issued - R); i < issued; ++i)
            mbar_wait_bounded(&full[i % R], (uint32_t)((i / R) & 1), again, a.status);
        const long long copied = *copied_s;
        again = false;
        if (copied > 0)
            mbar_wait_bounded(&freed[(copied - 1) % R], (uint32_t)(((copied - 1) / R) & 1), again, a.status);
    }
    tmem_fence_before();
    __syncthreads();
    if (warp == 0) {
        tmem_fence_after();
        tmem_dealloc_warp(tbase, kGtTmemCols);
    }
}

// Scratch, zeroed at launch: [next (8 B)][cnt N (4 B each)] then, at a 16-byte
// boundary, the accumulators [N][G] (S1, S2) in fp64.
struct GnTmemScratch {
    size_t cnt, acc, total;
};
static GnTmemScratch gn_tmem_scratch(int64_t N, int64_t G) {
    GnTmemScratch s;
    s.cnt = 16;
    s.acc = (s.cnt + (size_t)N * 4 + 15) / 16 * 16;
    s.total = s.acc + (size_t)N * G * 2 * sizeof(double);
    return s;
}

static size_t gn_tmem_smem(int C, int R, int TR) {
    return (size_t)R * C * kGtPix * 4 + (size_t)TR * C * sizeof(float4) +
           (size_t)2 * kGtApplyWarps * 32 * 8 * 4 +
           (size_t)(3 * kGtMaxSlots + 3 * kGtMaxTiles + 4 + 2 * kGtRing) * 8 + kGtRing * 8 + 8 +
           2 * kGtMaxC * sizeof(float) + 16;
}

bool gn_tmem_plan(const DeviceInfo& dev, const float* y, const float* out, int64_t N, int64_t C, int64_t HW,
                  int64_t G, GnTmemPlan* plan) {
    // (the tensor copy's coordinates are 32-bit: rows N*C and pixels HW below 2^31)
    if (HW % 4 != 0 || HW < 4 || C % 4 != 0 || C < 4 || C > kGtMaxC || N < 1 || N * C >= (1ll << 31) ||
        HW >= (1ll << 31) || (reinterpret_cast<uintptr_t>(y) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(out) & 15) != 0 || encode_tiled() == nullptr)
        return false;
    const int T = (int)((HW + kGtPix - 1) / kGtPix);
    const int TR = (int)std::min<int64_t>(kGtMaxTiles, kGtTmemCols / (2 * C));
    const size_t budget = (size_t)dev.max_smem_optin;
    int R = 0;
    for (int r = kGtMaxSlots; r >= 2; --r)
        if (gn_tmem_smem((int)C, r, TR) <= budget) {
            R = r;
            break;
        }
    const int slots_env = env_int("LSE_GNM_SLOTS", 0);
    if (slots_env >= 2 && slots_env < R) R = slots_env;
    const int grid = dev.sm_count;
    // deadlock bound (see the kernel's header): every CTA's buffers together exceed a sample
    if (R < 2 || (int64_t)TR * grid < T) return false;
    plan->grid = grid;
    plan->T = T;
    plan->TR = TR;
    plan->R = R;
    plan->threads = kGtThreads;
    plan->smem = std::max(gn_tmem_smem((int)C, R, TR), budget / 2 + 1024);  // one CTA per SM
    plan->scratch_bytes = gn_tmem_scratch(N, G).total;
    return plan->smem <= budget;
}

cudaError_t launch_gn_tmem(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                           int64_t N, int64_t C, int64_t HW, int64_t G, float eps, const GnTmemPlan& p, void* scratch,
                           cudaStream_t stream) {
    unsigned char* base = static_cast<unsigned char*>(scratch);
    const GnTmemScratch sc = gn_tmem_scratch(N, G);
    cudaError_t e = cudaMemsetAsync(base, 0, sc.total, stream);
    if (e != cudaSuccess) return e;
    GnTmemArgs args;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)HW, (cuuint64_t)(N * C)};
        const cuuint64_t strides[1] = {(cuuint64_t)HW * 4};
        const cuuint32_t box[2] = {(cuuint32_t)kGtPix, (cuuint32_t)C};
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
    args.T = p.T;
    args.TR = p.TR;
    args.R = p.R;
    args.eps = eps;
    args.next = reinterpret_cast<unsigned long long*>(base);
    args.cnt = reinterpret_cast<unsigned*>(base + sc.cnt);
    args.acc = reinterpret_cast<double2*>(base + sc.acc);
    args.status = dev.status;
    e = cudaFuncSetAttribute(gn_tmem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gn_tmem_kernel, p.threads, p.smem);
    if (e != cudaSuccess) return e;
    if (per_sm != 1) return cudaErrorNotSupported;  // each CTA holds all of the SM's tensor memory
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)p.grid);
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] gn_tmem: grid=%d T=%d TR=%d R=%d smem=%zu\n", p.grid, p.T, p.TR, p.R, p.smem);
    e = cudaLaunchKernelEx(&cfg, gn_tmem_kernel, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace lse
