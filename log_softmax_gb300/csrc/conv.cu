// Conv2d (3 x 3, stride 1, valid, bias) on the tensor cores: the layer that
// produces the y of the GroupNorm chain of the POPCORNBENCH page
// "Kimi-K2.6 / l2_p92" (8 -> 64 channels on 128 x 128 planes).
//
// conv2d_tc_kernel: persistent CTAs of NS tile slots (one warpgroup of 128
// threads each, NS = 1..4 by shared memory); a slot loops over tiles of 128
// wide pixels (conv_tile.cuh).  The weights are split (hi/lo tf32) into shared
// memory once per CTA; per tile the slot's threads stage the input window (hi
// and lo), one thread issues the tile's MMAs (18 with the hi and lo weights
// stacked for Cout <= 64, else 27) into the slot's tensor-memory columns, and
// after their commit every thread reads its pixel's Cout accumulators back
// (tcgen05.ld), adds the bias and stores y with coalesced rows per channel.
// The slots run independently, so one slot's loads overlap another's MMAs and
// epilogue.  With CPG > 0 the epilogue also takes each channel group's values
// of the tile to an exact (count, mean, M2) -- per thread over the group's
// channels, then across the tile's pixels in two passes through shared memory
// -- and stores one partial per (sample, tile, group); gn_tile_merge_kernel
// merges a sample's tiles.  The statistics mode uses one product of
// round-to-nearest tf32 operands (unbiased errors of ~2^-12 relative per
// product average out over the ~63,000 values of a group: mean and variance
// stay within ~1e-5 relative), the other modes the 3xTF32 split.
//
// conv_gn_act_lse runs, by default, the plain convolution and then the
// GroupNorm chain's work-queue kernel over y (gn_act_lse.cu); the statistics
// epilogue above and the form with y never in memory are its alternatives.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "conv_tile.cuh"
#include "gn_common.cuh"
#include "launch.h"

namespace lse {

struct ConvArgs {
    const float* x;
    const float* w;
    const float* b;
    float* y;
    int64_t N;
    int cin, H, W, cout, OH, OW;
    int64_t tiles;     // wide-pixel tiles per sample
    int S;             // staged window (pixels)
    int slots;         // tile slots per CTA
    int tma;           // raw windows fetched by bulk copies one tile ahead (else direct loads)
    int G, cpg;        // channel groups of the statistics (CPG > 0), cpg divides 16
    float4* partials;  // [N][tiles][G] (count, mean, M2, 0) (statistics mode)
    const float* stats;  // [N][G] (mean, 1/sqrt(var + eps)) (apply mode)
    const float* gamma;  // [cout] (apply mode)
    const float* beta;   // [cout] (apply mode)
    float* out;          // [N][OH * OW] channel lse (apply mode)
    int* status;
};

// What the epilogue does with the tile's accumulators.
//   kConvWriteY       y (3xTF32)
//   kConvStats        per-(tile, group) Welford partials only (one tf32 product)
//   kConvApplyLse     the chain finished from the accumulators (3xTF32)
//   kConvWriteYStats  y and the partials (3xTF32)
enum ConvMode { kConvWriteY = 0, kConvStats = 1, kConvApplyLse = 2, kConvWriteYStats = 3 };

constexpr int kConvMaxSlots = 4;

// Row stride (float2) of the statistics scratch [G][pixel]: 8 past the tile's
// 128 pixels, so that the rows of neighbouring groups start 16 banks apart.
constexpr int kConvWsmStride = kConvTileM + 8;

// Bytes of one slot: the window's hi and lo parts, or the statistics scratch
// [G][kConvWsmStride] float2 when that is larger (it reuses the same space).
__host__ __device__ static inline size_t conv_slot_bytes(int S, int G) {
    const size_t win = (size_t)S * 16 * 2 * 2, st = (size_t)G * kConvWsmStride * 8;
    return win > st ? win : st;
}

// The raw window buffer of one slot (TMA path): 8 channel rows of S floats.
__host__ __device__ static inline size_t conv_raw_bytes(int S) { return (size_t)S * 8 * 4; }

// The apply mode's per-channel table of one slot.
__host__ __device__ static inline size_t conv_tab_bytes(int cout) { return (size_t)cout * 16; }

__host__ __device__ static inline size_t conv_weight_bytes(int cout) {
    return (size_t)cout * 9 * 8 * 4 * 2 + (size_t)(cout * 4 + 127) / 128 * 128;
}

// Accumulator columns of one slot (2 Cout when the products are stacked), a
// power of two >= 32.
__host__ __device__ static inline uint32_t conv_tmem_cols(int cout) {
    const uint32_t need = (uint32_t)(conv_stacked(cout) ? 2 * cout : cout);
    uint32_t n = 32;
    while (n < need) n <<= 1;
    return n;
}

template <int CIN, int CPG, int MODE>
__global__ void __launch_bounds__(kConvMaxSlots * kConvTileM, 1) conv2d_tc_kernel(const ConvArgs a) {
    constexpr bool STATS = MODE == kConvStats || MODE == kConvWriteYStats;
    constexpr bool ONE_PRODUCT = MODE == kConvStats;
    constexpr bool APPLY = MODE == kConvApplyLse;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t bars[kConvMaxSlots];
    __shared__ uint64_t rawbars[kConvMaxSlots];
    __shared__ uint32_t tmem_slot;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int slot = tid / kConvTileM, wtid = tid - slot * kConvTileM;  // warpgroup and thread in it
    const int S = a.S, W = a.W;
    unsigned char* const bw = smem_raw;  // the nine B operands, hi and lo rows
    float* const bias = reinterpret_cast<float*>(bw + (size_t)a.cout * 9 * 8 * 4 * 2);
    const size_t win_bytes = conv_slot_bytes(S, STATS ? a.G : 0);
    const size_t slot_bytes = win_bytes + (a.tma ? conv_raw_bytes(S) : 0) + (APPLY ? conv_tab_bytes(a.cout) : 0);
    unsigned char* const ahi = smem_raw + conv_weight_bytes(a.cout) + (size_t)slot * slot_bytes;
    unsigned char* const alo = ahi + (size_t)S * 16 * 2;
    float* const raw = reinterpret_cast<float*>(ahi + win_bytes);
    // apply mode: the sample's per-channel table {mean, rstd*gamma*2log2e, beta*2log2e, 0}
    float4* const tab = reinterpret_cast<float4*>(ahi + win_bytes + (a.tma ? conv_raw_bytes(S) : 0));
    uint64_t* const rawbar = &rawbars[slot];
    float2* const wsm = reinterpret_cast<float2*>(ahi);  // [group][pixel] (mean, M2), after the MMAs
    const uint32_t ncols = conv_tmem_cols(a.cout);
    uint32_t alloc_cols = 32;
    while (alloc_cols < ncols * (uint32_t)a.slots) alloc_cols <<= 1;
    uint64_t* const bar = &bars[slot];

    if (warp == 0) tmem_alloc(&tmem_slot, alloc_cols);
    if (tid == 0) {
        for (int k = 0; k < a.slots; ++k) {
            mbar_init(&bars[k], 1);
            mbar_init(&rawbars[k], 1);
        }
        fence_mbar_init();
    }
    conv_stage_weights(a.w, a.cin, a.cout, bw);
    for (int c = tid; c < a.cout; c += blockDim.x) bias[c] = a.b[c];
    fence_proxy_async_smem();  // the weights are read by the tensor cores (async proxy)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot + (uint32_t)slot * ncols;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int64_t plane = (int64_t)a.H * W;
    const int64_t ohw = (int64_t)a.OH * a.OW;
    bool aborted = false;
    uint32_t phase = 0;
    const int bar_id = 1 + slot;  // named barrier of this warpgroup

    const int64_t first = (int64_t)blockIdx.x * a.slots + slot, step = (int64_t)gridDim.x * a.slots;
    const int64_t total = a.N * a.tiles;
    uint32_t raw_phase = 0;
    if (a.tma && wtid == 0 && first < total) {
        const int64_t n = first / a.tiles;
        conv_fetch_window<CIN>(a.x + n * a.cin * plane, plane, (first - n * a.tiles) * kConvTileM, S, raw, rawbar);
    }
    for (int64_t t = first; t < total; t += step) {
        const int64_t n = t / a.tiles;
        const int64_t q0 = (t - n * a.tiles) * kConvTileM;  // first wide pixel of the tile
        if (a.tma) {
            mbar_wait_bounded(rawbar, raw_phase, aborted, a.status);
            raw_phase ^= 1u;
            conv_split_window<CIN, !ONE_PRODUCT>(raw, plane, q0, S, wtid, kConvTileM, ahi, alo);
        } else {
            conv_stage_window<CIN>(a.x + n * a.cin * plane, plane, q0, S, wtid, kConvTileM, ahi, alo);
        }
        fence_proxy_async_smem();
        named_bar_sync(bar_id, kConvTileM);  // the window is in shared memory, the raw buffer free; D is free
        if (wtid == 0) {
            if (a.tma && t + step < total && !aborted) {  // the next tile's raw window, during this tile
                const int64_t n2 = (t + step) / a.tiles;
                conv_fetch_window<CIN>(a.x + n2 * a.cin * plane, plane, (t + step - n2 * a.tiles) * kConvTileM, S,
                                       raw, rawbar);
            }
            tc_fence_after();
            conv_issue_mma(tmem, ahi, alo, bw, W, S, a.cout, !ONE_PRODUCT, bar);
        }
        if constexpr (APPLY) {
            // the table of sample n, while the MMAs run (the previous tile's readers
            // passed the slot barrier at its end)
            const int cpg = a.cpg;
            for (int c = wtid; c < a.cout; c += kConvTileM) {
                const int64_t g = n * a.G + c / cpg;
                const float mean = a.stats[2 * g], rstd = a.stats[2 * g + 1];
                tab[c] = make_float4(mean, rstd * a.gamma[c] * (2.f * kLog2e), a.beta[c] * (2.f * kLog2e), 0.f);
            }
            named_bar_sync(bar_id, kConvTileM);
        }
        mbar_wait_bounded(bar, phase, aborted, a.status);
        phase ^= 1u;
        tc_fence_after();
        const int64_t q = q0 + wtid;
        const int64_t oh = q / W;
        const int ow = (int)(q - oh * W);
        const bool valid = ow < a.OW && oh < a.OH;
        const int64_t p = oh * a.OW + ow;
        MS st = ms_empty();
        for (int c0 = 0; c0 < a.cout; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + (uint32_t)c0, v);
            if (!ONE_PRODUCT && conv_stacked(a.cout)) {
                float vl[16];  // the A_hi B_lo half
                tmem_ld16(tmem + lane_base + (uint32_t)(a.cout + c0), vl);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += vl[j];
            } else {
                tmem_wait_ld();
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += bias[c0 + j];
            if constexpr (MODE == kConvWriteY || MODE == kConvWriteYStats) {
                if (valid) {
                    float* dst = a.y + n * a.cout * ohw + p;
#pragma unroll
                    for (int j = 0; j < 16; ++j) dst[(int64_t)(c0 + j) * ohw] = v[j];
                }
            }
            if constexpr (APPLY) {
                // z, tanh, hardswish, + y, then the online channel lse
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = act_residual(v[j], tab[c0 + j]);
                ms_fold<16>(st, v);
            }
            if constexpr (STATS) {
                // the 16 / CPG groups inside these 16 channels: exact mean and M2 of
                // this pixel's CPG values of each (the window is no longer read)
#pragma unroll
                for (int lo = 0; lo < 16; lo += CPG) {
                    float sum = 0.f;
#pragma unroll
                    for (int j = 0; j < CPG; ++j) sum += v[lo + j];
                    const float mean = sum * (1.f / CPG);
                    float m2 = 0.f;
#pragma unroll
                    for (int j = 0; j < CPG; ++j) m2 = fmaf(v[lo + j] - mean, v[lo + j] - mean, m2);
                    wsm[((c0 + lo) / CPG) * kConvWsmStride + wtid] = valid ? make_float2(mean, m2)
                                                                           : make_float2(0.f, -1.f);
                }
            }
        }
        if constexpr (APPLY) {
            if (valid) a.out[n * ohw + p] = ms_lse(st);
        }
        if constexpr (STATS) {
            // merge over the tile's pixels, tpg threads per group, each a strided share
            // of the pixels, reduced by shuffles within the tpg-lane block.  Every
            // valid pixel holds CPG values, so the merge is exact in two passes: the
            // group's mean is the mean of the pixel means, and its M2 the sum of the
            // pixel M2s plus CPG (mean_p - mean)^2 per pixel.
            named_bar_sync(bar_id, kConvTileM);
            const int G = a.G;
            int tpg = 1;
            while (tpg * 2 * G <= kConvTileM && tpg < 32) tpg *= 2;
            const int g = wtid / tpg, j = wtid - g * tpg;
            const float2* const row = wsm + (g < G ? g : 0) * kConvWsmStride;
            float cnt = 0.f, s1 = 0.f;
            if (g < G) {
                for (int m = j; m < kConvTileM; m += tpg) {
                    const float2 qv = row[m];
                    if (!(qv.y < 0.f)) {  // M2 < 0 marks no pixel; a NaN pixel counts
                        cnt += 1.f;
                        s1 += qv.x;
                    }
                }
            }
            for (int o = 1; o < tpg; o <<= 1) {
                cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
                s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            }
            const float mean = cnt > 0.f ? s1 / cnt : 0.f;
            float m2 = 0.f;
            if (g < G) {
                for (int m = j; m < kConvTileM; m += tpg) {
                    const float2 qv = row[m];
                    if (!(qv.y < 0.f)) {
                        const float d = qv.x - mean;
                        m2 += fmaf((float)CPG * d, d, qv.y);
                    }
                }
            }
            for (int o = 1; o < tpg; o <<= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
            if (g < G && j == 0)
                a.partials[(n * a.tiles + (q0 / kConvTileM)) * G + g] = make_float4(cnt * CPG, mean, m2, 0.f);
        }
        tc_fence_before();
        named_bar_sync(bar_id, kConvTileM);  // this slot is done reading D and its window / scratch
    }
    if (a.tma && wtid == 0 && aborted) {
        // after a timeout the last raw fetch may still be in flight: one more bounded
        // wait before the shared memory is released
        bool again = false;
        mbar_wait_bounded(rawbar, raw_phase, again, a.status);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_slot, alloc_cols);
}

// conv2d_ws_kernel: the y-writing convolution (Cout <= 96) as a pipeline of warp roles, so
// that the tensor cores, the hi / lo split and the y stores of different tiles overlap
// instead of running in series per tile slot:
//   load warp     bulk-copies tile i's raw window into raw[i % 4] once the split of
//                 tile i - 4 has released it;
//   split warps   two warpgroups, alternate tiles: raw[i % 4] into the hi / lo window
//                 win[i % 4] (once tile i - 4's MMAs are done with it);
//   MMA warps     two, alternate tiles: tile i's 18 MMAs (27 at Cout 80 and 96, products
//                 not stacked) from win[i % 4] into accumulator i % 4 of tensor memory
//                 (once tile i - 4's epilogue has read it), committed to the window's and
//                 the accumulator's barriers;
//   epilogue      four warpgroups, tiles in turn: the accumulator (its two halves added
//                 where the products are stacked) plus the bias, written to y (lane m of
//                 the accumulator is wide pixel m).
// Each ring is indexed by the CTA's tile number and every role's members divide the ring,
// so each entry has one member per role, and no barrier completes twice before its
// waiter has seen the first phase.
// Waits are bounded.
constexpr int kCwRing = 4;     // raw windows, split windows and accumulators in flight
constexpr int kCwMma = 2;      // MMA warps (alternate tiles; kCwRing a multiple)
constexpr int kCwSplitWG = 2;  // split warpgroups
constexpr int kCwEpiWG = 4;    // epilogue warpgroups
constexpr int kCwSplit0 = 1 + kCwMma, kCwEpi0 = kCwSplit0 + 4 * kCwSplitWG;  // first warp of each
constexpr int kCwThreads = 32 * (kCwEpi0 + 4 * kCwEpiWG);
// Ring ownership: tile i goes to member i mod (members) of each role, and the members
// divide the ring, so one member waits on each entry's barriers, in phase order.  A
// waiter that came to phase k + 1 of a barrier still in phase k would read the parity
// of phase k - 1 as its own; a timed-out run with three epilogue warpgroups (not a
// divisor of four) did exactly that.
static_assert(kCwRing % kCwMma == 0 && kCwRing % kCwSplitWG == 0 && kCwRing % kCwEpiWG == 0, "ring ownership");

__host__ __device__ static inline size_t conv_ws_smem(int cout, int S) {
    return conv_weight_bytes(cout) + (size_t)kCwRing * (conv_raw_bytes(S) + (size_t)S * 16 * 2 * 2);
}

template <int CIN>
__global__ void __launch_bounds__(kCwThreads, 1) conv2d_ws_kernel(const ConvArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t raw_full[kCwRing], raw_free[kCwRing], win_full[kCwRing], win_free[kCwRing];
    __shared__ uint64_t acc_full[kCwRing], acc_free[kCwRing];
    __shared__ uint32_t tmem_slot;
    __shared__ long long mma_done_s[kCwMma];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.S, W = a.W, cout = a.cout;
    unsigned char* const bw = smem_raw;  // the nine B operands, hi and lo rows
    float* const bias = reinterpret_cast<float*>(bw + (size_t)cout * 9 * 8 * 4 * 2);
    const size_t raw_bytes = conv_raw_bytes(S), win_bytes = (size_t)S * 16 * 2 * 2;
    unsigned char* const rawbase = smem_raw + conv_weight_bytes(cout);
    unsigned char* const winbase = rawbase + kCwRing * raw_bytes;
    auto rawp = [&](int r) { return reinterpret_cast<float*>(rawbase + (size_t)r * raw_bytes); };
    auto whi = [&](int w) { return winbase + (size_t)w * win_bytes; };
    auto wlo = [&](int w) { return winbase + (size_t)w * win_bytes + (size_t)S * 16 * 2; };
    const uint32_t ncols = conv_tmem_cols(cout);  // accumulator columns: 2 Cout (stacked) or Cout, at most 128

    if (warp == 0) tmem_alloc(&tmem_slot, 512);
    if (tid == 0) {
        for (int k = 0; k < kCwRing; ++k) {
            mbar_init(&raw_full[k], 1);
            mbar_init(&raw_free[k], kConvTileM);
            mbar_init(&win_full[k], kConvTileM);
            mbar_init(&win_free[k], 1);
            mbar_init(&acc_full[k], 1);
            mbar_init(&acc_free[k], 4);
        }
        for (int m = 0; m < kCwMma; ++m) mma_done_s[m] = 0;
        fence_mbar_init();
    }
    conv_stage_weights(a.w, a.cin, cout, bw);
    for (int c = tid; c < cout; c += blockDim.x) bias[c] = a.b[c];
    fence_proxy_async_smem();  // the weights are read by the tensor cores (async proxy)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int64_t plane = (int64_t)a.H * W;
    const int64_t ohw = (int64_t)a.OH * a.OW;
    const int64_t total = a.N * a.tiles;
    const int64_t nit = (int64_t)blockIdx.x < total ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto tile_of = [&](int64_t i) { return (int64_t)blockIdx.x + i * gridDim.x; };
    bool aborted = false;
    int64_t issued = 0;  // load warp: raw windows requested

    if (warp == 0) {
        // ---------------- load warp
        if (lane == 0) {
            for (int64_t i = 0; i < nit; ++i) {
                const int r = (int)(i % kCwRing);
                if (i >= kCwRing) mbar_wait_bounded(&raw_free[r], (uint32_t)((i / kCwRing - 1) & 1), aborted, a.status);
                if (aborted) break;
                const int64_t t = tile_of(i), n = t / a.tiles;
                conv_fetch_window<CIN>(a.x + n * a.cin * plane, plane, (t - n * a.tiles) * kConvTileM, S, rawp(r),
                                       &raw_full[r]);
                issued = i + 1;
            }
        }
    } else if (warp <= kCwMma) {
        // ---------------- MMA warps, alternate tiles: the whole warp runs the loop and its
        // waits (uniform branches), lane 0 issues.  The tensor pipe's queue is short: an
        // issuing warp's control between tiles (waits, fences, the lane-0 region) measured
        // 300 to 600 clocks per tile of idle pipe on GB300 with one issuing warp, and
        // about a tenth of that with two, each filling the other's gaps.
        const int mw = warp - 1;
        ConvTileMma mm;
        mm.init(bw, W, S, cout);
        long long done = 0;  // 1 + the last tile this warp issued
        for (int64_t i = mw; i < nit; i += kCwMma) {
            const int w = (int)(i % kCwRing);
            mbar_wait_bounded(&win_full[w], (uint32_t)((i / kCwRing) & 1), aborted, a.status);
            if (i >= kCwRing) mbar_wait_bounded(&acc_free[w], (uint32_t)((i / kCwRing - 1) & 1), aborted, a.status);
            if (__any_sync(0xffffffffu, aborted)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                mm.issue(tmem + (uint32_t)w * ncols, whi(w), wlo(w));
                umma_commit(&win_free[w]);
                umma_commit(&acc_full[w]);  // the same MMAs
            }
            __syncwarp();
            done = i + 1;
        }
        if (lane == 0) mma_done_s[mw] = done;
    } else if (warp < kCwEpi0) {
        // ---------------- split warpgroups: raw[i % 4] -> win[i % 4], alternate tiles
        const int sg = (warp - kCwSplit0) / 4, st = tid - 32 * kCwSplit0 - sg * kConvTileM;
        for (int64_t i = sg; i < nit; i += kCwSplitWG) {
            const int r = (int)(i % kCwRing);
            mbar_wait_bounded(&raw_full[r], (uint32_t)((i / kCwRing) & 1), aborted, a.status);
            if (i >= kCwRing) mbar_wait_bounded(&win_free[r], (uint32_t)((i / kCwRing - 1) & 1), aborted, a.status);
            const int64_t t = tile_of(i), n = t / a.tiles;
            conv_split_window<CIN, true>(rawp(r), plane, (t - n * a.tiles) * kConvTileM, S, st, kConvTileM, whi(r),
                                         wlo(r));
            fence_proxy_async_smem();  // the window is read by the tensor cores
            mbar_arrive(&raw_free[r]);
            mbar_arrive(&win_full[r]);
        }
    } else {
        // ---------------- epilogue warpgroups: accumulator i % 4 -> y, tiles in turn
        const int eg = (warp - kCwEpi0) / 4;
        const uint64_t drop = l2_policy_evict_first();
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int m = 32 * (warp & 3) + lane;  // accumulator lane of this thread: wide pixel q0 + m
        for (int64_t i = eg; i < nit; i += kCwEpiWG) {
            const int ac = (int)(i % kCwRing);
            mbar_wait_bounded(&acc_full[ac], (uint32_t)((i / kCwRing) & 1), aborted, a.status);
            tc_fence_after();
            __syncwarp();
            const int64_t t = tile_of(i), n = t / a.tiles;
            const int64_t q = (t - n * a.tiles) * kConvTileM + m;
            const int64_t oh = q / W;
            const int ow = (int)(q - oh * W);
            const bool valid = ow < a.OW && oh < a.OH;
            float* dst = a.y + n * cout * ohw + oh * a.OW + ow;
            const uint32_t d = tmem + (uint32_t)ac * ncols + lane_base;
            const bool stacked = conv_stacked(cout);
            for (int c0 = 0; c0 < cout; c0 += 16) {
                float v[16];
                tmem_ld16(d + (uint32_t)c0, v);
                if (stacked) {
                    float vl[16];  // stacked: the A_hi B_lo half, added into the first
                    tmem_ld16(d + (uint32_t)(cout + c0), vl);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] += vl[j];
                } else {
                    tmem_wait_ld();
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += bias[c0 + j];
                if (valid) {
                    // y is written once: evict-first lines (on GB300 2-3 % faster than plain
                    // stores on one box, equal on another; the chain that reads y back unchanged)
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(dst + (int64_t)(c0 + j) * ohw),
                                     "f"(v[j]), "l"(drop)
                                     : "memory");
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free[ac]);
        }
    }
    __syncthreads();
    if (tid == 0 && atomicAdd(a.status, 0) != 0) {
        // After a timeout anywhere: one more bounded wait for the raw windows and the MMAs
        // still in flight before shared and tensor memory are released (a commit
        // completes after every earlier MMA of its thread).
        bool again = false;
        for (int64_t i = std::max<int64_t>(0, issued - kCwRing); i < issued; ++i)
            mbar_wait_bounded(&raw_full[i % kCwRing], (uint32_t)((i / kCwRing) & 1), again, a.status);
        for (int m = 0; m < kCwMma; ++m) {  // a commit tracks its own thread's MMAs
            const long long done = mma_done_s[m];
            again = false;
            if (done > 0)
                mbar_wait_bounded(&acc_full[(done - 1) % kCwRing], (uint32_t)(((done - 1) / kCwRing) & 1), again,
                                  a.status);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// The pipelined kernel where it applies: y written, Cout <= 96 in multiples of 16, raw
// windows by bulk copies (16-byte aligned planes), its rings in shared memory;
// cudaErrorNotSupported otherwise (LSE_CONV_WS=0 forces that too).  Its rings take 96 S
// bytes per entry (S = conv_window(W)) beside the weights: up to W = 187 at Cout = 64.
// Measured on GB300 at x[128, 8, 128, 128] against the tile-slot kernel: Cout 64
// 0.129 / 0.168 ms, 96 0.212 / 0.225, but 128 0.313 / 0.279 (27 MMAs and 64 KB of y
// stores per tile: the tile slots overlap them better), so wider layers keep the slots.
template <int CIN>
static cudaError_t conv_ws_go(const DeviceInfo& dev, const ConvArgs& a0, cudaStream_t stream) {
    ConvArgs a = a0;
    if (env_int("LSE_CONV_WS", 1) == 0 || a.cout > 96 || a.cout % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(a.x) & 15) != 0 || ((int64_t)a.H * a.W) % 4 != 0 || env_int("LSE_CONV_TMA", 1) == 0)
        return cudaErrorNotSupported;
    const size_t need = conv_ws_smem(a.cout, a.S), budget = (size_t)dev.max_smem_optin - 1024;
    if (need > budget) return cudaErrorNotSupported;
    // more than half the shared memory: one CTA per SM (each allocates all of tensor memory)
    const size_t smem = std::max(need, std::min(budget, (size_t)dev.max_smem_optin / 2 + 1024));
    auto kern = conv2d_ws_kernel<CIN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kCwThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm != 1) return cudaErrorNotSupported;  // each CTA allocates all of tensor memory
    a.tma = 1;
    const int64_t total = a.N * a.tiles;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(total, dev.sm_count));
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] conv2d_ws: grid=%u window=%d tiles=%lld smem=%zu\n", grid, a.S, (long long)total, smem);
    kern<<<grid, kCwThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

bool conv_tc_supported(int64_t cin, int64_t cout, int64_t W) {
    return cin >= 1 && cin <= kConvMaxCin && cout >= 16 && cout <= 128 && cout % 16 == 0 && W <= kConvMaxW;
}

template <int CIN, int CPG, int MODE>
static cudaError_t conv_go(const DeviceInfo& dev, const ConvArgs& a, cudaStream_t stream);

template <int CIN>
static cudaError_t conv_write_y(const DeviceInfo& dev, const ConvArgs& a, cudaStream_t stream) {
    cudaError_t e = conv_ws_go<CIN>(dev, a, stream);
    if (e != cudaErrorNotSupported) return e;
    return conv_go<CIN, 0, kConvWriteY>(dev, a, stream);
}

static cudaError_t conv_dispatch(const DeviceInfo& dev, const ConvArgs& a, cudaStream_t stream) {
    switch (a.cin) {
        case 1: return conv_write_y<1>(dev, a, stream);
        case 2: return conv_write_y<2>(dev, a, stream);
        case 3: return conv_write_y<3>(dev, a, stream);
        case 4: return conv_write_y<4>(dev, a, stream);
        case 5: return conv_write_y<5>(dev, a, stream);
        case 6: return conv_write_y<6>(dev, a, stream);
        case 7: return conv_write_y<7>(dev, a, stream);
        default: return conv_write_y<8>(dev, a, stream);
    }
}

// The chain's epilogues are compiled for its own convolution (Cin = 8).
template <int MODE>
static cudaError_t conv_stats_dispatch(const DeviceInfo& dev, const ConvArgs& a, cudaStream_t stream) {
    switch (a.cpg) {
        case 1: return conv_go<8, 1, MODE>(dev, a, stream);
        case 2: return conv_go<8, 2, MODE>(dev, a, stream);
        case 4: return conv_go<8, 4, MODE>(dev, a, stream);
        case 8: return conv_go<8, 8, MODE>(dev, a, stream);
        default: return conv_go<8, 16, MODE>(dev, a, stream);
    }
}

static ConvArgs conv_args(const DeviceInfo& dev, const float* x, const float* w, const float* b, float* y, int64_t N,
                          int64_t cin, int64_t H, int64_t W, int64_t cout) {
    ConvArgs a;
    a.x = x;
    a.w = w;
    a.b = b;
    a.y = y;
    a.N = N;
    a.cin = (int)cin;
    a.H = (int)H;
    a.W = (int)W;
    a.cout = (int)cout;
    a.OH = (int)H - 2;
    a.OW = (int)W - 2;
    a.tiles = ((int64_t)a.OH * a.W + kConvTileM - 1) / kConvTileM;  // wide pixels
    a.S = conv_window(a.W);
    a.slots = 1;
    a.tma = 0;
    a.G = 1;
    a.cpg = (int)cout;
    a.partials = nullptr;
    a.stats = nullptr;
    a.gamma = nullptr;
    a.beta = nullptr;
    a.out = nullptr;
    a.status = dev.status;
    return a;
}

cudaError_t launch_conv2d_3x3(const DeviceInfo& dev, const float* x, const float* w, const float* b, float* y,
                              int64_t N, int64_t cin, int64_t H, int64_t W, int64_t cout, cudaStream_t stream) {
    return conv_dispatch(dev, conv_args(dev, x, w, b, y, N, cin, H, W, cout), stream);
}

template <int CIN, int CPG, int MODE>
static cudaError_t conv_go(const DeviceInfo& dev, const ConvArgs& a0, cudaStream_t stream) {
    auto kern = conv2d_tc_kernel<CIN, CPG, MODE>;
    ConvArgs a = a0;
    // as many tile slots (up to 4) as shared and tensor memory hold
    // raw windows by bulk copies when every plane starts 16-byte aligned
    a.tma = ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0 && ((int64_t)a.H * a.W) % 4 == 0 &&
             env_int("LSE_CONV_TMA", 1) != 0) ? 1 : 0;
    const size_t wbytes = conv_weight_bytes(a.cout);
    const size_t budget = (size_t)dev.max_smem_optin - 1024;
    auto slot_bytes = [&]() {
        return conv_slot_bytes(a.S, (MODE == kConvStats || MODE == kConvWriteYStats) ? a.G : 0) +
               (a.tma ? conv_raw_bytes(a.S) : 0) + (MODE == kConvApplyLse ? conv_tab_bytes(a.cout) : 0);
    };
    // wide rows: when the raw window buffer of the bulk-copy path does not fit
    // beside one slot's window, load the window directly instead
    if (a.tma && wbytes + slot_bytes() > budget) a.tma = 0;
    const size_t sbytes = slot_bytes();
    if (wbytes + sbytes > budget) return cudaErrorNotSupported;
    a.slots = (int)std::min<size_t>({(size_t)kConvMaxSlots, (budget - wbytes) / sbytes,
                                     (size_t)(512 / conv_tmem_cols(a.cout))});
    const size_t smem = wbytes + (size_t)a.slots * sbytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    const int threads = a.slots * kConvTileM;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    uint32_t alloc_cols = 32;
    while (alloc_cols < conv_tmem_cols(a.cout) * (uint32_t)a.slots) alloc_cols <<= 1;
    per_sm = std::min<int>(per_sm, (int)(512 / alloc_cols));  // tensor memory of co-resident CTAs
    const int64_t total = a.N * a.tiles;
    const int64_t blocks = (total + a.slots - 1) / a.slots;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)per_sm * dev.sm_count));
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] conv2d_tc: grid=%u (%d per SM) slots=%d window=%d tma=%d tiles=%lld smem=%zu\n", grid,
                per_sm, a.slots, a.S, a.tma, (long long)total, smem);
    kern<<<grid, threads, smem, stream>>>(a);
    return cudaGetLastError();
}

// One warp per (n, g): the sample's tile partials of group g merged in tile
// order (Chan et al.), then stats[2 (n G + g)] = mean, [+1] = 1/sqrt(var + eps).
__global__ void __launch_bounds__(256) gn_tile_merge_kernel(const float4* __restrict__ partials,
                                                            float* __restrict__ stats, int64_t NG, int64_t tiles,
                                                            int G, float eps) {
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (item >= NG) return;
    const int64_t n = item / G, g = item - n * G;
    Welford w{0.f, 0.f, 0.f};
    for (int64_t t = lane; t < tiles; t += 32) {
        const float4 q = partials[(n * tiles + t) * G + g];
        w = wf_merge(w, Welford{q.x, q.y, q.z});
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = wf_merge(w, wf_shfl_xor(w, o));
    if (lane == 0) {
        stats[2 * item] = w.mean;
        stats[2 * item + 1] = 1.f / sqrtf(w.m2 / w.n + eps);
    }
}

// Two ways through the chain: by default the convolution writes y with the
// partials and the GroupNorm apply pass reads y once (HBM: x, y twice, out);
// with LSE_CONV_CHAIN=2 y never reaches memory -- a one-product pass for the
// partials, then the convolution again, finishing the chain from tensor memory
// (HBM: x twice, out; twice the tensor work).
// 1: the convolution writes y and its tiles' statistics, then merge and apply;
// 2: y never in memory (statistics pass, then the convolution again);
// 3 (default): the convolution writes y, then the GroupNorm work queue over y.
static int conv_chain_mode() { return env_int("LSE_CONV_CHAIN", 3); }
static bool conv_chain_y_free() { return conv_chain_mode() == 2; }

size_t conv_chain_scratch_bytes(int64_t N, int64_t H, int64_t W, int64_t cout, int64_t G) {
    const int64_t tiles = ((H - 2) * W + kConvTileM - 1) / kConvTileM;  // wide pixels
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t y = conv_chain_y_free() ? 0 : up((size_t)N * cout * (H - 2) * (W - 2) * 4);
    return y + std::max(up((size_t)N * tiles * G * sizeof(float4)) + up((size_t)N * G * 8),
                        up(gn_fused_scratch_bytes(N, G, 0)));
}

cudaError_t launch_conv_gn_act_lse(const DeviceInfo& dev, const float* x, const float* w, const float* b,
                                   const float* gamma, const float* beta, float* out, int64_t N, int64_t cin,
                                   int64_t H, int64_t W, int64_t cout, int64_t G, float eps, void* scratch,
                                   cudaStream_t stream) {
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    const bool y_free = conv_chain_y_free();
    const int64_t ohw = (H - 2) * (W - 2);
    char* sp = static_cast<char*>(scratch);
    float* y = y_free ? nullptr : reinterpret_cast<float*>(sp);
    if (!y_free) sp += up((size_t)N * cout * ohw * 4);
    ConvArgs a = conv_args(dev, x, w, b, y, N, cin, H, W, cout);
    if (conv_chain_mode() == 3) {
        // y, then the one-kernel GroupNorm chain over it, samples last to first so
        // that its first statistics reads find the convolution's last samples in L2
        cudaError_t e = conv_write_y<8>(dev, a, stream);
        if (e != cudaSuccess) return e;
        return launch_gn_act_lse_fused(dev, y, gamma, beta, out, N, cout, ohw, G, eps, sp, stream, 0, true);
    }
    a.G = (int)G;
    a.cpg = (int)(cout / G);
    a.partials = reinterpret_cast<float4*>(sp);
    float* stats = reinterpret_cast<float*>(sp + up((size_t)N * a.tiles * G * sizeof(float4)));
    // 1: the convolution with each tile's per-group Welford partials (and y)
    cudaError_t e = y_free ? conv_stats_dispatch<kConvStats>(dev, a, stream)
                           : conv_stats_dispatch<kConvWriteYStats>(dev, a, stream);
    if (e != cudaSuccess) return e;
    // 2: per-(n, g) mean and 1/sqrt(var + eps)
    const int64_t NG = N * G;
    gn_tile_merge_kernel<<<(unsigned)((NG + 7) / 8), 256, 0, stream>>>(a.partials, stats, NG, a.tiles, (int)G, eps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 3: the GroupNorm apply pass over y, or the convolution again finishing the
    //    chain from tensor memory
    if (!y_free) return launch_gn_apply(dev, y, gamma, beta, out, N, cout, ohw, G, stats, stream);
    a.stats = stats;
    a.gamma = gamma;
    a.beta = beta;
    a.out = out;
    return conv_go<8, 0, kConvApplyLse>(dev, a, stream);
}

}  // namespace lse
