// Rows split over a group of CTAs and parked in tensor memory while the group merges
// their statistics: the kernel shared by the long-row log_softmax / softmax (a row of x)
// and GroupNorm (the contiguous slab of a sample's channel group, C / G x HW floats).
//
// A row's output is an element-wise transform of the row with constants from a statistic
// of the whole row ((max, sum of exponentials) for log_softmax, (mean, M2) for
// GroupNorm).  Each row is split over GS CTAs of a cooperative grid (one slice each);
// a slice lands chunk by chunk in shared memory (bulk copies), is folded into the CTA's
// partial statistic there, and is copied on into tensor memory (tcgen05.cp), where it
// waits for the group's statistic while the next chunks land.  Roles, per CTA:
//   fold warps   fold each landed chunk (shared-memory slot g % R, chunk g = j * nch + c of
//                the CTA) and arrive on folded[slot]; at the end of a row they publish the
//                CTA's partial through the group's tagged 64-bit slots.
//   copy warp    once a chunk is folded, copies it into row buffer j % TR of tensor
//                memory (after the store warps have released that buffer's previous
//                row) and commits the copy to freed[slot] (and, for the row's last
//                chunk, to tready[buffer]).
//   load warp    issues every bulk copy: chunk g + R into slot g % R once chunk g's
//                tensor-memory copy has completed.
//   merge warp   waits for this CTA's own partial of a row (pub), merges the group's
//                partials into the row's result and hands it over through res_s[j % 8]
//                and res_full[j % 8], so that the stores never wait for a round trip to
//                L2 and no warp polls L2 for a row long before it can be complete.
//   store warps  (SW = 4 or 8) wait for the row's result and its copies (tready), read
//                their lanes of the row buffer (with 8, two warps per quarter of the lanes
//                take alternate groups of four blocks), write the transform, and release
//                the buffer (tfree, one arrival per warp).
// Shared memory then holds only chunks in flight from HBM, being folded or being
// copied, and up to TR rows wait in tensor memory.  Fold warp 0 publishes row r only
// after this CTA's store of row r - TR, which implies every CTA's partials of r - TR,
// hence every CTA's store (and, the merge warp taking rows in order, every CTA's merge)
// of r - 2 TR: 2 TR < kRtSlots keeps the tagged slots safe.  The merge of row r in turn
// needs this CTA's store of r - TR, so res_s[r % 8] is never overwritten before it has
// been read, and pub[r % 8] completes again only after the merge of r (TR < 8).  Waits
// are bounded.
//
// An operation Op supplies (all device functions static):
//   Params                    its constants (a kernel argument);
//   S                         a partial statistic;  R  a row's result for the stores;
//   empty(), fold<K>(S&, v[K]), warp_allreduce(S), merge(S, S);
//   pack(S, tag) / unpack(word, count): a partial through one tagged 64-bit slot (bit
//                             32 carries the tag; count = the values the partial covers);
//   finish(S, Params) -> R;
//   Cursor cursor(R, Params, row); float4 out4(Cursor&, float4 x, col): the transform of
//                             four elements at columns col .. col + 3 of the row (a
//                             thread's columns increase from call to call).
#pragma once

#include "common.cuh"
#include "launch.h"
#include "tmem.cuh"

namespace lse {

constexpr int kRtSlots = 16;        // tagged partial slots per group member (tag = (r / 16) mod 2)
constexpr int kRtRingMax = 64;      // landing slots
constexpr int kRtMaxGroup = 64;     // CTAs per row
constexpr int kRtCols = 512;        // tensor-memory columns, all allocated by each CTA
constexpr int kRtMaxRows = 7;       // rows parked per CTA; 2 x 7 < kRtSlots
constexpr int kRtResRing = 8;       // row results handed from the merge warp to the stores (> kRtMaxRows)
constexpr int kRtFoldWarps = 8;
// threads of the kernel with SW store warps (4: one per quarter of the tensor-memory
// lanes; 8: two per quarter, taking alternate groups of four 1024-float blocks)
constexpr int row_tmem_threads(int SW) { return 32 * (kRtFoldWarps + SW + 3); }

// Polls a tagged slot until its tag is `tag`, at most ~1 s / 2^26 polls; on
// timeout records kStatusTimeout and sets `aborted`.
__device__ __forceinline__ unsigned long long poll_slot(const unsigned long long* p, uint32_t tag,
                                                        unsigned long long w, bool& aborted, int* status) {
    if (ms_tag_of(w) == tag || aborted) return w;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        __nanosleep(20);
        w = ld_relaxed_gpu_u64(p);
        if (ms_tag_of(w) == tag) return w;
        if ((it & 255u) == 255u && globaltimer_ns() - t0 > 1000000000ull) break;
    }
    aborted = true;
    atomicExch(status, kStatusTimeout);
    return w;
}

template <class Params>
struct RowTmemArgs {
    const float* x;
    float* out;
    int64_t rows, cols;
    int slice;                  // floats of a row owned by one CTA (multiple of 32)
    int chunk;                  // floats per landing chunk (multiple of 1024)
    int* status;                // device status word (bounded-wait timeouts)
    int group_size;             // CTAs per row; CTA b is rank b % group_size of group b / group_size
    unsigned long long* slots;  // [groups][kRtSlots][group_size] tagged partials, all bytes 0xFF at launch
    int ring;                   // landing slots of shared memory per CTA
    int trows;                  // row buffers in tensor memory
    Params op;
};

template <class Op, int SW>
__global__ void __launch_bounds__(row_tmem_threads(SW), 1) row_tmem_kernel(const RowTmemArgs<typename Op::Params> a) {
    using S = typename Op::S;
    using R = typename Op::R;
    constexpr int FW = kRtFoldWarps;
    static_assert(SW == 4 || SW == 8, "one or two store warps per quarter of the tensor-memory lanes");
    constexpr int kHalves = SW / 4;
    static_assert(kRtMaxRows < kRtResRing && 2 * kRtMaxRows < kRtSlots, "hand-over rings too small");
    constexpr int NF = 32 * FW;
    constexpr int kCopyWarp = FW + SW, kLoadWarp = FW + SW + 1, kMergeWarp = FW + SW + 2;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int chunk = a.chunk, Rg = a.ring, TR = a.trows;
    const int64_t rows = a.rows, cols = a.cols;
    float* const ring = reinterpret_cast<float*>(smem_raw);                                   // [Rg][chunk]
    uint64_t* const full = reinterpret_cast<uint64_t*>(smem_raw + (size_t)Rg * chunk * 4);   // [kRtRingMax]
    uint64_t* const freed = full + kRtRingMax;                                               // [kRtRingMax]
    uint64_t* const folded = freed + kRtRingMax;                                             // [kRtRingMax]
    uint64_t* const tfree = folded + kRtRingMax;                                             // [kRtMaxRows]
    uint64_t* const tready = tfree + kRtMaxRows;                                             // [kRtMaxRows]
    uint64_t* const res_full = tready + kRtMaxRows;                                          // [kRtResRing]
    uint64_t* const pub = res_full + kRtResRing;                                             // [kRtResRing]
    long long* const copied_s = reinterpret_cast<long long*>(pub + kRtResRing);              // [1]
    R* const res_s = reinterpret_cast<R*>(copied_s + 2);                                     // [kRtResRing]
    S* const red = reinterpret_cast<S*>(res_s + kRtResRing);                                 // [2][32]
    uint32_t* const tslot = reinterpret_cast<uint32_t*>(red + 64);                           // [1]

    const uint32_t GS = (uint32_t)a.group_size;
    const uint32_t rank = blockIdx.x % GS;
    const int64_t first_row = blockIdx.x / GS;
    const int64_t row_step = gridDim.x / GS;
    unsigned long long* const slots = a.slots + first_row * kRtSlots * GS;  // [kRtSlots][GS]
    const int64_t c_begin = (int64_t)rank * a.slice;
    const int len = (int)std::max<int64_t>(0, std::min<int64_t>(a.slice, cols - c_begin));
    const int nch = (len + chunk - 1) / chunk;
    const int cpr = (a.slice + 1023) / 1024 * 8;  // tensor-memory columns of one row buffer
    const int64_t nrows = first_row < rows ? (rows - first_row + row_step - 1) / row_step : 0;
    const int64_t total = nrows * nch;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    bool aborted = false;

    if (warp == 0) tmem_alloc_warp(tslot, kRtCols);
    if (tid == 0) {
        for (int r = 0; r < Rg; ++r) {
            mbar_init(&full[r], 1);
            mbar_init(&freed[r], 1);
            mbar_init(&folded[r], FW);
        }
        for (int b = 0; b < TR; ++b) {
            mbar_init(&tfree[b], SW);
            mbar_init(&tready[b], 1);
        }
        for (int k = 0; k < kRtResRing; ++k) {
            mbar_init(&res_full[k], 1);
            mbar_init(&pub[k], 1);
        }
        *copied_s = 0;
        fence_mbar_init();
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tbase = *tslot;

    int64_t issued = 0;  // load warp: chunks whose bulk copy has been issued
    auto issue = [&](int64_t g) {
        const int64_t j = g / nch;
        const int c = (int)(g - j * nch);
        const int sl = (int)(g % Rg);
        const int cb = c * chunk;
        const uint32_t bytes = (uint32_t)std::min(chunk, len - cb) * 4u;
        mbar_arrive_expect_tx(&full[sl], bytes);
        bulk_g2s(ring + (size_t)sl * chunk, a.x + (first_row + j * row_step) * cols + c_begin + cb, bytes, &full[sl]);
        issued = g + 1;
    };

    if (warp < FW) {
        // ---------------- fold warps
        for (int64_t j = 0; j < nrows; ++j) {
            S st = Op::empty();
            for (int c = 0; c < nch; ++c) {
                const int64_t g = j * nch + c;
                const int sl = (int)(g % Rg);
                mbar_wait_bounded(&full[sl], (uint32_t)((g / Rg) & 1), aborted, a.status);
                const int n = std::min(chunk, len - c * chunk);
                const int n4 = n >> 2;
                const float4* p = reinterpret_cast<const float4*>(ring + (size_t)sl * chunk);
                int i = tid;
                for (; i + 3 * NF < n4; i += 4 * NF) {
                    float v[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float4 q = p[i + k * NF];
                        v[4 * k + 0] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
                    }
                    Op::template fold<16>(st, v);
                }
                for (; i < n4; i += NF) {
                    float4 q = p[i];
                    float v[4] = {q.x, q.y, q.z, q.w};
                    Op::template fold<4>(st, v);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&folded[sl]);  // this warp is done reading slot sl
            }
            st = Op::warp_allreduce(st);
            if (lane == 0) red[(j & 1) * 32 + warp] = st;
            named_bar_sync(1, NF);  // every fold warp is done with this row and its red slot
            if (warp == 0) {
                S r = (lane < FW) ? red[(j & 1) * 32 + lane] : Op::empty();
                r = Op::warp_allreduce(r);
                // Not before this CTA's store of row j - TR: that bounds how far the partials
                // run ahead of every CTA's reads of the tagged slots (the fold warps alone
                // could run R / nch + TR rows ahead).  The phase cannot move on before
                // this publication, since it is the next use of the buffer.
                if (j >= TR)
                    mbar_wait_bounded(&tfree[j % TR], (uint32_t)(((j - TR) / TR) & 1), aborted, a.status);
                if (lane == 0) {
                    st_relaxed_gpu_u64(slots + (j % kRtSlots) * GS + rank, Op::pack(r, (uint32_t)(j / kRtSlots) & 1u));
                    mbar_arrive(&pub[j % kRtResRing]);
                }
            }
        }
    } else if (warp < FW + SW) {
        // ---------------- store warps: read the row from tensor memory, write its transform
        const uint32_t quarter = (uint32_t)(warp & 3);  // the lanes this warp may read
        const int half = (warp - FW) >> 2;               // its groups of four blocks: half, half + kHalves, ...
        const int l = (int)quarter * 32 + lane;          // tensor-memory lane of this thread
        for (int64_t j = 0; j < nrows; ++j) {
            const int b = (int)(j % TR);
            mbar_wait_bounded(&res_full[j % kRtResRing], (uint32_t)((j / kRtResRing) & 1), aborted, a.status);
            const R res = res_s[j % kRtResRing];
            mbar_wait_bounded(&tready[b], (uint32_t)((j / TR) & 1), aborted, a.status);
            tmem_fence_after();
            const int64_t row = first_row + j * row_step;
            float* dst = a.out + row * cols + c_begin;
            typename Op::Cursor cur = Op::cursor(res, a.op, row);
            const int nblk = (len + 1023) / 1024;
            const uint32_t taddr = tbase + (quarter << 21) + (uint32_t)(b * cpr);  // lane field: 32 q << 16
            // one block: lane l's floats [4l, 4l + 4) and [512 + 4l, 512 + 4l + 4) of it
            auto put = [&](int k, const uint32_t* r) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int e = 1024 * k + 512 * h + 4 * l;
                    if (e < len) {
                        const float4 q = make_float4(__uint_as_float(r[4 * h + 0]), __uint_as_float(r[4 * h + 1]),
                                                     __uint_as_float(r[4 * h + 2]), __uint_as_float(r[4 * h + 3]));
                        st_stream_f4(dst + e, Op::out4(cur, q, c_begin + e));
                    }
                }
            };
            const int ngrp = nblk / 4;  // whole groups of four blocks; the rest go to the next half in turn
            for (int q = half; q < ngrp; q += kHalves) {  // four blocks per load; never past the row's columns
                uint32_t r[32];
                tmem_ld32(taddr + 32u * q, r);
                tmem_wait_ld_all();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) put(4 * q + kk, r + 8 * kk);
            }
            if (half == ngrp % kHalves) {
                for (int k0 = 4 * ngrp; k0 < nblk; ++k0) {
                    uint32_t r[8];
                    tmem_ld8(taddr + 8u * k0, r);
                    tmem_wait_ld_all();
                    put(k0, r);
                }
            }
            tmem_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tfree[b]);
        }
    } else if (warp == kCopyWarp) {
        // ---------------- copy warp: folded chunks into tensor memory
        if (lane == 0) {
            int64_t copied = 0;
            for (int64_t g = 0; g < total && !aborted; ++g) {
                const int64_t j = g / nch;
                const int c = (int)(g - j * nch);
                const int sl = (int)(g % Rg);
                const int b = (int)(j % TR);
                mbar_wait_bounded(&folded[sl], (uint32_t)((g / Rg) & 1), aborted, a.status);
                if (c == 0 && j >= TR)  // the store warps have released row j - TR's buffer
                    mbar_wait_bounded(&tfree[b], (uint32_t)(((j - TR) / TR) & 1), aborted, a.status);
                tmem_fence_after();
                if (aborted) break;
                const int nblk = (std::min(chunk, len - c * chunk) + 1023) / 1024;
                const uint32_t col = (uint32_t)(b * cpr + c * (chunk / 1024) * 8);
                const float* slot = ring + (size_t)sl * chunk;
                for (int k = 0; k < nblk; ++k) tmem_cp_block(tbase + col + 8u * k, slot + 1024 * k);
                tmem_commit(&freed[sl]);
                if (c == nch - 1) tmem_commit(&tready[b]);
                copied = g + 1;
            }
            *copied_s = copied;
        }
    } else if (warp == kMergeWarp) {
        // ---------------- merge warp: the group's partials of each row into its result
        for (int64_t j = 0; j < nrows; ++j) {
            mbar_wait_bounded(&pub[j % kRtResRing], (uint32_t)((j / kRtResRing) & 1), aborted, a.status);
            S mine = Op::empty();
            for (uint32_t k = (uint32_t)lane; k < GS; k += 32) {
                const unsigned long long* p = slots + (j % kRtSlots) * GS + k;
                const int64_t cnt = std::max<int64_t>(0, std::min<int64_t>(a.slice, cols - (int64_t)k * a.slice));
                const S other = Op::unpack(
                    poll_slot(p, (uint32_t)(j / kRtSlots) & 1u, ld_relaxed_gpu_u64(p), aborted, a.status), cnt);
                mine = Op::merge(mine, other);
            }
            const R rv = Op::finish(Op::warp_allreduce(mine), a.op);
            if (lane == 0) {
                res_s[j % kRtResRing] = rv;
                mbar_arrive(&res_full[j % kRtResRing]);
            }
        }
    } else {
        // ---------------- load warp: chunk g + R into slot g % R once chunk g is in tensor memory
        if (lane == 0) {
            for (int64_t g = 0; g < std::min<int64_t>(Rg, total); ++g) issue(g);
            for (int64_t g = 0; g < total && !aborted; ++g) {
                if (!mbar_wait_bounded(&freed[g % Rg], (uint32_t)((g / Rg) & 1), aborted, a.status)) break;
                if (g + Rg < total) issue(g + Rg);
            }
        }
    }
    __syncthreads();
    if (warp == kLoadWarp && lane == 0 && atomicAdd(a.status, 0) != 0) {
        // After a timeout anywhere: one more bounded wait for every bulk copy and the
        // last tensor-memory copy still in flight before shared and tensor memory are
        // released (a commit completes after every earlier copy of its thread).
        bool again = false;
        for (int64_t g = std::max<int64_t>(0, issued - Rg); g < issued; ++g)
            mbar_wait_bounded(&full[g % Rg], (uint32_t)((g / Rg) & 1), again, a.status);
        const long long copied = *copied_s;
        again = false;
        if (copied > 0)
            mbar_wait_bounded(&freed[(copied - 1) % Rg], (uint32_t)(((copied - 1) / Rg) & 1), again, a.status);
    }
    tmem_fence_before();
    __syncthreads();
    if (warp == 0) {
        tmem_fence_after();
        tmem_dealloc_warp(tbase, kRtCols);
    }
}

// Shared memory of the kernel for R landing chunks of `chunk` floats; S and R of the
// operation at most 16 bytes each.
__host__ inline size_t row_tmem_smem(int chunk, int ring) {
    return (size_t)ring * chunk * 4 + (size_t)(3 * kRtRingMax + 2 * kRtMaxRows + 2 * kRtResRing) * 8 + 16 +
           (size_t)kRtResRing * 16 + 64 * 16 + 16;
}

// The launch plan of the kernel (rows x cols, 16-byte aligned x and out, cols % 4 == 0):
// group size GS (`forced` if non-zero), landing chunks of at most chunk_max floats
// (equal chunks, each a multiple of 1024), as many shared-memory slots as fit, and as
// many tensor-memory row buffers as 512 columns hold (8 columns per 1024 floats of the
// slice, at most kRtMaxRows, at least 2).  Where the CTAs loop over rows, slices
// shorter than min_slice floats are taken only when no group size gives a longer one:
// there each row's round trip through the group (publish, merge, store, release) costs
// more than its bytes (16384 for log_softmax, measured on GB300).  Every CTA allocates all of tensor memory, so
// the plan asks for more than half the SM's shared memory: one CTA per SM, and no CTA
// of the cooperative grid waits for another's allocation.  plan.nbuf holds 100 x
// landing slots + tensor-memory row buffers.
inline cudaError_t plan_row_tmem(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                                 int64_t cols, int forced, int chunk_max, int min_slice, GroupPlan* plan) {
    if (cols % 4 != 0 || rows < 1 || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return cudaErrorNotSupported;
    const int chunk_env = std::max(1024, chunk_max / 1024 * 1024);
    const size_t budget = (size_t)dev.max_smem_optin;
    double best = -1.0;
    for (int pass = 0; pass < 2 && best < 0; ++pass) {  // pass 0: slices of min_slice floats or more
        for (int GS = 1; GS <= kRtMaxGroup; ++GS) {
            if (forced && GS != forced) continue;
            const int64_t sl = ((cols + GS - 1) / GS + 31) / 32 * 32;
            if (sl * (GS - 1) >= cols || sl > 64 * 1024) continue;
            if (pass == 0 && !forced && sl < min_slice && rows > dev.sm_count / GS) continue;
            const int cpr = (int)((sl + 1023) / 1024) * 8;
            const int TR = std::min(kRtMaxRows, kRtCols / cpr);
            if (TR < 2) continue;
            // equal chunks of at most chunk_env floats, each a whole number of 1024-float blocks
            const int64_t nch0 = (sl + chunk_env - 1) / chunk_env;
            const int chunk = (int)(((sl + nch0 - 1) / nch0 + 1023) / 1024 * 1024);
            const int nch = (int)((sl + chunk - 1) / chunk);
            const int R = (int)std::min<int64_t>(kRtRingMax, (int64_t)(budget - row_tmem_smem(0, 0)) / ((int64_t)chunk * 4));
            if (R < 2) continue;
            const size_t smem = std::max(row_tmem_smem(chunk, R), budget / 2 + 1024);  // one CTA per SM
            if (smem > budget) continue;
            const int64_t groups = std::min<int64_t>(rows, dev.sm_count / GS);
            if (groups < 1) continue;
            const double score = (double)(groups * GS) / dev.sm_count - 0.002 * GS +
                                 0.01 * std::min(8.0, TR + (double)R / nch);
            if (score > best) {
                best = score;
                plan->threads = row_tmem_threads(4);  // the launch sets its own store-warp count
                plan->nbuf = R * 100 + TR;
                plan->group_size = GS;
                plan->groups = (int)groups;
                plan->slice = (int)sl;
                plan->chunk = chunk;
                plan->smem = smem;
                plan->scratch_bytes = (size_t)groups * kRtSlots * GS * sizeof(unsigned long long);
            }
        }
    }
    return best < 0 ? cudaErrorNotSupported : cudaSuccess;
}

template <class Op, int SW>
cudaError_t launch_row_tmem(const DeviceInfo& dev, const float* x, float* out, int64_t rows, int64_t cols,
                            const GroupPlan& p, void* scratch, cudaStream_t stream, const typename Op::Params& op,
                            const char* name) {
    cudaError_t e = cudaMemsetAsync(scratch, 0xFF, p.scratch_bytes, stream);
    if (e != cudaSuccess) return e;
    const int R = p.nbuf / 100, TR = p.nbuf % 100;
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] %s: GS=%d groups=%d slots=%d tmem_rows=%d slice=%d chunk=%d smem=%zu\n", name,
                p.group_size, p.groups, R, TR, p.slice, p.chunk, p.smem);
    RowTmemArgs<typename Op::Params> args{x, out, rows, cols, p.slice, p.chunk, dev.status, p.group_size,
                                          static_cast<unsigned long long*>(scratch), R, TR, op};
    auto kern = row_tmem_kernel<Op, SW>;
    constexpr int threads = row_tmem_threads(SW);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, p.smem);
    if (e != cudaSuccess) return e;
    if (per_sm != 1) return cudaErrorNotSupported;  // each CTA holds all of the SM's tensor memory
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the group waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)(p.groups * p.group_size));
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace lse
