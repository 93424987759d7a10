// Form 2: row-wise log_softmax over the last axis (and the row lse alone).
//
// out[r, j] = x[r, j] - lse_r, lse_r = max_r + log(sum_j exp(x[r, j] - max_r))
// (POPCORNBENCH page "Kimi-K2.6 / l1_p24", opening analysis).  That page's
// kernels give each row one block and read it two or three times from HBM;
// its traffic analysis judges the ideal of one read plus one write out of
// reach because a 1.5 MiB row does not fit on one SM.  On GB300 it fits in
// the shared memory of a group of CTAs, so the kernels here are:
//
//  rows_reg_kernel      rows up to 32K floats: the row lives in registers of
//                       one warp or one block; exact two-pass (max, then sum)
//                       over registers, one HBM read and one write.
//  row_tmem_kernel      (row_tmem.cuh, with LsmOp below; the default for long
//                       16-byte-aligned rows) a row split
//                       over a group of CTAs of a cooperative grid; each slice
//                       lands chunk by chunk in shared memory (bulk copies),
//                       is folded there and copied on into tensor memory
//                       (tcgen05.cp), where the row waits for its lse while
//                       the next chunks land.  Fold, copy, load, merge and
//                       store warps; the CTAs' pairs meet in tagged slots.
//                       One HBM read and one write, on all 152 SMs.
//  lsm_ws_kernel        the same split with each slice held in NB whole-slice
//                       shared-memory buffers (the default where the tensor-
//                       memory kernel has no plan); lsm_ring_kernel the same
//                       with a ring of chunk slots.
//  lsm_smem_kernel      the same staging with the pairs merged through a
//                       cluster's distributed shared memory or in lock step
//                       (selectable; slower on GB300).
//  lsm_l2_group_kernel  a group's slices read twice, the second time from L2
//                       (selectable; slower on GB300).
//  lsm_smem_cluster     rows up to 16 x ~226 KB: each CTA of a cluster copies
//                       its slice of the row into shared memory with bulk
//                       (TMA) copies, folds it into a running (max, sum) pair
//                       as the chunks land, the CTAs merge their pairs through
//                       distributed shared memory, and the output is written
//                       from shared memory.  Persistent: while chunk c of row
//                       i is written out, chunk c of the next row is already
//                       being copied into the same buffer.  One HBM read.
//  rows_stream_kernel   any row: each CTA of a cluster streams its slice twice
//                       (stats, then x - lse), merging pairs through
//                       distributed shared memory.  With mode 1 it makes one
//                       pass and writes the row lse only.
//
// The pair update is the online formulation of the same page (running max,
// running sum rescaled when the max grows, pairs merged as
// m = max(m1, m2), s = s1 e^(m1-m) + s2 e^(m2-m)).
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "row_tmem.cuh"
#include "tmem.cuh"

namespace lse {

// ------------------------------------------------------------------ helpers


__device__ __forceinline__ float lse_from_max_sum(float m, float s) {
    if (isnan(m)) return CUDART_NAN_F;
    if (m == CUDART_INF_F) return CUDART_INF_F;
    if (m == -CUDART_INF_F) return -CUDART_INF_F;
    return m + logf(s);
}

// ------------------------------------------------------------------ rows in registers

// Block (GT, RPB): GT threads per row (32, or the whole block when RPB == 1),
// RPB rows per block.  Each thread holds VPT vectors of VEC floats of its row.
template <int VEC, int VPT, int MODE>
__global__ void __launch_bounds__(1024) rows_reg_kernel(const float* __restrict__ x,
                                                        float* __restrict__ out, int64_t rows,
                                                        int64_t cols) {
    __shared__ float red[32];
    const int GT = blockDim.x;
    const int RPB = blockDim.y;
    const int t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5, nwarps = GT >> 5;
    for (int64_t row0 = (int64_t)blockIdx.x * RPB; row0 < rows; row0 += (int64_t)gridDim.x * RPB) {
        const int64_t row = row0 + threadIdx.y;
        const bool rv = row < rows;
        const float* src = x + row * cols;
        float v[VPT][VEC];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t j = ((int64_t)k * GT + t) * VEC;
            if (rv && j < cols) {
                if constexpr (VEC == 4) {
                    float4 a = ld_stream_f4(src + j);
                    v[k][0] = a.x; v[k][1] = a.y; v[k][2] = a.z; v[k][3] = a.w;
                } else {
                    v[k][0] = ld_stream_f1(src + j);
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = -CUDART_INF_F;
            }
        }
        float m = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = max_nan(m, v[k][e]);
        m = warp_allmax_nan(m);
        if (nwarps > 1) {
            __syncthreads();
            if (lane == 0) red[warp] = m;
            __syncthreads();
            m = warp_allmax_nan(lane < nwarps ? red[lane] : -CUDART_INF_F);
        }
        const float base = isfinite(m) ? m : 0.f;  // see ms_fold on why v - m comes first
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) s += ex2((v[k][e] - base) * kLog2e);
        s = warp_allsum(s);
        if (nwarps > 1) {
            __syncthreads();
            if (lane == 0) red[warp] = s;
            __syncthreads();
            s = warp_allsum(lane < nwarps ? red[lane] : 0.f);
        }
        const float lse = lse_from_max_sum(m, s);
        if constexpr (MODE != 1) {
            constexpr bool SM = (MODE == 2);
            if (rv) {
                float* dst = out + row * cols;
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int64_t j = ((int64_t)k * GT + t) * VEC;
                    if (j < cols) {
                        if constexpr (VEC == 4) {
                            st_stream_f4(dst + j, make_float4(row_out<SM>(v[k][0], lse), row_out<SM>(v[k][1], lse),
                                                              row_out<SM>(v[k][2], lse), row_out<SM>(v[k][3], lse)));
                        } else {
                            st_stream_f1(dst + j, row_out<SM>(v[k][0], lse));
                        }
                    }
                }
            }
        } else {
            if (rv && t == 0) out[row] = lse;
        }
    }
}

template <int VEC, int VPT, int MODE>
static cudaError_t rows_reg_go(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                               int64_t cols, int GT, cudaStream_t stream) {
    const int RPB = (GT == 32) ? 8 : 1;
    const int64_t nblk = (rows + RPB - 1) / RPB;
    const int per_sm = std::max(1, 2048 / (GT * RPB));
    const int64_t cap = (int64_t)dev.sm_count * per_sm * 32;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(nblk, cap));
    rows_reg_kernel<VEC, VPT, MODE><<<grid, dim3(GT, RPB), 0, stream>>>(x, out, rows, cols);
    return cudaGetLastError();
}

template <int MODE>
static cudaError_t rows_reg_dispatch(const DeviceInfo& dev, const float* x, float* out,
                                     int64_t rows, int64_t cols, bool vec4, cudaStream_t stream) {
    // Smallest configuration whose GT * VPT * VEC covers the row.
    if (vec4) {
        if (cols <= 32 * 4 * 1) return rows_reg_go<4, 1, MODE>(dev, x, out, rows, cols, 32, stream);
        if (cols <= 32 * 4 * 4) return rows_reg_go<4, 4, MODE>(dev, x, out, rows, cols, 32, stream);
        if (cols <= 128 * 4 * 4) return rows_reg_go<4, 4, MODE>(dev, x, out, rows, cols, 128, stream);
        if (cols <= 256 * 4 * 4) return rows_reg_go<4, 4, MODE>(dev, x, out, rows, cols, 256, stream);
        if (cols <= 256 * 4 * 8) return rows_reg_go<4, 8, MODE>(dev, x, out, rows, cols, 256, stream);
        if (cols <= 512 * 4 * 8) return rows_reg_go<4, 8, MODE>(dev, x, out, rows, cols, 512, stream);
        return rows_reg_go<4, 8, MODE>(dev, x, out, rows, cols, 1024, stream);
    }
    if (cols <= 32 * 1) return rows_reg_go<1, 1, MODE>(dev, x, out, rows, cols, 32, stream);
    if (cols <= 32 * 8) return rows_reg_go<1, 8, MODE>(dev, x, out, rows, cols, 32, stream);
    if (cols <= 256 * 8) return rows_reg_go<1, 8, MODE>(dev, x, out, rows, cols, 256, stream);
    if (cols <= 1024 * 8) return rows_reg_go<1, 8, MODE>(dev, x, out, rows, cols, 1024, stream);
    return rows_reg_go<1, 16, MODE>(dev, x, out, rows, cols, 1024, stream);
}

cudaError_t launch_rows_reg(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                            int64_t cols, int mode, cudaStream_t stream) {
    const bool vec4 = (cols % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0) &&
                      ((reinterpret_cast<uintptr_t>(out) & 15) == 0 || mode == 1);
    // Scalar rows hold 16 floats per thread at most (1024 threads).
    if (cols > kRegRowMaxCols || (!vec4 && cols > 1024 * 16))
        return launch_rows_stream(dev, x, out, rows, cols, mode, stream);
    if (mode == 0) return rows_reg_dispatch<0>(dev, x, out, rows, cols, vec4, stream);
    if (mode == 2) return rows_reg_dispatch<2>(dev, x, out, rows, cols, vec4, stream);
    return rows_reg_dispatch<1>(dev, x, out, rows, cols, vec4, stream);
}

// ------------------------------------------------------------------ rows in cluster shared memory

constexpr int kSmemMaxChunks = 64;

struct SmemLayout {
    int slice;      // floats of the row owned by one CTA (multiple of 4)
    int chunk;      // floats per bulk copy (multiple of 4)
    size_t bytes;   // dynamic shared memory per CTA
};

__host__ __device__ inline size_t smem_cluster_bytes(int slice, int nbuf = 1) {
    // [nbuf x slice floats][nbuf x kSmemMaxChunks mbarriers][2 MS partials][32 MS scratch][lse + pad]
    return (size_t)nbuf * ((size_t)slice * 4 + kSmemMaxChunks * 8) + 2 * sizeof(MS) + 32 * sizeof(MS) + 16;
}

struct SmemRowArgs {
    const float* x;
    float* out;
    int64_t rows, cols;
    int slice;           // floats of a row owned by one CTA (multiple of 4)
    int chunk;           // floats per bulk copy (multiple of 4)
    int* status;         // device status word (bounded-wait timeouts)
    // group variant only
    int group_size;            // CTAs per row; CTA b is rank b % group_size of group b / group_size
    unsigned long long* slots; // [groups][2][group_size] tagged pairs, all bytes 0xFF at launch
    int softmax;               // warp-specialised kernel: write exp(x - lse) instead of x - lse
    int ring;                  // ring / tensor-memory kernels: chunk slots of shared memory per CTA
    int trows;                 // tensor-memory kernel: row buffers in tensor memory
};

// Rows staged in shared memory, one slice per CTA, the CTAs of a row merging
// their (m, s) pairs either through distributed shared memory (GROUP = false:
// the CTAs of a thread-block cluster) or through global memory (GROUP = true:
// group_size CTAs of a cooperative grid, through tagged slots).
// Persistent: a group / cluster walks rows first, first + count, ...
//
// NBUF = 1: per row, fold the slice as its chunks land, merge (arrive + wait),
// write x - lse chunk by chunk, refilling each chunk with the next row.
// NBUF >= 2 (split phase): NBUF slices per CTA.  Step j folds row j, then waits
// for the merge of row j-1 (whose arrival was one fold earlier, so a straggler
// in the group costs nothing unless it is a whole row late), arrives for row j
// and writes row j-1, refilling its buffer with row j+1.  Because every CTA
// arrives for row j only after its wait for row j-1, no CTA is more than one
// arrival ahead: two tagged partial slots per CTA suffice.  Writing row j-1
// refills its buffer with row j-1+NBUF, so with NBUF = 3 the copies run two
// rows ahead: while row j is folded, row j+1 is already landing.
template <int THREADS, bool GROUP>
struct RowMerge {
    MS* part;                   // cluster: this CTA's two partial slots (shared memory)
    unsigned long long* slots;  // group: this group's [2][GS] tagged slots (global memory)
    unsigned long long pend;    // group: this lane's prefetched slot word
    uint32_t rank, GS;

    // Publishes this CTA's pair for step `it` (all threads call; st is the block
    // pair).  Group: one 64-bit relaxed store of the pair, tagged with the use
    // count of its slot mod 2 (slot it % 2 is reused two steps later, and no
    // CTA arrives for step it + 2 before every CTA has read step it).
    __device__ __forceinline__ void arrive(uint32_t it, const MS& st) {
        if constexpr (GROUP) {
            if (threadIdx.x == 0)
                st_relaxed_gpu_u64(slots + (it & 1u) * GS + rank, ms_pack_tagged(st, (it >> 1) & 1u));
        } else {
            if (threadIdx.x == 0) part[it & 1u] = st;
            asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        }
    }

    // Group: lanes 0..GS-1 of warp 0 issue their slot loads for step `it` early
    // (the result is only needed in wait()).
    __device__ __forceinline__ void prefetch(uint32_t it) {
        if constexpr (GROUP) {
            if (threadIdx.x < GS) pend = ld_relaxed_gpu_u64(slots + (it & 1u) * GS + threadIdx.x);
        }
    }

    // Group only, warp 0 only: waits for every CTA's pair of step `it` (after
    // prefetch(it)) and returns the merged lse in every lane; no block barrier.
    __device__ __forceinline__ float wait_warp0(uint32_t it, bool& aborted, int* status) {
        MS mine = ms_empty();
        if (threadIdx.x < GS) {
            const unsigned long long* p = slots + (it & 1u) * GS + threadIdx.x;
            mine = ms_unpack(poll_slot(p, (it >> 1) & 1u, pend, aborted, status));
        }
        return ms_lse(ms_warp_allreduce(mine));
    }

    // Waits for every CTA's pair of step `it` (after prefetch(it)), merges them
    // (same order in every CTA, so all compute the same lse) and returns the lse
    // to all threads.
    __device__ __forceinline__ float wait(uint32_t it, float* lse_sh, bool& aborted, int* status) {
        if constexpr (GROUP) {
            if (threadIdx.x < 32) {
                MS mine = ms_empty();
                if (threadIdx.x < GS) {
                    const unsigned long long* p = slots + (it & 1u) * GS + threadIdx.x;
                    mine = ms_unpack(poll_slot(p, (it >> 1) & 1u, pend, aborted, status));
                }
                const MS tot = ms_warp_allreduce(mine);
                if (threadIdx.x == 0) *lse_sh = ms_lse(tot);
            }
        } else {
            asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
            if (threadIdx.x == 0) {
                MS tot = ms_empty();
                for (uint32_t k = 0; k < GS; ++k) tot = ms_merge(tot, ld_peer_ms(&part[it & 1u], k));
                *lse_sh = ms_lse(tot);
            }
        }
        __syncthreads();
        return *lse_sh;
    }
};

template <int THREADS, bool GROUP, int NBUF>
__global__ void __launch_bounds__(THREADS, (1024 / THREADS > 0 ? 1024 / THREADS : 1))
    lsm_smem_kernel(const SmemRowArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int slice = a.slice, chunk = a.chunk;
    const int64_t rows = a.rows, cols = a.cols;
    float* const buf0 = reinterpret_cast<float*>(smem_raw);
    uint64_t* const bars0 = reinterpret_cast<uint64_t*>(smem_raw + (size_t)NBUF * slice * 4);
    MS* part = reinterpret_cast<MS*>(bars0 + NBUF * kSmemMaxChunks);
    MS* red = part + 2;
    float* lse_sh = reinterpret_cast<float*>(red + 32);

    RowMerge<THREADS, GROUP> mg;
    mg.pend = 0;
    int64_t first_row, row_step;
    if constexpr (GROUP) {
        mg.GS = (uint32_t)a.group_size;
        mg.rank = blockIdx.x % mg.GS;
        first_row = blockIdx.x / mg.GS;
        row_step = gridDim.x / mg.GS;
        mg.slots = a.slots + first_row * 2 * mg.GS;
        mg.part = nullptr;
    } else {
        mg.rank = cluster_ctarank();
        mg.GS = cluster_nctarank();
        first_row = cluster_id_x();
        row_step = nclusters_x();
        mg.part = part;
        mg.slots = nullptr;
    }
    const int64_t c_begin = (int64_t)mg.rank * slice;
    const int len = (int)std::max<int64_t>(0, std::min<int64_t>(slice, cols - c_begin));
    const int nch = (len + chunk - 1) / chunk;
    const int tid = threadIdx.x;
    const int64_t nrows = first_row < rows ? (rows - first_row + row_step - 1) / row_step : 0;
    bool aborted = false;
    uint32_t filled[NBUF], folded[NBUF];  // rows issued into / folded from each buffer (thread 0)
#pragma unroll
    for (int b = 0; b < NBUF; ++b) filled[b] = folded[b] = 0;

    if (tid == 0) {
        for (int c = 0; c < NBUF * kSmemMaxChunks; ++c) mbar_init(&bars0[c], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // Copies step j's row (if any) into buffer j % NBUF (thread 0; chunk c only,
    // or all chunks when c < 0).
    auto issue = [&](int64_t j, int c_only) {
        if (j >= nrows || aborted) return;
        const int b = (int)(j % NBUF);
        if (c_only <= 0) ++filled[b];
        const float* src = a.x + (first_row + j * row_step) * cols + c_begin;
        for (int c = (c_only < 0 ? 0 : c_only); c < (c_only < 0 ? nch : c_only + 1); ++c) {
            const int cb = c * chunk;
            const uint32_t bytes = (uint32_t)std::min(chunk, len - cb) * 4u;
            if (c_only >= 0) fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars0[b * kSmemMaxChunks + c], bytes);
            bulk_g2s(buf0 + (size_t)b * slice + cb, src + cb, bytes, &bars0[b * kSmemMaxChunks + c]);
        }
    };

    // Folds step j's slice into the block pair as its chunks land.
    auto fold = [&](int64_t j) -> MS {
        const int b = (int)(j % NBUF);
        const uint32_t phase = (uint32_t)((j / NBUF) & 1);
        const float* buf = buf0 + (size_t)b * slice;
        uint64_t* bars = bars0 + b * kSmemMaxChunks;
        MS st = ms_empty();
        for (int c = 0; c < nch; ++c) {
            mbar_wait_bounded(&bars[c], phase, aborted, a.status);
            const int cb = c * chunk;
            const int n4 = std::min(chunk, len - cb) >> 2;
            const float4* p = reinterpret_cast<const float4*>(buf + cb);
            int i = tid;
            for (; i + 3 * THREADS < n4; i += 4 * THREADS) {
                float v[16];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float4 q = p[i + k * THREADS];
                    v[4 * k + 0] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
                }
                ms_fold<16>(st, v);
            }
            for (; i < n4; i += THREADS) {
                float4 q = p[i];
                float v[4] = {q.x, q.y, q.z, q.w};
                ms_fold<4>(st, v);
            }
        }
        if (!aborted) ++folded[b];
        return ms_block_allreduce(st, red);
    };

    // Writes step j's row as x - lse from its buffer; as each chunk is consumed,
    // copies step j + NBUF's row into it.
    auto store = [&](int64_t j, float lse) {
        const int b = (int)(j % NBUF);
        const float* buf = buf0 + (size_t)b * slice;
        float* dst = a.out + (first_row + j * row_step) * cols + c_begin;
        for (int c = 0; c < nch; ++c) {
            const int cb = c * chunk;
            const int n4 = std::min(chunk, len - cb) >> 2;
            const float4* p = reinterpret_cast<const float4*>(buf + cb);
            for (int i = tid; i < n4; i += THREADS) {
                float4 q = p[i];
                st_stream_f4(dst + cb + 4 * i, make_float4(q.x - lse, q.y - lse, q.z - lse, q.w - lse));
            }
            __syncthreads();  // every thread is done reading chunk c
            if (tid == 0) issue(j + NBUF, c);
        }
    };

    if (tid == 0)
        for (int j = 0; j < NBUF; ++j) issue(j, -1);

    static_assert(NBUF >= 1 && NBUF <= 3, "one to three buffers");
    if constexpr (NBUF == 1) {
        for (int64_t j = 0; j < nrows; ++j) {
            const MS st = fold(j);
            mg.arrive((uint32_t)j, st);
            mg.prefetch((uint32_t)j);
            const float lse = mg.wait((uint32_t)j, lse_sh, aborted, a.status);
            store(j, lse);
        }
    } else {
        for (int64_t j = 0; j <= nrows; ++j) {
            if (j > 0) mg.prefetch((uint32_t)(j - 1));  // in flight during the fold
            MS st = ms_empty();
            if (j < nrows) st = fold(j);
            float lse_prev = 0.f;
            if (j > 0) lse_prev = mg.wait((uint32_t)(j - 1), lse_sh, aborted, a.status);
            if (j < nrows) mg.arrive((uint32_t)j, st);
            if (j > 0) store(j - 1, lse_prev);
        }
    }

    if (aborted && tid == 0) {
        // A copy never completed; none was issued after that.  Give each buffer's
        // fill still outstanding (at most one per buffer) one more bounded wait
        // before the CTA releases its shared memory.
        bool again = false;
        for (int bb = 0; bb < NBUF; ++bb) {
            if (filled[bb] <= folded[bb]) continue;
            for (int c = 0; c < nch; ++c)
                mbar_wait_bounded(&bars0[bb * kSmemMaxChunks + c], folded[bb] & 1u, again, a.status);
        }
    }
    if constexpr (!GROUP) cluster_sync();  // peers may still read part[] of this CTA
}

// Slice = ceil(cols / G) rounded up to 32 floats, so that every slice starts on
// a 128-byte line (neighbouring CTAs never share a line); chunk = floats per
// bulk copy (at most kSmemMaxChunks per slice).
// Warp-specialised group kernel, NB buffers per CTA.  FW fold warps fold each
// row (as its chunks land) and publish the CTA's pair; they never wait for the
// group.  SW store warps wait for the group's pairs of row j, merge them, write
// row j out of its buffer and refill each of its chunks with row j+NB.  Store
// back-pressure and the merge wait then stall only the store warps, while the
// fold warps run up to NB rows ahead.  A fold warp publishing row r implies
// every store warp of the group has read row r-2NB (r needs this CTA's store
// of r-NB, which needed every pair of r-NB, which needed every CTA's store of
// r-2NB), so kWsSlots = 16 >= 2NB tagged slots per CTA (tag = (r / 16) mod 2)
// suffice.  Groups of up to 64 CTAs: each lane of the merging warp reads two
// slots.
constexpr int kWsSlots = 16;
constexpr int kWsMaxGroup = 64;

template <int FW, int SW, int NB>
__global__ void __launch_bounds__(32 * (FW + SW), 1) lsm_ws_kernel(const SmemRowArgs a) {
    static_assert(2 * NB <= kWsSlots, "slots must cover two rounds of buffers");
    constexpr int NF = 32 * FW, NS = 32 * SW;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int slice = a.slice, chunk = a.chunk;
    const int64_t rows = a.rows, cols = a.cols;
    float* const buf0 = reinterpret_cast<float*>(smem_raw);
    uint64_t* const full = reinterpret_cast<uint64_t*>(smem_raw + (size_t)NB * slice * 4);  // [NB][K]
    float* const lse_s = reinterpret_cast<float*>(full + NB * kSmemMaxChunks);              // [1]
    MS* const red = reinterpret_cast<MS*>(lse_s + 4);                                      // [2][32]

    const uint32_t GS = (uint32_t)a.group_size;
    const uint32_t rank = blockIdx.x % GS;
    const int64_t first_row = blockIdx.x / GS;
    const int64_t row_step = gridDim.x / GS;
    unsigned long long* const slots = a.slots + first_row * kWsSlots * GS;  // [kWsSlots][GS]
    const int64_t c_begin = (int64_t)rank * slice;
    const int len = (int)std::max<int64_t>(0, std::min<int64_t>(slice, cols - c_begin));
    const int nch = (len + chunk - 1) / chunk;
    const int64_t nrows = first_row < rows ? (rows - first_row + row_step - 1) / row_step : 0;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    bool aborted = false;

    if (tid == 0) {
        for (int c = 0; c < NB * kSmemMaxChunks; ++c) mbar_init(&full[c], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // Issuer: the first store thread.  Copies step j's row into buffer j % NB.
    uint32_t filled[NB];
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) filled[bb] = 0;
    auto issue = [&](int64_t j, int c_only) {
        if (j >= nrows || aborted) return;
        const int b = (int)(j % NB);
        if (c_only <= 0) ++filled[b];
        const float* src = a.x + (first_row + j * row_step) * cols + c_begin;
        for (int c = (c_only < 0 ? 0 : c_only); c < (c_only < 0 ? nch : c_only + 1); ++c) {
            const int cb = c * chunk;
            const uint32_t bytes = (uint32_t)std::min(chunk, len - cb) * 4u;
            if (c_only >= 0) fence_proxy_async_smem();
            mbar_arrive_expect_tx(&full[b * kSmemMaxChunks + c], bytes);
            bulk_g2s(buf0 + (size_t)b * slice + cb, src + cb, bytes, &full[b * kSmemMaxChunks + c]);
        }
    };
    if (tid == NF)
        for (int j = 0; j < NB; ++j) issue(j, -1);

    if (warp < FW) {
        // ---------------- fold warps: fold, reduce, publish; never wait for the group
        for (int64_t j = 0; j < nrows; ++j) {
            const int b = (int)(j % NB);
            const uint32_t phase = (uint32_t)((j / NB) & 1);
            const float* buf = buf0 + (size_t)b * slice;
            MS st = ms_empty();
            for (int c = 0; c < nch; ++c) {
                mbar_wait_bounded(&full[b * kSmemMaxChunks + c], phase, aborted, a.status);
                const int cb = c * chunk;
                const int n4 = std::min(chunk, len - cb) >> 2;
                const float4* p = reinterpret_cast<const float4*>(buf + cb);
                int i = tid;
                for (; i + 3 * NF < n4; i += 4 * NF) {
                    float v[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float4 q = p[i + k * NF];
                        v[4 * k + 0] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
                    }
                    ms_fold<16>(st, v);
                }
                for (; i < n4; i += NF) {
                    float4 q = p[i];
                    float v[4] = {q.x, q.y, q.z, q.w};
                    ms_fold<4>(st, v);
                }
            }
            st = ms_warp_allreduce(st);
            if (lane == 0) red[(j & 1) * 32 + warp] = st;
            named_bar_sync(1, NF);  // every fold warp is done with this row and its red slot
            if (warp == 0) {
                MS r = (lane < FW) ? red[(j & 1) * 32 + lane] : ms_empty();
                r = ms_warp_allreduce(r);
                if (lane == 0)
                    st_relaxed_gpu_u64(slots + (j % kWsSlots) * GS + rank,
                                       ms_pack_tagged(r, (uint32_t)(j / kWsSlots) & 1u));
            }
        }
    } else {
        // ---------------- store warps: merge the group's pairs, write, refill
        const int sid = tid - NF;
        for (int64_t j = 0; j < nrows; ++j) {
            const int b = (int)(j % NB);
            if (sid < 32) {
                MS mine = ms_empty();
                for (uint32_t k = (uint32_t)sid; k < GS; k += 32) {
                    const unsigned long long* p = slots + (j % kWsSlots) * GS + k;
                    const MS other = ms_unpack(poll_slot(p, (uint32_t)(j / kWsSlots) & 1u,
                                                         ld_relaxed_gpu_u64(p), aborted, a.status));
                    mine = ms_merge(mine, other);
                }
                const float l = ms_lse(ms_warp_allreduce(mine));
                if (sid == 0) *lse_s = l;
            }
            named_bar_sync(2, NS);  // lse_s holds row j's lse
            const float lse = *lse_s;
            const float* buf = buf0 + (size_t)b * slice;
            float* dst = a.out + (first_row + j * row_step) * cols + c_begin;
            for (int c = 0; c < nch; ++c) {
                const int cb = c * chunk;
                const int n4 = std::min(chunk, len - cb) >> 2;
                const float4* p = reinterpret_cast<const float4*>(buf + cb);
                if (a.softmax) {
                    for (int i = sid; i < n4; i += NS) st_stream_f4(dst + cb + 4 * i, row_out4(p[i], lse, true));
                } else {
                    for (int i = sid; i < n4; i += NS) st_stream_f4(dst + cb + 4 * i, row_out4(p[i], lse, false));
                }
                named_bar_sync(2, NS);  // every store warp is done reading chunk c (and lse_s)
                if (sid == 0) issue(j + NB, c);
            }
        }
    }
    __syncthreads();
    if (tid == NF) {
        // After a timeout anywhere, give each buffer's last issued fill one more
        // bounded wait before the shared memory is released.
        if (atomicAdd(a.status, 0) != 0) {
            bool again = false;
            for (int bb = 0; bb < NB; ++bb) {
                if (filled[bb] == 0) continue;
                for (int c = 0; c < nch; ++c)
                    mbar_wait_bounded(&full[bb * kSmemMaxChunks + c], (filled[bb] - 1) & 1u, again, a.status);
            }
        }
    }
}

// Ring form of the warp-specialised group kernel: a CTA's shared memory is a ring of
// R chunk slots instead of NB whole-slice buffers, so that the rows in flight need not
// be a whole number.  Eight groups of 19 CTAs cover all 152 SMs with 81 KB slices, of
// which 3 would not fit in shared memory; a ring of 8 slots of 27 KB keeps 2.67 rows
// (216 KB) in flight instead.  Chunk c of the CTA's step j is its chunk
// g = j * nch + c, held in slot g % R (phase (g / R) & 1); the store warps refill a
// slot with chunk g + R as soon as they have written chunk g out.  The fold and store
// roles and the tagged pair slots are those of lsm_ws_kernel: a fold warp publishing
// row r implies every store warp of the group has read the pairs of row
// r - 2 ceil(R / nch), so ceil(R / nch) <= kWsSlots / 2 for every CTA of the group
// (the last, with the shortest slice and fewest chunks, runs furthest ahead) keeps
// the 16 slots safe.
constexpr int kRingMax = 64;

template <int FW, int SW>
__global__ void __launch_bounds__(32 * (FW + SW), 1) lsm_ring_kernel(const SmemRowArgs a) {
    constexpr int NF = 32 * FW, NS = 32 * SW;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int chunk = a.chunk, R = a.ring;
    const int64_t rows = a.rows, cols = a.cols;
    float* const ring = reinterpret_cast<float*>(smem_raw);                                 // [R][chunk]
    uint64_t* const full = reinterpret_cast<uint64_t*>(smem_raw + (size_t)R * chunk * 4);  // [R]
    float* const lse_s = reinterpret_cast<float*>(full + kRingMax);                        // [1]
    MS* const red = reinterpret_cast<MS*>(lse_s + 4);                                      // [2][32]

    const uint32_t GS = (uint32_t)a.group_size;
    const uint32_t rank = blockIdx.x % GS;
    const int64_t first_row = blockIdx.x / GS;
    const int64_t row_step = gridDim.x / GS;
    unsigned long long* const slots = a.slots + first_row * kWsSlots * GS;  // [kWsSlots][GS]
    const int64_t c_begin = (int64_t)rank * a.slice;
    const int len = (int)std::max<int64_t>(0, std::min<int64_t>(a.slice, cols - c_begin));
    const int nch = (len + chunk - 1) / chunk;
    const int64_t nrows = first_row < rows ? (rows - first_row + row_step - 1) / row_step : 0;
    const int64_t total = nrows * nch;  // chunks this CTA moves
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    bool aborted = false;

    if (tid == 0) {
        for (int r = 0; r < R; ++r) mbar_init(&full[r], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // Issuer: the first store thread.  Copies the CTA's chunk g into slot g % R.
    int64_t issued = 0;
    auto issue = [&](int64_t g) {
        if (g >= total || aborted) return;
        const int64_t j = g / nch;
        const int c = (int)(g - j * nch);
        const int sl = (int)(g % R);
        const int cb = c * chunk;
        const uint32_t bytes = (uint32_t)std::min(chunk, len - cb) * 4u;
        fence_proxy_async_smem();  // earlier generic reads of the slot come first
        mbar_arrive_expect_tx(&full[sl], bytes);
        bulk_g2s(ring + (size_t)sl * chunk, a.x + (first_row + j * row_step) * cols + c_begin + cb, bytes, &full[sl]);
        issued = g + 1;
    };
    if (tid == NF)
        for (int g = 0; g < R; ++g) issue(g);

    if (warp < FW) {
        // ---------------- fold warps: fold, reduce, publish; never wait for the group
        for (int64_t j = 0; j < nrows; ++j) {
            MS st = ms_empty();
            for (int c = 0; c < nch; ++c) {
                const int64_t g = j * nch + c;
                const int sl = (int)(g % R);
                mbar_wait_bounded(&full[sl], (uint32_t)((g / R) & 1), aborted, a.status);
                const int n4 = std::min(chunk, len - c * chunk) >> 2;
                const float4* p = reinterpret_cast<const float4*>(ring + (size_t)sl * chunk);
                int i = tid;
                for (; i + 3 * NF < n4; i += 4 * NF) {
                    float v[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float4 q = p[i + k * NF];
                        v[4 * k + 0] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
                    }
                    ms_fold<16>(st, v);
                }
                for (; i < n4; i += NF) {
                    float4 q = p[i];
                    float v[4] = {q.x, q.y, q.z, q.w};
                    ms_fold<4>(st, v);
                }
            }
            st = ms_warp_allreduce(st);
            if (lane == 0) red[(j & 1) * 32 + warp] = st;
            named_bar_sync(1, NF);  // every fold warp is done with this row and its red slot
            if (warp == 0) {
                MS r = (lane < FW) ? red[(j & 1) * 32 + lane] : ms_empty();
                r = ms_warp_allreduce(r);
                if (lane == 0)
                    st_relaxed_gpu_u64(slots + (j % kWsSlots) * GS + rank,
                                       ms_pack_tagged(r, (uint32_t)(j / kWsSlots) & 1u));
            }
        }
    } else {
        // ---------------- store warps: merge the group's pairs, write, refill
        const int sid = tid - NF;
        for (int64_t j = 0; j < nrows; ++j) {
            if (sid < 32) {
                MS mine = ms_empty();
                for (uint32_t k = (uint32_t)sid; k < GS; k += 32) {
                    const unsigned long long* p = slots + (j % kWsSlots) * GS + k;
                    const MS other = ms_unpack(poll_slot(p, (uint32_t)(j / kWsSlots) & 1u,
                                                         ld_relaxed_gpu_u64(p), aborted, a.status));
                    mine = ms_merge(mine, other);
                }
                const float l = ms_lse(ms_warp_allreduce(mine));
                if (sid == 0) *lse_s = l;
            }
            named_bar_sync(2, NS);  // lse_s holds row j's lse
            const float lse = *lse_s;
            float* dst = a.out + (first_row + j * row_step) * cols + c_begin;
            for (int c = 0; c < nch; ++c) {
                const int64_t g = j * nch + c;
                const int cb = c * chunk;
                const int n4 = std::min(chunk, len - cb) >> 2;
                const float4* p = reinterpret_cast<const float4*>(ring + (size_t)(g % R) * chunk);
                if (a.softmax) {
                    for (int i = sid; i < n4; i += NS) st_stream_f4(dst + cb + 4 * i, row_out4(p[i], lse, true));
                } else {
                    for (int i = sid; i < n4; i += NS) st_stream_f4(dst + cb + 4 * i, row_out4(p[i], lse, false));
                }
                named_bar_sync(2, NS);  // every store warp is done reading chunk g (and lse_s)
                if (sid == 0) issue(g + R);
            }
        }
    }
    __syncthreads();
    if (tid == NF && atomicAdd(a.status, 0) != 0) {
        // After a timeout anywhere, give each slot's last issued fill one more bounded
        // wait before the shared memory is released.
        bool again = false;
        for (int64_t g = std::max<int64_t>(0, issued - R); g < issued; ++g)
            mbar_wait_bounded(&full[g % R], (uint32_t)((g / R) & 1), again, a.status);
    }
}

// ---- rows parked in tensor memory while their lse is merged (row_tmem.cuh)

// The row statistic of log_softmax / softmax for the tensor-memory row kernel: the
// (max, sum of exponentials) pair, the row's lse, and x - lse or its exponential.
struct LsmOp {
    struct Params {
        int softmax;
    };
    using S = MS;
    using R = float;
    struct Cursor {
        float lse;
        bool softmax;
    };
    __device__ static S empty() { return ms_empty(); }
    template <int K>
    __device__ static void fold(S& st, const float (&v)[K]) {
        ms_fold<K>(st, v);
    }
    __device__ static S warp_allreduce(S st) { return ms_warp_allreduce(st); }
    __device__ static S merge(S x, S y) { return ms_merge(x, y); }
    __device__ static unsigned long long pack(S st, uint32_t tag) { return ms_pack_tagged(st, tag); }
    __device__ static S unpack(unsigned long long w, int64_t) { return ms_unpack(w); }
    __device__ static R finish(S st, const Params&) { return ms_lse(st); }
    __device__ static Cursor cursor(R lse, const Params& p, int64_t) { return Cursor{lse, p.softmax != 0}; }
    __device__ static float4 out4(Cursor& c, float4 x, int64_t) { return row_out4(x, c.lse, c.softmax); }
};

__host__ inline size_t smem_ring_bytes(int chunk, int ring) {
    return (size_t)ring * chunk * 4 + (size_t)kRingMax * 8 + 16 + 64 * sizeof(MS);
}

__host__ inline size_t smem_ws_bytes(int slice, int nb) {
    return (size_t)nb * slice * 4 + (size_t)nb * kSmemMaxChunks * 8 + 16 + 64 * sizeof(MS);
}

static void smem_chunking(int64_t cols, int G, int chunk_env, int* slice, int* chunk) {
    const int64_t sl = ((cols + G - 1) / G + 31) / 32 * 32;
    *slice = (int)std::min<int64_t>(sl, 1 << 26);
    int ch = std::min(std::max(1024, chunk_env & ~3), *slice);
    if ((*slice + ch - 1) / ch > kSmemMaxChunks) ch = ((*slice + kSmemMaxChunks - 1) / kSmemMaxChunks + 3) / 4 * 4;
    *chunk = ch;
}

template <int THREADS, int NBUF>
static cudaError_t smem_cluster_go(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                   int64_t cols, int CL, int slice, int chunk, size_t smem,
                                   cudaStream_t stream) {
    auto kern = lsm_smem_kernel<THREADS, false, NBUF>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (CL > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.gridDim = dim3(CL);
    int max_clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (max_clusters < 1) return cudaErrorNotSupported;
    const int64_t nclusters = std::min<int64_t>(rows, max_clusters);
    cfg.gridDim = dim3((unsigned)(nclusters * CL));
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] lsm_smem cluster: CL=%d nbuf=%d threads=%d slice=%d chunk=%d smem=%zu "
                "max_clusters=%d clusters=%lld\n", CL, NBUF, THREADS, slice, chunk, smem, max_clusters,
                (long long)nclusters);
    SmemRowArgs args{x, out, rows, cols, slice, chunk, dev.status, CL, nullptr};
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Picks the cluster size (smallest that stages the row; LSE_LSM_CLUSTER forces
// one), the CTA size (LSE_LSM_THREADS: 256, 512 or 1024) and the bulk-copy
// chunk (LSE_LSM_CHUNK floats).
cudaError_t launch_lsm_smem_cluster(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                    int64_t cols, cudaStream_t stream) {
    if (cols % 4 != 0 || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return cudaErrorNotSupported;
    const int threads = env_int("LSE_LSM_THREADS", 512);
    const int chunk_env = env_int("LSE_LSM_CHUNK", 8192);
    const int forced = env_int("LSE_LSM_CLUSTER", 0);
    const int nbuf = env_int("LSE_LSM_NBUF", 1) == 2 ? 2 : 1;
    const int cands[5] = {1, 2, 4, 8, 16};
    for (int ci = 0; ci < 5; ++ci) {
        const int CL = cands[ci];
        if (forced && CL != forced) continue;
        int slice, ch;
        smem_chunking(cols, CL, chunk_env, &slice, &ch);
        const size_t smem = smem_cluster_bytes(slice, nbuf);
        if ((int64_t)slice * CL < cols || smem > (size_t)dev.max_smem_optin) continue;
        cudaError_t e;
        if (nbuf == 2) {
            if (threads == 256)
                e = smem_cluster_go<256, 2>(dev, x, out, rows, cols, CL, slice, ch, smem, stream);
            else if (threads == 1024)
                e = smem_cluster_go<1024, 2>(dev, x, out, rows, cols, CL, slice, ch, smem, stream);
            else
                e = smem_cluster_go<512, 2>(dev, x, out, rows, cols, CL, slice, ch, smem, stream);
        } else if (threads == 256)
            e = smem_cluster_go<256, 1>(dev, x, out, rows, cols, CL, slice, ch, smem, stream);
        else if (threads == 1024)
            e = smem_cluster_go<1024, 1>(dev, x, out, rows, cols, CL, slice, ch, smem, stream);
        else
            e = smem_cluster_go<512, 1>(dev, x, out, rows, cols, CL, slice, ch, smem, stream);
        if (e == cudaErrorNotSupported || e == cudaErrorInvalidClusterSize) {
            (void)cudaGetLastError();
            continue;
        }
        return e;
    }
    return cudaErrorNotSupported;
}

// ---- group variant: plan (host), then launch with caller-provided scratch

template <int THREADS, int NBUF>
static cudaError_t group_occupancy(size_t smem, int* per_sm) {
    auto kern = lsm_smem_kernel<THREADS, true, NBUF>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, THREADS, smem);
}

static cudaError_t group_occupancy_any(int threads, int nbuf, size_t smem, int* per_sm) {
    if (nbuf == 3) {
        return threads == 256 ? group_occupancy<256, 3>(smem, per_sm)
             : threads == 1024 ? group_occupancy<1024, 3>(smem, per_sm)
                               : group_occupancy<512, 3>(smem, per_sm);
    }
    if (nbuf == 2) {
        return threads == 256 ? group_occupancy<256, 2>(smem, per_sm)
             : threads == 1024 ? group_occupancy<1024, 2>(smem, per_sm)
                               : group_occupancy<512, 2>(smem, per_sm);
    }
    return threads == 256 ? group_occupancy<256, 1>(smem, per_sm)
         : threads == 1024 ? group_occupancy<1024, 1>(smem, per_sm)
                           : group_occupancy<512, 1>(smem, per_sm);
}

namespace {
struct PlanKey {
    int device;
    int64_t rows, cols;
    int threads, chunk, group, nbuf;
    bool operator==(const PlanKey& o) const {
        return device == o.device && rows == o.rows && cols == o.cols && threads == o.threads &&
               chunk == o.chunk && group == o.group && nbuf == o.nbuf;
    }
};
std::mutex g_plan_mu;
PlanKey g_plan_keys[16];
GroupPlan g_plans[16];
int g_plan_n = 0, g_plan_next = 0;
}  // namespace

// Chooses the group size GS (CTAs per row, 1..32) and the buffering: the plan
// that keeps the most CTA slots of the GPU busy, preferring deeper buffering
// (each extra buffer is worth 4 % of coverage) and then the smallest group.
// LSE_LSM_GROUP forces GS, LSE_LSM_NBUF forces 1, 2 or 3 buffers,
// LSE_LSM_THREADS (256/512/1024) and LSE_LSM_CHUNK (floats per copy) tune.
cudaError_t plan_lsm_smem_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                                int64_t cols, GroupPlan* plan) {
    if (cols % 4 != 0 || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return cudaErrorNotSupported;
    const int threads = env_int("LSE_LSM_THREADS", 256);
    const int chunk_env = env_int("LSE_LSM_CHUNK", 8192);
    const int forced = env_int("LSE_LSM_GROUP", 0);
    const int nbuf_env = env_int("LSE_LSM_NBUF", 0);
    const PlanKey key{dev.device, rows, cols, threads, chunk_env, forced, nbuf_env};
    {
        std::lock_guard<std::mutex> lock(g_plan_mu);
        for (int i = 0; i < g_plan_n; ++i)
            if (g_plan_keys[i] == key) {
                *plan = g_plans[i];
                return cudaSuccess;
            }
    }
    double best_score = -1.0;
    GroupPlan best;
    for (int nbuf = 3; nbuf >= 1; --nbuf) {
        if (nbuf_env && nbuf != nbuf_env) continue;
        for (int GS = 1; GS <= 32; ++GS) {
            if (forced && GS != forced) continue;
            int slice, ch;
            smem_chunking(cols, GS, chunk_env, &slice, &ch);
            const size_t smem = smem_cluster_bytes(slice, nbuf);
            if ((int64_t)slice * GS < cols || smem > (size_t)dev.max_smem_optin) continue;
            if ((int64_t)slice * (GS - 1) >= cols) continue;  // a CTA would own nothing
            int per_sm = 0;
            cudaError_t e = group_occupancy_any(threads, nbuf, smem, &per_sm);
            if (e != cudaSuccess) return e;
            const int64_t slots = (int64_t)per_sm * dev.sm_count;
            const int64_t groups = std::min<int64_t>(rows, slots / GS);
            if (groups < 1) continue;
            const double cover = (double)(groups * GS) / (double)slots;
            const double score = cover + 0.04 * (nbuf - 1) - 1e-4 * GS;
            if (score > best_score) {
                best_score = score;
                best.threads = threads;
                best.nbuf = nbuf;
                best.group_size = GS;
                best.groups = (int)groups;
                best.slice = slice;
                best.chunk = ch;
                best.smem = smem;
                best.scratch_bytes = (size_t)groups * 2 * GS * sizeof(unsigned long long);
            }
        }
    }
    if (best_score < 0) return cudaErrorNotSupported;
    {
        std::lock_guard<std::mutex> lock(g_plan_mu);
        g_plan_keys[g_plan_next] = key;
        g_plans[g_plan_next] = best;
        g_plan_next = (g_plan_next + 1) % 16;
        g_plan_n = std::min(g_plan_n + 1, 16);
    }
    *plan = best;
    return cudaSuccess;
}

template <int THREADS, int NBUF>
static cudaError_t group_go(const SmemRowArgs& args, const GroupPlan& p, cudaStream_t stream) {
    auto kern = lsm_smem_kernel<THREADS, true, NBUF>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the group waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)(p.groups * p.group_size));
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_lsm_smem_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                  int64_t cols, const GroupPlan& p, void* scratch, cudaStream_t stream) {
    // every slot starts with tag 1, which no step's first use expects
    cudaError_t e = cudaMemsetAsync(scratch, 0xFF, p.scratch_bytes, stream);
    if (e != cudaSuccess) return e;
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] lsm_smem group: GS=%d groups=%d nbuf=%d threads=%d slice=%d chunk=%d "
                "smem=%zu\n", p.group_size, p.groups, p.nbuf, p.threads, p.slice, p.chunk, p.smem);
    SmemRowArgs args{x, out, rows, cols, p.slice, p.chunk, dev.status, p.group_size,
                     static_cast<unsigned long long*>(scratch)};
    if (p.nbuf == 3) {
        if (p.threads == 256) return group_go<256, 3>(args, p, stream);
        if (p.threads == 1024) return group_go<1024, 3>(args, p, stream);
        return group_go<512, 3>(args, p, stream);
    }
    if (p.nbuf == 2) {
        if (p.threads == 256) return group_go<256, 2>(args, p, stream);
        if (p.threads == 1024) return group_go<1024, 2>(args, p, stream);
        return group_go<512, 2>(args, p, stream);
    }
    if (p.threads == 256) return group_go<256, 1>(args, p, stream);
    if (p.threads == 1024) return group_go<1024, 1>(args, p, stream);
    return group_go<512, 1>(args, p, stream);
}

// ---- warp-specialised group variant

template <int FW, int SW, int NB>
static cudaError_t ws_occupancy(size_t smem, int* per_sm) {
    auto kern = lsm_ws_kernel<FW, SW, NB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, 32 * (FW + SW), smem);
}

// Warp splits compiled: (fold, store) = (4,4) (8,4) (8,8) (12,4) (16,4).
static int ws_split(int fw, int sw) {
    if (fw == 8 && sw == 4) return 1;
    if (fw == 8 && sw == 8) return 2;
    if (fw == 12 && sw == 4) return 3;
    if (fw == 16 && sw == 4) return 4;
    return 0;
}

template <int NB>
static cudaError_t ws_occupancy_nb(int fw, int sw, size_t smem, int* per_sm) {
    switch (ws_split(fw, sw)) {
        case 1: return ws_occupancy<8, 4, NB>(smem, per_sm);
        case 2: return ws_occupancy<8, 8, NB>(smem, per_sm);
        case 3: return ws_occupancy<12, 4, NB>(smem, per_sm);
        case 4: return ws_occupancy<16, 4, NB>(smem, per_sm);
        default: return ws_occupancy<4, 4, NB>(smem, per_sm);
    }
}

static cudaError_t ws_occupancy_any(int nb, int fw, int sw, size_t smem, int* per_sm) {
    switch (nb) {
        case 2: return ws_occupancy_nb<2>(fw, sw, smem, per_sm);
        case 4: return ws_occupancy_nb<4>(fw, sw, smem, per_sm);
        case 5: return ws_occupancy_nb<5>(fw, sw, smem, per_sm);
        default: return ws_occupancy_nb<3>(fw, sw, smem, per_sm);
    }
}

// Buffers NB (LSE_WS_NB: 2..5, default 3; 0 lets the planner choose) and group
// size GS (1..64): the plan that covers the most CTA slots (LSE_WS_GROUP forces
// GS); warps LSE_WS_FW / LSE_WS_SW (default 8 fold, 4 store).
cudaError_t plan_lsm_ws_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                              int64_t cols, GroupPlan* plan) {
    if (cols % 4 != 0 || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return cudaErrorNotSupported;
    int fw = env_int("LSE_WS_FW", 8);
    int sw = env_int("LSE_WS_SW", 4);
    if (ws_split(fw, sw) == 0) fw = sw = 4;
    const int chunk_env = env_int("LSE_LSM_CHUNK", 8192);
    const int forced = env_int("LSE_WS_GROUP", 0);
    const int nb_env = env_int("LSE_WS_NB", 3);
    double best_score = -1.0;
    for (int nb = 5; nb >= 2; --nb) {
        if (nb_env && nb != nb_env) continue;
        for (int GS = 1; GS <= kWsMaxGroup; ++GS) {
            if (forced && GS != forced) continue;
            int slice, ch;
            smem_chunking(cols, GS, chunk_env, &slice, &ch);
            const size_t smem = smem_ws_bytes(slice, nb);
            if ((int64_t)slice * GS < cols || smem > (size_t)dev.max_smem_optin) continue;
            if ((int64_t)slice * (GS - 1) >= cols) continue;
            int per_sm = 0;
            cudaError_t e = ws_occupancy_any(nb, fw, sw, smem, &per_sm);
            if (e != cudaSuccess) return e;
            const int64_t slots = (int64_t)per_sm * dev.sm_count;
            const int64_t groups = std::min<int64_t>(rows, slots / GS);
            if (groups < 1) continue;
            // Coverage of the SM slots, minus a cost per CTA of the group (smaller
            // slices and a wider merge: GS = 38 ran 25 % slower than GS = 24 on
            // 393,216-float rows), plus a bonus when the slices split the row
            // exactly on 4 KiB boundaries (equal work for every CTA of a group).
            const bool even = (cols % ((int64_t)GS * 1024) == 0);
            const double score = (double)(groups * GS) / (double)slots - 0.004 * GS + (even ? 0.05 : 0.0) +
                                 0.03 * (nb - 2);
            if (score > best_score) {
                best_score = score;
                plan->threads = 32 * (fw + sw);
                plan->nbuf = nb * 10000 + fw * 100 + sw;  // records buffers and the warp split
                plan->group_size = GS;
                plan->groups = (int)groups;
                plan->slice = slice;
                plan->chunk = ch;
                plan->smem = smem;
                plan->scratch_bytes = (size_t)groups * kWsSlots * GS * sizeof(unsigned long long);
            }
        }
    }
    return best_score < 0 ? cudaErrorNotSupported : cudaSuccess;
}

template <int FW, int SW, int NB>
static cudaError_t ws_go(const SmemRowArgs& args, const GroupPlan& p, cudaStream_t stream) {
    auto kern = lsm_ws_kernel<FW, SW, NB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the group waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(32 * (FW + SW));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)(p.groups * p.group_size));
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int NB>
static cudaError_t ws_go_nb(int fw, int sw, const SmemRowArgs& args, const GroupPlan& p,
                            cudaStream_t stream) {
    switch (ws_split(fw, sw)) {
        case 1: return ws_go<8, 4, NB>(args, p, stream);
        case 2: return ws_go<8, 8, NB>(args, p, stream);
        case 3: return ws_go<12, 4, NB>(args, p, stream);
        case 4: return ws_go<16, 4, NB>(args, p, stream);
        default: return ws_go<4, 4, NB>(args, p, stream);
    }
}

cudaError_t launch_lsm_ws_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                int64_t cols, const GroupPlan& p, void* scratch, cudaStream_t stream,
                                bool softmax) {
    cudaError_t e = cudaMemsetAsync(scratch, 0xFF, p.scratch_bytes, stream);
    if (e != cudaSuccess) return e;
    const int nb = p.nbuf / 10000, fw = (p.nbuf / 100) % 100, sw = p.nbuf % 100;
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] lsm_ws group: GS=%d groups=%d buffers=%d fold_warps=%d store_warps=%d "
                "slice=%d chunk=%d smem=%zu\n", p.group_size, p.groups, nb, fw, sw, p.slice, p.chunk, p.smem);
    SmemRowArgs args{x, out, rows, cols, p.slice, p.chunk, dev.status, p.group_size,
                     static_cast<unsigned long long*>(scratch), softmax ? 1 : 0};
    switch (nb) {
        case 2: return ws_go_nb<2>(fw, sw, args, p, stream);
        case 4: return ws_go_nb<4>(fw, sw, args, p, stream);
        case 5: return ws_go_nb<5>(fw, sw, args, p, stream);
        default: return ws_go_nb<3>(fw, sw, args, p, stream);
    }
}

// ---- ring form of the warp-specialised group kernel

// Group size GS (LSE_WS_GROUP forces it), chunk floats (LSE_RING_CHUNK: the
// smallest chunk count per slice with chunks of at most that many floats, default
// 6912 = 27 KB), as many ring slots as fit (at most kRingMax), and at least two
// slices' worth of slots.  The plan covering the most SM slots wins, then the one
// with the most rows in flight.  On the 4096 x 393,216 workload (GS = 19, three
// chunks per slice, 8 slots: 2.67 rows in flight on all 152 SMs) it measured 0.934
// of the copy peak against 0.950 for lsm_ws_kernel's 144 SMs with 3 rows in flight
// on the same GPU; 10 KB chunks 0.60, 40 KB chunks 0.90.
cudaError_t plan_lsm_ring_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                                int64_t cols, GroupPlan* plan) {
    if (cols % 4 != 0 || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return cudaErrorNotSupported;
    const int forced = env_int("LSE_WS_GROUP", 0);
    const int chunk_max = std::max(256, env_int("LSE_RING_CHUNK", 6912) & ~31);
    double best = -1.0;
    for (int GS = 1; GS <= kWsMaxGroup; ++GS) {
        if (forced && GS != forced) continue;
        const int64_t sl = ((cols + GS - 1) / GS + 31) / 32 * 32;
        if (sl * (GS - 1) >= cols || sl > (1 << 24)) continue;
        const int nch = (int)((sl + chunk_max - 1) / chunk_max);
        const int chunk = (int)(((sl + nch - 1) / nch + 31) / 32 * 32);
        // the group's last CTA owns the shortest slice, so the fewest chunks per row:
        // it runs furthest ahead, and bounds the ring (see lsm_ring_kernel)
        const int64_t last_len = cols - sl * (GS - 1);
        const int nch_min = (int)std::max<int64_t>(1, (last_len + chunk - 1) / chunk);
        int R = (int)std::min<int64_t>(kRingMax, ((int64_t)dev.max_smem_optin - (int64_t)smem_ring_bytes(0, 0)) /
                                                     ((int64_t)chunk * 4));
        R = std::min(R, (kWsSlots / 2) * nch_min);
        if (R < 2 * nch) continue;
        int per_sm = 0;
        auto kern = lsm_ring_kernel<8, 4>;
        const size_t smem = smem_ring_bytes(chunk, R);
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * 12, smem);
        if (e != cudaSuccess) return e;
        const int64_t slots = (int64_t)per_sm * dev.sm_count;
        const int64_t groups = std::min<int64_t>(rows, slots / GS);
        if (groups < 1) continue;
        const double score = (double)(groups * GS) / (double)slots + 0.01 * std::min(3.0, (double)R / nch) -
                             0.002 * GS;
        if (score > best) {
            best = score;
            plan->threads = 32 * 12;
            plan->nbuf = R;
            plan->group_size = GS;
            plan->groups = (int)groups;
            plan->slice = (int)sl;
            plan->chunk = chunk;
            plan->smem = smem;
            plan->scratch_bytes = (size_t)groups * kWsSlots * GS * sizeof(unsigned long long);
        }
    }
    return best < 0 ? cudaErrorNotSupported : cudaSuccess;
}

cudaError_t launch_lsm_ring_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows, int64_t cols,
                                  const GroupPlan& p, void* scratch, cudaStream_t stream, bool softmax) {
    (void)dev;
    cudaError_t e = cudaMemsetAsync(scratch, 0xFF, p.scratch_bytes, stream);
    if (e != cudaSuccess) return e;
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] lsm_ring group: GS=%d groups=%d ring=%d slice=%d chunk=%d smem=%zu\n", p.group_size,
                p.groups, p.nbuf, p.slice, p.chunk, p.smem);
    SmemRowArgs args{x, out, rows, cols, p.slice, p.chunk, dev.status, p.group_size,
                     static_cast<unsigned long long*>(scratch), softmax ? 1 : 0, p.nbuf};
    auto kern = lsm_ring_kernel<8, 4>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the group waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)(p.groups * p.group_size));
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---- rows parked in tensor memory (row_tmem.cuh): LSE_WS_GROUP forces the group size,
// LSE_TMEM_CHUNK (default 8192) bounds the landing chunks.
cudaError_t plan_lsm_tmem_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                                int64_t cols, GroupPlan* plan) {
    return plan_row_tmem(dev, x, out, rows, cols, env_int("LSE_WS_GROUP", 0), env_int("LSE_TMEM_CHUNK", 8192), 16384,
                         plan);
}

cudaError_t launch_lsm_tmem_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows, int64_t cols,
                                  const GroupPlan& p, void* scratch, cudaStream_t stream, bool softmax) {
    return launch_row_tmem<LsmOp, 4>(dev, x, out, rows, cols, p, scratch, stream, LsmOp::Params{softmax ? 1 : 0},
                                     "row_tmem (log_softmax)");
}

// ------------------------------------------------------------------ rows re-read from L2 by a group

// Each CTA of a group owns a slice of the row.  Pass 1 streams the slice from
// HBM into the running pair with loads that ask L2 to keep the lines; the
// group merges its pairs through tagged slots; pass 2 reads the slice again
// (from L2: the slices in flight across the GPU are sized to fit in it) and
// writes x - lse with streaming stores.  HBM sees one read and one write, and
// several CTAs per SM hide each other's merge waits.
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 2048 / THREADS) lsm_l2_group_kernel(const float* __restrict__ x,
                                                               float* __restrict__ out, int64_t rows,
                                                               int64_t cols, int group_size, int slice,
                                                               unsigned long long* slots, int* status) {
    __shared__ MS red[32];
    __shared__ float lse_sh;
    constexpr int T = THREADS;
    RowMerge<THREADS, true> mg;
    mg.GS = (uint32_t)group_size;
    mg.rank = blockIdx.x % mg.GS;
    const int64_t g = blockIdx.x / mg.GS;
    const int64_t NG = gridDim.x / mg.GS;
    mg.slots = slots + g * 2 * mg.GS;
    mg.part = nullptr;
    mg.pend = 0;
    const int64_t c_begin = (int64_t)mg.rank * slice;
    const int64_t len = std::max<int64_t>(0, std::min<int64_t>(slice, cols - c_begin));
    const int64_t n4 = len >> 2;
    const int tid = threadIdx.x;
    const uint64_t keep = l2_policy_evict_last();
    const uint64_t drop = l2_policy_evict_first();
    bool aborted = false;
    uint32_t j = 0;
    for (int64_t row = g; row < rows; row += NG, ++j) {
        const float* src = x + row * cols + c_begin;
        MS st = ms_empty();
        int64_t i = tid;
        for (; i + 3 * T < n4; i += 4 * T) {
            float v[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 q = ld_f4_l2hint(src + 4 * (i + k * T), keep);
                v[4 * k + 0] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
            }
            ms_fold<16>(st, v);
        }
        for (; i < n4; i += T) {
            const float4 q = ld_f4_l2hint(src + 4 * i, keep);
            float v[4] = {q.x, q.y, q.z, q.w};
            ms_fold<4>(st, v);
        }
        st = ms_block_allreduce(st, red);
        mg.arrive(j, st);
        mg.prefetch(j);
        const float lse = mg.wait(j, &lse_sh, aborted, status);
        float* dst = out + row * cols + c_begin;
        i = tid;
        for (; i + 3 * T < n4; i += 4 * T) {
            float4 q[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) q[k] = ld_f4_l2hint(src + 4 * (i + k * T), drop);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                st_stream_f4(dst + 4 * (i + k * T),
                             make_float4(q[k].x - lse, q[k].y - lse, q[k].z - lse, q[k].w - lse));
        }
        for (; i < n4; i += T) {
            const float4 q = ld_f4_l2hint(src + 4 * i, drop);
            st_stream_f4(dst + 4 * i, make_float4(q.x - lse, q.y - lse, q.z - lse, q.w - lse));
        }
    }
}

template <int THREADS>
static cudaError_t l2_occupancy(int* per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, lsm_l2_group_kernel<THREADS>, THREADS, 0);
}

// Group size LSE_L2_GROUP (default 16), CTA size LSE_L2_THREADS (256 / 512 / 1024,
// default 512).  Needs 16-byte-aligned rows.
cudaError_t plan_lsm_l2_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                              int64_t cols, GroupPlan* plan) {
    if (cols % 4 != 0 || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return cudaErrorNotSupported;
    const int threads = env_int("LSE_L2_THREADS", 512);
    int GS = std::min(32, std::max(1, env_int("LSE_L2_GROUP", 16)));
    int per_sm = 0;
    cudaError_t e = threads == 256 ? l2_occupancy<256>(&per_sm)
                  : threads == 1024 ? l2_occupancy<1024>(&per_sm)
                                    : l2_occupancy<512>(&per_sm);
    if (e != cudaSuccess) return e;
    const int64_t groups = std::min<int64_t>(rows, (int64_t)per_sm * dev.sm_count / GS);
    if (groups < 1) return cudaErrorNotSupported;
    const int64_t sl = ((cols + GS - 1) / GS + 31) / 32 * 32;
    if (sl > (int64_t)1 << 30) return cudaErrorNotSupported;
    plan->threads = threads;
    plan->nbuf = 0;
    plan->group_size = GS;
    plan->groups = (int)groups;
    plan->slice = (int)sl;
    plan->chunk = 0;
    plan->smem = 0;
    plan->scratch_bytes = (size_t)groups * 2 * GS * sizeof(unsigned long long);
    return cudaSuccess;
}

template <int THREADS>
static cudaError_t l2_go(const DeviceInfo& dev, const float* x, float* out, int64_t rows, int64_t cols,
                         const GroupPlan& p, unsigned long long* slots, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the group waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)(p.groups * p.group_size));
    cudaError_t e = cudaLaunchKernelEx(&cfg, lsm_l2_group_kernel<THREADS>, x, out, rows, cols,
                                       p.group_size, p.slice, slots, dev.status);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_lsm_l2_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                int64_t cols, const GroupPlan& p, void* scratch, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(scratch, 0xFF, p.scratch_bytes, stream);
    if (e != cudaSuccess) return e;
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] lsm_l2 group: GS=%d groups=%d threads=%d slice=%d\n", p.group_size,
                p.groups, p.threads, p.slice);
    auto* slots = static_cast<unsigned long long*>(scratch);
    if (p.threads == 256) return l2_go<256>(dev, x, out, rows, cols, p, slots, stream);
    if (p.threads == 1024) return l2_go<1024>(dev, x, out, rows, cols, p, slots, stream);
    return l2_go<512>(dev, x, out, rows, cols, p, slots, stream);
}

// ------------------------------------------------------------------ rows streamed by a cluster

template <int VEC, int MODE>
__global__ void __launch_bounds__(512) rows_stream_kernel(const float* __restrict__ x,
                                                          float* __restrict__ out, int64_t rows,
                                                          int64_t cols, int64_t slice) {
    __shared__ MS red[32];
    __shared__ MS part[2];
    __shared__ float lse_sh;
    constexpr int T = 512;
    const uint32_t rank = cluster_ctarank();
    const uint32_t CL = cluster_nctarank();
    const int64_t c_begin = (int64_t)rank * slice;
    const int64_t len = std::max<int64_t>(0, std::min<int64_t>(slice, cols - c_begin));
    const int64_t n = len / VEC;  // VEC == 4 implies len % 4 == 0
    const int tid = threadIdx.x;
    uint32_t it = 0;
    for (int64_t row = cluster_id_x(); row < rows; row += nclusters_x(), ++it) {
        const float* src = x + row * cols + c_begin;
        MS st = ms_empty();
        int64_t i = tid;
        for (; i + 3 * T < n; i += 4 * T) {
            float v[4 * VEC];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if constexpr (VEC == 4) {
                    float4 a = ld_stream_f4(src + (i + k * T) * 4);
                    v[4 * k + 0] = a.x; v[4 * k + 1] = a.y; v[4 * k + 2] = a.z; v[4 * k + 3] = a.w;
                } else {
                    v[k] = ld_stream_f1(src + i + k * T);
                }
            }
            ms_fold<4 * VEC>(st, v);
        }
        for (; i < n; i += T) {
            float v[VEC];
            if constexpr (VEC == 4) {
                float4 a = ld_stream_f4(src + i * 4);
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            } else {
                v[0] = ld_stream_f1(src + i);
            }
            ms_fold<VEC>(st, v);
        }
        st = ms_block_allreduce(st, red);
        if (CL > 1) {
            if (tid == 0) part[it & 1u] = st;
            cluster_sync();
            if (tid == 0) {
                MS tot = ms_empty();
                for (uint32_t k = 0; k < CL; ++k) tot = ms_merge(tot, ld_peer_ms(&part[it & 1u], k));
                lse_sh = ms_lse(tot);
            }
        } else if (tid == 0) {
            lse_sh = ms_lse(st);
        }
        __syncthreads();
        const float lse = lse_sh;
        if constexpr (MODE == 1) {
            if (rank == 0 && tid == 0) out[row] = lse;
        } else {
            constexpr bool SM = (MODE == 2);
            float* dst = out + row * cols + c_begin;
            for (int64_t j = tid; j < n; j += T) {
                if constexpr (VEC == 4) {
                    float4 a = ld_stream_f4(src + j * 4);
                    st_stream_f4(dst + j * 4, make_float4(row_out<SM>(a.x, lse), row_out<SM>(a.y, lse),
                                                          row_out<SM>(a.z, lse), row_out<SM>(a.w, lse)));
                } else {
                    st_stream_f1(dst + j, row_out<SM>(ld_stream_f1(src + j), lse));
                }
            }
        }
    }
    if (CL > 1) cluster_sync();
}

template <int VEC, int MODE>
static cudaError_t rows_stream_go(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                  int64_t cols, int CL, cudaStream_t stream) {
    auto kern = rows_stream_kernel<VEC, MODE>;
    const int64_t slice = ((cols + CL - 1) / CL + 3) / 4 * 4;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    const int64_t cap = std::max<int64_t>(1, (int64_t)dev.sm_count * 4 * 8 / CL);
    const int64_t nclusters = std::max<int64_t>(1, std::min<int64_t>(rows, cap));
    cfg.gridDim = dim3((unsigned)(nclusters * CL));
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, x, out, rows, cols, slice);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_rows_stream(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                               int64_t cols, int mode, cudaStream_t stream) {
    const bool vec4 = (cols % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0) &&
                      ((reinterpret_cast<uintptr_t>(out) & 15) == 0 || mode == 1);
    // Enough CTAs to cover the GPU a few times over, slices of at least 8K floats.
    const int64_t want = (int64_t)dev.sm_count * 8;
    int CL = 1;
    while (CL < 8 && rows * CL < want && (cols + 2 * CL - 1) / (2 * CL) >= 8192) CL *= 2;
    const int forced = env_int("LSE_STREAM_CLUSTER", 0);
    if (forced == 1 || forced == 2 || forced == 4 || forced == 8) CL = forced;
    if (vec4) {
        return mode == 0 ? rows_stream_go<4, 0>(dev, x, out, rows, cols, CL, stream)
             : mode == 2 ? rows_stream_go<4, 2>(dev, x, out, rows, cols, CL, stream)
                         : rows_stream_go<4, 1>(dev, x, out, rows, cols, CL, stream);
    }
    return mode == 0 ? rows_stream_go<1, 0>(dev, x, out, rows, cols, CL, stream)
         : mode == 2 ? rows_stream_go<1, 2>(dev, x, out, rows, cols, CL, stream)
                     : rows_stream_go<1, 1>(dev, x, out, rows, cols, CL, stream);
}

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::atoi(v);
}

}  // namespace lse
