// Form 2: row-wise log_softmax over the last axis (and the row lse alone).
//
// out[r, j] = x[r, j] - lse_r, lse_r = max_r + log(sum_j exp(x[r, j] - max_r))
// (POPCORNBENCH page "Kimi-K2.6 / l1_p24", opening analysis).  That page's
// kernels give each row one block and read it two or three times from HBM;
// its traffic analysis judges the ideal of one read plus one write out of
// reach because a 1.5 MiB row does not fit on one SM.  On GB300 it fits in
// the shared memory of a thread-block cluster, so the three kernels here are:
//
//  rows_reg_kernel      rows up to 32K floats: the row lives in registers of
//                       one warp or one block; exact two-pass (max, then sum)
//                       over registers, one HBM read and one write.
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
#include <cstdlib>

#include "common.cuh"
#include "launch.h"

namespace lse {

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

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
        m = warp_max_nan(m);
        if (nwarps > 1) {
            __syncthreads();
            if (lane == 0) red[warp] = m;
            __syncthreads();
            m = warp_max_nan(lane < nwarps ? red[lane] : -CUDART_INF_F);
        }
        const float base = isfinite(m) ? m : 0.f;  // see ms_fold on why v - m comes first
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) s += ex2((v[k][e] - base) * kLog2e);
        s = warp_sum(s);
        if (nwarps > 1) {
            __syncthreads();
            if (lane == 0) red[warp] = s;
            __syncthreads();
            s = warp_sum(lane < nwarps ? red[lane] : 0.f);
        }
        const float lse = lse_from_max_sum(m, s);
        if constexpr (MODE == 0) {
            if (rv) {
                float* dst = out + row * cols;
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int64_t j = ((int64_t)k * GT + t) * VEC;
                    if (j < cols) {
                        if constexpr (VEC == 4) {
                            st_stream_f4(dst + j, make_float4(v[k][0] - lse, v[k][1] - lse,
                                                              v[k][2] - lse, v[k][3] - lse));
                        } else {
                            st_stream_f1(dst + j, v[k][0] - lse);
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
    return rows_reg_dispatch<1>(dev, x, out, rows, cols, vec4, stream);
}

// ------------------------------------------------------------------ rows in cluster shared memory

constexpr int kSmemMaxChunks = 64;

struct SmemLayout {
    int slice;      // floats of the row owned by one CTA (multiple of 4)
    int chunk;      // floats per bulk copy (multiple of 4)
    size_t bytes;   // dynamic shared memory per CTA
};

__host__ __device__ inline size_t smem_cluster_bytes(int slice) {
    // [slice floats][kSmemMaxChunks mbarriers][2 MS partials][32 MS scratch][lse + pad]
    return (size_t)slice * 4 + kSmemMaxChunks * 8 + 2 * sizeof(MS) + 32 * sizeof(MS) + 16;
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS, 1) lsm_smem_cluster_kernel(
    const float* __restrict__ x, float* __restrict__ out, int64_t rows, int64_t cols, int slice,
    int chunk, int* status) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* buf = reinterpret_cast<float*>(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (size_t)slice * 4);
    MS* part = reinterpret_cast<MS*>(bars + kSmemMaxChunks);
    MS* red = part + 2;
    float* lse_sh = reinterpret_cast<float*>(red + 32);

    const uint32_t rank = cluster_ctarank();
    const uint32_t CL = cluster_nctarank();
    const int64_t c_begin = (int64_t)rank * slice;
    const int len = (int)std::max<int64_t>(0, std::min<int64_t>(slice, cols - c_begin));
    const int nch = (len + chunk - 1) / chunk;
    const int64_t first_row = cluster_id_x();
    const int64_t row_step = nclusters_x();
    const int tid = threadIdx.x;
    bool aborted = false;

    if (tid == 0) {
        for (int c = 0; c < nch; ++c) mbar_init(&bars[c], 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (tid == 0 && first_row < rows) {
        const float* src = x + first_row * cols + c_begin;
        for (int c = 0; c < nch; ++c) {
            const int cb = c * chunk;
            const uint32_t bytes = (uint32_t)std::min(chunk, len - cb) * 4u;
            mbar_arrive_expect_tx(&bars[c], bytes);
            bulk_g2s(buf + cb, src + cb, bytes, &bars[c]);
        }
    }

    uint32_t it = 0;
    uint32_t abort_par = 0;
    for (int64_t row = first_row; row < rows; row += row_step, ++it) {
        const uint32_t par = it & 1u;
        // ---- fold the slice into (m, s) as its chunks land
        MS st = ms_empty();
        for (int c = 0; c < nch; ++c) {
            if (!mbar_wait_bounded(&bars[c], par, aborted, status) && abort_par == 0) abort_par = par + 1;
            const int cb = c * chunk;
            const int n4 = std::min(chunk, len - cb) >> 2;
            const float4* p = reinterpret_cast<const float4*>(buf + cb);
            int i = tid;
            for (; i + 3 * THREADS < n4; i += 4 * THREADS) {
                float v[16];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float4 a = p[i + k * THREADS];
                    v[4 * k + 0] = a.x; v[4 * k + 1] = a.y; v[4 * k + 2] = a.z; v[4 * k + 3] = a.w;
                }
                ms_fold<16>(st, v);
            }
            for (; i < n4; i += THREADS) {
                float4 a = p[i];
                float v[4] = {a.x, a.y, a.z, a.w};
                ms_fold<4>(st, v);
            }
        }
        st = ms_block_allreduce(st, red);
        // ---- merge the CTAs' pairs through distributed shared memory
        if (tid == 0) part[par] = st;
        cluster_sync();
        if (tid == 0) {
            MS tot = ms_empty();
            for (uint32_t k = 0; k < CL; ++k) tot = ms_merge(tot, ld_peer_ms(&part[par], k));
            *lse_sh = ms_lse(tot);
        }
        __syncthreads();
        const float lse = *lse_sh;
        // ---- write x - lse from shared memory; refill each chunk with the next row
        const int64_t next = row + row_step;
        float* dst = out + row * cols + c_begin;
        const float* nsrc = x + next * cols + c_begin;
        for (int c = 0; c < nch; ++c) {
            const int cb = c * chunk;
            const int clen = std::min(chunk, len - cb);
            const int n4 = clen >> 2;
            const float4* p = reinterpret_cast<const float4*>(buf + cb);
            for (int i = tid; i < n4; i += THREADS) {
                float4 a = p[i];
                st_stream_f4(dst + cb + 4 * i, make_float4(a.x - lse, a.y - lse, a.z - lse, a.w - lse));
            }
            __syncthreads();  // every thread is done reading chunk c
            if (tid == 0 && next < rows && !aborted) {
                fence_proxy_async_smem();
                const uint32_t bytes = (uint32_t)clen * 4u;
                mbar_arrive_expect_tx(&bars[c], bytes);
                bulk_g2s(buf + cb, nsrc + cb, bytes, &bars[c]);
            }
        }
    }
    if (aborted && tid == 0 && abort_par != 0) {
        // A copy never completed: stop issuing (done above) and give the copies of
        // the abandoned row one more bounded wait before the CTA releases its
        // shared memory.
        bool again = false;
        for (int c = 0; c < nch; ++c) mbar_wait_bounded(&bars[c], abort_par - 1, again, status);
    }
    cluster_sync();  // peers may still read part[] of this CTA
}

template <int THREADS>
static cudaError_t smem_cluster_go(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                   int64_t cols, int CL, int slice, int chunk, size_t smem,
                                   cudaStream_t stream) {
    auto kern = lsm_smem_cluster_kernel<THREADS>;
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
    e = cudaLaunchKernelEx(&cfg, kern, x, out, rows, cols, slice, chunk, dev.status);
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
    int chunk = env_int("LSE_LSM_CHUNK", 8192);
    chunk = std::max(1024, chunk & ~3);
    const int forced = env_int("LSE_LSM_CLUSTER", 0);
    const int cands[5] = {1, 2, 4, 8, 16};
    for (int ci = 0; ci < 5; ++ci) {
        const int CL = cands[ci];
        if (forced && CL != forced) continue;
        const int64_t sl = ((cols + CL - 1) / CL + 3) / 4 * 4;
        const size_t smem = smem_cluster_bytes((int)std::min<int64_t>(sl, 1 << 26));
        if (sl > (1 << 26) || smem > (size_t)dev.max_smem_optin) continue;
        const int slice = (int)sl;
        int ch = std::min(chunk, slice);
        if ((slice + ch - 1) / ch > kSmemMaxChunks) ch = ((slice + kSmemMaxChunks - 1) / kSmemMaxChunks + 3) / 4 * 4;
        cudaError_t e;
        if (threads == 256)
            e = smem_cluster_go<256>(dev, x, out, rows, cols, CL, slice, ch, smem, stream);
        else if (threads == 1024)
            e = smem_cluster_go<1024>(dev, x, out, rows, cols, CL, slice, ch, smem, stream);
        else
            e = smem_cluster_go<512>(dev, x, out, rows, cols, CL, slice, ch, smem, stream);
        if (e == cudaErrorNotSupported || e == cudaErrorInvalidClusterSize) {
            (void)cudaGetLastError();
            continue;
        }
        return e;
    }
    return cudaErrorNotSupported;
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
            float* dst = out + row * cols + c_begin;
            for (int64_t j = tid; j < n; j += T) {
                if constexpr (VEC == 4) {
                    float4 a = ld_stream_f4(src + j * 4);
                    st_stream_f4(dst + j * 4, make_float4(a.x - lse, a.y - lse, a.z - lse, a.w - lse));
                } else {
                    st_stream_f1(dst + j, ld_stream_f1(src + j) - lse);
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
                         : rows_stream_go<4, 1>(dev, x, out, rows, cols, CL, stream);
    }
    return mode == 0 ? rows_stream_go<1, 0>(dev, x, out, rows, cols, CL, stream)
                     : rows_stream_go<1, 1>(dev, x, out, rows, cols, CL, stream);
}

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::atoi(v);
}

}  // namespace lse
