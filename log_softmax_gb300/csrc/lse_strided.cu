// Form 1: logsumexp over a strided (non-last) axis.
//
// x is contiguous (outer, R, inner); out[o, i] = lse over r of x[o, r, i]
// (the dim-0 logsumexp of the POPCORNBENCH page "FW-GLM-5-1 / l1_p29", task
// analysis).  That page gives each output one thread, which walks R twice
// (max pass, then sum pass).  Here each thread owns VEC adjacent columns, so a
// warp reads 32*VEC contiguous floats per r (one 512-byte transaction group
// for VEC=4) and keeps CH loads per column in flight; the pair (m, s) is
// updated online, once per batch of CH values ("Kimi-K2.6 / l1_p24",
// online-softmax derivation).  When R is long and inner is short, TY thread
// rows split R and their pairs are merged in shared memory.
//
// With LSM set the same kernel writes log_softmax over the strided axis
// instead of the lse (out has x's shape): the block publishes its columns'
// lse in shared memory and writes x - lse.  When R = CH * TY each thread's
// values are one load batch, kept in registers from the reduction to the
// write (ONE: the tile is read once).  Otherwise the block walks its tile a
// second time: the first walk marks its lines evict-last in L2 and the
// second evict-first, so the second walk is served from L2 while the tiles
// resident at once fit there.  Either way x is read from HBM once and out
// written once.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace lse {

template <int VEC>
__device__ __forceinline__ void load_cols(const float* p, float (&v)[VEC], uint64_t pol, bool hint) {
    if constexpr (VEC == 4) {
        float4 a = hint ? ld_f4_l2hint(p, pol) : ld_stream_f4(p);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else {
        v[0] = hint ? ld_f1_l2hint(p, pol) : ld_stream_f1(p);
    }
}

// ONE (with LSM, for R = CH * TY): a thread's rows ty, ty + TY, ... of its
// columns are one load batch, kept in registers for the write, so the tile is
// read once (no second walk through L2).
template <int VEC, int CH, bool LSM, bool ONE = false>
__global__ void __launch_bounds__(256) lse_strided_kernel(const float* __restrict__ x,
                                                          float* __restrict__ out, int64_t outer,
                                                          int64_t R, int64_t inner, int64_t tiles) {
    __shared__ MS red[256 * VEC];
    __shared__ float lse_s[LSM ? 256 * VEC : 1];
    const int TX = blockDim.x, TY = blockDim.y;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const uint64_t keep = LSM ? l2_policy_evict_last() : 0;
    const int64_t nblk = outer * tiles;
    for (int64_t b = blockIdx.x; b < nblk; b += gridDim.x) {
        const int64_t o = b / tiles;
        const int64_t tile = b - o * tiles;
        const int64_t c0 = (tile * TX + tx) * VEC;
        const bool valid = c0 < inner;
        MS st[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) st[j] = ms_empty();
        static_assert(!ONE || LSM, "the one-walk form writes log_softmax");
        constexpr bool one_walk = ONE;
        float keep_v[ONE ? VEC : 1][ONE ? CH : 1];
        if constexpr (ONE) {
            if (valid) {
                const float* base = x + o * R * inner + c0 + (int64_t)ty * inner;
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    float w[VEC];
                    load_cols<VEC>(base + (int64_t)k * TY * inner, w, 0, false);
#pragma unroll
                    for (int j = 0; j < VEC; ++j) keep_v[ONE ? j : 0][ONE ? k : 0] = w[j];
                }
                if constexpr (ONE) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) ms_fold<CH>(st[j], keep_v[j]);
                }
            }
        } else if (valid) {
            const float* base = x + o * R * inner + c0;
            int64_t r = ty;
            const int64_t step = (int64_t)CH * TY;
            for (; r + (int64_t)(CH - 1) * TY < R; r += step) {
                float v[VEC][CH];
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    float w[VEC];
                    load_cols<VEC>(base + (r + (int64_t)k * TY) * inner, w, keep, LSM);
#pragma unroll
                    for (int j = 0; j < VEC; ++j) v[j][k] = w[j];
                }
#pragma unroll
                for (int j = 0; j < VEC; ++j) ms_fold<CH>(st[j], v[j]);
            }
            for (; r < R; r += TY) {
                float w[VEC];
                load_cols<VEC>(base + r * inner, w, keep, LSM);
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    float v1[1] = {w[j]};
                    ms_fold<1>(st[j], v1);
                }
            }
        }
        if (TY > 1) {  // tree merge over the thread rows (TY is a power of two)
#pragma unroll
            for (int j = 0; j < VEC; ++j) red[(ty * TX + tx) * VEC + j] = st[j];
            __syncthreads();
            for (int h = TY >> 1; h > 0; h >>= 1) {
                if (ty < h) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        MS a = red[(ty * TX + tx) * VEC + j];
                        MS c = red[((ty + h) * TX + tx) * VEC + j];
                        red[(ty * TX + tx) * VEC + j] = ms_merge(a, c);
                    }
                }
                __syncthreads();
            }
            if (ty == 0) {
#pragma unroll
                for (int j = 0; j < VEC; ++j) st[j] = red[tx * VEC + j];
            }
            __syncthreads();  // red is reused by the next tile
        }
        if constexpr (LSM) {
            // every thread row needs the lse of its columns for the write walk
            if (ty == 0) {
#pragma unroll
                for (int j = 0; j < VEC; ++j) lse_s[tx * VEC + j] = ms_lse(st[j]);
            }
            __syncthreads();
            if (valid && one_walk) {  // constant: one of the two branches is compiled
                float l[VEC];
#pragma unroll
                for (int j = 0; j < VEC; ++j) l[j] = lse_s[tx * VEC + j];
                float* dst = out + o * R * inner + c0 + (int64_t)ty * inner;
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    const int kk = ONE ? k : 0;
                    if constexpr (VEC == 4)
                        st_stream_f4(dst + (int64_t)k * TY * inner,
                                     make_float4(keep_v[0][kk] - l[0], keep_v[ONE ? 1 : 0][kk] - l[1],
                                                 keep_v[ONE ? 2 : 0][kk] - l[2], keep_v[ONE ? 3 : 0][kk] - l[3]));
                    else
                        st_stream_f1(dst + (int64_t)k * TY * inner, keep_v[0][kk] - l[0]);
                }
            } else if (valid) {
                float l[VEC];
#pragma unroll
                for (int j = 0; j < VEC; ++j) l[j] = lse_s[tx * VEC + j];
                const uint64_t drop = l2_policy_evict_first();
                const int64_t off = o * R * inner + c0;
                for (int64_t r = ty; r < R; r += TY) {
                    float w[VEC];
                    load_cols<VEC>(x + off + r * inner, w, drop, true);
                    float* dst = out + off + r * inner;
                    if constexpr (VEC == 4)
                        st_stream_f4(dst, make_float4(w[0] - l[0], w[1] - l[1], w[2] - l[2], w[3] - l[3]));
                    else
                        st_stream_f1(dst, w[0] - l[0]);
                }
            }
            __syncthreads();  // lse_s is reused by the next tile
            continue;
        }
        if (ty == 0 && valid) {
            float* dst = out + o * inner + c0;
            if constexpr (VEC == 4) {
                float4 w = make_float4(ms_lse(st[0]), ms_lse(st[1]), ms_lse(st[2]), ms_lse(st[3]));
                *reinterpret_cast<float4*>(dst) = w;
            } else {
                dst[0] = ms_lse(st[0]);
            }
        }
    }
}

static int pow2_floor(int64_t v) {
    int p = 1;
    while ((int64_t)p * 2 <= v && p < (1 << 30)) p *= 2;
    return p;
}

static int pow2_ceil(int64_t v) {
    int p = 1;
    while ((int64_t)p < v && p < (1 << 30)) p *= 2;
    return p;
}

template <bool LSM>
static void strided_go(bool vec4, int CH, unsigned grid, dim3 block, const float* x, float* out, int64_t outer,
                       int64_t R, int64_t inner, int64_t tiles, cudaStream_t stream) {
    if (LSM && vec4 && CH == 8 && R == 8 * (int64_t)block.y && env_int("LSE_STRIDED_ONE_WALK", 1)) {
        lse_strided_kernel<4, 8, true, true><<<grid, block, 0, stream>>>(x, out, outer, R, inner, tiles);
        return;
    }
    if (vec4) {
        if (CH == 8)
            lse_strided_kernel<4, 8, LSM><<<grid, block, 0, stream>>>(x, out, outer, R, inner, tiles);
        else
            lse_strided_kernel<4, 4, LSM><<<grid, block, 0, stream>>>(x, out, outer, R, inner, tiles);
    } else {
        if (CH == 8)
            lse_strided_kernel<1, 8, LSM><<<grid, block, 0, stream>>>(x, out, outer, R, inner, tiles);
        else
            lse_strided_kernel<1, 4, LSM><<<grid, block, 0, stream>>>(x, out, outer, R, inner, tiles);
    }
}

cudaError_t launch_lse_strided(const DeviceInfo& dev, const float* x, float* out, int64_t outer,
                               int64_t R, int64_t inner, cudaStream_t stream, bool log_softmax) {
    const bool vec4 = (inner % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0) &&
                      ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    const int VEC = vec4 ? 4 : 1;
    const int64_t ncols = (inner + VEC - 1) / VEC;
    const int CH = (R >= 8) ? 8 : 4;
    const int ty_cap = pow2_floor(std::max<int64_t>(1, R / CH));
    // The log_softmax walk re-reads a tile of R x TX*VEC floats from L2, so it
    // splits R over as many thread rows as it can (up to 8): fewer bytes per
    // thread between the two walks, and a smaller set of tiles held in L2.
    const int tx_max = log_softmax ? 256 / std::min(8, ty_cap) : 256;
    const int TX = (int)std::min<int64_t>(tx_max, std::max<int64_t>(32, pow2_ceil(ncols)));
    const int TY = std::min(256 / TX, ty_cap);
    const int64_t tiles = (ncols + TX - 1) / TX;
    const int64_t nblk = outer * tiles;
    const int per_sm = std::max(1, 2048 / (TX * TY));
    const int64_t cap = (int64_t)dev.sm_count * per_sm * 64;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(nblk, cap));
    dim3 block(TX, TY);
    if (log_softmax)
        strided_go<true>(vec4, CH, grid, block, x, out, outer, R, inner, tiles, stream);
    else
        strided_go<false>(vec4, CH, grid, block, x, out, outer, R, inner, tiles, stream);
    return cudaGetLastError();
}

}  // namespace lse
