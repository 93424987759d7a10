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
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace lse {

template <int VEC, int CH>
__global__ void __launch_bounds__(256) lse_strided_kernel(const float* __restrict__ x,
                                                          float* __restrict__ out, int64_t outer,
                                                          int64_t R, int64_t inner, int64_t tiles) {
    __shared__ MS red[256 * VEC];
    const int TX = blockDim.x, TY = blockDim.y;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int64_t nblk = outer * tiles;
    for (int64_t b = blockIdx.x; b < nblk; b += gridDim.x) {
        const int64_t o = b / tiles;
        const int64_t tile = b - o * tiles;
        const int64_t c0 = (tile * TX + tx) * VEC;
        const bool valid = c0 < inner;
        MS st[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) st[j] = ms_empty();
        if (valid) {
            const float* base = x + o * R * inner + c0;
            int64_t r = ty;
            const int64_t step = (int64_t)CH * TY;
            for (; r + (int64_t)(CH - 1) * TY < R; r += step) {
                float v[VEC][CH];
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    const float* p = base + (r + (int64_t)k * TY) * inner;
                    if constexpr (VEC == 4) {
                        float4 a = ld_stream_f4(p);
                        v[0][k] = a.x; v[1][k] = a.y; v[2][k] = a.z; v[3][k] = a.w;
                    } else {
                        v[0][k] = ld_stream_f1(p);
                    }
                }
#pragma unroll
                for (int j = 0; j < VEC; ++j) ms_fold<CH>(st[j], v[j]);
            }
            for (; r < R; r += TY) {
                const float* p = base + r * inner;
                float v[VEC][1];
                if constexpr (VEC == 4) {
                    float4 a = ld_stream_f4(p);
                    v[0][0] = a.x; v[1][0] = a.y; v[2][0] = a.z; v[3][0] = a.w;
                } else {
                    v[0][0] = ld_stream_f1(p);
                }
#pragma unroll
                for (int j = 0; j < VEC; ++j) ms_fold<1>(st[j], v[j]);
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

cudaError_t launch_lse_strided(const DeviceInfo& dev, const float* x, float* out, int64_t outer,
                               int64_t R, int64_t inner, cudaStream_t stream) {
    const bool vec4 = (inner % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0) &&
                      ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    const int VEC = vec4 ? 4 : 1;
    const int64_t ncols = (inner + VEC - 1) / VEC;
    const int TX = (int)std::min<int64_t>(256, std::max<int64_t>(32, pow2_ceil(ncols)));
    const int CH = (R >= 8) ? 8 : 4;
    int TY = 256 / TX;
    TY = std::min(TY, pow2_floor(std::max<int64_t>(1, R / CH)));
    const int64_t tiles = (ncols + TX - 1) / TX;
    const int64_t nblk = outer * tiles;
    const int per_sm = std::max(1, 2048 / (TX * TY));
    const int64_t cap = (int64_t)dev.sm_count * per_sm * 64;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(nblk, cap));
    dim3 block(TX, TY);
    if (vec4) {
        if (CH == 8)
            lse_strided_kernel<4, 8><<<grid, block, 0, stream>>>(x, out, outer, R, inner, tiles);
        else
            lse_strided_kernel<4, 4><<<grid, block, 0, stream>>>(x, out, outer, R, inner, tiles);
    } else {
        if (CH == 8)
            lse_strided_kernel<1, 8><<<grid, block, 0, stream>>>(x, out, outer, R, inner, tiles);
        else
            lse_strided_kernel<1, 4><<<grid, block, 0, stream>>>(x, out, outer, R, inner, tiles);
    }
    return cudaGetLastError();
}

}  // namespace lse
