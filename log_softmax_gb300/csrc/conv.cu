// Conv2d (3 x 3, stride 1, valid, bias) on the tensor cores: the layer that
// produces the y of the GroupNorm chain of the POPCORNBENCH page
// "Kimi-K2.6 / l2_p92" (8 -> 64 channels on 128 x 128 planes).
//
// conv2d_tc_kernel: persistent CTAs of 128 threads loop over output tiles of
// 128 pixels x Cout channels.  The weights are split (hi/lo tf32) into shared
// memory once per CTA; per tile every thread writes the hi/lo patch row of one
// pixel, one thread issues the 3xTF32 MMAs into tensor memory, and after their
// commit every thread reads its pixel's Cout accumulators back (tcgen05.ld),
// adds the bias and stores y with coalesced rows per channel.  With STATS the
// epilogue also folds each channel group's values of the tile into a Welford
// (count, mean, M2) -- per thread over the group's channels, then across the
// tile's pixels by warp shuffles and shared memory -- and stores one partial
// per (sample, tile, group); gn_tile_merge_kernel merges a sample's tiles.
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
    int64_t tiles;  // pixel tiles per sample
    int G, cpg;     // channel groups of the statistics (STATS), cpg divides 16
    float4* partials;  // [N][tiles][G] (count, mean, M2, 0) (STATS)
    int* status;
};

// Tile slots per CTA: each slot is one warpgroup (128 threads) with its own
// patch buffers and accumulator, working on its own tiles, so one slot's MMAs
// and epilogue overlap the other's patch loads.
constexpr int kConvSlots = 2;

static size_t conv_smem_bytes(int cin, int cout) {
    const int Kp = conv_kpad(cin);
    return (size_t)kConvSlots * 2 * kConvTileM * Kp * 4 + (size_t)2 * cout * Kp * 4 + (size_t)(cout * 4 + 127) / 128 * 128;
}

__host__ __device__ static inline uint32_t conv_tmem_cols(int cout) { return cout <= 32 ? 32u : (cout <= 64 ? 64u : 128u); }

template <int CIN, int CPG>
__global__ void __launch_bounds__(kConvSlots * kConvTileM, 1) conv2d_tc_kernel(const ConvArgs a) {
    constexpr bool STATS = CPG > 0;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t bars[kConvSlots];
    __shared__ uint32_t tmem_slot;

    constexpr int Kp = conv_kpad(CIN);
    constexpr uint32_t kAbytes = kConvTileM * Kp * 4;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int slot = tid / kConvTileM, wtid = tid - slot * kConvTileM;  // warpgroup and thread in it
    unsigned char* const bhi = smem_raw;
    unsigned char* const blo = bhi + a.cout * Kp * 4;
    float* const bias = reinterpret_cast<float*>(blo + a.cout * Kp * 4);
    unsigned char* const ahi = smem_raw + (size_t)2 * a.cout * Kp * 4 + (size_t)((a.cout * 4 + 127) / 128 * 128) +
                               (size_t)slot * 2 * kAbytes;
    unsigned char* const alo = ahi + kAbytes;
    // [group][pixel] (mean, M2) of the statistics epilogue, in this slot's patch
    // buffers (free between the MMAs' completion and the next tile's patches)
    float2* const wsm = reinterpret_cast<float2*>(ahi);
    const uint32_t ncols = conv_tmem_cols(a.cout);
    uint64_t* const bar = &bars[slot];

    if (warp == 0) tmem_alloc(&tmem_slot, ncols * kConvSlots);
    if (tid == 0) {
        for (int k = 0; k < kConvSlots; ++k) mbar_init(&bars[k], 1);
        fence_mbar_init();
    }
    conv_stage_weights(a.w, a.cin, a.cout, bhi, blo, true);
    for (int c = tid; c < a.cout; c += blockDim.x) bias[c] = a.b[c];
    fence_proxy_async_smem();  // the weights are read by the tensor cores (async proxy)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot + (uint32_t)slot * ncols;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int64_t ohw = (int64_t)a.OH * a.OW;
    bool aborted = false;
    uint32_t phase = 0;
    const int bar_id = 1 + slot;  // named barrier of this warpgroup

    for (int64_t t = (int64_t)blockIdx.x * kConvSlots + slot; t < a.N * a.tiles;
         t += (int64_t)gridDim.x * kConvSlots) {
        const int64_t n = t / a.tiles;
        const int64_t p0 = (t - n * a.tiles) * kConvTileM;
        conv_stage_patches<CIN>(a.x + n * CIN * a.H * a.W, a.H, a.W, a.OW, ohw, p0, wtid, ahi, alo, true);
        fence_proxy_async_smem();
        named_bar_sync(bar_id, kConvTileM);  // the patches are in shared memory; D is free
        if (wtid == 0) {
            tc_fence_after();
            conv_issue_mma(tmem, ahi, alo, bhi, blo, a.cin, a.cout, true, bar);
        }
        mbar_wait_bounded(bar, phase, aborted, a.status);
        phase ^= 1u;
        tc_fence_after();
        const int64_t p = p0 + wtid;
        const bool valid = p < ohw;
        float* dst = a.y + n * a.cout * ohw + p;
        for (int c0 = 0; c0 < a.cout; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + (uint32_t)c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += bias[c0 + j];
            if (valid) {
#pragma unroll
                for (int j = 0; j < 16; ++j) dst[(int64_t)(c0 + j) * ohw] = v[j];
            }
            if constexpr (STATS) {
                // the 16 / CPG groups inside these 16 channels: exact mean and M2 of
                // this pixel's CPG values of each
#pragma unroll
                for (int lo = 0; lo < 16; lo += CPG) {
                    float sum = 0.f;
#pragma unroll
                    for (int j = 0; j < CPG; ++j) sum += v[lo + j];
                    const float mean = sum * (1.f / CPG);
                    float m2 = 0.f;
#pragma unroll
                    for (int j = 0; j < CPG; ++j) m2 = fmaf(v[lo + j] - mean, v[lo + j] - mean, m2);
                    wsm[((c0 + lo) / CPG) * kConvTileM + wtid] = make_float2(mean, m2);
                }
            }
        }
        if constexpr (STATS) {
            // merge over the tile's pixels: tpg threads per group, each a strided
            // share of the pixels, then shuffles within the tpg-lane block
            named_bar_sync(bar_id, kConvTileM);
            const int G = a.G;
            int tpg = 1;
            while (tpg * 2 * G <= kConvTileM && tpg < 32) tpg *= 2;
            const int g = wtid / tpg, j = wtid - g * tpg;
            Welford w{0.f, 0.f, 0.f};
            if (g < G) {
                for (int m = j; m < kConvTileM; m += tpg) {
                    const float2 q = wsm[g * kConvTileM + m];
                    if (p0 + m < ohw) w = wf_merge(w, Welford{(float)CPG, q.x, q.y});
                }
            }
            for (int o = 1; o < tpg; o <<= 1) {
                const Welford other = wf_shfl_xor(w, o);
                w = wf_merge(w, other);
            }
            if (g < G && j == 0)
                a.partials[(n * a.tiles + (p0 / kConvTileM)) * G + g] = make_float4(w.n, w.mean, w.m2, 0.f);
        }
        tc_fence_before();
        named_bar_sync(bar_id, kConvTileM);  // this slot is done reading D, the patches and wsm
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_slot, ncols * kConvSlots);
}

bool conv_tc_supported(int64_t cin, int64_t cout) {
    return cin >= 1 && cin <= kConvMaxCin && cout >= 16 && cout <= 128 && cout % 16 == 0;
}

template <int CIN, int CPG>
static cudaError_t conv_go(const DeviceInfo& dev, const ConvArgs& a, cudaStream_t stream);

static cudaError_t conv_dispatch(const DeviceInfo& dev, const ConvArgs& a, cudaStream_t stream) {
    switch (a.cin) {
        case 1: return conv_go<1, 0>(dev, a, stream);
        case 2: return conv_go<2, 0>(dev, a, stream);
        case 3: return conv_go<3, 0>(dev, a, stream);
        case 4: return conv_go<4, 0>(dev, a, stream);
        case 5: return conv_go<5, 0>(dev, a, stream);
        case 6: return conv_go<6, 0>(dev, a, stream);
        case 7: return conv_go<7, 0>(dev, a, stream);
        default: return conv_go<8, 0>(dev, a, stream);
    }
}

// The statistics epilogue is compiled for the chain's own convolution (Cin = 8).
static cudaError_t conv_stats_dispatch(const DeviceInfo& dev, const ConvArgs& a, cudaStream_t stream) {
    switch (a.cpg) {
        case 1: return conv_go<8, 1>(dev, a, stream);
        case 2: return conv_go<8, 2>(dev, a, stream);
        case 4: return conv_go<8, 4>(dev, a, stream);
        case 8: return conv_go<8, 8>(dev, a, stream);
        default: return conv_go<8, 16>(dev, a, stream);
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
    a.tiles = ((int64_t)a.OH * a.OW + kConvTileM - 1) / kConvTileM;
    a.G = 1;
    a.cpg = (int)cout;
    a.partials = nullptr;
    a.status = dev.status;
    return a;
}

cudaError_t launch_conv2d_3x3(const DeviceInfo& dev, const float* x, const float* w, const float* b, float* y,
                              int64_t N, int64_t cin, int64_t H, int64_t W, int64_t cout, cudaStream_t stream) {
    return conv_dispatch(dev, conv_args(dev, x, w, b, y, N, cin, H, W, cout), stream);
}

template <int CIN, int CPG>
static cudaError_t conv_go(const DeviceInfo& dev, const ConvArgs& a, cudaStream_t stream) {
    auto kern = conv2d_tc_kernel<CIN, CPG>;
    const size_t smem = conv_smem_bytes(a.cin, a.cout);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kConvSlots * kConvTileM, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    // tensor memory: per_sm CTAs x ncols columns must fit the SM's 512
    per_sm = std::min<int>(per_sm, (int)(512 / (kConvSlots * conv_tmem_cols(a.cout))));
    const int64_t total = a.N * a.tiles;
    const int64_t blocks = (total + kConvSlots - 1) / kConvSlots;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)per_sm * dev.sm_count));
    if (env_int("LSE_VERBOSE", 0)) {
        cudaFuncAttributes fa;
        cudaFuncGetAttributes(&fa, kern);
        int smem_sm = 0, resv = 0;
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev.device);
        cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, dev.device);
        fprintf(stderr,
                "[lse] conv2d_tc: grid=%u (%d per SM) tiles=%lld smem=%zu static=%zu regs=%d smem/SM=%d reserved=%d\n",
                grid, per_sm, (long long)total, smem, fa.sharedSizeBytes, fa.numRegs, smem_sm, resv);
    }
    kern<<<grid, kConvSlots * kConvTileM, smem, stream>>>(a);
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

size_t conv_chain_scratch_bytes(int64_t N, int64_t H, int64_t W, int64_t cout, int64_t G) {
    const int64_t ohw = (H - 2) * (W - 2);
    const int64_t tiles = (ohw + kConvTileM - 1) / kConvTileM;
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    return up((size_t)N * cout * ohw * 4) + up((size_t)N * tiles * G * sizeof(float4)) + up((size_t)N * G * 8);
}

cudaError_t launch_conv_gn_act_lse(const DeviceInfo& dev, const float* x, const float* w, const float* b,
                                   const float* gamma, const float* beta, float* out, int64_t N, int64_t cin,
                                   int64_t H, int64_t W, int64_t cout, int64_t G, float eps, void* scratch,
                                   cudaStream_t stream) {
    const int64_t ohw = (H - 2) * (W - 2);
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    char* sp = static_cast<char*>(scratch);
    float* y = reinterpret_cast<float*>(sp);
    sp += up((size_t)N * cout * ohw * 4);
    ConvArgs a = conv_args(dev, x, w, b, y, N, cin, H, W, cout);
    a.G = (int)G;
    a.cpg = (int)(cout / G);
    a.partials = reinterpret_cast<float4*>(sp);
    sp += up((size_t)N * a.tiles * G * sizeof(float4));
    float* stats = reinterpret_cast<float*>(sp);
    cudaError_t e = conv_stats_dispatch(dev, a, stream);
    if (e != cudaSuccess) return e;
    const int64_t NG = N * G;
    gn_tile_merge_kernel<<<(unsigned)((NG + 7) / 8), 256, 0, stream>>>(a.partials, stats, NG, a.tiles, (int)G, eps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_gn_apply(dev, y, gamma, beta, out, N, cout, ohw, G, stats, stream);
}

}  // namespace lse
