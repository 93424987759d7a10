// Form 3 (and GroupNorm alone, and the chain before its lse) on the work-queue
// schedule of gn_fused_kernel, with every item's data staged through a ring of
// shared-memory slots by bulk copies (TMA) instead of per-thread loads.
//
// Items, claimed from one counter in a fixed order (for k = 0, 1, ...: the G
// statistics items of sample k, then the apply tiles of sample k - lag):
//   statistics item (n, g)  the group's slab, cpg*HW contiguous floats, copied
//                           in 32 KB chunks; every thread folds a Welford
//                           (count, mean, M2) from shared memory; the block's
//                           merge is published and counted in (release).
//   apply tile (n, t)       pixels [t*TP, t*TP + TP) of every channel, copied
//                           in chunks of CC channel rows; the per-channel table
//                           of sample n is built while the first chunks land
//                           (after a bounded wait for the sample's statistics);
//                           each thread owns 4 adjacent pixels and either folds
//                           the channel lse (OUT 0) or writes the GroupNorm
//                           output (1) or y + hardswish(tanh(z)) (2, as two
//                           packed f32x2 pixel pairs).
// A CTA keeps up to R chunks (R x 32 KB) in flight, so a few CTAs per SM hide
// the HBM and L2 latency that per-thread loads could not.  The statistics
// chunks ask L2 to keep their lines (the apply tiles of the same sample read
// them again soon after) and the apply chunks to drop them.  All waits are
// bounded (about 1 s) and record a timeout in the device status word; the
// grid is cooperative, so every claimed statistics item is running.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "gn_common.cuh"
#include "launch.h"

namespace lse {

constexpr int kGntSlotBytes = 32768;
constexpr int kGntMaxSlots = 8;
constexpr int kGntThreads = 256;

struct GnTmaArgs {
    const float* y;
    const float* gamma;
    const float* beta;
    float* out;
    int64_t N, HW;
    int C, G, tiles, lag, nslot;
    float eps;
    float4* partials;          // [N][G] (count, mean, M2, 0)
    unsigned* done;            // [N] statistics items finished, zero at launch
    unsigned long long* next;  // work-item counter, zero at launch
    int* status;
};

template <int OUT, int T>
__global__ void __launch_bounds__(T) gn_tma_kernel(const GnTmaArgs a) {
    constexpr int TP = 4 * T;                  // apply tile width (pixels): 4 per thread
    constexpr int CF = kGntSlotBytes / 4;      // floats per slot
    constexpr int CC = CF / TP;                // channel rows per apply chunk
    static_assert(CC >= 1, "a slot must hold one apply row");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ Welford red[32];
    __shared__ long long item_sh;
    const int R = a.nslot;
    const int C = a.C, G = a.G, cpg = C / G;
    float* const ring = reinterpret_cast<float*>(smem_raw);                                   // [R][CF]
    // OUT 0 and 2 take the pair-form table [C] {mean, mean, sc, sc} then [C] {sh, sh};
    // OUT 1 [C] {mean, rstd * gamma, beta, 0}
    float4* const tab = reinterpret_cast<float4*>(smem_raw + (size_t)R * kGntSlotBytes);     // [C]
    float2* const tab_b = reinterpret_cast<float2*>(tab + C);                                // [C]
    uint64_t* const full = reinterpret_cast<uint64_t*>(tab_b + C);                           // [R]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t N = a.N, HW = a.HW;
    const int64_t GP = G, TT = a.tiles, lag = a.lag;
    const int64_t total = N * (GP + TT);
    const int64_t L = (int64_t)cpg * HW;  // floats of one statistics slab
    const int nck_stats = (int)((L + CF - 1) / CF);
    const int nck_apply = (C + CC - 1) / CC;
    const uint64_t keep = l2_policy_evict_last();
    const uint64_t drop = l2_policy_evict_first();
    bool aborted = false;
    uint64_t seq = 0;     // chunks consumed so far; every thread counts the same
    uint64_t issued = 0;  // chunks issued so far (thread 0)

    if (tid == 0) {
        for (int r = 0; r < R; ++r) mbar_init(&full[r], 1);
        fence_mbar_init();
    }
    __syncthreads();

    for (;;) {
        if (tid == 0) item_sh = (long long)atomicAdd(a.next, 1ull);
        __syncthreads();
        const int64_t t = item_sh;
        __syncthreads();
        if (t >= total) break;
        bool is_stats;
        int64_t n, idx;
        if (t < lag * GP) {
            is_stats = true;
            n = t / GP;
            idx = t - n * GP;
        } else if (t < lag * GP + (N - lag) * (GP + TT)) {
            const int64_t u = t - lag * GP;
            const int64_t k = lag + u / (GP + TT);
            const int64_t r = u - (k - lag) * (GP + TT);
            is_stats = r < GP;
            n = is_stats ? k : k - lag;
            idx = is_stats ? r : r - GP;
        } else {
            const int64_t u = t - lag * GP - (N - lag) * (GP + TT);
            n = N - lag + u / TT;
            idx = u - (n - (N - lag)) * TT;
            is_stats = false;
        }

        if (is_stats) {
            // ---------------- statistics item (n, g = idx)
            const float* slab = a.y + (n * C + idx * cpg) * HW;
            auto issue = [&](int i) {
                if (aborted) return;
                const uint64_t s = seq + i;
                const int r = (int)(s % R);
                const int64_t off = (int64_t)i * CF;
                const uint32_t bytes = (uint32_t)(std::min<int64_t>(CF, L - off) * 4);
                fence_proxy_async_smem();  // earlier generic reads of the slot come first
                mbar_arrive_expect_tx(&full[r], bytes);
                bulk_g2s_hint(ring + (size_t)r * CF, slab + off, bytes, &full[r], keep);
                issued = s + 1;
            };
            if (tid == 0)
                for (int i = 0; i < std::min(R, nck_stats); ++i) issue(i);
            Welford w{0.f, 0.f, 0.f};
            for (int i = 0; i < nck_stats; ++i) {
                const uint64_t s = seq + i;
                const int r = (int)(s % R);
                mbar_wait_bounded(&full[r], (uint32_t)((s / R) & 1), aborted, a.status);
                const int n4 = (int)(std::min<int64_t>(CF, L - (int64_t)i * CF) >> 2);
                const float4* p = reinterpret_cast<const float4*>(ring + (size_t)r * CF);
                int k = tid;
                for (; k + 3 * T < n4; k += 4 * T) {
                    float v[16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 q = p[k + u * T];
                        v[4 * u + 0] = q.x; v[4 * u + 1] = q.y; v[4 * u + 2] = q.z; v[4 * u + 3] = q.w;
                    }
                    w = wf_merge(w, wf_batch<16>(v));
                }
                for (; k < n4; k += T) {
                    const float4 q = p[k];
                    const float v[4] = {q.x, q.y, q.z, q.w};
                    w = wf_merge(w, wf_batch<4>(v));
                }
                __syncthreads();  // every thread is done with slot r
                if (tid == 0 && i + R < nck_stats) issue(i + R);
            }
            seq += nck_stats;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w = wf_merge(w, wf_shfl_xor(w, o));
            if (lane == 0) red[warp] = w;
            __syncthreads();
            if (warp == 0) {
                Welford r = (lane < T / 32) ? red[lane] : Welford{0.f, 0.f, 0.f};
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) r = wf_merge(r, wf_shfl_xor(r, o));
                if (lane == 0) {
                    float4* dst = a.partials + n * G + idx;
                    asm volatile("st.relaxed.gpu.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(r.n),
                                 "f"(r.mean), "f"(r.m2), "f"(0.f)
                                 : "memory");
                    red_release_gpu_add(a.done + n, 1u);
                }
            }
        } else {
            // ---------------- apply tile (n, idx)
            const int64_t px0 = idx * TP;
            const int tw = (int)std::min<int64_t>(TP, HW - px0);  // a multiple of 4
            auto issue = [&](int i) {
                if (aborted) return;
                const uint64_t s = seq + i;
                const int r = (int)(s % R);
                const int c0 = i * CC, nr = std::min(CC, C - c0);
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&full[r], (uint32_t)(nr * tw * 4));
                const float* src = a.y + (n * C + c0) * HW + px0;
                for (int cc = 0; cc < nr; ++cc)
                    bulk_g2s_hint(ring + (size_t)r * CF + cc * TP, src + cc * HW, (uint32_t)tw * 4u, &full[r], drop);
                issued = s + 1;
            };
            if (tid == 0) {
                for (int i = 0; i < std::min(R, nck_apply); ++i) issue(i);
                // the sample's statistics items were claimed earlier by running CTAs
                if (!aborted && ld_acquire_gpu_u32(a.done + n) < (unsigned)GP) {
                    const uint64_t t0 = globaltimer_ns();
                    bool ok = false;
                    for (uint32_t it = 0; it < (1u << 26); ++it) {
                        __nanosleep(64);
                        if (ld_acquire_gpu_u32(a.done + n) >= (unsigned)GP) {
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
            }
            __syncthreads();  // thread 0's acquire orders the partial reads below
            for (int c = tid; c < C; c += T) {
                const int g = c / cpg;
                float4 q;
                asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(q.x), "=f"(q.y), "=f"(q.z), "=f"(q.w)
                             : "l"(a.partials + n * G + g)
                             : "memory");
                const float rstd = 1.f / sqrtf(q.z / q.x + a.eps);
                if constexpr (OUT != 1)
                    gn_pair_entry(q.y, rstd * a.gamma[c] * (2.f * kLog2e), a.beta[c] * (2.f * kLog2e), tab, tab_b, c);
                else
                    tab[c] = make_float4(q.y, rstd * a.gamma[c], a.beta[c], 0.f);
            }
            __syncthreads();
            const bool on = 4 * tid < tw;
            Lse4 st = lse4_empty();
            for (int i = 0; i < nck_apply; ++i) {
                const uint64_t s = seq + i;
                const int r = (int)(s % R);
                mbar_wait_bounded(&full[r], (uint32_t)((s / R) & 1), aborted, a.status);
                const int c0 = i * CC, nr = std::min(CC, C - c0);
                const float* sl = ring + (size_t)r * CF + 4 * tid;
                if (on) {
                    if constexpr (OUT == 0) {
                        // the chain's residual in pair form (less 2/3), folded into the
                        // running channel lse of this thread's four pixels
                        auto residual = [&](int cc, f32x2& ra, f32x2& rb) {
                            const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(sl + cc * TP);
                            const float4 ta = tab[c0 + cc];
                            const float2 tb = tab_b[c0 + cc];
                            const f32x2 mean = f2_pack(ta.x, ta.y), sc = f2_pack(ta.z, ta.w);
                            const f32x2 sh = f2_pack(tb.x, tb.y);
                            ra = f2_residual_less_2_3(v.x, mean, sc, sh);
                            rb = f2_residual_less_2_3(v.y, mean, sc, sh);
                        };
                        if (nr == CC) {
                            f32x2 ra[CC], rb[CC];
#pragma unroll
                            for (int cc = 0; cc < CC; ++cc) residual(cc, ra[cc], rb[cc]);
                            lse4_fold<CC>(st, ra, rb);
                        } else {
                            for (int cc = 0; cc < nr; ++cc) {
                                f32x2 ra[1], rb[1];
                                residual(cc, ra[0], rb[0]);
                                lse4_fold<1>(st, ra, rb);
                            }
                        }
                    } else {
                        float* dst = a.out + (n * C + c0) * HW + px0 + 4 * tid;
                        for (int cc = 0; cc < nr; ++cc) {
                            float4 o;
                            if constexpr (OUT == 1) {
                                const float4 x = *reinterpret_cast<const float4*>(sl + cc * TP);
                                const float4 e = tab[c0 + cc];
                                o = make_float4(fmaf(x.x - e.x, e.y, e.z), fmaf(x.y - e.x, e.y, e.z),
                                                fmaf(x.z - e.x, e.y, e.z), fmaf(x.w - e.x, e.y, e.z));
                            } else {
                                // y + hardswish(tanh(z)) in pair form, plus the 2/3 it leaves out
                                const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(sl + cc * TP);
                                const float4 ta = tab[c0 + cc];
                                const float2 tb = tab_b[c0 + cc];
                                const f32x2 mean = f2_pack(ta.x, ta.y), sc = f2_pack(ta.z, ta.w);
                                const f32x2 sh = f2_pack(tb.x, tb.y), k23 = f2_pack(2.f / 3.f, 2.f / 3.f);
                                const f32x2 ra = f2_add(f2_residual_less_2_3(v.x, mean, sc, sh), k23);
                                const f32x2 rb = f2_add(f2_residual_less_2_3(v.y, mean, sc, sh), k23);
                                f2_unpack(ra, o.x, o.y);
                                f2_unpack(rb, o.z, o.w);
                            }
                            st_stream_f4(dst + cc * HW, o);
                        }
                    }
                }
                __syncthreads();  // every thread is done with slot r
                if (tid == 0 && i + R < nck_apply) issue(i + R);
            }
            seq += nck_apply;
            if constexpr (OUT == 0) {
                if (on) {
                    float m[4], sm[4];
                    lse4_unpack(st, m, sm);
                    *reinterpret_cast<float4*>(a.out + n * HW + px0 + 4 * tid) =
                        make_float4(m[0] + logf(sm[0]) + 2.f / 3.f, m[1] + logf(sm[1]) + 2.f / 3.f,
                                    m[2] + logf(sm[2]) + 2.f / 3.f, m[3] + logf(sm[3]) + 2.f / 3.f);
                }
            }
        }
    }
    if (tid == 0 && atomicAdd(a.status, 0) != 0) {
        // After a timeout anywhere, give each slot's last fill one more bounded
        // wait before the shared memory is released.
        bool again = false;
        for (uint64_t s = issued > (uint64_t)R ? issued - R : 0; s < issued; ++s)
            mbar_wait_bounded(&full[s % R], (uint32_t)((s / R) & 1), again, a.status);
    }
}

size_t gn_tma_scratch_bytes(int64_t N, int64_t G) {
    return (size_t)N * G * sizeof(float4) + ((size_t)N * sizeof(unsigned) + 15) / 16 * 16 + 16;
}

// Shared memory of one CTA with `slots` ring slots (the table takes 24 bytes per
// channel, enough for the pair form).
static size_t gn_tma_smem(int64_t C, int slots) {
    return (size_t)slots * kGntSlotBytes + (size_t)C * (sizeof(float4) + sizeof(float2)) +
           kGntMaxSlots * sizeof(uint64_t);
}

bool gn_tma_applies(const DeviceInfo& dev, const float* y, const float* out, int64_t C, int64_t HW) {
    if (HW % 4 != 0 || (reinterpret_cast<uintptr_t>(y) & 15) != 0 || (reinterpret_cast<uintptr_t>(out) & 15) != 0)
        return false;
    return gn_tma_smem(C, 2) <= (size_t)dev.max_smem_optin;
}

template <int OUT>
static cudaError_t gn_tma_go(const DeviceInfo& dev, const GnTmaArgs& args, size_t smem, int want_per_sm,
                            cudaStream_t stream) {
    auto kern = gn_tma_kernel<OUT, kGntThreads>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGntThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    if (want_per_sm > 0) per_sm = std::min(per_sm, want_per_sm);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the sample waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kGntThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    const int64_t items = args.N * ((int64_t)args.G + args.tiles);
    cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>(items, (int64_t)per_sm * dev.sm_count)));
    if (env_int("LSE_VERBOSE", 0))
        fprintf(stderr, "[lse] gn_tma: grid=%u slots=%d tiles=%d lag=%d smem=%zu\n", cfg.gridDim.x, args.nslot,
                args.tiles, args.lag, smem);
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_gn_tma(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                          int64_t N, int64_t C, int64_t HW, int64_t G, float eps, void* scratch, cudaStream_t stream,
                          int out_kind) {
    GnTmaArgs args;
    args.y = y;
    args.gamma = gamma;
    args.beta = beta;
    args.out = out;
    args.N = N;
    args.HW = HW;
    args.C = (int)C;
    args.G = (int)G;
    args.tiles = (int)((HW + 4 * kGntThreads - 1) / (4 * kGntThreads));
    args.lag = (int)std::min<int64_t>(N, std::max(0, env_int("LSE_GNT_LAG", 8)));
    args.eps = eps;
    // ring slots: LSE_GNT_SLOTS (default 3), as many as fit
    int slots = std::max(1, std::min(kGntMaxSlots, env_int("LSE_GNT_SLOTS", 3)));
    while (slots > 1 && gn_tma_smem(C, slots) > (size_t)dev.max_smem_optin) --slots;
    args.nslot = slots;
    char* sp = static_cast<char*>(scratch);
    args.partials = reinterpret_cast<float4*>(sp);
    sp += (size_t)N * G * sizeof(float4);
    args.done = reinterpret_cast<unsigned*>(sp);
    const size_t done_bytes = ((size_t)N * sizeof(unsigned) + 15) / 16 * 16;
    args.next = reinterpret_cast<unsigned long long*>(sp + done_bytes);
    args.status = dev.status;
    cudaError_t e = cudaMemsetAsync(args.done, 0, done_bytes + 16, stream);
    if (e != cudaSuccess) return e;
    const size_t smem = gn_tma_smem(C, slots);
    const int want = env_int("LSE_GNT_CTAS_PER_SM", 0);
    if (out_kind == 1) return gn_tma_go<1>(dev, args, smem, want, stream);
    if (out_kind == 2) return gn_tma_go<2>(dev, args, smem, want, stream);
    return gn_tma_go<0>(dev, args, smem, want, stream);
}

}  // namespace lse
