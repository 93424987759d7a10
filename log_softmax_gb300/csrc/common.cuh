// Device helpers shared by the logsumexp kernels: the (max, sum) pair and its
// merge, NaN-propagating max, base-2 exponentials, and the PTX wrappers for
// clusters, mbarriers and bulk (TMA) copies used on sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

namespace lse {

// log2(e) and ln(2): exp(v) = 2^(v * log2(e)).
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Value written to the device status word when a bounded wait gives up.
constexpr int kStatusTimeout = 7;

// ---------------------------------------------------------------- arithmetic

// max that returns NaN when either operand is NaN (fmaxf would drop it).
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// 2^t on the special-function unit; ex2(-inf) = +0, subnormal results flush to 0.
__device__ __forceinline__ float ex2(float t) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// The running pair of the online formulation: m is the largest value seen
// (natural units), s = sum of exp(v - m) over the values seen.  The empty set
// is (-inf, 0).
struct MS {
    float m;
    float s;
};

__device__ __forceinline__ MS ms_empty() { return MS{-CUDART_INF_F, 0.f}; }

// Pairwise merge: m = max(m1, m2), s = s1 * e^(m1 - m) + s2 * e^(m2 - m).
// An empty side contributes 0; NaN and +inf in m carry through (see ms_lse).
__device__ __forceinline__ MS ms_merge(MS a, MS b) {
    float m = max_nan(a.m, b.m);
    if (m == -CUDART_INF_F) return ms_empty();
    float fa = (a.m == -CUDART_INF_F) ? 0.f : ((a.m == m) ? 1.f : ex2((a.m - m) * kLog2e));
    float fb = (b.m == -CUDART_INF_F) ? 0.f : ((b.m == m) ? 1.f : ex2((b.m - m) * kLog2e));
    return MS{m, fmaf(a.s, fa, b.s * fb)};
}

// Folds K values into the running pair: one rescale for the batch, then one
// exponential per value.  v may hold -inf (it contributes 0) and NaN (it makes
// m NaN).
template <int K>
__device__ __forceinline__ float max_nan_tree(const float (&v)[K]) {
    float t[K];
#pragma unroll
    for (int k = 0; k < K; ++k) t[k] = v[k];
#pragma unroll
    for (int w = 1; w < K; w *= 2)
#pragma unroll
        for (int k = 0; k + w < K; k += 2 * w) t[k] = max_nan(t[k], t[k + w]);
    return t[0];
}

template <int K>
__device__ __forceinline__ void ms_fold(MS& st, const float (&v)[K]) {
    const float cm = max_nan_tree(v);
    float mn = max_nan(st.m, cm);
    if (mn != st.m) {  // also taken once m is NaN; s is NaN from then on anyway
        float f = (st.m == -CUDART_INF_F) ? 0.f : ex2((st.m - mn) * kLog2e);
        st.s *= f;
        st.m = mn;
    }
    // exp(v - m) = 2^((v - m) * log2 e).  The difference is taken first: it is exact
    // for v near m, whereas folding m into an fma shift would carry the rounding
    // error of m * log2 e (about 1e23 when |m| = 1e30).  An all -inf pair uses
    // base 0, so -inf - 0 = -inf contributes 0.
    const float base = (st.m == -CUDART_INF_F) ? 0.f : st.m;
    float acc0 = 0.f, acc1 = 0.f;  // two chains for more instructions in flight
#pragma unroll
    for (int k = 0; k < K; k += 2) {
        acc0 += ex2((v[k] - base) * kLog2e);
        if (k + 1 < K) acc1 += ex2((v[k + 1] - base) * kLog2e);
    }
    st.s += acc0 + acc1;
}

// Output of a row transform for one element: x - lse (log_softmax) or
// exp(x - lse) (softmax, as 2^((x - lse) log2 e); -inf gives 0, and the NaN
// cases of x - lse stay NaN).
template <bool SOFTMAX>
__device__ __forceinline__ float row_out(float v, float lse) {
    if constexpr (SOFTMAX) return ex2((v - lse) * kLog2e);
    return v - lse;
}

__device__ __forceinline__ float4 row_out4(float4 q, float lse, bool softmax) {
    if (softmax)
        return make_float4(row_out<true>(q.x, lse), row_out<true>(q.y, lse), row_out<true>(q.z, lse),
                           row_out<true>(q.w, lse));
    return make_float4(q.x - lse, q.y - lse, q.z - lse, q.w - lse);
}

// lse from the final pair, with the special-value rules: NaN, then +inf, then
// the empty / all -inf set gives -inf.
__device__ __forceinline__ float ms_lse(MS st) {
    if (isnan(st.m)) return CUDART_NAN_F;
    if (st.m == CUDART_INF_F) return CUDART_INF_F;
    if (st.m == -CUDART_INF_F) return -CUDART_INF_F;
    return st.m + logf(st.s);
}

// Rescale factor that brings a pair with max m to the reference max mr >= m:
// e^(m - mr); an empty pair (m = -inf) contributes 0.
__device__ __forceinline__ float ms_scale_to(float m, float mr) {
    return (m == -CUDART_INF_F) ? 0.f : ((m == mr) ? 1.f : ex2((m - mr) * kLog2e));
}

__device__ __forceinline__ float warp_allmax_nan(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Warp-wide merge, every lane ends with the result: the max first, then each
// lane rescales its sum once, then a plain sum (one exponential per lane
// instead of two per butterfly step).
__device__ __forceinline__ MS ms_warp_allreduce(MS st) {
    const float m = warp_allmax_nan(st.m);
    const float s = warp_allsum(st.s * ms_scale_to(st.m, m));
    return MS{m, s};
}

// Block-wide merge; every thread gets the result.  `scratch` holds >= 32 MS.
// Must be called by all threads of the block.
__device__ __forceinline__ MS ms_block_allreduce(MS st, MS* scratch) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    st = ms_warp_allreduce(st);
    __syncthreads();  // scratch may still be read from a previous call
    if (lane == 0) scratch[warp] = st;
    __syncthreads();
    MS r = (lane < nwarps) ? scratch[lane] : ms_empty();
    return ms_warp_allreduce(r);
}

// ---------------------------------------------------------------- memory

__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_stream_f1(const float* p) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// L2 eviction policies for loads: keep a line for a re-read soon after, or let
// it go first.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ float4 ld_f4_l2hint(const float* p, uint64_t policy) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ float ld_f1_l2hint(const float* p, uint64_t policy) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ void st_stream_f4(float* p, float4 v) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};"
                 :
                 : "l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_stream_f1(float* p, float v) {
    asm volatile("st.global.cs.f32 [%0], %1;" : : "l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t nclusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster; release/acquire orders shared memory
// writes before the barrier with peer reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Reads an MS pair from the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ MS ld_peer_ms(const MS* local_addr, uint32_t rank) {
    uint32_t a = smem_u32(local_addr), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    MS r;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(r.m), "=f"(r.s) : "r"(ra) : "memory");
    return r;
}

// ---------------------------------------------------------------- gpu-scope flags

__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A pair packed into one 64-bit word for a single-copy-atomic hand-over through
// global memory: low half the max, high half the sum with its lowest bit
// replaced by a 1-bit tag (relative change of the sum <= 2^-23; when the max is
// not finite the sum is not used).
__device__ __forceinline__ unsigned long long ms_pack_tagged(MS v, uint32_t tag) {
    const uint32_t sb = (__float_as_uint(v.s) & ~1u) | (tag & 1u);
    return ((unsigned long long)sb << 32) | __float_as_uint(v.m);
}

__device__ __forceinline__ uint32_t ms_tag_of(unsigned long long w) { return (uint32_t)(w >> 32) & 1u; }

__device__ __forceinline__ MS ms_unpack(unsigned long long w) {
    return MS{__uint_as_float((uint32_t)w), __uint_as_float((uint32_t)(w >> 32))};
}

__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_ms(MS* p, MS v) {
    asm volatile("st.relaxed.gpu.global.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(v.m), "f"(v.s) : "memory");
}

__device__ __forceinline__ MS ld_relaxed_gpu_ms(const MS* p) {
    MS v;
    asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];" : "=f"(v.m), "=f"(v.s) : "l"(p) : "memory");
    return v;
}

// ---------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier among `count` threads (a multiple of 32) of the CTA on hardware
// barrier `id` (1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for phase `parity` of `bar` to complete, for at most ~1 s (and at most
// 2^26 polls).  On timeout it records kStatusTimeout in the device status word
// `status`, sets `aborted` and returns false; once `aborted` is set it returns
// at once.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, bool& aborted,
                                                  int* status) {
    if (aborted) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && globaltimer_ns() - t0 > 1000000000ull) break;
    }
    aborted = true;
    atomicExch(status, kStatusTimeout);
    return false;
}

// Bulk copy (TMA, non-tensor) of `bytes` from this CTA's shared memory to
// global memory, tracked by the issuing thread's bulk async-groups.  Addresses
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until all of this thread's bulk groups are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bulk copy (TMA, non-tensor) of `bytes` from global to this CTA's shared
// memory, completing on `bar` by transaction count.  Addresses 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// bulk_g2s with an L2 eviction `policy` (createpolicy) for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

}  // namespace lse
