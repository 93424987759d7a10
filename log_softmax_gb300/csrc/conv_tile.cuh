// One output tile of a 3x3, stride-1, valid convolution as an implicit GEMM on
// the 5th-generation tensor cores (tcgen05, kind::tf32), for the Conv2d that
// feeds the GroupNorm chain of the POPCORNBENCH page "Kimi-K2.6 / l2_p92"
// (8 -> 64 channels, kernel 3, no padding, bias).
//
// Tile: M = 128 consecutive output pixels of one sample (flattened oh * OW + ow)
// by N = Cout output channels, K = Cin * 9 patch taps (padded with zeros to a
// multiple of 8).  A (the im2col patches) and B (the weights) sit in shared
// memory in the canonical K-major layout without swizzle: 8-row x 16-byte core
// matrices, core matrices along M (or N) 128 bytes apart (stride byte offset)
// and along K one full column of core matrices apart (leading byte offset).
// The accumulator D (128 lanes x Cout fp32 columns) lives in tensor memory;
// lane m holds pixel m, column c channel c, so an epilogue thread owns every
// channel of one pixel.
//
// Precision: a tf32 operand keeps 10 mantissa bits.  For results at fp32
// accuracy every operand is split, a = hi + lo with hi = rn_tf32(a) and
// lo = rn_tf32(a - hi), and D = A_hi B_hi + A_hi B_lo + A_lo B_hi ("3xTF32";
// the dropped A_lo B_lo term is ~2^-22 relative).  A single A_hi B_hi pass,
// with round-to-nearest operands (unbiased errors), serves where only sums
// over many outputs are needed.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace lse {

constexpr int kConvTileM = 128;
constexpr int kConvMaxCin = 8;
constexpr int kConvMaxK = 72;  // kConvMaxCin * 9, already a multiple of 8

// K padded to a multiple of 8 (one tf32 MMA consumes K = 8).
__host__ __device__ constexpr int conv_kpad(int cin) { return (cin * 9 + 7) / 8 * 8; }

// Byte offset of element (row r, tap k) in a K-major operand with `rows` rows
// (a multiple of 8): core matrix (k / 4, r / 8), 8 rows of 16 bytes.
__host__ __device__ constexpr uint32_t conv_kmajor_off(int r, int k, int rows) {
    return (uint32_t)(((k >> 2) * (rows >> 3) + (r >> 3)) * 128 + (r & 7) * 16 + (k & 3) * 4);
}

__device__ __forceinline__ uint32_t rn_tf32(float f) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
    return r;
}

// Shared-memory matrix descriptor: start address, leading (K) and stride (M/N)
// byte offsets, descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of a dense kind::tf32 MMA: fp32 accumulator, tf32 A
// and B, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_tf32(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Whole warp: allocate `ncols` tensor-memory columns (a power of two >= 32);
// the base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Whole warp: 16 consecutive fp32 columns of this warp's 32 lanes (thread i
// gets lane 32*(warp%4) + i); completes at tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The weights w [Cout][Cin][3][3] as the B operand (N = Cout rows, K taps):
// hi and lo parts (lo only when `split`), zero beyond K.  Whole CTA.
__device__ __forceinline__ void conv_stage_weights(const float* __restrict__ w, int cin, int cout, unsigned char* bhi,
                                                   unsigned char* blo, bool split) {
    const int K = cin * 9, Kp = conv_kpad(cin);
    for (int e = threadIdx.x; e < cout * Kp; e += blockDim.x) {
        const int n = e / Kp, k = e - n * Kp;
        const float v = k < K ? w[n * K + k] : 0.f;
        const uint32_t hi = rn_tf32(v);
        const uint32_t off = conv_kmajor_off(n, k, cout);
        *reinterpret_cast<uint32_t*>(bhi + off) = hi;
        if (split) *reinterpret_cast<uint32_t*>(blo + off) = rn_tf32(v - __uint_as_float(hi));
    }
}

// Thread m (0..127) writes row m of the A operand (the patch of output pixel
// p = p0 + m of sample plane xs = x + n*CIN*H*W), hi and lo parts (lo only
// when `split`); pixels past the plane's end get zero rows.  All of the row's
// loads are issued before the first is used (one latency per tile).
template <int CIN>
__device__ __forceinline__ void conv_stage_patches(const float* __restrict__ xs, int H, int W, int OW, int64_t ohw,
                                                   int64_t p0, int m, unsigned char* ahi, unsigned char* alo,
                                                   bool split) {
    constexpr int K = CIN * 9, KP = conv_kpad(CIN);
    const int64_t p = p0 + m;
    const bool valid = p < ohw;
    const int oh = valid ? (int)(p / OW) : 0, ow = valid ? (int)(p - (int64_t)oh * OW) : 0;
    const float* base = xs + (int64_t)oh * W + ow;
    const int64_t plane = (int64_t)H * W;
    float v[KP];
#pragma unroll
    for (int k = 0; k < KP; ++k) {
        const int ci = k / 9, t = k - (k / 9) * 9, u = t / 3, vv = t - (t / 3) * 3;
        v[k] = (valid && k < K) ? __ldg(base + ci * plane + u * W + vv) : 0.f;
    }
#pragma unroll
    for (int k0 = 0; k0 < KP; k0 += 4) {
        uint4 hi;
        hi.x = rn_tf32(v[k0]); hi.y = rn_tf32(v[k0 + 1]); hi.z = rn_tf32(v[k0 + 2]); hi.w = rn_tf32(v[k0 + 3]);
        const uint32_t off = conv_kmajor_off(m, k0, kConvTileM);
        *reinterpret_cast<uint4*>(ahi + off) = hi;
        if (split) {
            uint4 lo;
            lo.x = rn_tf32(v[k0] - __uint_as_float(hi.x));
            lo.y = rn_tf32(v[k0 + 1] - __uint_as_float(hi.y));
            lo.z = rn_tf32(v[k0 + 2] - __uint_as_float(hi.z));
            lo.w = rn_tf32(v[k0 + 3] - __uint_as_float(hi.w));
            *reinterpret_cast<uint4*>(alo + off) = lo;
        }
    }
}

// One thread: the MMAs of a tile into D at d_tmem.  split: A_hi B_hi + A_hi B_lo
// + A_lo B_hi per K-step of 8; else A_hi B_hi.  Then a commit on `bar`.
__device__ __forceinline__ void conv_issue_mma(uint32_t d_tmem, const unsigned char* ahi, const unsigned char* alo,
                                               const unsigned char* bhi, const unsigned char* blo, int cin, int cout,
                                               bool split, uint64_t* bar) {
    const int Kp = conv_kpad(cin);
    const uint32_t idesc = umma_idesc_tf32(kConvTileM, cout);
    const uint32_t lbo_a = (kConvTileM / 8) * 128, lbo_b = (uint32_t)(cout / 8) * 128;
    const uint32_t sa_hi = smem_u32(ahi), sa_lo = smem_u32(alo), sb_hi = smem_u32(bhi), sb_lo = smem_u32(blo);
    for (int i = 0; i < Kp / 8; ++i) {
        const uint32_t oa = 2u * i * lbo_a, ob = 2u * i * lbo_b;
        umma_tf32(d_tmem, umma_desc(sa_hi + oa, lbo_a, 128), umma_desc(sb_hi + ob, lbo_b, 128), idesc, i > 0);
        if (split) {
            umma_tf32(d_tmem, umma_desc(sa_hi + oa, lbo_a, 128), umma_desc(sb_lo + ob, lbo_b, 128), idesc, 1);
            umma_tf32(d_tmem, umma_desc(sa_lo + oa, lbo_a, 128), umma_desc(sb_hi + ob, lbo_b, 128), idesc, 1);
        }
    }
    umma_commit(bar);
}

}  // namespace lse
