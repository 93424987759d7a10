// One output tile of a 3x3, stride-1, valid convolution as nine shifted GEMMs
// on the 5th-generation tensor cores (tcgen05, kind::tf32), for the Conv2d that
// feeds the GroupNorm chain of the POPCORNBENCH page "Kimi-K2.6 / l2_p92"
// (8 -> 64 channels, kernel 3, no padding, bias).
//
// Tiles run over "wide" pixels q = oh * W + ow with ow in [0, W) (the two
// columns per row past OW are computed and dropped), so that output pixel q
// reads input pixel q + u*W + v at tap (u, v).  A tile of M = 128 wide pixels
// therefore needs only the input window [q0, q0 + 128 + 2W + 2) of each of the
// Cin (padded to 8) channels, staged once in shared memory as two K-groups of 4
// channels: element (channel c, window pixel s) at (c / 4) * LBO + s * 16 +
// (c % 4) * 4.  That is the canonical K-major, no-swizzle operand layout (8
// pixels x 16 bytes per core matrix, core matrices 128 bytes apart along M and
// LBO apart along K), and the A operand of tap (u, v) is the same window with
// its start address moved by (u*W + v) * 16 bytes: D += A_(u,v) B_(u,v) with
// K = 8 per tap, nine taps per tile.  B_(u,v) = w[:, :, u, v] (Cout x 8) sits
// in the same layout, one block per tap.  The accumulator D (128 lanes x Cout
// fp32 columns) lives in tensor memory; lane m holds wide pixel q0 + m.
//
// Precision: a tf32 operand keeps 10 mantissa bits.  For results at fp32
// accuracy every operand is split, a = hi + lo with hi = rn_tf32(a) and
// lo = rn_tf32(a - hi), and D = A_hi B_hi + A_hi B_lo + A_lo B_hi ("3xTF32";
// the dropped A_lo B_lo term is ~2^-22 relative).  B_hi and B_lo of a tap are
// stacked along N; for Cout <= 64 the first two products are one MMA of
// N = 2 Cout into columns [0, 2 Cout) and A_lo B_hi a second of N = Cout into
// [0, Cout), the epilogue adding the two halves (A_hi is read once per tap).
// Wider layers keep three MMAs of N = Cout into one accumulator, whose Cout
// columns leave room for more tile slots in tensor memory.
#pragma once

#include <algorithm>
#include <cstdint>

#include "common.cuh"

namespace lse {

constexpr int kConvTileM = 128;
constexpr int kConvMaxCin = 8;  // channels padded to 8: one tf32 MMA (K = 8) per tap
constexpr int kConvMaxW = 1024;

// Staged window length (pixels, a multiple of 8) for input width W.
__host__ __device__ constexpr int conv_window(int W) { return (kConvTileM + 2 * W + 2 + 7) / 8 * 8; }

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

// The weights w [Cout][Cin][3][3] as nine B operands, one per tap t = 3u + v,
// each 2 Cout rows (row co the hi part of output channel co, row Cout + co its
// lo part) by 8 channels: element (row r, channel c) of tap t at
// (2t + c / 4) * LBO_B + (r / 8) * 128 + (r % 8) * 16 + (c % 4) * 4 with
// LBO_B = 2 Cout / 8 * 128; zero for c >= cin.  Whole CTA.
__host__ __device__ constexpr uint32_t conv_lbo_b(int cout) { return (uint32_t)(2 * cout / 8) * 128; }

// Whether a tile's first two products run as one MMA of N = 2 Cout.
__host__ __device__ constexpr bool conv_stacked(int cout) { return cout <= 64; }

__device__ __forceinline__ void conv_stage_weights(const float* __restrict__ w, int cin, int cout,
                                                   unsigned char* b) {
    const uint32_t lbo = conv_lbo_b(cout);
    for (int e = threadIdx.x; e < cout * 9 * 8; e += blockDim.x) {
        const int co = e / 72, t = (e / 8) % 9, c = e % 8;
        const float v = c < cin ? w[(co * cin + c) * 9 + t] : 0.f;
        const uint32_t hi = rn_tf32(v);
        const uint32_t plane = (uint32_t)(2 * t + c / 4) * lbo + (c % 4) * 4;
        const int rlo = cout + co;
        *reinterpret_cast<uint32_t*>(b + plane + (uint32_t)(co / 8) * 128 + (co % 8) * 16) = hi;
        *reinterpret_cast<uint32_t*>(b + plane + (uint32_t)(rlo / 8) * 128 + (rlo % 8) * 16) =
            rn_tf32(v - __uint_as_float(hi));
    }
}

// The input window [q0, q0 + S) of one sample (planes xs[c * plane + q]) as
// the A operand, hi and lo parts; pixels past the plane and channels >= CIN are
// zero.  Threads t, t + nt, ... of the calling group each take one window pixel:
// CIN coalesced loads, then two 16-byte stores per part.
template <int CIN>
__device__ __forceinline__ void conv_stage_window(const float* __restrict__ xs, int64_t plane, int64_t q0, int S,
                                                  int t, int nt, unsigned char* ahi, unsigned char* alo) {
    const uint32_t lbo = (uint32_t)S * 16;
    for (int s = t; s < S; s += nt) {
        const int64_t q = q0 + s;
        const bool in = q < plane;
        float v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = (c < CIN && in) ? __ldg(xs + c * plane + q) : 0.f;
#pragma unroll
        for (int kg = 0; kg < 2; ++kg) {
            uint4 hi, lo;
            hi.x = rn_tf32(v[4 * kg + 0]); hi.y = rn_tf32(v[4 * kg + 1]);
            hi.z = rn_tf32(v[4 * kg + 2]); hi.w = rn_tf32(v[4 * kg + 3]);
            lo.x = rn_tf32(v[4 * kg + 0] - __uint_as_float(hi.x));
            lo.y = rn_tf32(v[4 * kg + 1] - __uint_as_float(hi.y));
            lo.z = rn_tf32(v[4 * kg + 2] - __uint_as_float(hi.z));
            lo.w = rn_tf32(v[4 * kg + 3] - __uint_as_float(hi.w));
            const uint32_t off = kg * lbo + (uint32_t)s * 16;
            *reinterpret_cast<uint4*>(ahi + off) = hi;
            *reinterpret_cast<uint4*>(alo + off) = lo;
        }
    }
}

// One thread: bulk copies (TMA) of the raw input window [q0, q0 + S) of CIN
// channel planes into raw[c][S] (the part inside the plane; the rest is never
// read), completing on `bar`.  Needs 16-byte aligned planes (x aligned,
// plane % 4 == 0) and q0 % 4 == 0.
template <int CIN>
__device__ __forceinline__ void conv_fetch_window(const float* __restrict__ xs, int64_t plane, int64_t q0, int S,
                                                  float* raw, uint64_t* bar) {
    const int64_t n = std::min<int64_t>(S, plane - q0);
    const uint32_t bytes = (uint32_t)n * 4u;
    mbar_arrive_expect_tx(bar, bytes * CIN);
#pragma unroll
    for (int c = 0; c < CIN; ++c) bulk_g2s(raw + (size_t)c * S, xs + c * plane + q0, bytes, bar);
}

// The raw window (raw[c][S], valid up to plane - q0) as the A operand, hi and
// lo parts, zero past the plane and for channels >= CIN.  Threads t, t + nt, ...
template <int CIN, bool SPLIT = true>
__device__ __forceinline__ void conv_split_window(const float* raw, int64_t plane, int64_t q0, int S, int t, int nt,
                                                  unsigned char* ahi, unsigned char* alo) {
    const uint32_t lbo = (uint32_t)S * 16;
    for (int s = t; s < S; s += nt) {
        const bool in = q0 + s < plane;
        float v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = (c < CIN && in) ? raw[c * S + s] : 0.f;
#pragma unroll
        for (int kg = 0; kg < 2; ++kg) {
            uint4 hi;
            hi.x = rn_tf32(v[4 * kg + 0]); hi.y = rn_tf32(v[4 * kg + 1]);
            hi.z = rn_tf32(v[4 * kg + 2]); hi.w = rn_tf32(v[4 * kg + 3]);
            const uint32_t off = kg * lbo + (uint32_t)s * 16;
            *reinterpret_cast<uint4*>(ahi + off) = hi;
            if constexpr (SPLIT) {
                uint4 lo;
                lo.x = rn_tf32(v[4 * kg + 0] - __uint_as_float(hi.x));
                lo.y = rn_tf32(v[4 * kg + 1] - __uint_as_float(hi.y));
                lo.z = rn_tf32(v[4 * kg + 2] - __uint_as_float(hi.z));
                lo.w = rn_tf32(v[4 * kg + 3] - __uint_as_float(hi.w));
                *reinterpret_cast<uint4*>(alo + off) = lo;
            }
        }
    }
}

// One thread: the MMAs of a tile into D at d_tmem, then a commit on `bar`.
// Without `split`, the hi parts alone (N = Cout).  With it, stacked: A_hi
// [B_hi; B_lo] (N = 2 Cout, columns [0, 2 Cout)) and A_lo B_hi (N = Cout,
// columns [0, Cout)); else A_hi B_hi, A_hi B_lo and A_lo B_hi, all N = Cout.
__device__ __forceinline__ void conv_issue_mma(uint32_t d_tmem, const unsigned char* ahi, const unsigned char* alo,
                                               const unsigned char* b, int W, int S, int cout, bool split,
                                               uint64_t* bar) {
    const bool stacked = split && conv_stacked(cout);
    const uint32_t idesc = umma_idesc_tf32(kConvTileM, cout), idesc2 = umma_idesc_tf32(kConvTileM, 2 * cout);
    const uint32_t lbo_a = (uint32_t)S * 16, lbo_b = conv_lbo_b(cout), lo_rows = (uint32_t)(cout / 8) * 128;
    const uint32_t sa_hi = smem_u32(ahi), sa_lo = smem_u32(alo), sb = smem_u32(b);
#pragma unroll
    for (int t = 0; t < 9; ++t) {
        const uint32_t oa = (uint32_t)((t / 3) * W + (t % 3)) * 16, ob = 2u * t * lbo_b;
        const uint64_t a_hi = umma_desc(sa_hi + oa, lbo_a, 128), b_hi = umma_desc(sb + ob, lbo_b, 128);
        umma_tf32(d_tmem, a_hi, b_hi, stacked ? idesc2 : idesc, t > 0);
        if (split) {
            if (!stacked) umma_tf32(d_tmem, a_hi, umma_desc(sb + ob + lo_rows, lbo_b, 128), idesc, 1);
            umma_tf32(d_tmem, umma_desc(sa_lo + oa, lbo_a, 128), b_hi, idesc, 1);
        }
    }
    umma_commit(bar);
}

// The tile MMAs with every descriptor but the window's built once: the nine B
// descriptors and the taps' window offsets stay in the issuing thread's registers, so a
// tile is 18 (stacked, Cout <= 64) or 27 MMAs with one add each.  An issue loop that
// rebuilds descriptors per MMA (several integer operations each, the tap's division by
// three) measured 1.5x to 3.5x slower on GB300 than the tensor pipe (56 clocks per MMA at
// M = 128, N = 128 / 64, K = 8).
struct ConvTileMma {
    uint64_t b[9];   // tap t: [B_hi; B_lo] (N = 2 Cout; its first Cout rows are B_hi)
    uint32_t oa[9];  // tap t's window offset, 16-byte units: (t / 3) W + t % 3
    uint32_t idesc, idesc2, lbo_a, lo16;
    bool stacked;

    __device__ __forceinline__ void init(const unsigned char* b_smem, int W, int S, int cout) {
        const uint32_t lbo_b = conv_lbo_b(cout), sb = smem_u32(b_smem);
#pragma unroll
        for (int t = 0; t < 9; ++t) {
            b[t] = umma_desc(sb + 2u * t * lbo_b, lbo_b, 128);
            oa[t] = (uint32_t)((t / 3) * W + (t % 3));
        }
        idesc = umma_idesc_tf32(kConvTileM, cout);
        idesc2 = umma_idesc_tf32(kConvTileM, 2 * cout);
        lbo_a = (uint32_t)S * 16;
        lo16 = (uint32_t)(cout / 8) * 128 / 16;  // B_lo's rows: the start field moved by Cout / 8 core matrices
        stacked = conv_stacked(cout);
    }
    // Stacked: A_hi [B_hi; B_lo] and A_lo B_hi of the nine taps into D at d_tmem; else
    // A_hi B_hi, A_hi B_lo and A_lo B_hi, all N = Cout (the windows' start fields plus an
    // offset: shared addresses stay below 2^18, no carry out of the field).
    __device__ __forceinline__ void issue(uint32_t d_tmem, const unsigned char* ahi, const unsigned char* alo) const {
        const uint64_t dh = umma_desc(smem_u32(ahi), lbo_a, 128), dl = umma_desc(smem_u32(alo), lbo_a, 128);
        if (stacked) {
#pragma unroll
            for (int t = 0; t < 9; ++t) {
                umma_tf32(d_tmem, dh + oa[t], b[t], idesc2, t > 0);
                umma_tf32(d_tmem, dl + oa[t], b[t], idesc, 1);
            }
        } else {
#pragma unroll
            for (int t = 0; t < 9; ++t) {
                umma_tf32(d_tmem, dh + oa[t], b[t], idesc, t > 0);
                umma_tf32(d_tmem, dh + oa[t], b[t] + lo16, idesc, 1);
                umma_tf32(d_tmem, dl + oa[t], b[t], idesc, 1);
            }
        }
    }
};

}  // namespace lse
