// tcgen05 building blocks shared by the tensor-core convolution kernels
// (conv_tc.cu, conv_tc_fused.cu): operand kinds, shared-memory matrix and
// instruction descriptors, MMA / commit / tensor-memory wrappers, the
// epilogue's swizzle key, and the in-CTA rearrangement of OIHW filters into
// the B operand layout.  See conv_tc.cu for the GEMM formulation.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace sc {

namespace tc {

constexpr int NTHREADS = 320;   // warps 4 producer, 5 MMA; 0-3 and 6-9 epilogue (two sets, TMEM lane quadrant = warp % 4)
constexpr int WP = 32;          // padded row pitch (pixels) = lanes of a warp
constexpr int TC = 30;          // output columns per tile
constexpr int CH = 32;          // channels per stage (one swizzled row per pixel)

// Operand kinds.  Either way a K step (one MMA's K) is 32 bytes of a pixel's
// channels and one 16-byte chunk of a B row holds CU = KC / 2 channels.  A
// 32-channel stage is SUB sub-buffers, each filled by one TMA box, with one
// ROWB-byte swizzled row per padded pixel.  With the row width equal to the
// swizzle span (128-byte rows with 128-byte swizzling, 64-byte rows with
// 64-byte swizzling), the tensor core's read of a 32-byte K slice of 8
// consecutive rows touches every 16-byte bank group exactly twice (no
// conflicts; tests/test_kernel_swizzle.py checks each layout).
//  * OpTF32: fp32 activations, TF32 MMA (kind::tf32), K step = 8 channels;
//    one 128-byte row of 32 channels per pixel (4 K steps per row).
//  * OpBF16: bf16 activations, BF16 MMA (kind::f16), K step = 16 channels;
//    one 64-byte row of 32 channels per pixel (2 K steps per row; two
//    32-byte-row sub-buffers, one TMA box each, took 37.1 against 36.1 us on
//    the 32 -> 32 layer, with the same results).  The fp32 filters are
//    rounded to bf16 (to nearest even) when the CTA stages them.
//  * OpTF32x3: OpTF32's layout with every operand split into a TF32 head and
//    a remainder, v = hi(v) + lo(v), hi(v) = v with its 13 low mantissa bits
//    cleared (exactly a TF32 value), lo(v) = v - hi(v) (exact in fp32, at most
//    2^-10 |v|).  Each product is x_hi w_hi + (x_hi w_lo + x_lo w_hi): the
//    dropped x_lo w_lo is below 2^-20 |x w|, and the remainders lose at most
//    2^-10 of themselves to the TF32 conversion, so every product is within
//    ~3 * 2^-20 of exact ("split" or "3xTF32" tensor-core arithmetic, as in
//    Ootomo and Yokota, "Recovering single precision accuracy from Tensor
//    Cores while surpassing the FP32 theoretical peak performance", 2022).
//    The head products and the two correction products go to separate
//    accumulators, added once in the epilogue, so the small corrections are
//    not rounded against the large running sum.  The filter bank stacks
//    heads and remainders in N, so x_hi [w_hi | w_lo] is one MMA of twice
//    the width (head and first correction side by side in tensor memory)
//    and x_lo w_hi a second one into the correction columns.  The MMA
//    itself drops an fp32 operand's 13 low mantissa bits (truncation), so
//    the activations' heads are the copied values as they are; only their
//    remainders are written.
struct OpTF32 {
    static constexpr int ESZ = 4, KC = 8, ROWB = 128, SUB = 1;
    static constexpr uint32_t A_LAYOUT = 2, FMT = 2;   // descriptor layout 128B swizzle; TF32
    static constexpr bool X3 = false;
};
struct OpBF16 {
    static constexpr int ESZ = 2, KC = 16, ROWB = 64, SUB = 1;
    static constexpr uint32_t A_LAYOUT = 4, FMT = 1;   // descriptor layout 64B swizzle; BF16
    static constexpr bool X3 = false;
};
struct OpTF32x3 {
    static constexpr int ESZ = 4, KC = 8, ROWB = 128, SUB = 1;
    static constexpr uint32_t A_LAYOUT = 2, FMT = 2;
    static constexpr bool X3 = true;
};

// The TF32 head of an fp32 value (13 low mantissa bits cleared) and the
// remainder v - head, both as raw bits.
__device__ __forceinline__ uint32_t tf32_head(uint32_t v) { return v & 0xFFFFE000u; }
__device__ __forceinline__ uint32_t tf32_rest(uint32_t v)
{
    return __float_as_uint(__fsub_rn(__uint_as_float(v), __uint_as_float(tf32_head(v))));
}

// Instruction descriptor: D = F32, A = B = FMT (TF32 2, BF16 1), both
// K-major, dense, M = 128.
__host__ __device__ constexpr uint32_t idesc_mma(uint32_t fmt, int n)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) | ((128u >> 4) << 24);
}

// Shared-memory matrix descriptors as two 32-bit words: low = start address
// (16-byte units, bits 0-13) | LBO (16-byte units) << 16; high = SBO
// (16-byte units) | version 1 << 14 | layout type << 29 (bits 61-63 of the
// descriptor; 0 = no swizzle, 2 = 128-byte swizzle); base offset 0.  Shared
// addresses stay below 2^18, so stepping a start address is one 32-bit add
// that cannot carry into the LBO field.
template <class OP>
__host__ __device__ constexpr uint32_t a_hi() { return ((8u * OP::ROWB) >> 4) | (1u << 14) | (OP::A_LAYOUT << 29); }   // SBO = 8 rows
constexpr uint32_t B_HI = (128u >> 4) | (1u << 14);

template <class OP>
__device__ __forceinline__ void mma_w(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                      uint32_t idesc, uint32_t acc)
{
    if constexpr (OP::FMT == 2) {
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            ".reg .b64 da, db;\n"
            "setp.ne.b32 p, %6, 0;\n"
            "mov.b64 da, {%1, %2};\n"
            "mov.b64 db, {%3, %4};\n"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], da, db, %5, p;\n"
            "}\n" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc)
            : "memory");
    } else {
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            ".reg .b64 da, db;\n"
            "setp.ne.b32 p, %6, 0;\n"
            "mov.b64 da, {%1, %2};\n"
            "mov.b64 db, {%3, %4};\n"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n"
            "}\n" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc)
            : "memory");
    }
}

// Two floats -> two bf16 (round to nearest even), `lo` at the lower address.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// CW consecutive fp32 TMEM columns (4, 8, 16 or 32) of this thread's lane;
// the caller waits with tmem_wait_ld before using them.
template <int CW>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[CW])
{
    if constexpr (CW == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr));
    } else if constexpr (CW == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr));
    } else if constexpr (CW == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
              "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
              "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
              "=r"(r[30]), "=r"(r[31])
            : "r"(taddr));
    }
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Swizzle key of pixel row p of an epilogue output buffer (rows of ROWB =
// 128 or 64 bytes, 1024-byte aligned): 16-byte chunk q of row p is stored at
// chunk q ^ key(p).  This is the TMA's own 128-byte or 64-byte swizzle
// pattern, so the buffer is a valid source for a swizzled TMA store, and the
// row-wise writes (one row per lane) of every 8-lane phase touch 8 distinct
// 16-byte bank groups.
template <int ROWB>
__device__ __forceinline__ int stg_key(int p)
{
    return ROWB == 128 ? (p & 7) : ((p >> 1) & 3);
}


// Rearrange one CTA's staged OIHW filters into the MMA's B layout: the
// [k][r][cb][n][CU] bank whose element (k, r, cb, n, j) with n = s * CG + co
// is w[co0 + co][KC k + CU cb + j][r - (3 - R) / 2][s - (3 - S) / 2] (as TF32
// or rounded to bf16), zero for n >= 3 * CG, taps the R x S filter lacks,
// channels beyond Cin and co >= co_n.  raw holds output channel co's
// Cin * R * S floats at raw + co * raw_pitch * 4 (raw_pitch: an odd number of
// 16-byte units, so that the 16-byte reads below are free of bank conflicts).
// One unit is one output channel and one block of CU input channels (one
// 16-byte chunk); neighbouring threads take neighbouring output channels,
// whose B rows are neighbours.  Threads lt = 0 .. LT-1 share the work.
// OP::X3: each (k, r, cb) block has 2 NB rows, the TF32 heads in rows
// [0, NB) and the remainders in rows [NB, 2 NB), so that one MMA of
// N = 2 NB multiplies A by both.
template <int CG, class OP>
__device__ __forceinline__ void stage_filter_bank(const float *raw, uint4 *bank, int raw_pitch, int co_n, int Cin, int R,
                                                  int S, int nk, int lt, int LT)
{
    constexpr int NB = (3 * CG + 15) / 16 * 16;
    constexpr int RB = OP::X3 ? 2 * NB : NB;   // rows per (k, r, cb) block
    constexpr int CU = OP::KC / 2;
    const int RS = R * S;
    const int units = CG * 2 * nk;
    for (int u = lt; u < units; u += LT) {
        const int co = u % CG, cib = u / CG;
        const int k = cib >> 1, cb = cib & 1, ci0 = CU * cib;
        const int nj = co < co_n ? (Cin - ci0 < CU ? Cin - ci0 : CU) : 0;   // real channels of this unit
        const float *src = raw + (size_t)co * raw_pitch * 4 + (size_t)ci0 * RS;   // [j][rr][ss]
        float f[CU * 9];   // [j][r][s] of the 3 x 3 taps
        if (R == 3 && S == 3 && nj == CU) {
#pragma unroll
            for (int q = 0; q < CU * 9 / 4; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(src + 4 * q);
                f[4 * q] = v.x;
                f[4 * q + 1] = v.y;
                f[4 * q + 2] = v.z;
                f[4 * q + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < CU; ++j)
#pragma unroll
                for (int t = 0; t < 9; ++t) {
                    const int rr = t / 3 - (3 - R) / 2, ss = t % 3 - (3 - S) / 2;
                    f[j * 9 + t] = (j < nj && rr >= 0 && rr < R && ss >= 0 && ss < S) ? src[j * RS + rr * S + ss] : 0.f;
                }
        }
#pragma unroll
        for (int t = 0; t < 9; ++t) {
            const int r = t / 3, s = t % 3;
            uint4 o;
            const int at = ((k * 3 + r) * 2 + cb) * RB + s * CG + co;
            if constexpr (CU == 4) {
                o = make_uint4(__float_as_uint(f[t]), __float_as_uint(f[9 + t]), __float_as_uint(f[18 + t]),
                               __float_as_uint(f[27 + t]));
                if constexpr (OP::X3) {
                    bank[at + NB] = make_uint4(tf32_rest(o.x), tf32_rest(o.y), tf32_rest(o.z), tf32_rest(o.w));
                    o = make_uint4(tf32_head(o.x), tf32_head(o.y), tf32_head(o.z), tf32_head(o.w));
                }
            } else {
                o = make_uint4(pack_bf16(f[t], f[9 + t]), pack_bf16(f[18 + t], f[27 + t]), pack_bf16(f[36 + t], f[45 + t]),
                               pack_bf16(f[54 + t], f[63 + t]));
            }
            bank[at] = o;
        }
    }
    // B rows n >= 3 * CG (N rounded up to a multiple of 16) are zero
    constexpr int PADN = NB - 3 * CG;
    if constexpr (PADN > 0) {
        for (int e = lt; e < nk * 3 * 2 * PADN; e += LT) {
            bank[(e / PADN) * RB + 3 * CG + e % PADN] = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (OP::X3) bank[(e / PADN) * RB + NB + 3 * CG + e % PADN] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// The same rearrangement with all nine taps stacked in N: the [k][cb][n][CU]
// bank whose element (k, cb, n, j) with n = (3 r + s) * CG + co is
// w[co][KC k + CU cb + j][r][s] (3 x 3 filters), zero for n >= 9 * CG,
// channels beyond Cin and co >= co_n.  One MMA per K step then covers every
// tap; the taps' row shifts are summed by the epilogue.
template <int CG, class OP>
__device__ __forceinline__ void stage_filter_bank_taps_in_n(const float *raw, uint4 *bank, int raw_pitch, int co_n,
                                                            int Cin, int nk, int lt, int LT)
{
    constexpr int NB = (9 * CG + 15) / 16 * 16;
    constexpr int RB = OP::X3 ? 2 * NB : NB;   // rows per (k, cb) block (X3: heads, then remainders)
    constexpr int CU = OP::KC / 2;
    const int units = CG * 2 * nk;
    for (int u = lt; u < units; u += LT) {
        const int co = u % CG, cib = u / CG;
        const int k = cib >> 1, cb = cib & 1, ci0 = CU * cib;
        const int nj = co < co_n ? (Cin - ci0 < CU ? Cin - ci0 : CU) : 0;
        const float *src = raw + (size_t)co * raw_pitch * 4 + (size_t)ci0 * 9;   // [j][r][s]
        float f[CU * 9];
#pragma unroll
        for (int j = 0; j < CU; ++j)
#pragma unroll
            for (int t = 0; t < 9; ++t) f[j * 9 + t] = j < nj ? src[j * 9 + t] : 0.f;
#pragma unroll
        for (int t = 0; t < 9; ++t) {
            uint4 o;
            const int at = (k * 2 + cb) * RB + t * CG + co;
            if constexpr (CU == 4) {
                o = make_uint4(__float_as_uint(f[t]), __float_as_uint(f[9 + t]), __float_as_uint(f[18 + t]),
                               __float_as_uint(f[27 + t]));
                if constexpr (OP::X3) {
                    bank[at + NB] = make_uint4(tf32_rest(o.x), tf32_rest(o.y), tf32_rest(o.z), tf32_rest(o.w));
                    o = make_uint4(tf32_head(o.x), tf32_head(o.y), tf32_head(o.z), tf32_head(o.w));
                }
            } else {
                o = make_uint4(pack_bf16(f[t], f[9 + t]), pack_bf16(f[18 + t], f[27 + t]), pack_bf16(f[36 + t], f[45 + t]),
                               pack_bf16(f[54 + t], f[63 + t]));
            }
            bank[at] = o;
        }
    }
    constexpr int PADN = NB - 9 * CG;
    if constexpr (PADN > 0) {
        for (int e = lt; e < nk * 2 * PADN; e += LT) {
            bank[(e / PADN) * RB + 9 * CG + e % PADN] = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (OP::X3) bank[(e / PADN) * RB + NB + 9 * CG + e % PADN] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// Odd pitch, in 16-byte units, of one output channel's staged OIHW filters.
__host__ __device__ inline int filter_raw_pitch(int Cin, int RS) { return (Cin * RS / 4) | 1; }

}  // namespace tc

}  // namespace sc
