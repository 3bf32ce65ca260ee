// Shared device helpers for the stencilconv kernels (sm_103a).
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define SC_HD __host__ __device__ __forceinline__
#else
#define SC_HD inline
#endif

namespace sc {

// ---------------------------------------------------------------------------
// XOR swizzle of shared-memory chunks ("CUDA共有メモリのスウィズリング",
// section "スウィズリングの公式"): for an array whose rows are SW bytes
// (a power of two >= 32) split into equal chunks (16 bytes for the float4
// activation tiles, 4 bytes for the float transpose tile), chunk x of row y
// is stored at chunk (y XOR x) mod (chunks per row).  The element offset
// inside a chunk is kept.
//
// swz16(i, log2_chunks_per_row): physical 16-byte chunk index of logical
// chunk i in a linear array viewed as rows of 2^L chunks.  L = 3 is the
// 128-byte row used for the activation tiles.
// ---------------------------------------------------------------------------
SC_HD int swz16(int i, int log2_chunks_per_row)
{
    const int mask = (1 << log2_chunks_per_row) - 1;
    return (i & ~mask) | ((i ^ (i >> log2_chunks_per_row)) & mask);
}

// Same map on a [row][chunk] array with 2^L chunks per row: returns the
// physical chunk column of logical chunk `c` in row `row`.
SC_HD int swz_col(int row, int c, int log2_chunks_per_row)
{
    const int mask = (1 << log2_chunks_per_row) - 1;
    return (row ^ c) & mask;
}

// TMA swizzle of a staged pixel of c_sh fp32 channels (c_sh = 8, 16 or 32:
// 32-, 64- or 128-byte pixels, copied with the TMA swizzle of that span, in
// stage rows of a multiple of 8 pixels from a 1024-byte-aligned base): the
// copy XORs address bits 4.. with bits 7.., so 16-byte chunk q of pixel p is
// stored at chunk q ^ tma_swz_key(p, c_sh) of that pixel.
SC_HD int tma_swz_key(int p, int c_sh) { return (p * c_sh / 32) & (c_sh / 4 - 1); }

// Physical 16-byte chunk of logical chunk L of a staged input row of the
// tiled single-channel kernel (conv_c1.cu).  A thread's window starts 2
// chunks after its left neighbour's, so without a swizzle pixel lanes pl and
// pl + 4 of a quarter-warp read the same bank group.  Swapping the two
// chunks of each pair in every odd group of 8 ("CUDA共有メモリのスウィズリング":
// chunk x of row y at x XOR y, with y = bit 3 of L and x's lowest bit) puts
// the 8 pixel lanes' chunks in 8 distinct bank groups for every chunk of the
// window.  It only swaps chunks 2k and 2k + 1, so it is one-to-one on a row
// of an even number of chunks.
SC_HD int c1_band_chunk(int L) { return L ^ ((L >> 3) & 1); }

// conv_small.cu stages a tile row of 66 pixels x 4 16-byte chunks (16
// channels); lanes 8 c + q read pixel 8 q + k, so the eight pixel runs of
// a quarter-warp ask for chunks 32 apart, all in one bank group (chunk mod
// 8).  Chunk 4 p + cb is stored at (4 p + cb) XOR ((p / 8) mod 8): the XOR
// only touches the low 3 bits, so it permutes each aligned group of 8
// chunks (one pixel pair), and over q it adds q mod 8 to the bank group.
SC_HD int small_tile_chunk(int p, int cb) { return (4 * p + cb) ^ ((p >> 3) & 7); }

#if defined(__CUDACC__)

// ---------------------------------------------------------------------------
// cp.async (global -> shared, asynchronous, completion tracked per thread by
// commit groups).  src_bytes < size zero-fills the rest: used for halo
// pixels outside the image (zero "same" padding) with src_bytes = 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ float4 ldg_stream(const float4 *p)
{
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void stg_stream(float4 *p, float4 v)
{
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};\n" ::"l"(p), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ float relu_if(float v, int act) { return act ? fmaxf(v, 0.0f) : v; }

// ---------------------------------------------------------------------------
// mbarrier + TMA (cp.async.bulk.tensor) helpers.  Every wait is bounded in
// time: a wait that runs out returns false and the caller records
// SC_ERR_DEVICE_TIMEOUT in the device status word instead of spinning on.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Wait for phase `parity` of the barrier to complete, at most timeout_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long timeout_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > timeout_ns) return false;
    }
}

// As mbar_wait_bounded, for a thread with nothing else to do (a producer
// waiting for a stage to be released): between polls it sleeps about
// sleep_ns, so that its polling takes few issue slots from the warps that
// share its scheduler.
__device__ __forceinline__ bool mbar_wait_bounded_idle(uint32_t bar, uint32_t parity,
                                                       unsigned long long timeout_ns, unsigned sleep_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > timeout_ns) return false;
    }
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// 4-D tiled TMA load of the tensor map's box at (c0, c1, c2, c3) into shared
// memory; completion is signalled on the mbarrier as transaction bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, int c0, int c1, int c2, int c3,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::
            "r"(dst),
        "l"(reinterpret_cast<unsigned long long>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Contiguous bulk copy (cp.async.bulk) of `bytes` (a multiple of 16; both
// addresses 16-byte aligned) from global to shared memory, signalled on the
// mbarrier as transaction bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// 2-D tiled TMA load of the tensor map's box at (x, y) into shared memory;
// completion is signalled on the mbarrier as transaction bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::
            "r"(dst),
        "l"(reinterpret_cast<unsigned long long>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 4-D tiled TMA store of a shared-memory box to the tensor map's box at
// (c0, c1, c2, c3); elements outside the tensor are not written.  The store
// joins this thread's current bulk group (see bulk_commit / bulk_wait_*).
// The coordinates must not be negative.
__device__ __forceinline__ void tma_store_4d(const void *tmap, uint32_t src, int c0, int c1, int c2, int c3)
{
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];\n" ::"l"(
                     reinterpret_cast<unsigned long long>(tmap)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
                 : "memory");
}

// 5-D tiled TMA store, as tma_store_4d.
__device__ __forceinline__ void tma_store_5d(const void *tmap, uint32_t src, int c0, int c1, int c2, int c3, int c4)
{
    asm volatile("cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4, %5}], [%6];\n" ::"l"(
                     reinterpret_cast<unsigned long long>(tmap)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;\n" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

#endif  // __CUDACC__

}  // namespace sc
