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

#endif  // __CUDACC__

}  // namespace sc
