// Layout change between NCHW and NHWC as a batched 2-D transpose through a
// shared-memory tile ("Optimizing convolution kernels - CNNs in Vulkan
// Part 2/3", section "Vectorization": channels of a pixel stored
// contiguously; the staged transpose is the shared-memory tile method of
// the shared-memory bank-conflict page, with the XOR swizzle of
// "CUDA共有メモリのスウィズリング" in place of a padding column).
//
// dst[n][b][a] = src[n][a][b] for a < A, b < B.  A 32 x 32 tile is read
// with lanes along b (coalesced) and stored as logical element [a][b] at
// physical column (a XOR b) of row a; it is read back with lanes along a
// (logical column b of rows a = lane) and written coalesced.  With 32 floats
// per tile row (128 bytes, 4-byte chunks), both the row write and the
// swizzled column read put the 32 lanes in 32 different banks.
#include "common.cuh"
#include "launch.h"

namespace sc {

__global__ void __launch_bounds__(256)
    transpose_batched_kernel(const float *__restrict__ src, float *__restrict__ dst, long long A,
                             long long B, long long tiles_b)
{
    __shared__ float tile[32][32];
    const int tx = threadIdx.x & 31;
    const int ty = threadIdx.x >> 5;  // 0..7
    const long long n = blockIdx.y;
    const long long ta = blockIdx.x / tiles_b;
    const long long tb = blockIdx.x % tiles_b;
    const long long a0 = ta * 32, b0 = tb * 32;
    const float *s = src + n * A * B;
    float *d = dst + n * A * B;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int ra = ty + 8 * i;          // tile row = a offset
        const long long a = a0 + ra, b = b0 + tx;
        float v = 0.f;
        if (a < A && b < B) v = s[a * B + b];
        tile[ra][swz_col(ra, tx, 5)] = v;   // logical [ra][tx]
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int rb = ty + 8 * i;          // b offset
        const long long a = a0 + tx, b = b0 + rb;
        const float v = tile[tx][swz_col(tx, rb, 5)];  // logical [tx][rb]
        if (a < A && b < B) d[b * A + a] = v;
    }
}

// The same transpose with 16-byte accesses on both sides, for A % 4 == 0,
// B % 4 == 0 and 16-byte aligned pointers: a 32 (a) x 128 (b) tile, each
// thread reading four 4-element runs along b and writing four along a, so
// four times the bytes are in flight per load instruction (the scalar
// kernel above reaches about half the HBM bandwidth).  Shared layout:
// element [a][b] at row a, column b ^ (4 * (a / 4)) (an XOR on bits 2..4 of
// the column, "CUDA共有メモリのスウィズリング"): a row write of 16-byte
// runs stays one run per lane, and the column reads of the write-back (8
// lanes over a / 4, 4 over b) land in 32 distinct banks.
__global__ void __launch_bounds__(256)
    transpose_batched_v4_kernel(const float *__restrict__ src, float *__restrict__ dst, long long A, long long B,
                                long long tiles_b)
{
    __shared__ __align__(16) float tile[32][128];
    const int tid = threadIdx.x;
    const long long n = blockIdx.y;
    const long long a0 = (blockIdx.x / tiles_b) * 32, b0 = (blockIdx.x % tiles_b) * 128;
    const float *s = src + n * A * B;
    float *d = dst + n * A * B;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int ra = (tid >> 5) + 8 * i, cb = 4 * (tid & 31);   // tile row, first column
        const long long a = a0 + ra, b = b0 + cb;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a < A && b < B) v = ldg_stream(reinterpret_cast<const float4 *>(s + a * B + b));
        *reinterpret_cast<float4 *>(&tile[ra][cb ^ (4 * (ra >> 2))]) = v;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int qa = tid & 7, rb = (tid >> 3) + 32 * i;   // a run qa (4 a's), tile column rb
        const long long a = a0 + 4 * qa, b = b0 + rb;
        float4 v;
        v.x = tile[4 * qa + 0][rb ^ (4 * qa)];
        v.y = tile[4 * qa + 1][rb ^ (4 * qa)];
        v.z = tile[4 * qa + 2][rb ^ (4 * qa)];
        v.w = tile[4 * qa + 3][rb ^ (4 * qa)];
        if (a < A && b < B) stg_stream(reinterpret_cast<float4 *>(d + b * A + a), v);
    }
}

cudaError_t launch_transpose_batched(const float *src, float *dst, int N, long long A, long long B,
                                     cudaStream_t st)
{
    if ((A & 3) == 0 && (B & 3) == 0 && ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0) {
        const long long ta = (A + 31) / 32, tb = (B + 127) / 128;
        if (ta * tb > 0x7fffffffLL || N > 65535) return cudaErrorInvalidConfiguration;
        transpose_batched_v4_kernel<<<dim3((unsigned)(ta * tb), N), 256, 0, st>>>(src, dst, A, B, tb);
        return cudaGetLastError();
    }
    const long long ta = (A + 31) / 32, tb = (B + 31) / 32;
    if (ta * tb > 0x7fffffffLL || N > 65535) return cudaErrorInvalidConfiguration;
    transpose_batched_kernel<<<dim3((unsigned)(ta * tb), N), 256, 0, st>>>(src, dst, A, B, tb);
    return cudaGetLastError();
}

}  // namespace sc
