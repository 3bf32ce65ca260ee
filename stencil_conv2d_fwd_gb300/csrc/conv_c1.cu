// Special-case direct convolution: one input channel.
//
// Method: "Optimizing Memory Efficiency for Convolution Kernels on Kepler
// GPUs", Section 3.2 (special case) and Algorithm 1:
//  * a CTA owns a block of image columns and a band of rows; its threads
//    sweep the band downward one output row per step (Fig. 5a);
//  * vertical reuse lives in registers: each thread keeps the K input rows
//    its outputs need and loads one new row per step (Algorithm 1, lines
//    3-6);
//  * each thread computes n = 4 contiguous output pixels and reads them as
//    one 16-byte unit (Section 3.2.3, Fig. 5b: W_CD matched to W_SMB);
//  * every thread of a warp reads the same filter tap at the same time, so
//    filter reads are broadcasts (Section 3.2.2 puts them in constant
//    memory; here the CTA stages them once in shared memory, which gives
//    the same broadcast without a per-call constant-bank upload; a
//    constant-bank variant, one weight operand per FMA, measured 2x slower
//    on GB300).
// Groups of 32 output channels use a tiled form of the same sweep
// (conv_c1_tile_kernel below): the band's input rows are staged in shared
// memory once, and each thread computes 8 channels x 8 pixels.
// The FMAs run as packed dual-FP32 FMAs (__ffma2_rn) on pairs of output
// channels; each component rounds like fmaf.
// Horizontal sharing between neighbouring threads goes through warp
// shuffles instead of a shared-memory row: a lane's left and right halo
// pixels are the edge values its neighbour lanes already hold in registers;
// only the two outermost pixel lanes of a warp load their halo from global.
//
// Output channels: each thread computes F_T of them for its 4 pixels;
// CL lanes of a warp split a group of CL*F_T channels (F_T = 8: channels
// g*4*CL + 4*cl + e, g in {0,1}) so one warp store writes 4*CL contiguous
// NHWC channels of each of its pixels.  Filters of an R x S kernel sit centred in a
// K x K register window (K = max(R, S), zero taps around them).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace sc {

template <int K, int F_T, int CL_>
struct C1Cfg {
    static constexpr int CL = CL_;              // lanes along output channels
    static constexpr int PL = 32 / CL;          // pixel lanes per warp
    static constexpr int HALO = K / 2;
    static constexpr int WIN = 4 + K - 1;       // pixels a thread needs per row
    static constexpr int CO_CTA = F_T * CL;     // output channels per CTA
    static constexpr int NG = F_T >= 4 ? F_T / 4 : 1;
    static_assert(HALO <= 4, "halo must come from the adjacent lane");
};

// Raw loads of one input row for this thread (Algorithm 1's register
// prefetch): the 4 own pixels x0..x0+3 and, for the two outermost pixel
// lanes of the warp, their halo pixels.  Zero outside the image.
struct C1Raw {
    float own[4];
    float edge[4];  // halo pixels loaded from global (outermost lanes only)
};

__device__ __forceinline__ float ldg_nc_f32(const float *p)
{
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];\n" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ldg_nc_f32x4(const float *p)
{
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

template <class C>
__device__ __forceinline__ void c1_issue_row(C1Raw &raw, const float *__restrict__ xrow, bool row_ok,
                                             int x0, int W, bool vec, int pl)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) raw.own[j] = 0.f;
#pragma unroll
    for (int h = 0; h < 4; ++h) raw.edge[h] = 0.f;
    if (!row_ok) return;
    if (vec && x0 + 3 < W) {
        const float4 t = ldg_nc_f32x4(xrow + x0);
        raw.own[0] = t.x; raw.own[1] = t.y; raw.own[2] = t.z; raw.own[3] = t.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (x0 + j < W) raw.own[j] = ldg_nc_f32(xrow + x0 + j);
    }
    if (pl == 0) {
#pragma unroll
        for (int h = 0; h < C::HALO; ++h) {
            const int gx = x0 - C::HALO + h;
            if (gx >= 0 && gx < W) raw.edge[h] = ldg_nc_f32(xrow + gx);
        }
    } else if (pl == C::PL - 1) {
#pragma unroll
        for (int h = 0; h < C::HALO; ++h) {
            const int gx = x0 + 4 + h;
            if (gx < W) raw.edge[h] = ldg_nc_f32(xrow + gx);
        }
    }
}

// Window of one row: win[0..WIN) = x[row][x0 - HALO .. x0 + 3 + HALO].  The
// halo pixels are the neighbour lanes' own pixels, passed by shuffle.
template <class C>
__device__ __forceinline__ void c1_finish_row(float (&win)[C::WIN], const C1Raw &raw, int pl,
                                              int lane)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) win[C::HALO + j] = raw.own[j];
    if constexpr (C::HALO > 0) {
        const int left = lane - C::CL;    // neighbour lane to the left (same channels)
        const int right = lane + C::CL;
#pragma unroll
        for (int h = 0; h < C::HALO; ++h) {
            // left halo pixel x0 - HALO + h is the left neighbour's own[4 - HALO + h]
            const float l = __shfl_sync(0xffffffffu, raw.own[4 - C::HALO + h], left < 0 ? lane : left);
            // right halo pixel x0 + 4 + h is the right neighbour's own[h]
            const float r = __shfl_sync(0xffffffffu, raw.own[h], right > 31 ? lane : right);
            win[h] = pl == 0 ? raw.edge[h] : l;
            win[C::HALO + 4 + h] = pl == C::PL - 1 ? raw.edge[h] : r;
        }
    }
}

template <int K, int F_T, int CL>
__global__ void __launch_bounds__(256)
    conv_c1_kernel(const float *__restrict__ x, const float *__restrict__ w,
                   const float *__restrict__ bias, float *__restrict__ y, int N, int H, int W,
                   int Cout, int R, int S, int act, int rows_per_cta, int col_tiles, int vec)
{
    using C = C1Cfg<K, F_T, CL>;
    __shared__ __align__(16) float ws[K * K * C::CO_CTA];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int cl = lane % CL;
    const int pl = lane / CL;
    const int co0 = blockIdx.y * C::CO_CTA;
    const int n = blockIdx.z;
    const int ct = blockIdx.x % col_tiles;
    const int rt = blockIdx.x / col_tiles;
    const int x0 = (ct * nwarps + warp) * (C::PL * 4) + pl * 4;
    const int y0 = rt * rows_per_cta;
    const int y1 = min(H, y0 + rows_per_cta);

    // Stage the CTA's filters as [K*K taps][CO_CTA], centred, zero elsewhere.
    for (int e = tid; e < K * K * C::CO_CTA; e += blockDim.x) {
        const int col = e % C::CO_CTA;
        const int tap = e / C::CO_CTA;
        const int r = tap / K - (K - R) / 2;
        const int s = tap % K - (K - S) / 2;
        const int co = co0 + col;
        float v = 0.f;
        if (r >= 0 && r < R && s >= 0 && s < S && co < Cout) v = w[((long long)co * R + r) * S + s];
        ws[e] = v;
    }
    __syncthreads();

    // this thread's output channels (CTA-local), and their bias
    int col_of[F_T];
#pragma unroll
    for (int f = 0; f < F_T; ++f)
        col_of[f] = F_T >= 4 ? (f / 4) * (4 * CL) + 4 * cl + (f % 4) : cl * F_T + f;
    float bv[F_T];
#pragma unroll
    for (int f = 0; f < F_T; ++f) {
        const int co = co0 + col_of[f];
        bv[f] = (bias && co < Cout) ? bias[co] : 0.f;
    }

    const float *xn = x + (long long)n * H * W;
    float win[K][C::WIN];
    // prologue: rows y0 - HALO .. y0 + HALO - 1 into window rows 0 .. K-2
#pragma unroll
    for (int t = 0; t < K - 1; ++t) {
        const int yy = y0 - C::HALO + t;
        const bool ok = yy >= 0 && yy < H;
        C1Raw raw;
        c1_issue_row<C>(raw, xn + (long long)(ok ? yy : 0) * W, ok, x0, W, vec, pl);
        c1_finish_row<C>(win[t], raw, pl, lane);
    }

    for (int oy = y0; oy < y1; ++oy) {
        // prefetch the new bottom row (oy + HALO) into registers
        C1Raw raw;
        {
            const int yy = oy + C::HALO;
            const bool ok = yy < H;
            c1_issue_row<C>(raw, xn + (long long)(ok ? yy : 0) * W, ok, x0, W, vec, pl);
        }
        float acc[F_T][4];
#pragma unroll
        for (int f = 0; f < F_T; ++f)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[f][j] = 0.f;
        // kernel rows 0 .. K-2 use rows already in registers; the last
        // kernel row uses the prefetched row once its halo is exchanged
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            if (ky == K - 1) c1_finish_row<C>(win[ky], raw, pl, lane);
            // keep one kernel row of filter loads in flight at a time
            asm volatile("" ::: "memory");
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const float *wt = ws + (ky * K + kx) * C::CO_CTA;
                float wv[F_T];
                if constexpr (F_T >= 4) {
#pragma unroll
                    for (int g = 0; g < F_T / 4; ++g) {
                        const float4 t = *reinterpret_cast<const float4 *>(wt + g * 4 * CL + 4 * cl);
                        wv[4 * g + 0] = t.x;
                        wv[4 * g + 1] = t.y;
                        wv[4 * g + 2] = t.z;
                        wv[4 * g + 3] = t.w;
                    }
                } else {
#pragma unroll
                    for (int f = 0; f < F_T; ++f) wv[f] = wt[cl * F_T + f];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float v = win[ky][j + kx];
                    if constexpr (F_T % 2 == 0) {
                        // packed FP32 FMA on pairs of output channels
                        const float2 vv = make_float2(v, v);
#pragma unroll
                        for (int f = 0; f < F_T; f += 2) {
                            float2 a2 = make_float2(acc[f][j], acc[f + 1][j]);
                            a2 = __ffma2_rn(make_float2(wv[f], wv[f + 1]), vv, a2);
                            acc[f][j] = a2.x;
                            acc[f + 1][j] = a2.y;
                        }
                    } else {
#pragma unroll
                        for (int f = 0; f < F_T; ++f) acc[f][j] = fmaf(wv[f], v, acc[f][j]);
                    }
                }
            }
        }
        // epilogue
        float *yrow = y + ((long long)n * H + oy) * W * Cout;
        if constexpr (F_T >= 4) {
#pragma unroll
            for (int g = 0; g < F_T / 4; ++g) {
                const int co = co0 + g * 4 * CL + 4 * cl;
                if (co < Cout) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (x0 + j < W) {
                            float4 o;
                            o.x = relu_if(acc[4 * g + 0][j] + bv[4 * g + 0], act);
                            o.y = relu_if(acc[4 * g + 1][j] + bv[4 * g + 1], act);
                            o.z = relu_if(acc[4 * g + 2][j] + bv[4 * g + 2], act);
                            o.w = relu_if(acc[4 * g + 3][j] + bv[4 * g + 3], act);
                            *reinterpret_cast<float4 *>(yrow + (long long)(x0 + j) * Cout + co) = o;
                        }
                    }
                }
            }
        } else {
            // F_T == 1 (Cout == 1): four contiguous pixels of one channel
            if (co0 + cl < Cout) {
                float o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) o[j] = relu_if(acc[0][j] + bv[0], act);
                if (vec && x0 + 3 < W) {
                    *reinterpret_cast<float4 *>(yrow + x0) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (x0 + j < W) yrow[x0 + j] = o[j];
                }
            }
        }
        // slide the register window down one row
#pragma unroll
        for (int t = 0; t < K - 1; ++t)
#pragma unroll
            for (int j = 0; j < C::WIN; ++j) win[t][j] = win[t + 1][j];
    }
}

// The same computation for W % 4 == 0 and 16-byte aligned x and y (every
// thread's 4 pixels are all inside or all outside the image), without the
// per-row window shift: the K window rows live in a ring of registers, and
// the row loop is unrolled K times so that the ring slot of every window row
// is a compile-time constant (input row q of the band sits in slot q mod K).
// Each input row is fetched two output rows before its first use (the rows
// of all warps of an SM otherwise wait on the same fetch latency together).
// The accumulators start at the bias (the sum's first term instead of its
// last; the rounding stays within the FP32 bound), read from shared memory
// with the filters, and the stores need one in-image test per thread.
template <int K, int F_T, int CL>
__global__ void __launch_bounds__(256, (K >= 7 && F_T >= 8) ? 1 : 2)
    conv_c1_ring_kernel(const float *__restrict__ x, const float *__restrict__ w,
                        const float *__restrict__ bias, float *__restrict__ y, int N, int H, int W,
                        int Cout, int R, int S, int act, int rows_per_cta, int col_tiles)
{
    using C = C1Cfg<K, F_T, CL>;
    __shared__ __align__(16) float ws[K * K * C::CO_CTA];
    __shared__ __align__(16) float bs[C::CO_CTA];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int cl = lane % CL;
    const int pl = lane / CL;
    const int co0 = blockIdx.y * C::CO_CTA;
    const int n = blockIdx.z;
    const int ct = blockIdx.x % col_tiles;
    const int rt = blockIdx.x / col_tiles;
    const int x0 = (ct * nwarps + warp) * (C::PL * 4) + pl * 4;
    const int y0 = rt * rows_per_cta;
    const int y1 = min(H, y0 + rows_per_cta);
    const bool px_ok = x0 < W;   // W % 4 == 0: all 4 pixels or none

    for (int e = tid; e < K * K * C::CO_CTA; e += blockDim.x) {
        const int col = e % C::CO_CTA;
        const int tap = e / C::CO_CTA;
        const int r = tap / K - (K - R) / 2;
        const int s = tap % K - (K - S) / 2;
        const int co = co0 + col;
        float v = 0.f;
        if (r >= 0 && r < R && s >= 0 && s < S && co < Cout) v = w[((long long)co * R + r) * S + s];
        ws[e] = v;
    }
    for (int e = tid; e < C::CO_CTA; e += blockDim.x) bs[e] = (bias && co0 + e < Cout) ? bias[co0 + e] : 0.f;
    __syncthreads();

    const float *xn = x + (long long)n * H * W;
    auto issue = [&](C1Raw &raw, int yy) {   // image row yy (zeros outside the image)
        const bool ok = yy >= 0 && yy < H;
        c1_issue_row<C>(raw, xn + (long long)(ok ? yy : 0) * W, ok, x0, W, true, pl);
    };
    float win[K][C::WIN];
    // prologue: band rows q = 0 .. K - 2 (image rows y0 - HALO + q) into
    // slots q, all fetches in flight together; row K - 1 stays in flight
    C1Raw raw_c;   // band row i + K - 1, fetched during row i - 1
    {
        C1Raw pro[K > 1 ? K - 1 : 1];
#pragma unroll
        for (int t = 0; t < K - 1; ++t) issue(pro[t], y0 - C::HALO + t);
        issue(raw_c, y0 + C::HALO);
#pragma unroll
        for (int t = 0; t < K - 1; ++t) c1_finish_row<C>(win[t], pro[t], pl, lane);
    }

    const int nrows = y1 - y0;
    for (int m = 0; m < nrows; m += K) {
#pragma unroll
        for (int u = 0; u < K; ++u) {
            const int i = m + u;
            if (i < nrows) {   // the same for the whole CTA
            // one output row at a time: keeps the unrolled rows from
            // overlapping (their registers would not fit)
            asm volatile("" ::: "memory");
            const int oy = y0 + i;
            C1Raw raw_n;   // band row i + K (image row oy + HALO + 1)
            issue(raw_n, oy + C::HALO + 1);
            float acc[F_T][4];
            if constexpr (F_T >= 4) {
#pragma unroll
                for (int g = 0; g < F_T / 4; ++g) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(bs + g * 4 * CL + 4 * cl);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[4 * g + 0][j] = b4.x;
                        acc[4 * g + 1][j] = b4.y;
                        acc[4 * g + 2][j] = b4.z;
                        acc[4 * g + 3][j] = b4.w;
                    }
                }
            } else {
#pragma unroll
                for (int f = 0; f < F_T; ++f)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[f][j] = bs[cl * F_T + f];
            }
#pragma unroll
            for (int ky = 0; ky < K; ++ky) {
                float(&wr)[C::WIN] = win[(u + ky) % K];   // band row i + ky
                if (ky == K - 1) c1_finish_row<C>(wr, raw_c, pl, lane);
                asm volatile("" ::: "memory");
#pragma unroll
                for (int kx = 0; kx < K; ++kx) {
                    const float *wt = ws + (ky * K + kx) * C::CO_CTA;
                    float wv[F_T];
                    if constexpr (F_T >= 4) {
#pragma unroll
                        for (int g = 0; g < F_T / 4; ++g) {
                            const float4 t = *reinterpret_cast<const float4 *>(wt + g * 4 * CL + 4 * cl);
                            wv[4 * g + 0] = t.x;
                            wv[4 * g + 1] = t.y;
                            wv[4 * g + 2] = t.z;
                            wv[4 * g + 3] = t.w;
                        }
                    } else {
#pragma unroll
                        for (int f = 0; f < F_T; ++f) wv[f] = wt[cl * F_T + f];
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float v = wr[j + kx];
                        if constexpr (F_T % 2 == 0) {
                            const float2 vv = make_float2(v, v);
#pragma unroll
                            for (int f = 0; f < F_T; f += 2) {
                                float2 a2 = make_float2(acc[f][j], acc[f + 1][j]);
                                a2 = __ffma2_rn(make_float2(wv[f], wv[f + 1]), vv, a2);
                                acc[f][j] = a2.x;
                                acc[f + 1][j] = a2.y;
                            }
                        } else {
#pragma unroll
                            for (int f = 0; f < F_T; ++f) acc[f][j] = fmaf(wv[f], v, acc[f][j]);
                        }
                    }
                }
            }
            raw_c = raw_n;
            if (px_ok) {
                float *yrow = y + ((long long)n * H + oy) * W * Cout;
                if constexpr (F_T >= 4) {
#pragma unroll
                    for (int g = 0; g < F_T / 4; ++g) {
                        const int co = co0 + g * 4 * CL + 4 * cl;
                        if (co < Cout) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                float4 o;
                                o.x = relu_if(acc[4 * g + 0][j], act);
                                o.y = relu_if(acc[4 * g + 1][j], act);
                                o.z = relu_if(acc[4 * g + 2][j], act);
                                o.w = relu_if(acc[4 * g + 3][j], act);
                                *reinterpret_cast<float4 *>(yrow + (long long)(x0 + j) * Cout + co) = o;
                            }
                        }
                    }
                } else if (co0 + cl < Cout) {
                    // F_T == 1 (Cout == 1): four contiguous pixels of one channel
                    *reinterpret_cast<float4 *>(yrow + x0) =
                        make_float4(relu_if(acc[0][0], act), relu_if(acc[0][1], act), relu_if(acc[0][2], act),
                                    relu_if(acc[0][3], act));
                }
            }
            }
        }
    }
}

// The driver's tensor-map encoder (conv_tma_k3.cu), or nullptr.
PFN_cuTensorMapEncodeTiled_v12000 conv_tma_encoder();



// Tiled variant for groups of 32 output channels (F_T = 8, CL = 4), W % 4
// == 0 and 16-byte aligned x and y.  A CTA of four warps owns 256 image
// columns and a band of rows; it stages the band's input rows (plus the
// vertical halo) in shared memory once, then each thread computes 8 output
// channels x 8 contiguous pixels of one row at a time (32 accumulator pairs),
// reading the K rows of its window from the staged tile (four 16-byte loads
// a row) instead of keeping a K-row ring in registers.  The FMA order is the
// ring kernel's (bias first, then the taps row by row), so both give the
// same bits.  Each warp stores its output row (64 pixels x 32 channels)
// through a swizzled shared-memory buffer with one TMA copy; one buffer per
// warp suffices (a row's arithmetic takes far longer than its copy's read of
// the buffer), so four CTAs fit per SM.  Measured against the ring kernel
// (1 -> 32, 5 x 5 on 1280 x 720): 38.6 -> 34.4 us (33.4 us with the
// staggered buffer writes below); with two buffers and two CTAs per SM
// 36.0 us, three CTAs 35.4 us; CTAs of 2 warps at 8 per SM 34.5 us, of 8
// warps at 2 per SM 40.8 us.
constexpr int kC1TileWarps = 4;
constexpr int kC1TileCtas = 4;                 // resident CTAs per SM the grid is sized for
constexpr int kC1TilePx = 64 * kC1TileWarps;   // tile columns
constexpr int kC1TilePitch = kC1TilePx + 8;    // staged floats per row: image columns tx0 - 4 .. tx0 + 259
constexpr int kC1TileOutBuf = 64 * 128;        // one output row of a warp: 64 pixels x 128 bytes

template <int K>
__global__ void __launch_bounds__(32 * kC1TileWarps, kC1TileCtas)
    conv_c1_tile_kernel(const float *__restrict__ x, const float *__restrict__ w, const float *__restrict__ bias,
                        int N, int H, int W, int Cout, int R, int S, int act, int rows_per_cta, int col_tiles,
                        const __grid_constant__ CUtensorMap tmy)
{
    constexpr int HALO = K / 2;
    constexpr int CO = 32;   // output channels per CTA
    constexpr int PX = 8;    // pixels per thread
    static_assert(HALO <= 4, "the staged row keeps 4 columns of halo room on each side");
    extern __shared__ __align__(1024) unsigned char c1t_raw[];
    __shared__ __align__(16) float ws[K * K * CO];
    __shared__ __align__(16) float bs[CO];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // 4 channel lanes x 8 pixel lanes; the 8 lanes of a quarter-warp share
    // a channel lane, so a filter load asks for one 16-byte chunk per
    // quarter-warp (2 shared-memory wavefronts where one chunk per lane of
    // a quarter takes 4)
    const int cl = lane >> 3, pl = lane & 7;
    const int co0 = blockIdx.y * CO;
    const int n = blockIdx.z;
    const int ct = blockIdx.x % col_tiles, rt = blockIdx.x / col_tiles;
    const int tx0 = ct * kC1TilePx;
    const int y0 = rt * rows_per_cta;
    const int y1 = min(H, y0 + rows_per_cta);
    const int nrows = y1 - y0, nin = nrows + K - 1;
    // dynamic shared memory: [an output buffer per warp][input tile]
    const uint32_t raw_u = smem_u32(c1t_raw);
    const uint32_t obase = (raw_u + 1023) & ~1023u;
    float *tile = reinterpret_cast<float *>(c1t_raw + (obase - raw_u) + kC1TileWarps * kC1TileOutBuf);

    // staged column c of row r is image pixel (y0 - HALO + r, tx0 - 4 + c);
    // 16-byte pieces are wholly inside or outside the image (W % 4 == 0)
    // two copy groups: the K rows of the first output row, then the rest,
    // which land while the first row is computed
    const float *xn = x + (long long)n * H * W;
    constexpr int CPR = kC1TilePitch / 4;
    auto stage_rows = [&](int r0, int r1) {
        for (int e = r0 * CPR + tid; e < r1 * CPR; e += 32 * kC1TileWarps) {
            const int r = e / CPR, q = e % CPR;
            const int iy = y0 - HALO + r, ix = tx0 - 4 + 4 * q;
            const bool ok = iy >= 0 && iy < H && ix >= 0 && ix + 3 < W;
            cp_async16(smem_u32(tile + r * kC1TilePitch + 4 * c1_band_chunk(q)), ok ? xn + (long long)iy * W + ix : x,
                       ok ? 16 : 0);
        }
        cp_async_commit();
    };
    // the band's copies first, so that their latency overlaps the filter
    // and bias loads below
    stage_rows(0, K);
    stage_rows(K, nin);
    for (int e = tid; e < K * K * CO; e += 32 * kC1TileWarps) {
        const int col = e % CO, tap = e / CO;
        const int r = tap / K - (K - R) / 2, s = tap % K - (K - S) / 2;
        const int co = co0 + col;
        float v = 0.f;
        if (r >= 0 && r < R && s >= 0 && s < S && co < Cout) v = w[((long long)co * R + r) * S + s];
        ws[e] = v;
    }
    for (int e = tid; e < CO; e += 32 * kC1TileWarps) bs[e] = (bias && co0 + e < Cout) ? bias[co0 + e] : 0.f;
    cp_async_wait<1>();
    __syncthreads();

    const int xw = tx0 + warp * 64;             // the warp's first column
    // staged 16-byte chunks of this thread's window (image columns x - 4 ..
    // x + 11): logical chunks 16 * warp + 2 * pl + q, q = 0..3
    int woff[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) woff[q] = 4 * c1_band_chunk(16 * warp + 2 * pl + q);
    const uint32_t buf = obase + (uint32_t)(warp * kC1TileOutBuf);
    for (int i = 0; i < nrows; ++i) {
        const int oy = y0 + i;
        if (i == 1) {   // the rest of the band has landed
            cp_async_wait<0>();
            __syncthreads();
        }
        float acc[8][PX];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const float4 b4 = *reinterpret_cast<const float4 *>(bs + g * 16 + 4 * cl);
#pragma unroll
            for (int j = 0; j < PX; ++j) {
                acc[4 * g + 0][j] = b4.x;
                acc[4 * g + 1][j] = b4.y;
                acc[4 * g + 2][j] = b4.z;
                acc[4 * g + 3][j] = b4.w;
            }
        }
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            // image columns x - 4 .. x + 11 of input row oy - HALO + ky
            const float *trow = tile + (i + ky) * kC1TilePitch;
            float win[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 t = *reinterpret_cast<const float4 *>(trow + woff[q]);
                win[4 * q] = t.x;
                win[4 * q + 1] = t.y;
                win[4 * q + 2] = t.z;
                win[4 * q + 3] = t.w;
            }
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const float *wt = ws + (ky * K + kx) * CO;
                float wv[8];
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const float4 t = *reinterpret_cast<const float4 *>(wt + g * 16 + 4 * cl);
                    wv[4 * g + 0] = t.x;
                    wv[4 * g + 1] = t.y;
                    wv[4 * g + 2] = t.z;
                    wv[4 * g + 3] = t.w;
                }
#pragma unroll
                for (int j = 0; j < PX; ++j) {
                    const float v = win[4 - HALO + j + kx];
                    const float2 vv = make_float2(v, v);
#pragma unroll
                    for (int f = 0; f < 8; f += 2) {
                        float2 a2 = make_float2(acc[f][j], acc[f + 1][j]);
                        a2 = __ffma2_rn(make_float2(wv[f], wv[f + 1]), vv, a2);
                        acc[f][j] = a2.x;
                        acc[f + 1][j] = a2.y;
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_read<0>();   // the store that last read this buffer is done
        __syncwarp();
        if (xw < W) {
            // the buffer holds the warp's 64 pixels in the order the output
            // copy's box walks them: pixel 8 * pl + j in 128-byte row
            // 8 * j + pl, 16-byte chunk q at q ^ pl (the 128-byte TMA
            // swizzle of that row), so the 8 pixel lanes of a quarter-warp
            // write 8 distinct bank groups
#pragma unroll
            for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int j = 0; j < PX; ++j) {
                    const int q = g * 4 + cl;   // 16-byte chunk: channels 4q .. 4q + 3
                    float o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = relu_if(acc[4 * g + e][j], act);
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(buf + (8 * j + pl) * 128 +
                                                                                     ((q ^ pl) << 4)),
                                 "f"(o[0]), "f"(o[1]), "f"(o[2]), "f"(o[3])
                                 : "memory");
                }
        }
        fence_proxy_async_smem();   // these writes -> visible to the copy
        __syncwarp();
        if (lane == 0 && xw < W) {
            tma_store_5d(&tmy, buf, co0, xw / 8, 0, oy, n);
            bulk_commit();
        }
    }
    // the buffers must outlive the stores' reads of them; the stores' writes
    // to global memory complete before the grid does
    if (lane == 0) bulk_wait_read<0>();
}

template <int K>
static cudaError_t launch_c1_tile(const ConvArgs &a, cudaStream_t st)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = conv_tma_encoder();
    if (!encode) return cudaErrorNotSupported;
    const int col_tiles = (a.W + kC1TilePx - 1) / kC1TilePx;
    const int groups = (a.Cout + 31) / 32;
    // one wave: bands of rows so that every CTA is resident at once
    const long long per_band = (long long)col_tiles * groups * a.N;
    long long bands = (long long)kC1TileCtas * device_sm_count() / per_band;
    if (bands < 1) bands = 1;
    int rows_per_cta = (int)((a.H + bands - 1) / bands);
    if (rows_per_cta > 48) rows_per_cta = 48;   // bounds the staged tile
    const long long nb = (long long)col_tiles * ((a.H + rows_per_cta - 1) / rows_per_cta);
    if (nb > 0x7fffffffLL || groups > 65535 || a.N > 65535) return cudaErrorInvalidConfiguration;
    // The output as a 5-D tensor (channel, pixel group of 8, pixel in the
    // group, row, image): the box (32 channels, 8 groups, 8 pixels) of a
    // warp's row lands in shared memory with group fastest, i.e. pixel
    // 8 * g + j in 128-byte row 8 * j + g.  Needs W % 8 == 0.
    if (a.W % 8) return cudaErrorNotSupported;
    CUtensorMap tm;
    const cuuint64_t dims[5] = {(cuuint64_t)a.Cout, (cuuint64_t)(a.W / 8), 8, (cuuint64_t)a.H, (cuuint64_t)a.N};
    const cuuint64_t strides[4] = {(cuuint64_t)a.Cout * 32, (cuuint64_t)a.Cout * 4, (cuuint64_t)a.W * a.Cout * 4,
                                   (cuuint64_t)a.H * a.W * a.Cout * 4};
    const cuuint32_t box[5] = {32, 8, 8, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, a.y, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    const int smem = kC1TileWarps * kC1TileOutBuf + 1024 + (rows_per_cta + K - 1) * kC1TilePitch * 4;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static KernelCache cache;
    e = ensure_dynamic_smem(cache, dev, conv_c1_tile_kernel<K>, smem);
    if (e != cudaSuccess) return e;
    conv_c1_tile_kernel<K><<<dim3((unsigned)nb, groups, a.N), 32 * kC1TileWarps, smem, st>>>(
        a.x, a.w, a.b, a.N, a.H, a.W, a.Cout, a.R, a.S, a.act, rows_per_cta, col_tiles, tm);
    return cudaGetLastError();
}

template <int K, int F_T, int CL>
static cudaError_t launch_c1_cfg(const ConvArgs &a, cudaStream_t st)
{
    using C = C1Cfg<K, F_T, CL>;
    const int warp_cols = C::PL * 4;
    const int warps_needed = (a.W + warp_cols - 1) / warp_cols;
    const int nwarps = warps_needed < 8 ? warps_needed : 8;
    const int col_tiles = (a.W + nwarps * warp_cols - 1) / (nwarps * warp_cols);
    const int groups = (a.Cout + C::CO_CTA - 1) / C::CO_CTA;
    // Enough CTAs for two per SM, but bands of at least 2K rows so the
    // K - 1 rows of vertical halo stay a small share of each band's loads.
    const long long per_band = (long long)col_tiles * groups * a.N;
    const long long want = 2LL * device_sm_count();
    long long bands = (want + per_band - 1) / per_band;
    int min_rows = 2 * K;
    long long max_bands = (a.H + min_rows - 1) / min_rows;
    if (bands > max_bands) bands = max_bands;
    if (bands < 1) bands = 1;
    const int rows_per_cta = (int)((a.H + bands - 1) / bands);
    const long long nb = (long long)col_tiles * ((a.H + rows_per_cta - 1) / rows_per_cta);
    if (nb > 0x7fffffffLL || groups > 65535 || a.N > 65535) return cudaErrorInvalidConfiguration;
    const int vec = ((a.W & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0) &&
                    ((reinterpret_cast<uintptr_t>(a.y) & 15) == 0);
    if (vec) {
        // groups of 32 channels: the tiled kernel (any filter size up to 7)
        if constexpr (F_T == 8 && CL == 4) {
            const cudaError_t e = launch_c1_tile<K>(a, st);
            if (e != cudaErrorNotSupported) return e;
        }
        // the ring needs more registers than 7 x 7 filters with 8 channels
        // per thread leave at 2 CTAs per SM; those keep the shifting window
        if (!(K >= 7 && F_T >= 8)) {
            conv_c1_ring_kernel<K, F_T, CL><<<dim3((unsigned)nb, groups, a.N), nwarps * 32, 0, st>>>(
                a.x, a.w, a.b, a.y, a.N, a.H, a.W, a.Cout, a.R, a.S, a.act, rows_per_cta, col_tiles);
            return cudaGetLastError();
        }
    }
    conv_c1_kernel<K, F_T, CL><<<dim3((unsigned)nb, groups, a.N), nwarps * 32, 0, st>>>(
        a.x, a.w, a.b, a.y, a.N, a.H, a.W, a.Cout, a.R, a.S, a.act, rows_per_cta, col_tiles, vec);
    return cudaGetLastError();
}

template <int K>
static cudaError_t launch_c1_k(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout == 1) return launch_c1_cfg<K, 1, 1>(a, st);
    if (a.Cout == 4) return launch_c1_cfg<K, 4, 1>(a, st);
    if (a.Cout <= 8) return launch_c1_cfg<K, 8, 1>(a, st);
    if (a.Cout <= 16) return launch_c1_cfg<K, 8, 2>(a, st);
    return launch_c1_cfg<K, 8, 4>(a, st);
}

// Small images with one output channel (a few thousand pixels): the row
// sweep above would leave most SMs idle and walk its rows one after another,
// each behind a load.  Here each thread computes 4 horizontally adjacent
// output pixels of one row on its own and issues all its loads (the K x K
// filter, the bias and K rows of 4 + K - 1 pixels, zero outside the image)
// at once, so a launch costs about one load latency after the launch
// itself.  FMA order as in the kernels above: bias, then the taps row by
// row.
constexpr int kC1SmallThreads = 64;
constexpr long long kC1SmallPixels = 1LL << 16;   // N * H * W up to which it is used

template <int K>
__global__ void __launch_bounds__(kC1SmallThreads)
    conv_c1_small_kernel(const float *__restrict__ x, const float *__restrict__ w, const float *__restrict__ bias,
                         float *__restrict__ y, int N, int H, int W, int R, int S, int act)
{
    constexpr int HALO = K / 2, WIN = 4 + K - 1;
    const int qw = (W + 3) / 4;
    const long long t = (long long)blockIdx.x * kC1SmallThreads + threadIdx.x;
    if (t >= (long long)N * H * qw) return;
    const int x0 = 4 * (int)(t % qw);
    const long long row = t / qw;   // n * H + oy
    const int oy = (int)(row % H);
    const float *xn = x + (row - oy) * W;
    float wv[K * K];
#pragma unroll
    for (int ky = 0; ky < K; ++ky)
#pragma unroll
        for (int kx = 0; kx < K; ++kx) {
            const int r = ky - (K - R) / 2, s = kx - (K - S) / 2;
            wv[ky * K + kx] = (r >= 0 && r < R && s >= 0 && s < S) ? __ldg(w + r * S + s) : 0.f;
        }
    float win[K][WIN];
#pragma unroll
    for (int ky = 0; ky < K; ++ky) {
        const int iy = oy - HALO + ky;
#pragma unroll
        for (int c = 0; c < WIN; ++c) {
            const int ix = x0 - HALO + c;
            win[ky][c] = (iy >= 0 && iy < H && ix >= 0 && ix < W) ? __ldg(xn + (long long)iy * W + ix) : 0.f;
        }
    }
    const float b = bias ? __ldg(bias) : 0.f;
    float acc[4] = {b, b, b, b};
#pragma unroll
    for (int ky = 0; ky < K; ++ky)
#pragma unroll
        for (int kx = 0; kx < K; ++kx)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = fmaf(wv[ky * K + kx], win[ky][j + kx], acc[j]);
    float *yr = y + row * W;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (x0 + j < W) yr[x0 + j] = relu_if(acc[j], act);
}

template <int K>
static cudaError_t launch_c1_small(const ConvArgs &a, cudaStream_t st)
{
    const long long threads = (long long)a.N * a.H * ((a.W + 3) / 4);
    const long long blocks = (threads + kC1SmallThreads - 1) / kC1SmallThreads;
    conv_c1_small_kernel<K><<<(unsigned)blocks, kC1SmallThreads, 0, st>>>(a.x, a.w, a.b, a.y, a.N, a.H, a.W, a.R,
                                                                         a.S, a.act);
    return cudaGetLastError();
}

cudaError_t launch_conv_c1(const ConvArgs &a, cudaStream_t st)
{
    const int K = a.R > a.S ? a.R : a.S;
    if (a.Cout == 1 && (long long)a.N * a.H * a.W <= kC1SmallPixels) {
        switch (K) {
        case 1: return launch_c1_small<1>(a, st);
        case 3: return launch_c1_small<3>(a, st);
        case 5: return launch_c1_small<5>(a, st);
        case 7: return launch_c1_small<7>(a, st);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (K) {
    case 1: return launch_c1_k<1>(a, st);
    case 3: return launch_c1_k<3>(a, st);
    case 5: return launch_c1_k<5>(a, st);
    case 7: return launch_c1_k<7>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sc
