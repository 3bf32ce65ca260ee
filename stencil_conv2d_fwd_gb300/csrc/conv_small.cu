// Direct convolution for small images (up to 64 K pixels in all) with up to
// 16 input and 16 output channels and 3 x 3 filters: the shape of a
// single small CNN layer, whose whole work (16 -> 16 on 128 x 128: 75
// MFLOP) is about a microsecond of the GPU's FP32 rate, so that a launch is
// dominated by its fixed costs (starting the CTAs, one round trip to memory,
// barriers, address arithmetic) unless these are kept few.
//
// Method: "Optimizing Memory Efficiency for Convolution Kernels on Kepler
// GPUs", Section 3.3 (a CTA stages its tile's input channels plus halo and
// its filters in shared memory; each thread keeps a register row of W + 2
// pixels reused over the taps of a filter row), laid out for latency:
//  * one CTA of 8 warps per 2 x 64 pixel tile and all (up to 16) output
//    channels, one tile per SM (128 CTAs for a 128 x 128 image); its warps
//    split the tile's rows (2) and the input channels (4 groups of 4), so a
//    thread computes 8 pixels x 4 output channels over 4 input channels;
//  * every copy is issued at once and waited for once: the input tile by
//    16-byte asynchronous copies, the filter bank by loads along its OIHW
//    order (a warp-wide load is one 128-byte line; loads with a lane per
//    output channel touched 32 lines each and took 1.4 us of L1 lookups per
//    CTA) stored transposed to [ci][tap][co] at a row pitch of 20 floats;
//  * the four input-channel groups' partial sums are exchanged through
//    shared memory so that each warp finishes and stores 2 of its row's 8
//    pixels per thread: two barriers in all.
// Lane mapping: lane = 8 * c + q, c = output-channel quad (one per
// quarter-warp, so a filter load is one 16-byte chunk per quarter-warp, two
// wavefronts a warp), q = pixel run (pixels 8 q .. 8 q + 7 of the tile
// row).  The eight runs of a quarter-warp read eight 16-byte chunks 32
// chunks apart, all in one bank group unless swizzled: the staged row is
// stored through small_tile_chunk (common.cuh), which puts them in eight
// bank groups (four wavefronts a warp, the fewest for eight distinct chunks
// per quarter-warp).
// FMA order: for each output, each input-channel group's taps (channels
// ascending, then filter row, then column) into its own partial sum; the
// four partial sums then added in group order, and the bias last.
#include "common.cuh"
#include "launch.h"

namespace sc {

namespace {
constexpr int SM_TH = 2, SM_TW = 64;                              // output tile
constexpr int SM_PT = 8;                                          // output pixels per thread
constexpr int SM_CIG = 4;                                         // input-channel groups = warps per tile row
constexpr int SM_NT = 32 * SM_TH * SM_CIG;                        // 256 threads
constexpr int SM_PW = SM_TW + 2;                                  // staged pixels per row: x0 - 1 .. x0 + 64
constexpr int SM_MAXC = 16;                                       // input and output channels at most
constexpr long long SM_MAX_PIXELS = 1LL << 16;                    // N * H * W up to which it is used
constexpr int SM_XS_FLOATS = (SM_TH + 2) * SM_PW * SM_MAXC;       // staged input rows
constexpr int SM_WP = 20;                                         // filter row pitch: 16 outputs + 4
constexpr int SM_WS_FLOATS = SM_MAXC * 9 * SM_WP;                 // filters [ci][tap][co]
constexpr int SM_PART_F4 = SM_TH * SM_CIG * (SM_CIG - 1) * 2 * 32; // exchanged partial sums
constexpr int SM_SMEM = (SM_XS_FLOATS + SM_WS_FLOATS) * 4 + SM_PART_F4 * 16;
static_assert(SM_PW * 4 % 8 == 0, "a staged row is whole groups of 8 chunks (small_tile_chunk)");
}  // namespace

template <int CB>   // input channels / 4
__global__ void __launch_bounds__(SM_NT, 1)
    conv_small_kernel(const float *__restrict__ x, const float *__restrict__ w, const float *__restrict__ bias,
                      float *__restrict__ y, int H, int W, int Cout, int act, int tiles_x, int tiles_y)
{
    constexpr int Cin = 4 * CB;
    extern __shared__ __align__(16) float small_smem[];
    float *xs = small_smem;                                              // [row][small_tile_chunk(p, cb)]
    float *ws = xs + SM_XS_FLOATS;                                       // [ci * 9 + tap][co], pitch SM_WP
    float4 *part = reinterpret_cast<float4 *>(ws + SM_WS_FLOATS);       // [row][owner][slot][pair][lane]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = blockIdx.x;
    const int tx = t % tiles_x, ty = (t / tiles_x) % tiles_y, n = t / (tiles_x * tiles_y);
    const int y0 = ty * SM_TH, x0 = tx * SM_TW;

    // the input tile, zero outside the image (the "same" padding)
    const float *xn = x + (long long)n * H * W * Cin;
    for (int e = tid; e < (SM_TH + 2) * SM_PW * CB; e += SM_NT) {
        const int cb = e % CB, p = (e / CB) % SM_PW, r = e / (CB * SM_PW);
        const int iy = y0 - 1 + r, ix = x0 - 1 + p;
        const bool ok = iy >= 0 && iy < H && ix >= 0 && ix < W;
        cp_async16(smem_u32(xs + r * SM_PW * SM_MAXC + 4 * small_tile_chunk(p, cb)),
                   ok ? xn + ((long long)iy * W + ix) * Cin + 4 * cb : x, ok ? 16 : 0);
    }
    cp_async_commit();

    const int row = warp / SM_CIG, grp = warp % SM_CIG;   // tile row, input-channel group
    const int c = lane >> 3, q = lane & 7;                // output-channel quad, pixel run
    float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (bias && 4 * c < Cout) bv = make_float4(bias[4 * c], bias[4 * c + 1], bias[4 * c + 2], bias[4 * c + 3]);
    {
        // the filter bank in its OIHW order, element e = co * 9 Cin + k with
        // k = ci * 9 + tap, to word k * SM_WP + co: a warp's 32 stores fall
        // in 8 banks (the 20-float pitch; 16 would put them in one)
        constexpr int KK = Cin * 9, NV = (SM_MAXC * KK + SM_NT - 1) / SM_NT;
        float wv[NV];
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            const int e = tid + m * SM_NT;
            wv[m] = e < Cout * KK ? __ldg(w + e) : 0.f;
        }
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            const int e = tid + m * SM_NT;
            if (e < Cout * KK) ws[(e % KK) * SM_WP + e / KK] = wv[m];
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    float acc[4][SM_PT];   // [output channel][pixel]
#pragma unroll
    for (int f = 0; f < 4; ++f)
#pragma unroll
        for (int j = 0; j < SM_PT; ++j) acc[f][j] = 0.f;
    if (grp < CB && 4 * c < Cout) {
        const float *xrow = xs + row * SM_PW * SM_MAXC;
        const float *wg = ws + (4 * grp * 9) * SM_WP + 4 * c;
#pragma unroll
        for (int r = 0; r < 3; ++r) {
            // staged pixels 8 q .. 8 q + 9 (image columns x - 1 .. x + 8), channels 4 grp .. 4 grp + 3
            float4 px[SM_PT + 2];
#pragma unroll
            for (int k = 0; k < SM_PT + 2; ++k)
                px[k] = *reinterpret_cast<const float4 *>(xrow + r * SM_PW * SM_MAXC +
                                                          4 * small_tile_chunk(SM_PT * q + k, grp));
#pragma unroll
            for (int ci = 0; ci < 4; ++ci)
#pragma unroll
                for (int s = 0; s < 3; ++s) {
                    const float4 wv = *reinterpret_cast<const float4 *>(wg + (ci * 9 + 3 * r + s) * SM_WP);
#pragma unroll
                    for (int j = 0; j < SM_PT; ++j) {
                        const float4 p = px[j + s];
                        const float v = ci == 0 ? p.x : (ci == 1 ? p.y : (ci == 2 ? p.z : p.w));
                        const float2 vv = make_float2(v, v);
                        float2 a2 = __ffma2_rn(make_float2(wv.x, wv.y), vv, make_float2(acc[0][j], acc[1][j]));
                        acc[0][j] = a2.x;
                        acc[1][j] = a2.y;
                        a2 = __ffma2_rn(make_float2(wv.z, wv.w), vv, make_float2(acc[2][j], acc[3][j]));
                        acc[2][j] = a2.x;
                        acc[3][j] = a2.y;
                    }
                }
        }
    }

    // pixel pair o (pixels 2 o, 2 o + 1 of each run) is finished by group o
    // of the row; the other three groups hand it their partial sums, in
    // slot g (g < o) or g - 1 (g > o)
    auto part_at = [&](int owner, int g, int pp) {
        return part + (((row * SM_CIG + owner) * (SM_CIG - 1) + (g < owner ? g : g - 1)) * 2 + pp) * 32 + lane;
    };
#pragma unroll
    for (int o = 0; o < SM_CIG; ++o)
        if (o != grp)
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
                const int j = 2 * o + pp;
                *part_at(o, grp, pp) = make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
            }
    __syncthreads();
    const int gy = y0 + row;
    if (gy >= H || 4 * c >= Cout) return;
    float4 mine[2];   // this group's own partial sums of its pair (register indices fixed at compile time)
#pragma unroll
    for (int o = 0; o < SM_CIG; ++o)
        if (o == grp)
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
                mine[pp] = make_float4(acc[0][2 * o + pp], acc[1][2 * o + pp], acc[2][2 * o + pp], acc[3][2 * o + pp]);
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        const int j = 2 * grp + pp;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int g = 0; g < SM_CIG; ++g) {
            const float4 v = g == grp ? mine[pp] : *part_at(grp, g, pp);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        const int gx = x0 + SM_PT * q + j;
        if (gx < W) {
            float4 o;
            o.x = relu_if(s.x + bv.x, act);
            o.y = relu_if(s.y + bv.y, act);
            o.z = relu_if(s.z + bv.z, act);
            o.w = relu_if(s.w + bv.w, act);
            *reinterpret_cast<float4 *>(y + (((long long)n * H + gy) * W + gx) * Cout + 4 * c) = o;
        }
    }
}

template <int CB>
static cudaError_t launch_small(const ConvArgs &a, int tiles_x, int tiles_y, unsigned nb, cudaStream_t st)
{
    static KernelCache cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = ensure_dynamic_smem(cache, dev, conv_small_kernel<CB>, SM_SMEM);
    if (e != cudaSuccess) return e;
    conv_small_kernel<CB><<<nb, SM_NT, SM_SMEM, st>>>(a.x, a.w, a.b, a.y, a.H, a.W, a.Cout, a.act, tiles_x,
                                                      tiles_y);
    return cudaGetLastError();
}

// NHWC, Cin and Cout multiples of 4 up to 16, 3 x 3 filters, at most 64 K
// pixels in all; cudaErrorNotSupported otherwise.
cudaError_t launch_conv_small(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cin % 4 || a.Cout % 4 || a.Cin > SM_MAXC || a.Cout > SM_MAXC || a.R != 3 || a.S != 3 ||
        (long long)a.N * a.H * a.W > SM_MAX_PIXELS)
        return cudaErrorNotSupported;
    const int tiles_x = (a.W + SM_TW - 1) / SM_TW, tiles_y = (a.H + SM_TH - 1) / SM_TH;
    const long long nb = (long long)tiles_x * tiles_y * a.N;
    if (nb > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    switch (a.Cin / 4) {
    case 1: return launch_small<1>(a, tiles_x, tiles_y, (unsigned)nb, st);
    case 2: return launch_small<2>(a, tiles_x, tiles_y, (unsigned)nb, st);
    case 3: return launch_small<3>(a, tiles_x, tiles_y, (unsigned)nb, st);
    default: return launch_small<4>(a, tiles_x, tiles_y, (unsigned)nb, st);
    }
}

}  // namespace sc
