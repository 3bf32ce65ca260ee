// General-case direct convolution, FP32 FFMA, NHWC activations.
//
// Method: "Optimizing Memory Efficiency for Convolution Kernels on Kepler
// GPUs", Section 3.3 (general case) and Algorithm 2:
//  * a CTA owns F_TB output channels ("filters") of one TH x TW block of
//    output pixels (the 2-D TB layout, Section 3.3.1);
//  * C_SH input channels of the block plus its halo, and the matching
//    filter slice, are staged in shared memory per step (Fig. 6), with the
//    next step's copy in flight while the current one is consumed
//    (Algorithm 2's prefetch, here as cp.async double buffering);
//  * each thread accumulates F_T filters x W_T horizontally contiguous
//    pixels in registers; for one input row it keeps W_T + S - 1 pixels in
//    registers and reuses them over the S taps of that row (Section 3.3.2);
//  * filter values are read as 16-byte units of 4 output channels and
//    pixels as 16-byte units of 4 input channels, so the shared-memory access
//    width matches the bank width (Section 2.1, W_CD = W_SMB) and a single
//    LDS.128 feeds 4 x W_T FMAs;
//  * pixels are read by the lanes of one warp that own different pixels,
//    filters by the lanes that own different output channels; lanes that
//    share a pixel (or a filter unit) read the same address (broadcast,
//    Section 3.3.2).
// Activations use the packed 4-channel layout of "Optimizing convolution
// kernels - CNNs in Vulkan Part 2/3", section "Vectorization" (channels of
// a pixel contiguous), so every global->shared copy is one 16-byte cp.async.
//
// Shared-memory activation tile, per stage: [C_SH/4][TH+R-1][TWP] chunks of
// float4, TWP = TW + S - 1, linear chunk index q, stored at chunk swz16(q, 3)
// (XOR swizzle over 128-byte rows, "CUDA共有メモリのスウィズリング").  The
// lanes of a warp read chunks W_T apart in one tile row; without the XOR they
// would all fall into the same four banks.
// Filter tile, per stage: [C_SH][R][S][F_TB] floats (filters transposed so a
// thread's 4 output channels are one 16-byte unit).  It is written by lanes
// that run along output channels, which is conflict-free without padding.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace sc {

template <int S_, int F_TB_, int W_T_, int TH_, int TW_, int C_SH_, int MINB_>
struct GenCfg {
    static constexpr int S = S_;
    static constexpr int F_TB = F_TB_;
    static constexpr int W_T = W_T_;
    static constexpr int TH = TH_;
    static constexpr int TW = TW_;
    static constexpr int C_SH = C_SH_;
    static constexpr int MINB = MINB_;
    static constexpr int F_T = F_TB >= 8 ? 8 : 4;       // output channels per thread
    static constexpr int NG = F_T / 4;                   // float4 groups per thread
    static constexpr int T_X = F_TB / F_T;               // lanes along output channels
    static constexpr int PXL = 32 / T_X;                 // lanes along pixels
    static constexpr int WARP_COLS = PXL * W_T;
    static constexpr int WARPS_PER_ROW = TW / WARP_COLS;
    static constexpr int NWARPS = WARPS_PER_ROW * TH;
    static constexpr int NT = NWARPS * 32;
    static constexpr int CB = C_SH / 4;
    static constexpr int TWP = TW + S - 1;
    static constexpr int WIN = W_T + S - 1;
    static_assert(F_TB % F_T == 0 && 32 % T_X == 0, "bad channel split");
    static_assert(TW % WARP_COLS == 0, "tile width must hold whole warps");
    static_assert(C_SH % 4 == 0, "C_SH must be a multiple of 4");
    static_assert(NT <= 1024, "too many threads");

    // Activation chunks per stage for R rows of taps.  The swizzle permutes
    // chunks inside rows of 8, so the tile is padded to whole rows of 8: the
    // physical index of logical chunk q < used_chunks stays below this.
    static __host__ __device__ int used_chunks(int R) { return CB * (TH + R - 1) * TWP; }
    static __host__ __device__ int in_chunks(int R) { return (used_chunks(R) + 7) & ~7; }
    // floats per stage: activation chunks * 4 + filters
    static __host__ __device__ int w_floats(int R) { return C_SH * R * S * F_TB; }
    static __host__ __device__ int stage_floats(int R) { return in_chunks(R) * 4 + w_floats(R); }
    static size_t smem_bytes(int R) { return 2 * size_t(stage_floats(R)) * sizeof(float); }
};

template <class C>
__device__ __forceinline__ void gen_issue_stage(float *stage, const float *__restrict__ x,
                                                const float *__restrict__ w, int n, int y0,
                                                int x0, int co0, int c0, int H, int W, int Cin,
                                                int Cout, int R, int tid)
{
    float4 *in_s = reinterpret_cast<float4 *>(stage);
    float *w_s = stage + C::in_chunks(R) * 4;
    const int THh = C::TH + R - 1;
    const int nq = C::used_chunks(R);
    // activation halo tile: one 16-byte chunk (4 channels of a pixel) per copy
    for (int q = tid; q < nq; q += C::NT) {
        const int xx = q % C::TWP;
        const int t = q / C::TWP;
        const int yy = t % THh;
        const int cb = t / THh;
        const int gy = y0 - R / 2 + yy;
        const int gx = x0 - C::S / 2 + xx;
        const int ci = c0 + 4 * cb;
        const bool ok = (gy >= 0) & (gy < H) & (gx >= 0) & (gx < W) & (ci < Cin);
        const float *src = ok ? x + ((((long long)n * H + gy) * W + gx) * Cin + ci) : x;
        cp_async16(smem_u32(in_s + swz16(q, 3)), src, ok ? 16 : 0);
    }
    // filter slice [C_SH][R][S][F_TB], lanes along output channels
    const int RS = R * C::S;
    const int nw = C::C_SH * RS * C::F_TB;
    for (int e = tid; e < nw; e += C::NT) {
        const int col = e % C::F_TB;
        const int row = e / C::F_TB;  // = ci_l * RS + rs
        const int ci = c0 + row / RS;
        const int rs = row % RS;
        const int co = co0 + col;
        const bool ok = (co < Cout) & (ci < Cin);
        const float *src = ok ? w + (((long long)co * Cin + ci) * RS + rs) : w;
        cp_async4(smem_u32(w_s + e), src, ok ? 4 : 0);
    }
}

template <class C>
__global__ void __launch_bounds__(C::NT, C::MINB)
    conv_general_kernel(const float *__restrict__ x, const float *__restrict__ w,
                        const float *__restrict__ bias, float *__restrict__ y, int N, int H,
                        int W, int Cin, int Cout, int R, int act, int tiles_x, int tiles_y)
{
    extern __shared__ __align__(16) float smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tx = lane % C::T_X;        // output-channel lane
    const int pl = lane / C::T_X;        // pixel lane

    int tile = blockIdx.x;
    const int txi = tile % tiles_x;
    tile /= tiles_x;
    const int tyi = tile % tiles_y;
    const int n = tile / tiles_y;
    const int co0 = blockIdx.y * C::F_TB;
    const int y0 = tyi * C::TH;
    const int x0 = txi * C::TW;

    const int ry = warp / C::WARPS_PER_ROW;                                   // tile row
    const int cx0 = (warp % C::WARPS_PER_ROW) * C::WARP_COLS + pl * C::W_T;   // tile col

    const int stage_f = C::stage_floats(R);
    const int THh = C::TH + R - 1;
    const int nk = (Cin + C::C_SH - 1) / C::C_SH;

    float acc[C::F_T][C::W_T];
#pragma unroll
    for (int f = 0; f < C::F_T; ++f)
#pragma unroll
        for (int j = 0; j < C::W_T; ++j) acc[f][j] = 0.0f;

    gen_issue_stage<C>(smem, x, w, n, y0, x0, co0, 0, H, W, Cin, Cout, R, tid);
    cp_async_commit();

    for (int k = 0; k < nk; ++k) {
        if (k + 1 < nk) {
            gen_issue_stage<C>(smem + ((k + 1) & 1) * stage_f, x, w, n, y0, x0, co0,
                               (k + 1) * C::C_SH, H, W, Cin, Cout, R, tid);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        const float *stage = smem + (k & 1) * stage_f;
        const float4 *in_s = reinterpret_cast<const float4 *>(stage);
        const float4 *w_s4 = reinterpret_cast<const float4 *>(stage + C::in_chunks(R) * 4);

#pragma unroll 1
        for (int cb = 0; cb < C::CB; ++cb) {
#pragma unroll 1
            for (int r = 0; r < R; ++r) {
                // one input row of W_T + S - 1 pixels x 4 channels
                const int base = (cb * THh + ry + r) * C::TWP + cx0;
                float4 px[C::WIN];
#pragma unroll
                for (int j = 0; j < C::WIN; ++j) px[j] = in_s[swz16(base + j, 3)];
                // filter rows of (ci = 4cb + c, r, s): ((4cb + c) * R + r) * S + s
                const float4 *wr = w_s4 + ((4 * cb * R + r) * C::S) * (C::F_TB / 4) + tx;
#pragma unroll
                for (int s = 0; s < C::S; ++s) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float4 *wp = wr + (c * R * C::S + s) * (C::F_TB / 4);
                        float wv[C::F_T];
#pragma unroll
                        for (int g = 0; g < C::NG; ++g) {
                            const float4 t = wp[g * C::T_X];
                            wv[4 * g + 0] = t.x;
                            wv[4 * g + 1] = t.y;
                            wv[4 * g + 2] = t.z;
                            wv[4 * g + 3] = t.w;
                        }
#pragma unroll
                        for (int j = 0; j < C::W_T; ++j) {
                            const float4 p = px[j + s];
                            const float v = c == 0 ? p.x : (c == 1 ? p.y : (c == 2 ? p.z : p.w));
#pragma unroll
                            for (int f = 0; f < C::F_T; ++f) acc[f][j] = fmaf(wv[f], v, acc[f][j]);
                        }
                    }
                }
            }
        }
        __syncthreads();
    }

    // epilogue: bias, activation, 16-byte NHWC stores of 4 output channels
    const int gy = y0 + ry;
    if (gy >= H) return;
#pragma unroll
    for (int g = 0; g < C::NG; ++g) {
        const int co = co0 + g * (C::F_TB / C::NG) + 4 * tx;
        if (co >= Cout) continue;
        float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (bias) bv = make_float4(bias[co], bias[co + 1], bias[co + 2], bias[co + 3]);
#pragma unroll
        for (int j = 0; j < C::W_T; ++j) {
            const int gx = x0 + cx0 + j;
            if (gx < W) {
                float4 o;
                o.x = relu_if(acc[4 * g + 0][j] + bv.x, act);
                o.y = relu_if(acc[4 * g + 1][j] + bv.y, act);
                o.z = relu_if(acc[4 * g + 2][j] + bv.z, act);
                o.w = relu_if(acc[4 * g + 3][j] + bv.w, act);
                *reinterpret_cast<float4 *>(y + ((((long long)n * H + gy) * W + gx) * Cout + co)) = o;
            }
        }
    }
}

template <class C>
cudaError_t launch_gen(const ConvArgs &a, cudaStream_t st)
{
    const int tiles_x = (a.W + C::TW - 1) / C::TW;
    const int tiles_y = (a.H + C::TH - 1) / C::TH;
    const long long nt = (long long)tiles_x * tiles_y * a.N;
    const int groups = (a.Cout + C::F_TB - 1) / C::F_TB;
    if (nt > 0x7fffffffLL || groups > 65535) return cudaErrorInvalidConfiguration;
    const size_t smem = C::smem_bytes(a.R);
    if (smem > 48 * 1024) {
        // opt in to more than 48 KB once per device (largest size seen so far)
        static int allowed[64] = {0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || allowed[dev] < (int)smem) {
            e = cudaFuncSetAttribute(conv_general_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) allowed[dev] = (int)smem;
        }
    }
    conv_general_kernel<C><<<dim3((unsigned)nt, groups), C::NT, smem, st>>>(
        a.x, a.w, a.b, a.y, a.N, a.H, a.W, a.Cin, a.Cout, a.R, a.act, tiles_x, tiles_y);
    return cudaGetLastError();
}

// Tile table.  Chosen per output-channel count; the width of a warp's pixel
// run (PXL * W_T) and the tile height set how many CTAs a layer gets.
template <int S>
cudaError_t dispatch_general(const ConvArgs &a, cudaStream_t st)
{
    // C_SH = 8 channels per stage for all; smaller Cin is zero-padded in smem.
    if (a.Cout > 48) return launch_gen<GenCfg<S, 64, 8, 8, 32, 8, 1>>(a, st);
    if (a.Cout > 16) return launch_gen<GenCfg<S, 32, 8, 8, 64, 8, 1>>(a, st);
    if (a.Cout > 8) return launch_gen<GenCfg<S, 16, 4, 4, 64, 8, 2>>(a, st);
    if (a.Cout > 4) return launch_gen<GenCfg<S, 8, 4, 4, 128, 8, 2>>(a, st);
    return launch_gen<GenCfg<S, 4, 8, 4, 256, 8, 2>>(a, st);
}

}  // namespace sc
