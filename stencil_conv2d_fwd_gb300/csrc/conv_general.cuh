// General-case direct convolution, FP32 FFMA, NHWC activations.
//
// Method: "Optimizing Memory Efficiency for Convolution Kernels on Kepler
// GPUs", Section 3.3 (general case) and Algorithm 2:
//  * a CTA owns F_TB output channels ("filters") and walks over TH x TW
//    blocks of output pixels (the 2-D TB layout, Section 3.3.1);
//  * C_SH input channels of a block plus its halo are staged in shared
//    memory per step (Fig. 6), with the next step's copy in flight while the
//    current one is consumed (Algorithm 2's prefetch, here cp.async double
//    buffering that runs on across block boundaries);
//  * each thread accumulates F_T filters x W_T horizontally contiguous
//    pixels in registers; for one input row it keeps W_T + K - 1 pixels in
//    registers and reuses them over the K taps of that row (Section 3.3.2);
//  * filter values are read as 16-byte units of 4 output channels and
//    pixels as 16-byte units of 4 input channels, so the shared-memory access
//    width matches the bank width (Section 2.1, W_CD = W_SMB) and one LDS.128
//    feeds 4 x W_T FMAs;
//  * lanes of a warp that own different pixels read different pixel units,
//    lanes that own different filters read different filter units, and lanes
//    sharing either read the same address (broadcast, Section 3.3.2).
// Activations use the packed 4-channel layout of "Optimizing convolution
// kernels - CNNs in Vulkan Part 2/3", section "Vectorization", so each
// global->shared copy is one 16-byte cp.async with zero fill at the border.
//
// GB300 changes to the method:
//  * The FMAs are issued as packed dual-FP32 FMAs (__ffma2_rn, sm_100 and
//    later), each component rounding like fmaf.  Both operands of such an
//    FMA are register pairs, and the pairing axis is chosen by the thread's
//    accumulator count:
//    - many accumulators (F_T x W_T > 32): pairs of output channels.  The
//      two filter values are one half of a 16-byte filter unit; the pixel
//      value is used twice, which costs one register copy per value and is
//      spread over the F_T / 2 channel pairs.
//    - few accumulators (PAIRC): pairs of input channels.  Each output keeps
//      two partial sums, over the even and over the odd input channels,
//      added once at the end; the pixel pair is one half of a 16-byte pixel
//      unit and the filter pair one half of a 16-byte unit of 4 input
//      channels (the filter bank is staged as [ci/4][r][s][F_TB][4]), so no
//      operand needs a copy.  With 4 output channels the copies of the other
//      pairing were half as many instructions as the FMAs themselves.
//  * Persistent CTAs: the grid is sized to the resident CTAs, and each CTA
//    keeps its whole filter bank (all input channels, transposed to
//    [ci][r][s][F_TB]) in shared memory for all the blocks it computes, when
//    it fits (RESIDENT); otherwise the filter slice is staged per step.
//  * The kernel size is a template parameter K (square); an R x S filter
//    with R, S <= K sits centred in the K x K taps with zeros around it.
//
// Shared-memory activation tile per stage: C_SH/4 planes of [TH+K-1][TWP]
// chunks of 16 bytes, TWP = TW + K - 1 rounded up to a multiple of 8.  The
// pixel lanes of a warp read chunks W_T apart in one tile row.  Chunk `col`
// of a tile row is stored at column phys_col(col): inside each group of 8
// chunks (128 bytes) the chunk index is XORed with the group index, the
// swizzle of "CUDA共有メモリのスウィズリング" with 128-byte swizzle rows, keeping
// as many low bits of the group index as the lane stride needs (none for odd
// W_T, whose plain layout is already conflict-free).  Each lane's key is a
// constant over the run.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace sc {

template <int K_, int F_TB_, int W_T_, int TH_, int TW_, int C_SH_, bool RESIDENT_, int MINB_>
struct GenCfg {
    static constexpr int K = K_;
    static constexpr int F_TB = F_TB_;
    static constexpr int W_T = W_T_;
    static constexpr int TH = TH_;
    static constexpr int TW = TW_;
    static constexpr int C_SH = C_SH_;
    static constexpr bool RESIDENT = RESIDENT_;
    static constexpr int MINB = MINB_;                   // CTAs per SM the registers must allow
    // Pixel lanes read chunks W_T apart, and a 16-byte shared load is served
    // 8 lanes at a time.  An odd stride already puts 8 lanes in 8 bank groups;
    // a stride of 2, 4 or 8 needs the chunk index XORed with the low 1, 2 or
    // 3 bits of its 8-chunk group index (SWZ_MASK), which makes any 8
    // consecutive lanes conflict-free for every kernel size.
    static constexpr int SWZ_MASK = (W_T % 8 == 0) ? 7 : (W_T % 4 == 0) ? 3 : (W_T % 2 == 0) ? 1 : 0;
    static constexpr int F_T = F_TB >= 8 ? 8 : 4;       // output channels per thread
    static constexpr bool PAIRC = F_T * W_T_ <= 32;       // FMA pairs along input channels
    static constexpr int NG = F_T / 4;                   // float4 groups per thread
    static constexpr int T_X = F_TB / F_T;               // lanes along output channels
    static constexpr int PXL = 32 / T_X;                 // lanes along pixels
    static constexpr int WARP_COLS = PXL * W_T;
    static constexpr int WARPS_PER_ROW = TW / WARP_COLS;
    static constexpr int NWARPS = WARPS_PER_ROW * TH;
    static constexpr int NT = NWARPS * 32;
    static constexpr int CB = C_SH / 4;
    static constexpr int KK = K * K;
    static constexpr int THh = TH + K - 1;
    static constexpr int TWU = TW + K - 1;               // tile row width used
    static constexpr int TWP = (TWU + 7) & ~7;           // tile row pitch (chunks)
    static constexpr int WIN = W_T + K - 1;
    // Channel-block planes are THh * TWP + 8 / CB chunks apart: the 8 lanes
    // of one copy phase hold 8 / CB consecutive pixels x CB blocks, and the
    // stagger puts each block's pixels in their own bank groups.
    static constexpr int PLANE = THh * TWP + (CB >= 8 ? 1 : 8 / CB);
    static constexpr int IN_CHUNKS = (CB * PLANE + 7) & ~7;
    static constexpr int STAGE_W = RESIDENT ? 0 : C_SH * KK * F_TB;
    static constexpr int STAGE_FLOATS = IN_CHUNKS * 4 + STAGE_W;
    static_assert(F_TB % F_T == 0 && 32 % T_X == 0, "bad channel split");
    static_assert(TW % WARP_COLS == 0, "tile width must hold whole warps");
    static_assert(C_SH % 4 == 0, "C_SH must be a multiple of 4");
    static_assert(NT <= 1024, "too many threads");

    // shared memory: [resident filters][stage 0][stage 1]
    static __host__ __device__ size_t w_res_floats(int cin_pad)
    {
        return RESIDENT ? (size_t)cin_pad * KK * F_TB : 0;
    }
    static size_t smem_bytes(int cin_pad) { return (w_res_floats(cin_pad) + 2 * (size_t)STAGE_FLOATS) * 4; }
};

// Physical chunk column of logical chunk column `col` in a tile row: inside
// each group of 8 chunks (128 bytes), the chunk index XOR the low bits of
// the group index.
template <class C>
__host__ __device__ __forceinline__ int phys_col(int col)
{
    return (col & ~7) | ((col ^ ((col >> 3) & C::SWZ_MASK)) & 7);
}

// Copy filters for input channels [c0, c0 + nci) into shared memory, zero
// where the R x S filter has no tap, where co >= Cout or ci >= Cin:
//  * channel pairing: ws[(ci-c0)*KK + r*K + s][F_TB] (transposed, output
//    channels contiguous);
//  * PAIRC: ws[((ci-c0)/4)*KK + r*K + s][F_TB][4] (4 consecutive input
//    channels of one output channel and tap contiguous).
// Consecutive threads write consecutive shared-memory words.
template <class C>
__device__ __forceinline__ void gen_issue_filters(float *ws, const float *__restrict__ w, int co0,
                                                  int c0, int nci, int Cin, int Cout, int R, int S,
                                                  int tid)
{
    const int n = nci * C::KK * C::F_TB;
    const int dr = (C::K - R) / 2, ds = (C::K - S) / 2;
    for (int e = tid; e < n; e += C::NT) {
        int col, ci, rs;
        if constexpr (C::PAIRC) {
            col = (e >> 2) % C::F_TB;
            const int t = e / (4 * C::F_TB);
            rs = t % C::KK;
            ci = c0 + (t / C::KK) * 4 + (e & 3);
        } else {
            col = e % C::F_TB;
            const int row = e / C::F_TB;
            ci = c0 + row / C::KK;
            rs = row % C::KK;
        }
        const int r = rs / C::K - dr;
        const int s = rs % C::K - ds;
        const int co = co0 + col;
        const bool ok = (co < Cout) & (ci < Cin) & (r >= 0) & (r < R) & (s >= 0) & (s < S);
        const float *src = ok ? w + ((((long long)co * Cin + ci) * R + r) * S + s) : w;
        cp_async4(smem_u32(ws + e), src, ok ? 4 : 0);
    }
}

// Activation halo tile of output block (n, y0, x0), input channels
// [c0, c0 + C_SH): one 16-byte cp.async per (channel block, row, column),
// zero-filled outside the image and beyond Cin.  Each warp copies whole
// tile rows; its lanes run over (column, channel block) with the channel
// block fastest, so the 32 copies of one instruction read whole 32-byte
// sectors of consecutive pixels (NHWC keeps a pixel's channels together)
// and the per-copy index arithmetic stays a few adds.
template <class C>
__device__ __forceinline__ void gen_issue_tile(float4 *in_s, const float *__restrict__ x, int n, int y0,
                                               int x0, int c0, int H, int W, int Cin, int warp, int lane)
{
    for (int yy = warp; yy < C::THh; yy += C::NWARPS) {
        const int gy = y0 - C::K / 2 + yy;
        const bool row_ok = (gy >= 0) & (gy < H);
        const float *grow = x + ((((long long)n * H + (row_ok ? gy : 0)) * W) * Cin + c0);
        for (int q = lane; q < C::TWU * C::CB; q += 32) {
            const int cb = q % C::CB;
            const int xx = q / C::CB;
            const int gx = x0 - C::K / 2 + xx;
            const bool ok = row_ok & (gx >= 0) & (gx < W) & (c0 + 4 * cb < Cin);
            const float *src = ok ? grow + (long long)gx * Cin + 4 * cb : x;
            cp_async16(smem_u32(in_s + cb * C::PLANE + yy * C::TWP + phys_col<C>(xx)), src, ok ? 16 : 0);
        }
    }
}

template <class C>
__global__ void __launch_bounds__(C::NT, C::MINB)
    conv_general_kernel(const float *__restrict__ x, const float *__restrict__ w,
                        const float *__restrict__ bias, float *__restrict__ y, int N, int H, int W,
                        int Cin, int Cout, int R, int S, int act, int tiles_x, int tiles_y)
{
    extern __shared__ __align__(128) float smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tx = lane % C::T_X;        // output-channel lane
    const int pl = lane / C::T_X;        // pixel lane
    const int co0 = blockIdx.y * C::F_TB;
    const int ry = warp / C::WARPS_PER_ROW;                                   // tile row
    const int cx0 = (warp % C::WARPS_PER_ROW) * C::WARP_COLS + pl * C::W_T;   // tile col

    const int cin_pad = (Cin + C::C_SH - 1) / C::C_SH * C::C_SH;
    const int nk = cin_pad / C::C_SH;
    const int ntiles = tiles_x * tiles_y * N;
    float *w_res = smem;
    float *stage0 = smem + C::w_res_floats(cin_pad);

    // pixel-column offsets of this lane's row window (constant over the run)
    int pcol[C::WIN];
#pragma unroll
    for (int j = 0; j < C::WIN; ++j) pcol[j] = phys_col<C>(cx0 + j);

    float bv[C::F_T];
#pragma unroll
    for (int g = 0; g < C::NG; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int co = co0 + g * (C::F_TB / C::NG) + 4 * tx + e;
            bv[4 * g + e] = (bias && co < Cout) ? bias[co] : 0.0f;
        }

    int tile = blockIdx.x;
    if (tile >= ntiles) return;
    auto decode = [&](int t, int &n, int &y0, int &x0) {
        x0 = (t % tiles_x) * C::TW;
        t /= tiles_x;
        y0 = (t % tiles_y) * C::TH;
        n = t / tiles_y;
    };
    auto issue = [&](int t, int k, int buf) {
        int n, y0, x0;
        decode(t, n, y0, x0);
        float *st = stage0 + buf * C::STAGE_FLOATS;
        gen_issue_tile<C>(reinterpret_cast<float4 *>(st), x, n, y0, x0, k * C::C_SH, H, W, Cin, warp, lane);
        if constexpr (!C::RESIDENT)
            gen_issue_filters<C>(st + C::IN_CHUNKS * 4, w, co0, k * C::C_SH, C::C_SH, Cin, Cout, R, S, tid);
    };

    if constexpr (C::RESIDENT) gen_issue_filters<C>(w_res, w, co0, 0, cin_pad, Cin, Cout, R, S, tid);
    issue(tile, 0, 0);
    cp_async_commit();

    int it = 0;
    // accumulators: channel pairing uses acc, PAIRC the (even, odd input
    // channel) partial sums acc2
    constexpr int AF = C::PAIRC ? 1 : C::F_T, AW = C::PAIRC ? 1 : C::W_T;
    constexpr int PF = C::PAIRC ? C::F_T : 1, PW = C::PAIRC ? C::W_T : 1;
    for (; tile < ntiles; tile += gridDim.x) {
        float acc[AF][AW];
        float2 acc2[PF][PW];
#pragma unroll
        for (int f = 0; f < AF; ++f)
#pragma unroll
            for (int j = 0; j < AW; ++j) acc[f][j] = 0.0f;
#pragma unroll
        for (int f = 0; f < PF; ++f)
#pragma unroll
            for (int j = 0; j < PW; ++j) acc2[f][j] = make_float2(0.0f, 0.0f);

        for (int k = 0; k < nk; ++k, ++it) {
            // prefetch the next step: the next channel chunk, or the first
            // chunk of this CTA's next block
            const int nt = (k + 1 < nk) ? tile : tile + (int)gridDim.x;
            const int nkk = (k + 1 < nk) ? k + 1 : 0;
            if (nt < ntiles) {
                issue(nt, nkk, (it + 1) & 1);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();

            const float *st = stage0 + (it & 1) * C::STAGE_FLOATS;
            const float4 *in_s = reinterpret_cast<const float4 *>(st);
            const float4 *w_s4 =
                C::RESIDENT ? reinterpret_cast<const float4 *>(w_res) + (size_t)k * C::C_SH * C::KK * (C::F_TB / 4)
                            : reinterpret_cast<const float4 *>(st + C::IN_CHUNKS * 4);
            if constexpr (C::PAIRC) {
                // the whole step unrolled: every shared-memory address is a
                // per-lane base plus a constant
#pragma unroll
                for (int cb = 0; cb < C::CB; ++cb) {
#pragma unroll
                    for (int r = 0; r < C::K; ++r) {
                        // one input row: W_T + K - 1 pixels x 4 channels
                        const float4 *row = in_s + cb * C::PLANE + (ry + r) * C::TWP;
                        float4 px[C::WIN];
#pragma unroll
                        for (int j = 0; j < C::WIN; ++j) px[j] = row[pcol[j]];
                        // filter units ((cb * K + r) * K + s) * F_TB + co, 4 input channels each
                        const float4 *wr = w_s4 + (cb * C::KK + r * C::K) * C::F_TB + 4 * tx;
#pragma unroll
                        for (int s = 0; s < C::K; ++s) {
                            float4 wv[C::F_T];
#pragma unroll
                            for (int g = 0; g < C::NG; ++g)
#pragma unroll
                                for (int e = 0; e < 4; ++e) wv[4 * g + e] = wr[s * C::F_TB + g * (C::F_TB / C::NG) + e];
                            // input channels 0, 1 of the unit, then 2, 3
#pragma unroll
                            for (int j = 0; j < C::W_T; ++j)
#pragma unroll
                                for (int f = 0; f < C::F_T; ++f)
                                    acc2[f][j] = __ffma2_rn(make_float2(wv[f].x, wv[f].y),
                                                            make_float2(px[j + s].x, px[j + s].y), acc2[f][j]);
#pragma unroll
                            for (int j = 0; j < C::W_T; ++j)
#pragma unroll
                                for (int f = 0; f < C::F_T; ++f)
                                    acc2[f][j] = __ffma2_rn(make_float2(wv[f].z, wv[f].w),
                                                            make_float2(px[j + s].z, px[j + s].w), acc2[f][j]);
                        }
                    }
                }
            } else {
#pragma unroll 1
            for (int cb = 0; cb < C::CB; ++cb) {
#pragma unroll 1
                for (int r = 0; r < C::K; ++r) {
                    // one input row: W_T + K - 1 pixels x 4 channels
                    const float4 *row = in_s + cb * C::PLANE + (ry + r) * C::TWP;
                    float4 px[C::WIN];
#pragma unroll
                    for (int j = 0; j < C::WIN; ++j) px[j] = row[pcol[j]];
                    // filter rows ((4cb + c) * K + r) * K + s
                    const float4 *wr = w_s4 + (4 * cb * C::KK + r * C::K) * (C::F_TB / 4) + tx;
#pragma unroll
                    for (int s = 0; s < C::K; ++s) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float4 *wp = wr + (c * C::KK + s) * (C::F_TB / 4);
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
                                const float2 vv = make_float2(v, v);
                                // packed FP32 FMA on pairs of output channels
#pragma unroll
                                for (int f = 0; f < C::F_T; f += 2) {
                                    float2 a2 = make_float2(acc[f][j], acc[f + 1][j]);
                                    a2 = __ffma2_rn(make_float2(wv[f], wv[f + 1]), vv, a2);
                                    acc[f][j] = a2.x;
                                    acc[f + 1][j] = a2.y;
                                }
                            }
                        }
                    }
                }
            }
            }
            __syncthreads();
        }
        auto res = [&](int f, int j) {
            if constexpr (C::PAIRC) return acc2[f][j].x + acc2[f][j].y;
            else return acc[f][j];
        };

        // epilogue: bias, activation, 16-byte NHWC stores of 4 output channels
        int n, y0, x0;
        decode(tile, n, y0, x0);
        const int gy = y0 + ry;
        if (gy < H) {
#pragma unroll
            for (int g = 0; g < C::NG; ++g) {
                const int co = co0 + g * (C::F_TB / C::NG) + 4 * tx;
                if (co < Cout) {
#pragma unroll
                    for (int j = 0; j < C::W_T; ++j) {
                        const int gx = x0 + cx0 + j;
                        if (gx < W) {
                            float4 o;
                            o.x = relu_if(res(4 * g + 0, j) + bv[4 * g + 0], act);
                            o.y = relu_if(res(4 * g + 1, j) + bv[4 * g + 1], act);
                            o.z = relu_if(res(4 * g + 2, j) + bv[4 * g + 2], act);
                            o.w = relu_if(res(4 * g + 3, j) + bv[4 * g + 3], act);
                            *reinterpret_cast<float4 *>(y + ((((long long)n * H + gy) * W + gx) * Cout + co)) = o;
                        }
                    }
                }
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
    const int cin_pad = (a.Cin + C::C_SH - 1) / C::C_SH * C::C_SH;
    const size_t smem = C::smem_bytes(cin_pad);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static KernelCache cache;
    e = ensure_dynamic_smem(cache, dev, conv_general_kernel<C>, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 1;
    e = resident_ctas(cache, dev, conv_general_kernel<C>, C::NT, (int)smem, &per_sm);
    if (e != cudaSuccess) return e;
    // persistent grid: the resident CTAs, shared out among the output-channel groups
    const long long slots = (long long)per_sm * device_sm_count();
    long long gx = (slots + groups - 1) / groups;
    if (gx > nt) gx = nt;
    if (gx < 1) gx = 1;
    conv_general_kernel<C><<<dim3((unsigned)gx, groups), C::NT, smem, st>>>(
        a.x, a.w, a.b, a.y, a.N, a.H, a.W, a.Cin, a.Cout, a.R, a.S, a.act, tiles_x, tiles_y);
    return cudaGetLastError();
}

// Filters of one output-channel group stay resident in shared memory when
// they take at most this much.
constexpr size_t kResidentFilterBytes = 160 * 1024;

template <int K, int F_TB, int W_T, int TH, int TW, int C_SH, int MINB>
cudaError_t launch_gen_auto(const ConvArgs &a, cudaStream_t st)
{
    const size_t cin_pad = (size_t)(a.Cin + C_SH - 1) / C_SH * C_SH;
    if (cin_pad * K * K * F_TB * 4 <= kResidentFilterBytes)
        return launch_gen<GenCfg<K, F_TB, W_T, TH, TW, C_SH, true, MINB>>(a, st);
    return launch_gen<GenCfg<K, F_TB, W_T, TH, TW, C_SH, false, MINB>>(a, st);
}

// Columns computed beyond the image edge when rows are cut into tiles of tw.
inline int tile_waste(int W, int tw) { return (W + tw - 1) / tw * tw - W; }

// Tiles for more than 16 output channels (measured on GB300, 3x3 layers).
// One CTA per SM with ~160 registers per thread beats two CTAs at 128: with
// fewer registers the FMA stream stalls more at dispatch.  The pixel run per
// thread is 8 or 7, whichever wastes fewer columns at the image edge, and a
// stage holds 16 input channels when Cin is a multiple of 16.
template <int K, int CS>
cudaError_t dispatch_wide(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout > 32) {
        if (tile_waste(a.W, 28) < tile_waste(a.W, 32)) return launch_gen_auto<K, 64, 7, 8, 28, CS, 1>(a, st);
        return launch_gen_auto<K, 64, 8, 8, 32, CS, 1>(a, st);
    }
    if (tile_waste(a.W, 56) < tile_waste(a.W, 64)) return launch_gen_auto<K, 32, 7, 8, 56, CS, 1>(a, st);
    return launch_gen_auto<K, 32, 8, 8, 64, CS, 1>(a, st);
}

// Tiles for 16 or fewer output channels.
template <int K, int CS>
cudaError_t dispatch_narrow(const ConvArgs &a, cudaStream_t st)
{
    if (a.Cout > 8) return launch_gen_auto<K, 16, 4, 4, 64, CS, 2>(a, st);
    if (a.Cout > 4) return launch_gen_auto<K, 8, 4, 4, 128, CS, 2>(a, st);
    return launch_gen_auto<K, 4, 4, 4, 128, CS, 2>(a, st);
}

// Channels per stage: 16 when Cin is a multiple of 16 (3x3 only), else 8;
// 7x7 filter slices staged per step need 4.
template <int K>
constexpr int stage_channels_small() { return K >= 7 ? 4 : 8; }

}  // namespace sc
