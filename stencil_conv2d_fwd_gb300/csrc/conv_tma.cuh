// General-case direct convolution, FP32 FFMA, NHWC activations, with the
// activation tiles staged by the Tensor Memory Accelerator (TMA).
//
// Method: "Optimizing Memory Efficiency for Convolution Kernels on Kepler
// GPUs", Section 3.3 (general case) and Algorithm 2, as in
// conv_general.cuh: a CTA owns F_TB output channels and walks over TH x TW
// blocks of output pixels; C_SH input channels of a block plus its halo are
// staged in shared memory per step while later steps are in flight; each
// thread accumulates F_T filters x W_T horizontally contiguous pixels and
// reuses a register row of W_T + K - 1 pixels over the K taps of that row.
//
// What differs from conv_general.cuh:
//  * Staging.  One thread of a producer warp stages a whole step (C_SH
//    channels of the (TH + K - 1) x (TW + K - 1) halo tile) with one 4-D TMA
//    copy into a ring of NSTAGE shared-memory stages.  The copy's zero fill
//    gives the zero "same" padding, the channels beyond Cin and the ragged
//    right and bottom edges.  Consumer warps wait on the stage's mbarrier and
//    release it with one arrive per warp.  There are no per-element copy
//    instructions (with 4 output channels those cost as many instructions
//    as the FMAs) and no block-wide barriers.
//  * Layout and bank conflicts.  A pixel takes C_SH * 4 bytes of a stage
//    (32, 64 or 128), and the copy uses the TMA swizzle of that span
//    ("CUDA共有メモリのスウィズリング": 16-byte chunk q of pixel p is stored at
//    chunk q ^ key(p), key(p) = (p * C_SH / 32) mod (C_SH / 4)).  A stage row
//    holds a multiple of 8 pixels, so key depends on p only.  The 16-byte
//    bank group of (p, q) is then a one-to-one function of p mod 8 for
//    each q, and a thread owns W_T consecutive pixels with W_T odd, so the
//    8 lanes of a 16-byte load phase (8 consecutive pixel lanes) read
//    pixels that differ mod 8: 8 distinct bank groups.
//  * The FMAs are packed dual-FP32 FMAs (__ffma2_rn), each component
//    rounding like fmaf.  PAIRC pairs input channels: each output keeps two
//    partial sums (even and odd input channels, added once at the end), so
//    both operands are halves of 16-byte units (4 channels of a pixel; 4
//    input channels of one output channel's tap, the filter bank staged as
//    [ci / 4][r][s][F_TB][4]).  Otherwise pairs of output channels, as in
//    conv_general.cuh.
//  * Rows per consumer warp (H_T): a warp may compute H_T tile rows; the
//    input rows it reads sit in a register ring (row q in slot q mod H_T),
//    so each filter unit is loaded once for H_T rows and each input row
//    once for up to H_T output rows.
//  * Every wait is bounded: on expiry the kernel records
//    SC_ERR_DEVICE_TIMEOUT in the status word, the producer lets its copies
//    still in flight land, and the CTA returns.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace sc {

template <int K_, int F_TB_, int W_T_, int TH_, int H_T_, int C_SH_, int NSTAGE_, int MINB_, bool PAIRC_>
struct TmaCfg {
    static constexpr int K = K_;
    static constexpr int F_TB = F_TB_;
    static constexpr int W_T = W_T_;
    static constexpr int TH = TH_;                      // tile rows
    static constexpr int H_T = H_T_;                    // tile rows per consumer warp
    static constexpr int C_SH = C_SH_;                  // channels per step
    static constexpr int NSTAGE = NSTAGE_;
    static constexpr int MINB = MINB_;
    static constexpr bool PAIRC = PAIRC_;
    static constexpr int F_T = F_TB >= 8 ? 8 : 4;       // output channels per thread
    static constexpr int NG = F_T / 4;                   // float4 groups per thread
    static constexpr int T_X = F_TB / F_T;               // lanes along output channels
    static constexpr int PXL = 32 / T_X;                 // lanes along pixels
    static constexpr int TW = PXL * W_T;                 // tile columns
    static constexpr int TWU = TW + K - 1;
    static constexpr int TWB = (TWU + 7) & ~7;           // staged columns (box width)
    static constexpr int THh = TH + K - 1;
    static constexpr int CB = C_SH / 4;                  // 16-byte chunks per pixel
    static constexpr int PXB = C_SH * 4;                 // bytes per staged pixel (= swizzle span)
    static constexpr int PITCH = TWB * PXB;              // bytes per stage row
    static constexpr int BOX_BYTES = THh * PITCH;
    static constexpr int STAGE_BYTES = (BOX_BYTES + 1023) & ~1023;
    static constexpr int KK = K * K;
    static constexpr int WIN = W_T + K - 1;
    static constexpr int NC = TH / H_T;                  // consumer warps
    static constexpr int NT = (NC + 1) * 32;             // + the producer warp
    static_assert(W_T % 2 == 1, "W_T must be odd (bank-conflict-free pixel loads)");
    static_assert(TH % H_T == 0, "whole rows per consumer warp");
    static_assert(C_SH == 8 || C_SH == 16 || C_SH == 32, "C_SH must be 8, 16 or 32");
    static_assert(F_TB % F_T == 0 && 32 % T_X == 0, "bad channel split");
    static_assert(TWB <= 256 && THh <= 256, "TMA box dimensions are at most 256");
    static_assert(NT <= 1024, "too many threads");
    // swizzle key of staged pixel p (a stage row holds a multiple of 8 pixels)
    static __host__ __device__ int key(int p) { return tma_swz_key(p, C_SH); }
    // shared memory: [NSTAGE stages][filter bank][barriers]
    static __host__ __device__ size_t w_floats(int cin_pad) { return (size_t)cin_pad * KK * F_TB; }
    static size_t smem_bytes(int cin_pad)
    {
        return (size_t)NSTAGE * STAGE_BYTES + w_floats(cin_pad) * 4 + 2 * NSTAGE * 8 + 1024;
    }
};

// Filters of input channels [0, cin_pad) into the resident bank, zero where
// the R x S filter has no tap, where co >= Cout or ci >= Cin:
//  * PAIRC: ws[(ci / 4) * KK + r * K + s][F_TB][4];
//  * else:  ws[ci * KK + r * K + s][F_TB].
// Consecutive threads write consecutive shared-memory words.
template <class C>
__device__ __forceinline__ void tma_issue_filters(float *ws, const float *__restrict__ w, int co0, int cin_pad,
                                                  int Cin, int Cout, int R, int S, int tid)
{
    const int n = cin_pad * C::KK * C::F_TB;
    const int dr = (C::K - R) / 2, ds = (C::K - S) / 2;
    for (int e = tid; e < n; e += C::NT) {
        int col, ci, rs;
        if constexpr (C::PAIRC) {
            col = (e >> 2) % C::F_TB;
            const int t = e / (4 * C::F_TB);
            rs = t % C::KK;
            ci = (t / C::KK) * 4 + (e & 3);
        } else {
            col = e % C::F_TB;
            const int row = e / C::F_TB;
            ci = row / C::KK;
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

// The same bank from 16-byte loads, for R = S = K (so the bank's row index
// ci * KK + rs is the OIHW row's own element index) and a 16-byte-aligned w
// with Cin % 4 == 0: each thread reads 4 consecutive elements of one output
// channel's OIHW row and writes them to 4 bank rows; the lanes of a warp
// take consecutive output channels, so each 4-byte shared store of the warp
// fills 32 consecutive words.  Four times fewer global requests than one per
// element, and no 4-byte asynchronous copies.  Not for PAIRC banks.
template <class C>
__device__ __forceinline__ void tma_load_filters_v4(float *ws, const float *__restrict__ w, int co0, int cin_pad,
                                                    int Cin, int Cout, int tid)
{
    const int row = Cin * C::KK;              // floats of one output channel's OIHW row
    const int nq = cin_pad * C::KK / 4;       // 4-element pieces of a bank column
    const int n = nq * C::F_TB;
    // four pieces a thread in flight before any is stored, so that the
    // loads' latencies overlap
    constexpr int B = 4;
    for (int e0 = tid; e0 < n; e0 += B * C::NT) {
        float4 v[B];
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int e = e0 + b * C::NT;
            const int col = e % C::F_TB, m = e / C::F_TB;
            const int co = co0 + col;
            v[b] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < n && co < Cout && 4 * m < row) v[b] = __ldg(reinterpret_cast<const float4 *>(w + (long long)co * row) + m);
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int e = e0 + b * C::NT;
            if (e < n) {
                const int col = e % C::F_TB, m = e / C::F_TB;
                float *dst = ws + (size_t)(4 * m) * C::F_TB + col;
                dst[0] = v[b].x;
                dst[C::F_TB] = v[b].y;
                dst[2 * C::F_TB] = v[b].z;
                dst[3 * C::F_TB] = v[b].w;
            }
        }
    }
}

template <class C>
__global__ void __launch_bounds__(C::NT, C::MINB)
    conv_tma_kernel(const __grid_constant__ CUtensorMap tm, const float *__restrict__ w,
                    const float *__restrict__ bias, float *__restrict__ y, int N, int H, int W, int Cin, int Cout,
                    int R, int S, int act, int tiles_x, int tiles_y, int *status, unsigned long long timeout_ns,
                    int drop_copy)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the dynamic buffer is 1024-byte aligned in practice; align explicitly
    // (smem_bytes reserves the slack)
    const uint32_t raw_u32 = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw_u32 + 1023) & ~1023u) - raw_u32);
    const uint32_t stage0 = smem_u32(smem);
    const int cin_pad = (Cin + C::C_SH - 1) / C::C_SH * C::C_SH;
    float *w_res = reinterpret_cast<float *>(smem + (size_t)C::NSTAGE * C::STAGE_BYTES);
    const uint32_t bars = smem_u32(w_res + C::w_floats(cin_pad));   // full[NSTAGE], empty[NSTAGE]
    auto full = [&](int i) { return bars + 8 * i; };
    auto empty = [&](int i) { return bars + 8 * (C::NSTAGE + i); };

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int co0 = blockIdx.y * C::F_TB;
    const int nk = cin_pad / C::C_SH;
    const int ntiles = tiles_x * tiles_y * N;

    auto decode = [&](int t, int &n, int &y0, int &x0) {
        x0 = (t % tiles_x) * C::TW;
        t /= tiles_x;
        y0 = (t % tiles_y) * C::TH;
        n = t / tiles_y;
    };
    // copy i of this CTA: step i % nk of tile blockIdx.x + (i / nk) * gridDim.x
    auto issue = [&](int i, int t, int k) {
        int n, y0, x0;
        decode(t, n, y0, x0);
        const int slot = i % C::NSTAGE;
        mbar_arrive_expect_tx(full(slot), C::BOX_BYTES);
        if (i != drop_copy)   // test hook: that copy is never issued
            tma_load_4d(stage0 + slot * C::STAGE_BYTES, &tm, k * C::C_SH, x0 - C::K / 2, y0 - C::K / 2, n, full(slot));
    };
    const int my_tiles = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int pre = my_tiles * nk < C::NSTAGE ? my_tiles * nk : C::NSTAGE;
    const int pre0 = pre < 1 ? pre : 1;   // issued before the filters
    if (warp == C::NC && lane == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), C::NC);
        }
        fence_mbar_init();
        // the first copy goes out before the filters are staged, so the two
        // loads overlap
        for (int i = 0; i < pre0; ++i) issue(i, blockIdx.x + (i / nk) * gridDim.x, i % nk);
    }
    // large banks (64 -> 64: 147 KB a CTA, 146.7 -> 128.4 us) from 16-byte
    // loads; small ones (16 -> 16: 9 KB) keep the asynchronous copies, which
    // overlap the first activation copies entirely
    bool v4 = false;
    if constexpr (!C::PAIRC)
        v4 = R == C::K && S == C::K && (Cin & 3) == 0 && (reinterpret_cast<uintptr_t>(w) & 15) == 0 &&
             C::w_floats(cin_pad) >= 8192;
    if (v4) {
        tma_load_filters_v4<C>(w_res, w, co0, cin_pad, Cin, Cout, tid);
    } else {
        tma_issue_filters<C>(w_res, w, co0, cin_pad, Cin, Cout, R, S, tid);
        cp_async_commit();
        cp_async_wait<0>();
    }
    __syncthreads();   // the last block-wide barrier: roles split below

    if (warp == C::NC) {
        // ---------------- producer: one thread issues every copy ----------
        if (lane != 0) return;
        int issued = 0;
        bool failed = false;
        if (pre > pre0) {   // the ring's first fill, once the first copy has landed
            (void)mbar_wait_bounded_idle(full(0), 0, timeout_ns, 64);
            for (int i = pre0; i < pre; ++i) issue(i, blockIdx.x + (i / nk) * gridDim.x, i % nk);
        }
        for (int t = blockIdx.x; t < ntiles && !failed; t += gridDim.x) {
            for (int k = 0; k < nk; ++k, ++issued) {
                if (issued < pre) continue;   // issued before the filters
                const int slot = issued % C::NSTAGE;
                if (issued >= C::NSTAGE &&
                    !mbar_wait_bounded_idle(empty(slot), ((issued / C::NSTAGE) - 1) & 1, timeout_ns, 64)) {
                    failed = true;
                    break;
                }
                // the consumers' reads of this stage come before the copy's writes
                fence_proxy_async_smem();
                issue(issued, t, k);
            }
        }
        if (failed) atomicExch(status, kDeviceTimeout);
        // copies still in flight land before the CTA may exit (each wait
        // returns at once for a stage the consumers already took)
        for (int i = issued - C::NSTAGE > 0 ? issued - C::NSTAGE : 0; i < issued; ++i)
            (void)mbar_wait_bounded(full(i % C::NSTAGE), (i / C::NSTAGE) & 1, timeout_ns);
        return;
    }

    // ---------------- consumers: warp `warp` computes tile rows warp * H_T .. + H_T - 1
    const int tx = lane % C::T_X;   // output-channel lane
    const int pl = lane / C::T_X;   // pixel lane
    const int cx0 = pl * C::W_T;    // first tile column of this lane
    // byte offset in a stage of (tile row warp * H_T, pixel cx0 + j, chunk cb)
    uint32_t poff[C::WIN][C::CB];
#pragma unroll
    for (int j = 0; j < C::WIN; ++j)
#pragma unroll
        for (int cb = 0; cb < C::CB; ++cb)
            poff[j][cb] = warp * C::H_T * C::PITCH + (cx0 + j) * C::PXB + ((cb ^ C::key(cx0 + j)) << 4);

    float bv[C::F_T];
#pragma unroll
    for (int g = 0; g < C::NG; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int co = co0 + g * (C::F_TB / C::NG) + 4 * tx + e;
            bv[4 * g + e] = (bias && co < Cout) ? bias[co] : 0.0f;
        }
    const unsigned char *wbase = reinterpret_cast<const unsigned char *>(w_res);
    auto ld4 = [](const unsigned char *p) { return *reinterpret_cast<const float4 *>(p); };

    // accumulators [output row][channel][pixel]: channel pairing uses acc,
    // PAIRC the (even, odd input channel) partial sums acc2
    constexpr int AH = C::PAIRC ? 1 : C::H_T, AF = C::PAIRC ? 1 : C::F_T, AW = C::PAIRC ? 1 : C::W_T;
    constexpr int PH = C::PAIRC ? C::H_T : 1, PF = C::PAIRC ? C::F_T : 1, PW = C::PAIRC ? C::W_T : 1;
    int it = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        float acc[AH][AF][AW];
        float2 acc2[PH][PF][PW];
#pragma unroll
        for (int h = 0; h < AH; ++h)
#pragma unroll
            for (int f = 0; f < AF; ++f)
#pragma unroll
                for (int j = 0; j < AW; ++j) acc[h][f][j] = 0.0f;
#pragma unroll
        for (int h = 0; h < PH; ++h)
#pragma unroll
            for (int f = 0; f < PF; ++f)
#pragma unroll
                for (int j = 0; j < PW; ++j) acc2[h][f][j] = make_float2(0.0f, 0.0f);

        for (int k = 0; k < nk; ++k, ++it) {
            const int slot = it % C::NSTAGE;
            if (!mbar_wait_bounded(full(slot), (it / C::NSTAGE) & 1, timeout_ns)) {
                if (lane == 0) atomicExch(status, kDeviceTimeout);
                return;
            }
            const unsigned char *sbase = smem + slot * C::STAGE_BYTES;
            const unsigned char *pa[C::WIN][C::CB];
#pragma unroll
            for (int j = 0; j < C::WIN; ++j)
#pragma unroll
                for (int cb = 0; cb < C::CB; ++cb) pa[j][cb] = sbase + poff[j][cb];
            // filters of this step's channels: float4 units
            const unsigned char *wk = wbase + (size_t)k * (C::CB * C::KK * C::F_TB * 16);
#pragma unroll
            for (int cb = 0; cb < C::CB; ++cb) {
                // register ring of input rows: row q (from the warp's first
                // tile row) in pw[q % H_T]; output row h uses rows h .. h + K - 1
                float4 pw[C::H_T][C::WIN];
#pragma unroll
                for (int q = 0; q < C::H_T - 1; ++q)
#pragma unroll
                    for (int j = 0; j < C::WIN; ++j) pw[q % C::H_T][j] = ld4(pa[j][cb] + q * C::PITCH);
#pragma unroll
                for (int r = 0; r < C::K; ++r) {
                    const int qn = r + C::H_T - 1;   // the row this filter row brings in
#pragma unroll
                    for (int j = 0; j < C::WIN; ++j) pw[qn % C::H_T][j] = ld4(pa[j][cb] + qn * C::PITCH);
                    if constexpr (C::PAIRC) {
#pragma unroll
                        for (int s = 0; s < C::K; ++s) {
                            // unit ((cb * K + r) * K + s) * F_TB + co: 4 input channels
                            const unsigned char *wu = wk + (((cb * C::K + r) * C::K + s) * C::F_TB + 4 * tx) * 16;
                            float4 wv[C::F_T];
#pragma unroll
                            for (int g = 0; g < C::NG; ++g)
#pragma unroll
                                for (int e = 0; e < 4; ++e) wv[4 * g + e] = ld4(wu + (g * (C::F_TB / C::NG) + e) * 16);
#pragma unroll
                            for (int h = 0; h < C::H_T; ++h) {
                                const float4(&px)[C::WIN] = pw[(r + h) % C::H_T];
#pragma unroll
                                for (int j = 0; j < C::W_T; ++j)
#pragma unroll
                                    for (int f = 0; f < C::F_T; ++f)
                                        acc2[h][f][j] = __ffma2_rn(make_float2(wv[f].x, wv[f].y),
                                                                   make_float2(px[j + s].x, px[j + s].y), acc2[h][f][j]);
#pragma unroll
                                for (int j = 0; j < C::W_T; ++j)
#pragma unroll
                                    for (int f = 0; f < C::F_T; ++f)
                                        acc2[h][f][j] = __ffma2_rn(make_float2(wv[f].z, wv[f].w),
                                                                   make_float2(px[j + s].z, px[j + s].w), acc2[h][f][j]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int s = 0; s < C::K; ++s) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                // filter row ((4 cb + c) * K + r) * K + s: F_TB output channels
                                const unsigned char *wu = wk + ((((4 * cb + c) * C::K + r) * C::K + s) * (C::F_TB / 4) + tx) * 16;
                                float wv[C::F_T];
#pragma unroll
                                for (int g = 0; g < C::NG; ++g) {
                                    const float4 q = ld4(wu + g * C::T_X * 16);
                                    wv[4 * g + 0] = q.x;
                                    wv[4 * g + 1] = q.y;
                                    wv[4 * g + 2] = q.z;
                                    wv[4 * g + 3] = q.w;
                                }
#pragma unroll
                                for (int h = 0; h < C::H_T; ++h) {
                                    const float4(&px)[C::WIN] = pw[(r + h) % C::H_T];
#pragma unroll
                                    for (int j = 0; j < C::W_T; ++j) {
                                        const float4 p = px[j + s];
                                        const float v = c == 0 ? p.x : (c == 1 ? p.y : (c == 2 ? p.z : p.w));
                                        const float2 vv = make_float2(v, v);
#pragma unroll
                                        for (int f = 0; f < C::F_T; f += 2) {
                                            float2 a2 = make_float2(acc[h][f][j], acc[h][f + 1][j]);
                                            a2 = __ffma2_rn(make_float2(wv[f], wv[f + 1]), vv, a2);
                                            acc[h][f][j] = a2.x;
                                            acc[h][f + 1][j] = a2.y;
                                        }
                                    }
                                }
                            }
                        }
                    }
                }
            }
            // every lane's reads of this stage are done: release it
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(slot));
        }

        // epilogue: bias, activation, 16-byte NHWC stores of 4 output
        // channels; a group's W_T values are formed before its first store,
        // and rows inside the image store without per-pixel tests (32 -> 32
        // on 1280 x 720: 279.6 -> 275.1 us)
        auto res = [&](int h, int f, int j) {
            if constexpr (C::PAIRC) return acc2[h][f][j].x + acc2[h][f][j].y;
            else return acc[h][f][j];
        };
        int n, y0, x0;
        decode(t, n, y0, x0);
        const bool full_row = x0 + cx0 + C::W_T <= W;
#pragma unroll
        for (int h = 0; h < C::H_T; ++h) {
            const int gy = y0 + warp * C::H_T + h;
            if (gy < H) {
#pragma unroll
                for (int g = 0; g < C::NG; ++g) {
                    const int co = co0 + g * (C::F_TB / C::NG) + 4 * tx;
                    if (co < Cout) {
                        float4 o[C::W_T];
#pragma unroll
                        for (int j = 0; j < C::W_T; ++j) {
                            o[j].x = relu_if(res(h, 4 * g + 0, j) + bv[4 * g + 0], act);
                            o[j].y = relu_if(res(h, 4 * g + 1, j) + bv[4 * g + 1], act);
                            o[j].z = relu_if(res(h, 4 * g + 2, j) + bv[4 * g + 2], act);
                            o[j].w = relu_if(res(h, 4 * g + 3, j) + bv[4 * g + 3], act);
                        }
                        float *yp = y + ((((long long)n * H + gy) * W + x0 + cx0) * Cout + co);
                        if (full_row) {
#pragma unroll
                            for (int j = 0; j < C::W_T; ++j) *reinterpret_cast<float4 *>(yp + (long long)j * Cout) = o[j];
                        } else {
#pragma unroll
                            for (int j = 0; j < C::W_T; ++j)
                                if (x0 + cx0 + j < W) *reinterpret_cast<float4 *>(yp + (long long)j * Cout) = o[j];
                        }
                    }
                }
            }
        }
    }
}

// The driver's tensor-map encoder (cached), or nullptr.
PFN_cuTensorMapEncodeTiled_v12000 conv_tma_encoder();

// Filters of one output-channel group stay resident in shared memory when
// they take at most this much; larger banks are not supported here.
constexpr size_t kTmaFilterBytes = 160 * 1024;
// Opt-in shared memory per CTA on sm_103.
constexpr size_t kTmaMaxSmem = 227 * 1024;

// drop_copy >= 0 leaves that copy of every CTA (0-based, in issue order)
// un-issued, so the waits for it expire after timeout_ns (tests of the
// device-status path).
template <class C>
cudaError_t launch_conv_tma(const ConvArgs &a, cudaStream_t st, int drop_copy = -1,
                            unsigned long long timeout_ns = 1000000000ull)
{
    const int cin_pad = (a.Cin + C::C_SH - 1) / C::C_SH * C::C_SH;
    if ((size_t)cin_pad * C::KK * C::F_TB * 4 > kTmaFilterBytes || a.R > C::K || a.S > C::K || (a.Cin & 3))
        return cudaErrorNotSupported;
    const int tiles_x = (a.W + C::TW - 1) / C::TW;
    const int tiles_y = (a.H + C::TH - 1) / C::TH;
    const long long nt = (long long)tiles_x * tiles_y * a.N;
    const int groups = (a.Cout + C::F_TB - 1) / C::F_TB;
    if (nt > 0x7fffffffLL || groups > 65535) return cudaErrorInvalidConfiguration;
    PFN_cuTensorMapEncodeTiled_v12000 encode = conv_tma_encoder();
    int *status = device_status_ptr();
    if (!encode || !status) return cudaErrorNotSupported;
    // NHWC activations as a 4-D tensor (C, W, H, N); box = C_SH channels x
    // TWB columns x THh rows of one image, swizzled with the span of one
    // staged pixel
    CUtensorMap tm;
    const cuuint64_t dims[4] = {(cuuint64_t)a.Cin, (cuuint64_t)a.W, (cuuint64_t)a.H, (cuuint64_t)a.N};
    const cuuint64_t strides[3] = {(cuuint64_t)a.Cin * 4, (cuuint64_t)a.W * a.Cin * 4,
                                   (cuuint64_t)a.H * a.W * a.Cin * 4};
    const cuuint32_t box[4] = {(cuuint32_t)C::C_SH, (cuuint32_t)C::TWB, (cuuint32_t)C::THh, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle swz = C::PXB == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                   : C::PXB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    // L2 fills promoted to 64 bytes: a step copies C_SH channels (32 or 64
    // bytes) of each pixel, and 128-byte promotion fetched the other steps'
    // channels with the first step (32 -> 32: 276.3 -> 275.0 us)
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(a.x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    const size_t smem = C::smem_bytes(cin_pad);
    if (smem > kTmaMaxSmem) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static KernelCache cache;
    e = ensure_dynamic_smem(cache, dev, conv_tma_kernel<C>, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 1;
    e = resident_ctas(cache, dev, conv_tma_kernel<C>, C::NT, (int)smem, &per_sm);
    if (e != cudaSuccess) return e;
    // persistent grid: the resident CTAs, shared out among the output-channel groups
    const long long slots = (long long)per_sm * device_sm_count();
    long long gx = (slots + groups - 1) / groups;
    if (gx > nt) gx = nt;
    if (gx < 1) gx = 1;
    conv_tma_kernel<C><<<dim3((unsigned)gx, groups), C::NT, smem, st>>>(
        tm, a.w, a.b, a.y, a.N, a.H, a.W, a.Cin, a.Cout, a.R, a.S, a.act, tiles_x, tiles_y, status, timeout_ns,
        drop_copy);
    return cudaGetLastError();
}

}  // namespace sc
