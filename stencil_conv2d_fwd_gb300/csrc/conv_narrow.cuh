// Direct convolution for narrow outputs: 3 x 3 filters, at most 4 output
// channels, FP32 FFMA, NHWC activations staged by TMA.
//
// Method: "Optimizing Memory Efficiency for Convolution Kernels on Kepler
// GPUs", Section 3.3 and Algorithm 2, as conv_tma.cuh (a CTA walks over
// TH x TW blocks of output pixels, C_SH input channels of a block plus its
// halo staged per step, each thread reusing a register row of W_T + 2
// pixels over the 3 taps of a filter row), with the changes a layer of 4
// output channels needs on GB300:
//  * With 4 output channels a step holds little arithmetic per staged byte
//    (each 16-byte weight load feeds only W_T x 2 packed FMAs), so the
//    latency of a step's first loads, paid again at every step boundary,
//    is a large share of the step.  Here a consumer warp, while it computes
//    the last filter row of a step, already waits for the next step's stage
//    and loads that step's first input row and first weights into
//    registers, so the next step starts on data in hand.  The steps of a
//    tile are unrolled (NK = Cin / C_SH of them), so the prefetched rows
//    need no register moves.
//  * The producer issues the first copy before the CTA stages its filters,
//    so the filter loads and the first activation copies overlap, and the
//    rest of the ring's first fill once that copy has landed: at the start
//    of a launch every CTA's copies arrive together, and a CTA whose whole
//    ring is in flight waits for most of it before its first stage is
//    complete (per-CTA timestamps on 1280 x 720: the first stage landed
//    6.1 us into the launch, then a tile every 7.7 us).
//  * The tensor map promotes L2 fills to 64 bytes, not 128: a step's copy
//    takes 32 bytes (8 channels) of each 128-byte pixel, and 128-byte
//    promotion made the first step of a tile fetch all 32 channels at once
//    (49.4 -> 48.2 us with the staggered fill, 46.8 us with both).
// The copy protocol (one 4-D TMA box per step into a ring of NSTAGE
// swizzled stages, full/empty mbarriers, bounded waits that record
// SC_ERR_DEVICE_TIMEOUT) and the shared-memory layout are conv_tma.cuh's
// for F_TB = 4: one pixel lane per lane, pixels W_T apart with W_T odd, so
// the 8 lanes of a load phase read 8 distinct bank groups.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace sc {

template <int W_T_, int TH_, int C_SH_, int NSTAGE_, int MINB_, int NK_>
struct N4Cfg {
    static constexpr int K = 3;
    static constexpr int F = 4;                          // output channels per thread (and CTA)
    static constexpr int W_T = W_T_;
    static constexpr int TH = TH_;                       // tile rows = consumer warps
    static constexpr int C_SH = C_SH_;                   // channels per step
    static constexpr int NSTAGE = NSTAGE_;
    static constexpr int MINB = MINB_;
    static constexpr int NK = NK_;                       // steps per tile: Cin = NK * C_SH
    static constexpr int TW = 32 * W_T;
    static constexpr int TWB = (TW + K - 1 + 7) & ~7;    // staged columns (box width)
    static constexpr int THh = TH + K - 1;
    static constexpr int CB = C_SH / 4;
    static constexpr int PXB = C_SH * 4;
    static constexpr int PITCH = TWB * PXB;
    static constexpr int BOX_BYTES = THh * PITCH;
    static constexpr int STAGE_BYTES = (BOX_BYTES + 1023) & ~1023;
    static constexpr int WIN = W_T + K - 1;
    static constexpr int NT = (TH + 1) * 32;
    static constexpr int CIN = NK * C_SH;
    static constexpr int W_UNITS = CIN * K * K;          // float4 filter units [ci][r][s] (4 outputs)
    static_assert(W_T % 2 == 1, "W_T must be odd (bank-conflict-free pixel loads)");
    static_assert(C_SH == 8 || C_SH == 16, "C_SH must be 8 or 16");
    static_assert(TWB <= 256 && THh <= 256, "TMA box dimensions are at most 256");
    static __host__ __device__ int key(int p) { return tma_swz_key(p, C_SH); }
    static size_t smem_bytes() { return (size_t)NSTAGE * STAGE_BYTES + (size_t)W_UNITS * 16 + 2 * NSTAGE * 8 + 1024; }
};

template <class C>
__global__ void __launch_bounds__(C::NT, C::MINB)
    conv_n4_kernel(const __grid_constant__ CUtensorMap tm, const float *__restrict__ w,
                   const float *__restrict__ bias, float *__restrict__ y, int N, int H, int W, int Cout, int R,
                   int S, int act, int tiles_x, int tiles_y, int *status, unsigned long long timeout_ns)
{
    extern __shared__ __align__(1024) unsigned char n4_raw[];
    const uint32_t raw_u32 = smem_u32(n4_raw);
    unsigned char *smem = n4_raw + (((raw_u32 + 1023) & ~1023u) - raw_u32);
    const uint32_t stage0 = smem_u32(smem);
    float4 *w_res = reinterpret_cast<float4 *>(smem + (size_t)C::NSTAGE * C::STAGE_BYTES);
    const uint32_t bars = smem_u32(w_res + C::W_UNITS);   // full[NSTAGE], empty[NSTAGE]
    auto full = [&](int i) { return bars + 8 * i; };
    auto empty = [&](int i) { return bars + 8 * (C::NSTAGE + i); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = tiles_x * tiles_y * N;
    // steps of this CTA: NK per tile of its tiles blockIdx.x, + gridDim.x, ...
    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_tiles * C::NK;
    auto decode = [&](int t, int &n, int &y0, int &x0) {
        x0 = (t % tiles_x) * C::TW;
        t /= tiles_x;
        y0 = (t % tiles_y) * C::TH;
        n = t / tiles_y;
    };
    auto issue = [&](int i) {   // copy i of this CTA: tile blockIdx.x + (i / NK) * gridDim.x, step i % NK
        int n, y0, x0;
        decode(blockIdx.x + (i / C::NK) * gridDim.x, n, y0, x0);
        const int slot = i % C::NSTAGE;
        mbar_arrive_expect_tx(full(slot), C::BOX_BYTES);
        tma_load_4d(stage0 + slot * C::STAGE_BYTES, &tm, (i % C::NK) * C::C_SH, x0 - 1, y0 - 1, n, full(slot));
    };
    const int pre = total < C::NSTAGE ? total : C::NSTAGE;
    const int pre0 = pre < 1 ? pre : 1;   // issued before the filters
    if (warp == C::TH && lane == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), C::TH);
        }
        fence_mbar_init();
        for (int i = 0; i < pre0; ++i) issue(i);
    }
    // filters as float4 units [ci][r][s] of 4 output channels, zero where
    // the R x S filter has no tap or co >= Cout
    for (int e = tid; e < C::W_UNITS * 4; e += C::NT) {
        const int co = e & 3, u = e >> 2;
        const int ci = u / 9, rs = u % 9;
        const int r = rs / 3 - (3 - R) / 2, s = rs % 3 - (3 - S) / 2;
        const bool ok = (co < Cout) & (r >= 0) & (r < R) & (s >= 0) & (s < S);
        const float *src = ok ? w + ((((long long)co * C::CIN + ci) * R + r) * S + s) : w;
        cp_async4(smem_u32(reinterpret_cast<float *>(w_res) + e), src, ok ? 4 : 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();   // barriers initialised and filters staged: roles split below

    if (warp == C::TH) {
        // ---------------- producer: the remaining copies, each into a stage
        // the consumers have released
        if (lane != 0) return;
        bool failed = false;
        if (pre > pre0) {   // the ring's first fill, once the first copy has landed
            (void)mbar_wait_bounded_idle(full(0), 0, timeout_ns, 64);
            for (int k = pre0; k < pre; ++k) issue(k);
        }
        int i = pre;
        for (; i < total; ++i) {
            const int slot = i % C::NSTAGE;
            if (!mbar_wait_bounded_idle(empty(slot), ((i / C::NSTAGE) - 1) & 1, timeout_ns, 64)) {
                failed = true;
                break;
            }
            fence_proxy_async_smem();   // the consumers' reads come before the copy's writes
            issue(i);
        }
        if (failed) atomicExch(status, kDeviceTimeout);
        for (int k = i - C::NSTAGE > 0 ? i - C::NSTAGE : 0; k < i; ++k)
            (void)mbar_wait_bounded(full(k % C::NSTAGE), (k / C::NSTAGE) & 1, timeout_ns);
        return;
    }

    // ---------------- consumers: warp `warp` computes tile row `warp`
    const int cx0 = lane * C::W_T;
    uint32_t poff[C::WIN][C::CB];   // byte offset in a stage of (tile row warp, pixel cx0 + j, chunk cb)
#pragma unroll
    for (int j = 0; j < C::WIN; ++j)
#pragma unroll
        for (int cb = 0; cb < C::CB; ++cb)
            poff[j][cb] = warp * C::PITCH + (cx0 + j) * C::PXB + ((cb ^ C::key(cx0 + j)) << 4);
    float bv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) bv[e] = (bias && e < Cout) ? bias[e] : 0.0f;

    auto ld4 = [](const unsigned char *p) { return *reinterpret_cast<const float4 *>(p); };
    auto wait_full = [&](int i) { return mbar_wait_bounded(full(i % C::NSTAGE), (i / C::NSTAGE) & 1, timeout_ns); };
    // input row q (0..2) of chunk cb of step i's stage
    auto row_ptr = [&](int i, int j, int cb, int q) {
        return smem + (i % C::NSTAGE) * C::STAGE_BYTES + poff[j][cb] + q * C::PITCH;
    };
    const float4 *wq = w_res;

    // step i's first row (chunk 0, filter row 0) and its first weight units,
    // loaded ahead of the step
    float4 nrow[C::WIN];
    float4 nw0 = make_float4(0.f, 0.f, 0.f, 0.f), nw1 = nw0;
    if (total > 0) {
        if (!wait_full(0)) {
            if (lane == 0) atomicExch(status, kDeviceTimeout);
            return;
        }
#pragma unroll
        for (int j = 0; j < C::WIN; ++j) nrow[j] = ld4(row_ptr(0, j, 0, 0));
        nw0 = wq[0];
        nw1 = wq[C::K * C::K];
    }
    int i = 0;   // this CTA's step counter
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        float acc[4][C::W_T];
#pragma unroll
        for (int f = 0; f < 4; ++f)
#pragma unroll
            for (int j = 0; j < C::W_T; ++j) acc[f][j] = 0.0f;
        const bool more_tiles = t + (int)gridDim.x < ntiles;
#pragma unroll
        for (int k = 0; k < C::NK; ++k, ++i) {
            const bool has_next = (k + 1 < C::NK) || more_tiles;
#pragma unroll
            for (int cb = 0; cb < C::CB; ++cb) {
#pragma unroll
                for (int r = 0; r < C::K; ++r) {
                    float4 px[C::WIN];
                    if (cb == 0 && r == 0) {
#pragma unroll
                        for (int j = 0; j < C::WIN; ++j) px[j] = nrow[j];
                    } else {
#pragma unroll
                        for (int j = 0; j < C::WIN; ++j) px[j] = ld4(row_ptr(i, j, cb, r));
                    }
#pragma unroll
                    for (int s = 0; s < C::K; ++s) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            // unit of (channel k * C_SH + 4 cb + c, r, s)
                            const int u = ((k * C::C_SH + 4 * cb + c) * C::K + r) * C::K + s;
                            float4 wv;
                            if (cb == 0 && r == 0 && s == 0 && c < 2)
                                wv = c == 0 ? nw0 : nw1;
                            else
                                wv = wq[u];
                            if (cb == C::CB - 1 && r == C::K - 1 && s == 1 && c == 0 && has_next) {
                                // the next step's stage and first loads, while
                                // this step's last filter row is still computing
                                if (!wait_full(i + 1)) {
                                    if (lane == 0) atomicExch(status, kDeviceTimeout);
                                    return;
                                }
                                const int kn = k + 1 < C::NK ? k + 1 : 0;
#pragma unroll
                                for (int j = 0; j < C::WIN; ++j) nrow[j] = ld4(row_ptr(i + 1, j, 0, 0));
                                nw0 = wq[(kn * C::C_SH * C::K) * C::K];
                                nw1 = wq[((kn * C::C_SH + 1) * C::K) * C::K];
                            }
#pragma unroll
                            for (int j = 0; j < C::W_T; ++j) {
                                const float4 p = px[j + s];
                                const float v = c == 0 ? p.x : (c == 1 ? p.y : (c == 2 ? p.z : p.w));
                                const float2 vv = make_float2(v, v);
                                float2 a = __ffma2_rn(make_float2(wv.x, wv.y), vv, make_float2(acc[0][j], acc[1][j]));
                                acc[0][j] = a.x;
                                acc[1][j] = a.y;
                                a = __ffma2_rn(make_float2(wv.z, wv.w), vv, make_float2(acc[2][j], acc[3][j]));
                                acc[2][j] = a.x;
                                acc[3][j] = a.y;
                            }
                        }
                    }
                }
            }
            // every lane's reads of this stage are done: release it
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(i % C::NSTAGE));
        }

        // epilogue: bias, activation, 16-byte NHWC stores of the 4 outputs,
        // all W_T values formed before the first store and the stores of a
        // row inside the image issued without per-pixel tests (1.0-1.6 us
        // less on 1280 x 720 than forming and storing pixel by pixel)
        int n, y0, x0;
        decode(t, n, y0, x0);
        const int gy = y0 + warp;
        if (gy < H) {
            float4 o[C::W_T];
#pragma unroll
            for (int j = 0; j < C::W_T; ++j) {
                o[j].x = relu_if(acc[0][j] + bv[0], act);
                o[j].y = relu_if(acc[1][j] + bv[1], act);
                o[j].z = relu_if(acc[2][j] + bv[2], act);
                o[j].w = relu_if(acc[3][j] + bv[3], act);
            }
            float4 *yp = reinterpret_cast<float4 *>(y + (((long long)n * H + gy) * W + x0 + cx0) * 4);
            if (x0 + cx0 + C::W_T <= W) {
#pragma unroll
                for (int j = 0; j < C::W_T; ++j) yp[j] = o[j];
            } else {
#pragma unroll
                for (int j = 0; j < C::W_T; ++j)
                    if (x0 + cx0 + j < W) yp[j] = o[j];
            }
        }
    }
}

// The driver's tensor-map encoder (conv_tma_k3.cu), or nullptr.
PFN_cuTensorMapEncodeTiled_v12000 conv_tma_encoder();

// Launch for NHWC x with Cin == C::CIN and Cout == 4, 3 x 3 (or smaller,
// centred) filters; cudaErrorNotSupported where it does not apply.
template <class C>
cudaError_t launch_conv_n4(const ConvArgs &a, cudaStream_t st, unsigned long long timeout_ns = 1000000000ull)
{
    if (a.Cin != C::CIN || a.Cout != 4 || a.R > 3 || a.S > 3) return cudaErrorNotSupported;
    const int tiles_x = (a.W + C::TW - 1) / C::TW;
    const int tiles_y = (a.H + C::TH - 1) / C::TH;
    const long long nt = (long long)tiles_x * tiles_y * a.N;
    if (nt > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    PFN_cuTensorMapEncodeTiled_v12000 encode = conv_tma_encoder();
    int *status = device_status_ptr();
    if (!encode || !status) return cudaErrorNotSupported;
    CUtensorMap tm;
    const cuuint64_t dims[4] = {(cuuint64_t)a.Cin, (cuuint64_t)a.W, (cuuint64_t)a.H, (cuuint64_t)a.N};
    const cuuint64_t strides[3] = {(cuuint64_t)a.Cin * 4, (cuuint64_t)a.W * a.Cin * 4,
                                   (cuuint64_t)a.H * a.W * a.Cin * 4};
    const cuuint32_t box[4] = {(cuuint32_t)C::C_SH, (cuuint32_t)C::TWB, (cuuint32_t)C::THh, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle swz = C::PXB == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(a.x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    const size_t smem = C::smem_bytes();
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static KernelCache cache;
    e = ensure_dynamic_smem(cache, dev, conv_n4_kernel<C>, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 1;
    e = resident_ctas(cache, dev, conv_n4_kernel<C>, C::NT, (int)smem, &per_sm);
    if (e != cudaSuccess) return e;
    long long gx = (long long)per_sm * device_sm_count();
    if (gx > nt) gx = nt;
    if (gx < 1) gx = 1;
    conv_n4_kernel<C><<<(unsigned)gx, C::NT, smem, st>>>(tm, a.w, a.b, a.y, a.N, a.H, a.W, a.Cout, a.R, a.S, a.act,
                                                         tiles_x, tiles_y, status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace sc
