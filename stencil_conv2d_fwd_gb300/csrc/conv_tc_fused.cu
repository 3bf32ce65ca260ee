// Two 3 x 3 convolution layers fused in one pass on the tensor cores: the
// intermediate activation never reaches HBM ("Optimizing convolution kernels -
// CNNs in Vulkan Part 2/3", section "Reducing memory traffic": most of a
// network's traffic is activations written by one layer and read back by the
// next; "Model-Based Warp Overlapped Tiling for Image Processing Programs on
// GPUs", Abstract: overlapped tiles recompute a producer stage's halo so a
// consumer stage can run from on-chip data).
//
//   t = act1(conv3x3(x, w1) + b1)   C0 -> C1 = 32 channels, TF32 operands
//   y = act2(conv3x3(t, w2) + b2)   32 -> C2 <= 8 channels, TF32 operands
//
// Tiles overlap: each tile computes layer 1 for 8 rows x 30 columns and
// layer 2 for the interior 6 rows x 28 columns (layer 2 reads a 1-pixel halo
// of layer 1's output), so tiles step by 6 rows and 28 columns and layer 1 is
// recomputed on the overlap (1.43x).  Layer 1 is the kernel of conv_tc.cu
// (horizontal taps stacked in N = 96, vertical taps as A row offsets, two
// M-tiles of 128 rows); its epilogue adds b1, applies act1, writes zero for
// pixels outside the image (layer 2's zero padding) and stores the 8 x 32
// pixels x 32 channels into a shared tile T laid out exactly like a stage
// (128-byte swizzled rows, row pitch 32 pixels): T is layer 2's A operand.
// Layer 2 then runs the same scheme (N = 3 * CG2 rounded to 16) from T; its
// epilogue adds b2, applies act2 and writes y.
//
// Roles (352 threads, one persistent CTA per SM): the producer streams layer
// 1's 32-channel input stages by TMA; one MMA lane issues layer 1 tile by
// tile, another layer 2 (each waits on its own barriers while the other's
// MMAs keep the tensor core busy); the eight epilogue warps (TMEM lane
// quadrant = warp % 4, M-tile = warp set) finish layer 1 of tile u into T,
// then layer 2 of tile u - 1.  Layer 1's accumulators, T and layer 2's accumulators are
// each double-buffered.  Every wait is bounded in time; on expiry the CTA
// records SC_ERR_DEVICE_TIMEOUT, lets its own copies and MMAs land, frees
// tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace sc {

namespace fz {

constexpr int C1 = 32;          // layer-1 output channels = one group
constexpr int NB1 = 96;         // layer-1 MMA N
constexpr int MT = 2;           // M-tiles per tile (both layers)
constexpr int TR1 = 8;          // layer-1 rows per tile
constexpr int TR2 = 6, TC2 = 28;   // layer-2 output rows / columns per tile
constexpr int THh = TR1 + 2;    // staged input rows
constexpr uint32_t STAGE_BYTES = THh * tc::WP * 128;   // one 32-channel stage (40 KB); T has the same shape
constexpr int MAX_STAGE = 4;
// warps 0-3, 6-9 epilogue; 4 producer; 5 issues layer 1's MMAs, 10 layer 2's
// (two issuing threads: while one waits on a barrier, the other's MMAs keep
// the tensor core busy)
constexpr int NTHREADS = 352;

struct Geom {
    int tiles_x, tiles_y, ntiles, nk1, nstg1, nstage, raw_pitch1, raw_pitch2;
    uint32_t w1_bytes, w2_bytes, smem_bytes;
};

}  // namespace fz

template <int CG2>
__global__ void __launch_bounds__(fz::NTHREADS, 1)
    conv_tc_fused2_kernel(const __grid_constant__ CUtensorMap tmx, const float *__restrict__ w1,
                          const float *__restrict__ b1, int act1, const float *__restrict__ w2,
                          const float *__restrict__ b2, int act2, float *__restrict__ y, int H, int W, int C0, int C2,
                          fz::Geom g, int *status, unsigned long long timeout_ns)
{
    using OP = tc::OpTF32;
    // Layer 2 with 4 output channels stacks all nine taps in N (8 MMAs per
    // tile; the vertical taps' row shifts, which cross warps, are summed
    // through shared memory); with 8 it stacks the horizontal taps only (24
    // MMAs; lane shifts only), as layer 1 does.
    constexpr bool RSN = CG2 == 4;
    constexpr int NB2 = RSN ? (9 * CG2 + 15) / 16 * 16 : (3 * CG2 + 15) / 16 * 16;
    constexpr int D3BUF = RSN ? 1 : 2;              // layer-2 accumulator buffers
    constexpr int KS = tc::CH / OP::KC;             // K steps per 32-channel stage
    constexpr uint32_t AR = 2 * OP::ROWB, AM = 8 * OP::ROWB;   // A units per vertical tap, per M-tile
    constexpr uint32_t D3COL = 2 * fz::MT * fz::NB1;           // first TMEM column of layer 2's accumulators
    static_assert(D3COL + D3BUF * fz::MT * NB2 <= 512, "tensor memory holds both layers' accumulator buffers");
    extern __shared__ __align__(1024) unsigned char smem_dyn[];
    __shared__ __align__(8) unsigned long long full_bar[fz::MAX_STAGE], empty_bar[fz::MAX_STAGE];
    __shared__ __align__(8) unsigned long long acc1_full[2], acc1_empty[2], t_full[2], t_empty[2], acc2_full[2],
        acc2_empty[2], rs_bar[2], w_bar, wt_bar, fin_bar, fin2_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ns = g.nstage;
    unsigned char *smem_raw = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    unsigned char *abuf = smem_raw;                                     // ns input stages
    unsigned char *tbuf = abuf + (size_t)ns * fz::STAGE_BYTES;          // two intermediate tiles T
    unsigned char *wsm1 = tbuf + 2 * (size_t)fz::STAGE_BYTES;           // layer-1 filter bank
    unsigned char *wsm2 = wsm1 + g.w1_bytes;                            // layer-2 filter bank
    float *rsum = reinterpret_cast<float *>(wsm2 + g.w2_bytes);          // layer-2 vertical-tap partial sums (RSN)

    // Filters of both layers, staged (OIHW rows, bulk copies) into the T
    // buffers, which are idle until the first tile's layer 1 is done, then
    // rearranged into the two B banks by every warp but the producer.
    const uint32_t raw1_bytes = (uint32_t)(fz::C1 * g.raw_pitch1 * 16);
    unsigned char *raw1 = tbuf, *raw2 = tbuf + raw1_bytes;
    if (warp == 0) tc::tmem_alloc(smem_u32(&tmem_base_sh), 512);
    if (tid == 0) {
        for (int j = 0; j < ns; ++j) {
            mbar_init(smem_u32(&full_bar[j]), 1);
            mbar_init(smem_u32(&empty_bar[j]), 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(smem_u32(&acc1_full[j]), 1);
            mbar_init(smem_u32(&acc1_empty[j]), 8);
            mbar_init(smem_u32(&t_full[j]), 8);
            mbar_init(smem_u32(&t_empty[j]), 1);
            mbar_init(smem_u32(&acc2_full[j]), 1);
            mbar_init(smem_u32(&acc2_empty[j]), 8);
            mbar_init(smem_u32(&rs_bar[j]), 8);   // one arrive per epilogue warp
        }
        mbar_init(smem_u32(&w_bar), 1);
        mbar_init(smem_u32(&wt_bar), fz::NTHREADS / 32 - 1);   // every warp but the producer
        mbar_init(smem_u32(&fin_bar), 1);
        mbar_init(smem_u32(&fin2_bar), 1);
        abort_sh = 0;
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    auto aborted = [&]() { return *reinterpret_cast<volatile int *>(&abort_sh) != 0; };
    auto give_up = [&]() { atomicExch(&abort_sh, 1); };
    if (warp == 4) {
        const uint32_t row1 = (uint32_t)(C0 * 9 * 4), row2 = (uint32_t)(fz::C1 * 9 * 4);
        if (lane == 0) mbar_arrive_expect_tx(smem_u32(&w_bar), row1 * fz::C1 + row2 * (uint32_t)C2);
        __syncwarp();
        for (int co = lane; co < fz::C1 + C2; co += 32) {
            if (co < fz::C1)
                bulk_load(smem_u32(raw1) + (uint32_t)(co * g.raw_pitch1 * 16), w1 + (size_t)co * C0 * 9, row1,
                          smem_u32(&w_bar));
            else
                bulk_load(smem_u32(raw2) + (uint32_t)((co - fz::C1) * g.raw_pitch2 * 16),
                          w2 + (size_t)(co - fz::C1) * fz::C1 * 9, row2, smem_u32(&w_bar));
        }
    } else {
        const bool landed = mbar_wait_bounded(smem_u32(&w_bar), 0, timeout_ns);
        if (!landed) give_up();
        constexpr int LT = fz::NTHREADS - 32;
        const int lt = warp < 4 ? tid : tid - 32;
        if (landed) {
            tc::stage_filter_bank<fz::C1, OP>(reinterpret_cast<const float *>(raw1), reinterpret_cast<uint4 *>(wsm1),
                                              g.raw_pitch1, fz::C1, C0, 3, 3, g.nk1, lt, LT);
            if constexpr (RSN)
                tc::stage_filter_bank_taps_in_n<CG2, OP>(reinterpret_cast<const float *>(raw2),
                                                         reinterpret_cast<uint4 *>(wsm2), g.raw_pitch2, C2, fz::C1,
                                                         fz::C1 / OP::KC, lt, LT);
            else
                tc::stage_filter_bank<CG2, OP>(reinterpret_cast<const float *>(raw2), reinterpret_cast<uint4 *>(wsm2),
                                               g.raw_pitch2, C2, fz::C1, 3, 3, fz::C1 / OP::KC, lt, LT);
        }
        fence_proxy_async_smem();   // the banks -> the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&wt_bar));
    }

    const int my_tiles = (g.ntiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    // tile u's layer-2 output origin (n, Y, X); its layer-1 rows start at Y - 1, columns at X - 1
    auto tile_origin = [&](int u, int &n, int &Y, int &X) {
        int t = (int)blockIdx.x + u * (int)gridDim.x;
        X = (t % g.tiles_x) * fz::TC2;
        t /= g.tiles_x;
        Y = (t % g.tiles_y) * fz::TR2;
        n = t / g.tiles_y;
    };

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const int total = my_tiles * g.nstg1;
            int issued = 0, s = 0, c = 0, u = 0;
            uint32_t ph = 0;
            int n, Y, X;
            tile_origin(0, n, Y, X);
            for (int j = 0; j < total && !aborted(); ++j) {
                if (j >= ns && !mbar_wait_bounded(smem_u32(&empty_bar[s]), ph ^ 1u, timeout_ns)) {
                    give_up();
                    break;
                }
                mbar_arrive_expect_tx(smem_u32(&full_bar[s]), fz::STAGE_BYTES);
                tma_load_4d(smem_u32(abuf + (size_t)s * fz::STAGE_BYTES), &tmx, tc::CH * c, X - 2, Y - 2, n,
                            smem_u32(&full_bar[s]));
                issued = j + 1;
                if (++s == ns) {
                    s = 0;
                    ph ^= 1u;
                }
                if (++c == g.nstg1) {
                    c = 0;
                    if (++u < my_tiles) tile_origin(u, n, Y, X);
                }
            }
            for (int j = (issued > ns ? issued - ns : 0); j < issued; ++j)
                (void)mbar_wait_bounded(smem_u32(&full_bar[j % ns]), (j / ns) & 1, timeout_ns);
        }
    } else if (warp == 5 || warp == 10) {
        // ------------------------------------------- MMA issuers (layer 1: warp 5, layer 2: warp 10)
        if (lane == 0) {
            constexpr uint32_t idesc1 = tc::idesc_mma(OP::FMT, fz::NB1), idesc2 = tc::idesc_mma(OP::FMT, NB2);
            constexpr uint32_t A_HI = tc::a_hi<OP>();
            const uint32_t a_base = smem_u32(abuf) >> 4, t_base = smem_u32(tbuf) >> 4;
            const uint32_t w1_base = smem_u32(wsm1) >> 4, w2_base = smem_u32(wsm2) >> 4;
            const uint32_t a_lbo = 1u << 16;
            // nks K steps x 3 vertical taps x 2 M-tiles (innermost) from A rows
            // a0, B bank b0 with N rows, into accumulators d0, d0 + n
            auto issue = [&](uint32_t d0, uint32_t a0, uint32_t b0, uint32_t n, uint32_t idesc, int nks, uint32_t acc0) {
#pragma unroll 1
                for (int kk = 0; kk < nks; ++kk)
#pragma unroll
                    for (int r = 0; r < 3; ++r)
#pragma unroll
                        for (int gi = 0; gi < fz::MT; ++gi)
                            tc::mma_w<OP>(d0 + (uint32_t)gi * n, a0 + (uint32_t)(kk * 2 + r * AR + gi * AM), A_HI,
                                          b0 + (uint32_t)((kk * 3 + r) * 2) * n, tc::B_HI, idesc,
                                          (kk > 0 || r > 0) ? 1u : acc0);
            };
            int s = 0, j = 0, committed = -1;
            uint32_t ph = 0;
            bool ok = mbar_wait_bounded(smem_u32(&wt_bar), 0, timeout_ns);   // both banks complete
            if (!ok) give_up();
            // layer 2 of tile v: A = T[v & 1], B = the layer-2 bank
            auto layer2 = [&](int v) -> bool {
                const int bb = v & 1;
                if (!mbar_wait_bounded(smem_u32(&t_full[bb]), (v >> 1) & 1, timeout_ns)) return false;
                const uint32_t ta = (t_base + (uint32_t)bb * (fz::STAGE_BYTES >> 4)) | a_lbo;
                if constexpr (RSN) {
                    // one accumulator buffer: the epilogue has read tile v - 1's
                    if (v >= 1 && !mbar_wait_bounded(smem_u32(&acc2_empty[0]), (v - 1) & 1, timeout_ns)) return false;
                    tc::fence_after_sync();
                    const uint32_t b2 = w2_base | ((uint32_t)NB2 << 16);
#pragma unroll
                    for (int kk = 0; kk < fz::C1 / OP::KC; ++kk)
#pragma unroll
                        for (int gi = 0; gi < fz::MT; ++gi)
                            tc::mma_w<OP>(tmem + D3COL + (uint32_t)(gi * NB2), ta + (uint32_t)(kk * 2 + gi * AM), A_HI,
                                          b2 + (uint32_t)(kk * 2 * NB2), tc::B_HI, idesc2, kk > 0 ? 1u : 0u);
                    tc::mma_commit(smem_u32(&acc2_full[0]));
                } else {
                    if (v >= 2 && !mbar_wait_bounded(smem_u32(&acc2_empty[bb]), ((v >> 1) - 1) & 1, timeout_ns))
                        return false;
                    tc::fence_after_sync();
                    issue(tmem + D3COL + (uint32_t)(bb * fz::MT * NB2), ta, w2_base | ((uint32_t)NB2 << 16), NB2, idesc2,
                          fz::C1 / OP::KC, 0u);
                    tc::mma_commit(smem_u32(&acc2_full[bb]));
                }
                tc::mma_commit(smem_u32(&t_empty[bb]));
                return true;
            };
            if (warp == 5) {
                for (int u = 0; ok && u < my_tiles && !aborted(); ++u) {
                    const int b = u & 1;
                    if (u >= 2 && !mbar_wait_bounded(smem_u32(&acc1_empty[b]), ((u >> 1) - 1) & 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t d1 = tmem + (uint32_t)(b * fz::MT * fz::NB1);
                    for (int c = 0; c < g.nstg1; ++c, ++j) {
                        if (!mbar_wait_bounded(smem_u32(&full_bar[s]), ph, timeout_ns)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        const int nks = g.nk1 - KS * c < KS ? g.nk1 - KS * c : KS;
                        issue(d1, (a_base + (uint32_t)s * (fz::STAGE_BYTES >> 4)) | a_lbo,
                              (w1_base + (uint32_t)(c * KS * 3 * 2 * fz::NB1)) | ((uint32_t)fz::NB1 << 16), fz::NB1,
                              idesc1, nks, c > 0 ? 1u : 0u);
                        tc::mma_commit(smem_u32(&empty_bar[s]));
                        committed = j;
                        if (++s == ns) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    tc::mma_commit(smem_u32(&acc1_full[b]));
                }
            } else {
                for (int v = 0; ok && v < my_tiles && !aborted(); ++v)
                    if (!layer2(v)) ok = false;
            }
            if (!ok) give_up();
            // MMAs still executing must finish before tensor memory is freed:
            // a commit after everything issued, then its wait
            unsigned long long *fb = warp == 5 ? &fin_bar : &fin2_bar;
            tc::mma_commit(smem_u32(fb));
            (void)mbar_wait_bounded(smem_u32(fb), 0, timeout_ns);
            (void)committed;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3, mt = warp < 4 ? 0 : 1;   // TMEM lane quadrant, M-tile (both layers)
        float bias1[fz::C1], bias2[CG2];
#pragma unroll
        for (int i = 0; i < fz::C1; ++i) bias1[i] = b1 ? __ldg(b1 + i) : 0.f;
#pragma unroll
        for (int i = 0; i < CG2; ++i) bias2[i] = (b2 && i < C2) ? __ldg(b2 + i) : 0.f;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        // layer 2 of tile v: y rows Y + 4 mt + q4 (< Y + 6), columns X + lane (lane < 28)
        auto layer2 = [&](int v) -> bool {
            const int bb = RSN ? 0 : (v & 1);
            const uint32_t par = RSN ? (uint32_t)(v & 1) : (uint32_t)((v >> 1) & 1);
            const bool got = mbar_wait_bounded(smem_u32(&acc2_full[bb]), par, timeout_ns);
            if (__any_sync(0xffffffffu, !got)) return false;
            tc::fence_after_sync();
            int n, Y, X;
            tile_origin(v, n, Y, X);
            const uint32_t d = tmem + D3COL + (uint32_t)(bb * fz::MT * NB2 + mt * NB2) + lane_off;
            if constexpr (RSN) {
                // this warp holds T row ty = 4 mt + q4; per vertical tap r its
                // lane-shift sums c_r belong to output row ty - r
                uint32_t rv[9][CG2];
#pragma unroll
                for (int t = 0; t < 9; ++t) tc::tmem_ld<CG2>(d + (uint32_t)(t * CG2), rv[t]);
                tc::tmem_wait_ld();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc2_empty[0]));
                const int ty = mt * 4 + q4;
                float *rb = rsum + (size_t)(v & 1) * (3 * fz::TR2 * 32 * CG2);   // [r][row][px][co], two tiles' worth
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    float c[CG2];
#pragma unroll
                    for (int i = 0; i < CG2; ++i)
                        c[i] = __uint_as_float(rv[3 * r][i]) +
                               __shfl_down_sync(0xffffffffu, __uint_as_float(rv[3 * r + 1][i]), 1) +
                               __shfl_down_sync(0xffffffffu, __uint_as_float(rv[3 * r + 2][i]), 2);
                    const int ty3 = ty - r;
                    if (ty3 >= 0 && ty3 < fz::TR2)
                        *reinterpret_cast<float4 *>(rb + ((r * fz::TR2 + ty3) * 32 + lane) * CG2) =
                            make_float4(c[0], c[1], c[2], c[3]);
                }
                // every epilogue warp's partial sums are in place (a bounded
                // wait on an mbarrier, not bar.sync: a warp that gave up must
                // not leave the others waiting forever)
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&rs_bar[v & 1]));
                const bool all = mbar_wait_bounded(smem_u32(&rs_bar[v & 1]), (v >> 1) & 1, timeout_ns);
                if (__any_sync(0xffffffffu, !all)) return false;
                const int e = warp < 4 ? warp : warp - 2;   // output row of this warp
                const int oy = Y + e, ox = X + lane;
                if (e < fz::TR2 && lane < fz::TC2 && oy < H && ox < W) {
                    float o[CG2];
#pragma unroll
                    for (int i = 0; i < CG2; ++i) o[i] = 0.f;
#pragma unroll
                    for (int r = 0; r < 3; ++r) {
                        const float4 p = *reinterpret_cast<const float4 *>(rb + ((r * fz::TR2 + e) * 32 + lane) * CG2);
                        o[0] += p.x;
                        o[1] += p.y;
                        o[2] += p.z;
                        o[3] += p.w;
                    }
                    float *yp = y + (((long long)n * H + oy) * W + ox) * C2;
                    *reinterpret_cast<float4 *>(yp) =
                        make_float4(relu_if(o[0] + bias2[0], act2), relu_if(o[1] + bias2[1], act2),
                                    relu_if(o[2] + bias2[2], act2), relu_if(o[3] + bias2[3], act2));
                }
                return true;
            } else {
                uint32_t r0[CG2], r1[CG2], r2[CG2];
                tc::tmem_ld<CG2>(d, r0);
                tc::tmem_ld<CG2>(d + CG2, r1);
                tc::tmem_ld<CG2>(d + 2 * CG2, r2);
                tc::tmem_wait_ld();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc2_empty[bb]));
                float v2[CG2];
#pragma unroll
                for (int i = 0; i < CG2; ++i)
                    v2[i] = relu_if(__uint_as_float(r0[i]) +
                                        __shfl_down_sync(0xffffffffu, __uint_as_float(r1[i]), 1) +
                                        __shfl_down_sync(0xffffffffu, __uint_as_float(r2[i]), 2) + bias2[i],
                                    act2);
                const int ty = mt * 4 + q4, oy = Y + ty, ox = X + lane;
                if (ty < fz::TR2 && lane < fz::TC2 && oy < H && ox < W) {
                    float *yp = y + (((long long)n * H + oy) * W + ox) * C2;
#pragma unroll
                    for (int qq = 0; qq < CG2 / 4; ++qq)
                        if (4 * qq < C2)
                            *reinterpret_cast<float4 *>(yp + 4 * qq) =
                                make_float4(v2[4 * qq], v2[4 * qq + 1], v2[4 * qq + 2], v2[4 * qq + 3]);
                }
                return true;
            }
        };
        bool ok = true;
        for (int u = 0; u < my_tiles; ++u) {
            const int b = u & 1;
            if (aborted()) {
                ok = false;
                break;
            }
            // layer 1 of tile u -> T[b]
            bool got = mbar_wait_bounded(smem_u32(&acc1_full[b]), (u >> 1) & 1, timeout_ns);
            if (got && u >= 2) got = mbar_wait_bounded(smem_u32(&t_empty[b]), ((u >> 1) - 1) & 1, timeout_ns);
            if (__any_sync(0xffffffffu, !got)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            int n, Y, X;
            tile_origin(u, n, Y, X);
            const uint32_t d = tmem + (uint32_t)(b * fz::MT * fz::NB1 + mt * fz::NB1) + lane_off;
            uint32_t r0[fz::C1], r1[fz::C1], r2[fz::C1];
            tc::tmem_ld<fz::C1>(d, r0);
            tc::tmem_ld<fz::C1>(d + fz::C1, r1);
            tc::tmem_ld<fz::C1>(d + 2 * fz::C1, r2);
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc1_empty[b]));
            // this lane's layer-1 pixel: row Y - 1 + 4 mt + q4, column X - 1 + lane;
            // zero outside the image (layer 2's zero padding) and in the two pad lanes
            const int ty = mt * 4 + q4, py = Y - 1 + ty, px = X - 1 + lane;
            const bool inside = lane < tc::TC && py >= 0 && py < H && px >= 0 && px < W;
            float v1[fz::C1];
#pragma unroll
            for (int i = 0; i < fz::C1; ++i) {
                const float s = __uint_as_float(r0[i]) + __shfl_down_sync(0xffffffffu, __uint_as_float(r1[i]), 1) +
                                __shfl_down_sync(0xffffffffu, __uint_as_float(r2[i]), 2);
                v1[i] = inside ? relu_if(s + bias1[i], act1) : 0.f;
            }
            const uint32_t trow = smem_u32(tbuf) + (uint32_t)b * fz::STAGE_BYTES + (uint32_t)((ty * tc::WP + lane) * 128);
#pragma unroll
            for (int qq = 0; qq < 8; ++qq)
                tc::st_shared_v4(trow + ((qq ^ (lane & 7)) << 4), __float_as_uint(v1[4 * qq]),
                                 __float_as_uint(v1[4 * qq + 1]), __float_as_uint(v1[4 * qq + 2]),
                                 __float_as_uint(v1[4 * qq + 3]));
            fence_proxy_async_smem();   // T -> the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&t_full[b]));
            // layer 2 of the previous tile
            if (u >= 1 && !layer2(u - 1)) {
                ok = false;
                break;
            }
        }
        if (ok && my_tiles >= 1 && !aborted() && !layer2(my_tiles - 1)) ok = false;
        if (!ok && lane == 0) give_up();
    }

    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) (void)mbar_wait_bounded(smem_u32(&w_bar), 0, timeout_ns);   // the weight copies have landed
    if (aborted() && tid == 0 && status) atomicExch(status, kDeviceTimeout);
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

constexpr size_t kFusedSmemCap = 227 * 1024 - 1024;

static PFN_cuTensorMapEncodeTiled_v12000 fused_tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

template <int CG2>
static cudaError_t launch_fused_cg(const FusedArgs &a, cudaStream_t st)
{
    constexpr bool RSN = CG2 == 4;
    constexpr int NB2 = RSN ? (9 * CG2 + 15) / 16 * 16 : (3 * CG2 + 15) / 16 * 16;
    constexpr size_t RSUM_BYTES = RSN ? 2 * 3 * fz::TR2 * 32 * CG2 * 4 : 0;
    fz::Geom g;
    g.nk1 = (a.C0 + 7) / 8;
    g.nstg1 = (a.C0 + tc::CH - 1) / tc::CH;
    g.raw_pitch1 = tc::filter_raw_pitch(a.C0, 9);
    g.raw_pitch2 = tc::filter_raw_pitch(fz::C1, 9);
    g.w1_bytes = (uint32_t)(((size_t)g.nk1 * 3 * 2 * fz::NB1 * 16 + 1023) & ~(size_t)1023);
    g.w2_bytes = (uint32_t)(((size_t)(fz::C1 / 8) * (RSN ? 1 : 3) * 2 * NB2 * 16 + 1023) & ~(size_t)1023);
    const size_t fixed = 2 * (size_t)fz::STAGE_BYTES + g.w1_bytes + g.w2_bytes + RSUM_BYTES + 1024;
    if (fixed + 2 * (size_t)fz::STAGE_BYTES > kFusedSmemCap) return cudaErrorNotSupported;
    // the staged OIHW filters of both layers go into the two T buffers
    if ((size_t)fz::C1 * g.raw_pitch1 * 16 + (size_t)CG2 * g.raw_pitch2 * 16 > 2 * (size_t)fz::STAGE_BYTES)
        return cudaErrorNotSupported;
    int ns = (int)((kFusedSmemCap - fixed) / fz::STAGE_BYTES);
    g.nstage = ns < fz::MAX_STAGE ? ns : fz::MAX_STAGE;
    g.smem_bytes = (uint32_t)(fixed + (size_t)g.nstage * fz::STAGE_BYTES);
    g.tiles_x = (a.W + fz::TC2 - 1) / fz::TC2;
    g.tiles_y = (a.H + fz::TR2 - 1) / fz::TR2;
    const long long nt = (long long)g.tiles_x * g.tiles_y * a.N;
    if (nt > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    g.ntiles = (int)nt;
    PFN_cuTensorMapEncodeTiled_v12000 encode = fused_tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tm;
    const cuuint64_t dims[4] = {(cuuint64_t)a.C0, (cuuint64_t)a.W, (cuuint64_t)a.H, (cuuint64_t)a.N};
    const cuuint64_t strides[3] = {(cuuint64_t)a.C0 * 4, (cuuint64_t)a.W * a.C0 * 4, (cuuint64_t)a.H * a.W * a.C0 * 4};
    const cuuint32_t box[4] = {(cuuint32_t)tc::CH, (cuuint32_t)tc::WP, (cuuint32_t)fz::THh, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(a.x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static KernelCache cache;
    e = ensure_dynamic_smem(cache, dev, conv_tc_fused2_kernel<CG2>, (int)g.smem_bytes);
    if (e != cudaSuccess) return e;
    const int grid = g.ntiles < device_sm_count() ? g.ntiles : device_sm_count();
    conv_tc_fused2_kernel<CG2><<<grid, fz::NTHREADS, g.smem_bytes, st>>>(
        tm, a.w1, a.b1, a.act1, a.w2, a.b2, a.act2, a.y, a.H, a.W, a.C0, a.C2, g, device_status_ptr(), 1000000000ull);
    return cudaGetLastError();
}

cudaError_t launch_conv_tc_fused2(const FusedArgs &a, cudaStream_t st)
{
    // tensor memory: layer 1's two accumulator buffers take 2 x 192 of the
    // 512 columns, layer 2's two take 2 x 2 x NB2 (32 or 64 for C2 <= 4 / 8)
    if (a.C1 != fz::C1 || a.C2 > 8) return cudaErrorNotSupported;
    if (a.C2 <= 4) return launch_fused_cg<4>(a, st);
    return launch_fused_cg<8>(a, st);
}

}  // namespace sc
