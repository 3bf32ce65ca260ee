// Tensor-core variant of the direct convolution: implicit GEMM on the 5th
// generation tensor cores (tcgen05, accumulators in tensor memory), TF32
// operands, fp32 accumulation.  It computes the same operation as
// conv2d_fwd (stride 1, zero "same" padding, bias, ReLU; R, S in {1, 3}) with
// x and w truncated to TF32 by the MMA, so it is checked with its own
// tolerance (5e-3 * sum|x*w|).
//
// GEMM view ("Optimizing Memory Efficiency for Convolution Kernels on Kepler
// GPUs", Section 3.3, compares direct convolution with the GEMM
// formulation; the reuse argument of Section 3.3.2 is kept: each input pixel
// is staged once per tile and every tap reads it again from shared memory).
// With 3 x 3 taps (r, s) and a group of Cg output channels per CTA:
//
//   D_mt[m][(s, co)] = sum_r sum_ci A[mt*128 + r*WP + m][ci] * w[co][ci][r][s]
//   y[pixel m of M-tile mt][co] = sum_s D_mt[m + s][(s, co)]
//
// A holds the tile's padded pixels (row pitch WP = 32: padded pixel
// q = py * 32 + px is image pixel (y0 - 1 + py, x0 - 1 + px), zero outside
// the image), so the vertical tap r is an A start address r * WP rows
// further, while the three horizontal taps s sit side by side in the MMA's N
// dimension (N = 3 * Cg rounded up to 16).  Stacking the taps in N instead of
// issuing one MMA per tap matters because an M = 128 MMA costs about
// (A bytes + B bytes) / 128 B per clock of shared-memory reads, at least
// ~44 clocks, whatever N: with N = Cg <= 64 the tensor core would stay below
// two thirds of its rate.  The sum over s is a shift by s GEMM rows, i.e. by
// s TMEM lanes: the epilogue adds the columns of lane l + s with a warp
// shuffle.  Output column tx of a tile is lane tx of a warp; with WP = 32
// each warp's 32 lanes are one padded image row and lanes 30 and 31 (which
// would need the next warp's lanes) are exactly the two padding columns, so
// a tile is TC = 30 output columns wide and 4 image rows per M-tile.
//
// Operand layouts (K-major): A is staged 32 channels at a time by one 4-D TMA
// box per stage with 128-byte swizzling: one 128-byte row per padded pixel,
// 8-row atoms (SBO = 1024 bytes); a K step of 8 channels is +32 bytes of the
// start address, a vertical tap +4 KB, an M-tile +16 KB, so every start
// address keeps the swizzle phase of its 1024-byte-aligned stage buffer.  B
// (filters, no swizzle): per (8-channel step, r), two 4-channel blocks of N
// rows x 16 bytes (core matrices of 8 rows, SBO 128 bytes, LBO N * 16 bytes);
// row n = s * Cg + co.  One MMA is M = 128 x N x K = 8.
//
// Pipeline: persistent CTAs (one per SM and channel group), the group's
// filter bank resident in shared memory, warp-specialised roles linked by
// mbarriers:
//  * all warps first stage the group's filters (bulk copy of the OIHW rows,
//    then a transpose in shared memory into the B layout).
//  * producer (warp 4, one lane): per stage one TMA box of (32 channels, 32 pixels, THh rows) of the
//    tile's padded activations; the TMA zero fill outside the image (and
//    past Cin) is the convolution's zero padding.  A stage buffer is
//    refilled once the MMAs that read it have completed (`empty`).
//  * MMA issuer (warp 5, one lane): waits for a stage (`full`), issues its
//    (K steps) x 3 x MT MMAs, commits them to the stage's `empty` barrier,
//    and after a tile's last stage commits to the tile's accumulator
//    barrier.  Each barrier wait leaves the tensor core idle for ~100-200
//    clocks, so stages are large (32 channels).
//  * epilogue (warps 0-3 and 6-9, one TMEM lane quadrant each, the two sets
//    on alternate M-tiles): waits for a tile's accumulators, reads the
//    three s-blocks with tcgen05.ld, sums them with lane shifts, transposes
//    through a swizzled per-warp shared-memory buffer so that each store
//    instruction writes whole pixel records, adds bias, applies ReLU,
//    writes NHWC, and frees the accumulator buffer.  Accumulators are
//    double-buffered in tensor memory, so a tile's epilogue overlaps the
//    next tile's MMAs.
// Two modes change this (template parameters of the kernel):
//  * split TF32 (OpTF32x3): warps 6-9 write each stage's TF32 remainders
//    instead (the MMA reads the copied values as their TF32 heads); every
//    (K step, tap) issues x_hi [w_hi | w_lo] and x_lo w_hi into a head and
//    a correction accumulator, which the epilogue adds (warps 0-3 alone).
//  * nine taps in N (RSN, 4-channel groups, 3 x 3): one MMA per K step and
//    M-tile over the tile's staged rows; the epilogue sums the horizontal
//    taps by lane shifts and the vertical ones through shared memory.
// Every wait is bounded in time; on expiry the CTA records
// SC_ERR_DEVICE_TIMEOUT, lets its own copies and MMAs land, frees tensor
// memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace sc {

namespace tc {
constexpr int MIN_STAGE = 2;
constexpr int MAX_STAGE = 8;                 // 6 -> 8: BF16 32 -> 32 37.1 -> 36.3 us (its copies are latency-bound)
constexpr int TMEM_BUF = 256;   // tensor-memory columns per accumulator buffer (two buffers)
constexpr int OUT_BUF = 4096;                // one epilogue output buffer: 30 pixel rows of up to 128 bytes
constexpr int STG_BYTES = 8 * OUT_BUF;       // one per epilogue warp
constexpr int X3_LO = 2;                     // split TF32: buffers for the stages' remainders (a ring of its own)
constexpr int X3_STG_BYTES = 4 * OUT_BUF;    // split TF32: four epilogue warps

struct TcGeom {
    int MT, TR, THh;                // M-tiles per tile, tile rows (4 MT; RSN 4 MT - 2), staged rows (TR + 2)
    int tiles_x, tiles_y, ntiles;   // tiles of TC x TR output pixels, per image and in all
    int nk, nstg, nstage;           // K steps, 32-channel stages per tile, stage buffers
    int raw_pitch;                  // 16-byte units per output channel of the staged OIHW filters
    uint32_t stage_bytes, w_bytes, smem_bytes, tmem_cols;
};

}  // namespace tc

__device__ __forceinline__ void give_up_flag(int &flag) { atomicExch(&flag, 1); }

// CG: output channels per CTA (4, 8, 16 or 32); NB = MMA N = 3 * CG rounded
// up to 16.  OP: operand kind (tc::OpTF32, tc::OpTF32x3, tc::OpBF16).
// YBF16: y is bf16 (else fp32).  RSN (CG = 4, 3 x 3 filters): all nine taps
// stacked in N (NB = 48), one MMA per K step and M-tile, the M rows being
// the tile's staged rows (4 MT of them for 4 MT - 2 output rows); the
// horizontal shifts are lane shuffles and the vertical ones, which cross
// warps, are summed through shared memory in the epilogue.  With 4 output
// channels the per-tap MMAs of N = 16 sit at the tensor core's fixed cost
// per instruction; stacking the taps issues a third as many.
template <int CG, class OP, bool YBF16, bool RSN = false>
__global__ void __launch_bounds__(tc::NTHREADS, 1)
    conv_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                   const float *__restrict__ w, const float *__restrict__ bias, void *__restrict__ yv, int H, int W,
                   int Cin, int Cout, int R, int S, int act, tc::TcGeom g, int *status, unsigned long long timeout_ns)
{
    static_assert(!RSN || CG == 4, "nine taps in N for 4-channel groups");
    constexpr int NB = RSN ? (9 * CG + 15) / 16 * 16 : (3 * CG + 15) / 16 * 16;
    constexpr int NR = RSN ? 1 : 3;                // vertical taps issued as A row offsets
    constexpr int KS = tc::CH / OP::KC;            // K steps per stage
    constexpr int KSUB = KS / OP::SUB;             // K steps per sub-buffer
    constexpr int CU = OP::KC / 2;                 // input channels per 16-byte B chunk
    constexpr int CW = CG;                         // epilogue column chunk = the group
    constexpr int OSZ = YBF16 ? 2 : 4;             // bytes per output element
    constexpr int OROWB = CW * OSZ;                // bytes of one pixel's group of outputs
    constexpr bool TMA_OUT = OROWB >= 64;          // store through a swizzled shared-memory buffer and TMA
    constexpr int OCH = OROWB >= 16 ? OROWB / 16 : 1;   // 16-byte chunks per pixel (or one 8-byte piece)
    constexpr bool X3 = OP::X3;                    // split TF32: head and correction accumulators
    constexpr int DSTR = X3 ? 2 * NB : NB;         // tensor-memory columns per M-tile
    constexpr int RB = X3 ? 2 * NB : NB;           // filter-bank rows per (K step, tap, 4-channel block)
    extern __shared__ __align__(1024) unsigned char smem_dyn[];
    __shared__ __align__(8) unsigned long long full_bar[tc::MAX_STAGE], empty_bar[tc::MAX_STAGE];
    __shared__ __align__(8) unsigned long long conv_bar[X3 ? tc::MAX_STAGE : 1];   // X3: a stage is split
    __shared__ __align__(8) unsigned long long lo_empty[X3 ? tc::X3_LO : 1];       // X3: a remainder buffer is free
    __shared__ __align__(8) unsigned long long rs_bar[RSN ? 2 : 1];                // RSN: a tile's row partial sums are in place
    __shared__ __align__(8) unsigned long long acc_full[2], acc_empty[2], w_bar, wt_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int co0 = blockIdx.y * CG;                     // this CTA's output channels co0 .. co0+CG-1
    const int ns = g.nstage;
    // stage buffers need 1024-byte alignment (the 128-byte swizzle pattern)
    unsigned char *smem_raw = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    unsigned char *abuf = smem_raw;                      // ns activation stages (X3: read as their TF32 heads)
    // X3: X3_LO buffers for the remainders, same layout as a stage; stage j
    // (head buffer j % ns) puts its remainders in buffer j % X3_LO
    unsigned char *alo = abuf + (size_t)ns * g.stage_bytes;
    unsigned char *wsm = alo + (X3 ? (size_t)tc::X3_LO * g.stage_bytes : 0);   // resident filters (X3: heads and remainders)
    unsigned char *stg = wsm + g.w_bytes;                // epilogue transpose buffers
    float *rsum = reinterpret_cast<float *>(stg);         // RSN: [2 tiles][3 taps r][TR rows][32 px][CG]

    // Filters, once per CTA.  The producer warp bulk-copies the group's OIHW
    // weights (one contiguous run of Cin * R * S floats per output channel)
    // into the top of the stage buffers, rows g.raw_pitch 16-byte units apart
    // (an odd number, so that the 16-byte reads below are free of bank
    // conflicts); the other warps then rearrange them into the MMA's B
    // layout: the [k][r][cb][n][CU] bank whose element (k, r, cb, n, j) with
    // n = s * CG + co is w[co0 + co][KC k + CU cb + j][r - (3 - R) / 2][s - (3 - S) / 2]
    // (as TF32 or rounded to bf16), zero for n >= 3 * CG, taps the R x S
    // filter lacks, channels beyond Cin and co beyond Cout.  One unit is one
    // output channel and one block of CU input channels (one 16-byte chunk);
    // neighbouring lanes take neighbouring output channels, whose B rows are
    // neighbours.  Meanwhile the producer already fills the
    // stage buffers below the staged weights; `wt_bar` (one arrive per
    // rearranging warp) releases the rest, and the bank, to the MMA warp.
    const int RS = R * S;
    const int co_n = Cout - co0 < CG ? Cout - co0 : CG;   // output channels this CTA copies
    const uint32_t raw_bytes = (uint32_t)(CG * g.raw_pitch * 16);
    unsigned char *raw_sm = abuf + (size_t)ns * g.stage_bytes - raw_bytes;
    if (warp == 0) tc::tmem_alloc(smem_u32(&tmem_base_sh), g.tmem_cols);
    if (tid == 0) {
        for (int j = 0; j < ns; ++j) {
            mbar_init(smem_u32(&full_bar[j]), 1);
            mbar_init(smem_u32(&empty_bar[j]), 1);
        }
        if constexpr (X3) {
            for (int j = 0; j < ns; ++j) mbar_init(smem_u32(&conv_bar[j]), 4);   // one arrive per converting warp
            for (int j = 0; j < tc::X3_LO; ++j) mbar_init(smem_u32(&lo_empty[j]), 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(smem_u32(&acc_full[j]), 1);
            mbar_init(smem_u32(&acc_empty[j]), X3 ? 4 : 8);   // one arrive per epilogue warp
            if constexpr (RSN) mbar_init(smem_u32(&rs_bar[j]), X3 ? 4 : 8);
        }
        mbar_init(smem_u32(&w_bar), 1);
        mbar_init(smem_u32(&wt_bar), tc::NTHREADS / 32 - 1);   // every warp but the producer
        abort_sh = 0;
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    if (warp == 4) {
        const uint32_t row = (uint32_t)(Cin * RS * 4);
        if (lane == 0) mbar_arrive_expect_tx(smem_u32(&w_bar), row * (uint32_t)co_n);
        __syncwarp();
        for (int co = lane; co < co_n; co += 32)
            bulk_load(smem_u32(raw_sm) + (uint32_t)(co * g.raw_pitch * 16), w + (size_t)(co0 + co) * Cin * RS, row,
                      smem_u32(&w_bar));
    } else {
        const bool landed = mbar_wait_bounded(smem_u32(&w_bar), 0, timeout_ns);
        if (!landed) give_up_flag(abort_sh);
        constexpr int LT = tc::NTHREADS - 32;   // threads of every warp but the producer
        if (landed) {
            if constexpr (RSN)
                tc::stage_filter_bank_taps_in_n<CG, OP>(reinterpret_cast<const float *>(raw_sm),
                                                        reinterpret_cast<uint4 *>(wsm), g.raw_pitch, co_n, Cin, g.nk,
                                                        warp < 4 ? tid : tid - 32, LT);
            else
                tc::stage_filter_bank<CG, OP>(reinterpret_cast<const float *>(raw_sm), reinterpret_cast<uint4 *>(wsm),
                                              g.raw_pitch, co_n, Cin, R, S, g.nk, warp < 4 ? tid : tid - 32, LT);
        }
        // the staged weights' buffers go to the TMA (async proxy) next, the
        // bank to the tensor core
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&wt_bar));
    }

    const int my_tiles = (g.ntiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int total = my_tiles * g.nstg;
    auto tile_origin = [&](int u, int &n, int &y0, int &x0) {
        int t = (int)blockIdx.x + u * (int)gridDim.x;
        x0 = (t % g.tiles_x) * tc::TC;
        t /= g.tiles_x;
        y0 = (t % g.tiles_y) * g.TR;
        n = t / g.tiles_y;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int *>(&abort_sh) != 0; };
    auto give_up = [&]() { give_up_flag(abort_sh); };

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0, s = 0, c = 0, u = 0;
            uint32_t ph = 0;
            int n, y0, x0;
            tile_origin(0, n, y0, x0);
            const int first_raw = (int)((ns * g.stage_bytes - raw_bytes) / g.stage_bytes);   // lowest buffer under the staged weights
            for (int j = 0; j < total && !aborted(); ++j) {
                if (j >= ns && !mbar_wait_bounded(smem_u32(&empty_bar[s]), ph ^ 1u, timeout_ns)) {
                    give_up();
                    break;
                }
                if (j == first_raw && !mbar_wait_bounded(smem_u32(&wt_bar), 0, timeout_ns)) {
                    give_up();
                    break;
                }
                mbar_arrive_expect_tx(smem_u32(&full_bar[s]), g.stage_bytes);
#pragma unroll
                for (int sb = 0; sb < OP::SUB; ++sb)
                    tma_load_4d(smem_u32(abuf + (size_t)s * g.stage_bytes + (size_t)sb * (g.stage_bytes / OP::SUB)), &tmx,
                                tc::CH * c + sb * (tc::CH / OP::SUB), x0 - 1, y0 - 1, n, smem_u32(&full_bar[s]));
                issued = j + 1;
                if (++s == ns) {
                    s = 0;
                    ph ^= 1u;
                }
                if (++c == g.nstg) {
                    c = 0;
                    if (++u < my_tiles) tile_origin(u, n, y0, x0);
                }
            }
            // every copy this lane issued has landed before the CTA may exit
            for (int j = (issued > ns ? issued - ns : 0); j < issued; ++j)
                (void)mbar_wait_bounded(smem_u32(&full_bar[j % ns]), (j / ns) & 1, timeout_ns);
        }
    } else if (warp == 5) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_mma(OP::FMT, NB);
            constexpr uint32_t A_HI = tc::a_hi<OP>();
            constexpr uint32_t AR = 2 * OP::ROWB, AM = 8 * OP::ROWB;   // A units per vertical tap (32 rows), per M-tile (128 rows)
            const uint32_t asub = (g.stage_bytes / OP::SUB) >> 4;         // A units per sub-buffer
            const uint32_t a_base = smem_u32(abuf) >> 4, w_base = smem_u32(wsm) >> 4;
            const uint32_t a_lbo = 1u << 16, b_lbo = (uint32_t)RB << 16;
            // X3: the current stage's remainders, in 16-byte units from its
            // heads (set per stage; start addresses stay below 2^14 units)
            uint32_t alo_off = 0;
            constexpr uint32_t idesc2 = tc::idesc_mma(OP::FMT, 2 * NB);
            // One (K step, tap, M-tile): the head product into the M-tile's
            // first NB columns.  X3: x_hi [w_hi | w_lo] (N = 2 NB) puts the
            // head product and x_hi w_lo side by side, then x_lo w_hi (the
            // bank's first NB rows) adds into the correction columns.
            auto mma1 = [&](uint32_t d, uint32_t ad, uint32_t bd, uint32_t acc) {
                if constexpr (X3) {
                    tc::mma_w<OP>(d, ad, A_HI, bd, tc::B_HI, idesc2, acc);
                    tc::mma_w<OP>(d + NB, ad + alo_off, A_HI, bd, tc::B_HI, idesc, 1u);
                } else {
                    tc::mma_w<OP>(d, ad, A_HI, bd, tc::B_HI, idesc, acc);
                }
            };
            // G M-tiles at a time, M-tiles innermost: consecutive MMAs go to
            // different accumulators (back-to-back MMAs into one accumulator
            // issue more slowly); a full stage (KS K steps) is unrolled so that
            // every descriptor is a register plus a constant.  A: +2 units
            // (32 B) per K step within a row, asub per sub-buffer, AR per
            // vertical tap, AM per M-tile.  B:
            // 2 * RB units per (K step, tap).
            auto issue = [&](auto gsz, uint32_t d0, uint32_t a0, uint32_t b0, int nks, uint32_t acc0) {
                constexpr int G = decltype(gsz)::value;
                if (nks == KS) {
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk)
#pragma unroll
                        for (int r = 0; r < NR; ++r)
#pragma unroll
                            for (int gi = 0; gi < G; ++gi)
                                mma1(d0 + (uint32_t)(gi * DSTR), a0 + (uint32_t)(kk / KSUB) * asub + (uint32_t)((kk % KSUB) * 2 + r * AR + gi * AM),
                                     b0 + (uint32_t)((kk * NR + r) * 2 * RB), (kk > 0 || r > 0) ? 1u : acc0);
                    return;
                }
#pragma unroll 1
                for (int kk = 0; kk < nks; ++kk) {
#pragma unroll
                    for (int r = 0; r < NR; ++r)
#pragma unroll
                        for (int gi = 0; gi < G; ++gi)
                            mma1(d0 + (uint32_t)(gi * DSTR), a0 + (uint32_t)(kk / KSUB) * asub + (uint32_t)((kk % KSUB) * 2 + r * AR + gi * AM),
                                 b0 + (uint32_t)((kk * NR + r) * 2 * RB), (kk > 0 || r > 0) ? 1u : acc0);
                }
            };
            int s = 0, j = 0, committed = -1;
            uint32_t ph = 0;
            if (!mbar_wait_bounded(smem_u32(&wt_bar), 0, timeout_ns)) give_up();   // the bank is complete
            for (int u = 0; u < my_tiles && !aborted(); ++u) {
                const int b = u & 1;
                if (u >= 2 && !mbar_wait_bounded(smem_u32(&acc_empty[b]), ((u >> 1) - 1) & 1, timeout_ns)) {
                    give_up();
                    break;
                }
                tc::fence_after_sync();
                const uint32_t dbase = tmem + (uint32_t)(b * tc::TMEM_BUF);
                bool ok = true;
                for (int c = 0; c < g.nstg; ++c, ++j) {
                    // X3: the stage once its heads and remainders are written
                    if (!mbar_wait_bounded(smem_u32(X3 ? &conv_bar[s] : &full_bar[s]), ph, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t a_lo = (a_base + (uint32_t)s * (g.stage_bytes >> 4)) | a_lbo;
                    if constexpr (X3)
                        alo_off = (uint32_t)(((size_t)(ns - s + j % tc::X3_LO) * g.stage_bytes) >> 4);
                    const uint32_t b_lo = (w_base + (uint32_t)(c * KS * NR * 2 * RB)) | b_lbo;
                    const int nks = g.nk - KS * c < KS ? g.nk - KS * c : KS;
                    const uint32_t acc0 = c > 0 ? 1u : 0u;
                    int mt = 0;
                    if (g.MT == 1) {
                        issue(std::integral_constant<int, 1>{}, dbase, a_lo, b_lo, nks, acc0);
                        mt = 1;
                    } else if (g.MT & 1) {
                        issue(std::integral_constant<int, 3>{}, dbase, a_lo, b_lo, nks, acc0);
                        mt = 3;
                    }
#pragma unroll 1
                    for (; mt < g.MT; mt += 2)
                        issue(std::integral_constant<int, 2>{}, dbase + (uint32_t)(mt * DSTR), a_lo + (uint32_t)(mt * AM),
                              b_lo, nks, acc0);
                    tc::mma_commit(smem_u32(&empty_bar[s]));
                    if constexpr (X3) tc::mma_commit(smem_u32(&lo_empty[j % tc::X3_LO]));
                    committed = j;
                    if (++s == ns) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) {
                    give_up();
                    break;
                }
                tc::mma_commit(smem_u32(&acc_full[b]));
            }
            // MMAs still executing must finish before tensor memory is freed
            if (committed >= 0)
                (void)mbar_wait_bounded(smem_u32(&empty_bar[committed % ns]), (committed / ns) & 1, timeout_ns);
        }
    } else if (X3 && warp >= 6) {
        // ---------------------------------------------------- X3: converters
        // Warps 6-9 write each landed stage's remainders into a remainder
        // buffer (the same offsets, so the same swizzle phase), make the
        // writes visible to the tensor core and pass the stage to the MMA
        // warp.  The heads need no pass: the TF32 MMA drops an fp32
        // operand's 13 low mantissa bits (truncation, measured on sm_103a
        // and pinned by tests/test_parity_tc.py), so it reads the copied
        // values as exactly their heads.
        const int ct = tid - 6 * 32;
        const uint32_t nchunk = g.stage_bytes >> 4;
        constexpr int CB = 4;   // 16-byte chunks a thread loads before it writes
        int s = 0;
        uint32_t ph = 0;
        for (int j = 0; j < total; ++j) {
            if (aborted()) break;
            const int l = j % tc::X3_LO;
            // the stage has landed, and the MMAs of stage j - X3_LO have read
            // this remainder buffer
            bool got = mbar_wait_bounded(smem_u32(&full_bar[s]), ph, timeout_ns);
            if (got && j >= tc::X3_LO)
                got = mbar_wait_bounded(smem_u32(&lo_empty[l]), (uint32_t)((j / tc::X3_LO - 1) & 1), timeout_ns);
            if (__any_sync(0xffffffffu, !got)) {
                if (lane == 0) give_up();
                break;
            }
            uint4 *hp = reinterpret_cast<uint4 *>(abuf + (size_t)s * g.stage_bytes);
            uint4 *lp = reinterpret_cast<uint4 *>(alo + (size_t)l * g.stage_bytes);
            for (uint32_t c0 = (uint32_t)ct; c0 < nchunk; c0 += 128 * CB) {
                uint4 v[CB];
#pragma unroll
                for (int q = 0; q < CB; ++q)
                    if (c0 + 128 * q < nchunk) v[q] = hp[c0 + 128 * q];
#pragma unroll
                for (int q = 0; q < CB; ++q) {
                    const uint32_t c = c0 + 128 * q;
                    if (c < nchunk)
                        lp[c] = make_uint4(tc::tf32_rest(v[q].x), tc::tf32_rest(v[q].y), tc::tf32_rest(v[q].z),
                                           tc::tf32_rest(v[q].w));
                }
            }
            fence_proxy_async_smem();   // these writes -> visible to the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&conv_bar[s]));
            if (++s == ns) {
                s = 0;
                ph ^= 1u;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Two sets of four warps (0-3 and 6-9); warp w reads TMEM lane
        // quadrant q = w % 4, set 0 the even M-tiles of a tile, set 1 the odd
        // ones.  Lane l holds GEMM row m = mt * 128 + 32 q + l, i.e. padded
        // column l of tile row 4 mt + q; its output column l (l < 30) is the
        // sum over s of the s-block of lane l + s.  With TMA_OUT each lane
        // writes its pixel (bias and ReLU applied) into the warp's output
        // buffer and lane 0 stores the row with one TMA copy (image edges and
        // channels past Cout are clipped by the TMA), waiting first for its
        // previous store to have read the buffer.  Otherwise (outputs of 16
        // or 32 bytes per pixel) each lane stores its pixel directly:
        // neighbouring lanes write neighbouring pixels.
        // (X3: warps 0-3 only, every M-tile; warps 6-9 convert)
        const int q4 = warp & 3, set = warp < 4 ? 0 : 1;
        constexpr int MSTEP = X3 ? 1 : 2;
        float bias_r[CW];
#pragma unroll
        for (int i = 0; i < CW; ++i) bias_r[i] = (bias && co0 + i < Cout) ? __ldg(bias + co0 + i) : 0.f;
        const uint32_t wst = smem_u32(stg + (warp < 4 ? warp : warp - 2) * tc::OUT_BUF);
        for (int u = 0; u < my_tiles; ++u) {
            const int b = u & 1;
            if (aborted()) break;
            const bool got = mbar_wait_bounded(smem_u32(&acc_full[b]), (u >> 1) & 1, timeout_ns);
            if (__any_sync(0xffffffffu, !got) || aborted()) {
                if (lane == 0) give_up();
                break;
            }
            tc::fence_after_sync();
            int n, y0, x0;
            tile_origin(u, n, y0, x0);
            const uint32_t tbuf = tmem + (uint32_t)(b * tc::TMEM_BUF) + ((uint32_t)(q4 * 32) << 16);
            if constexpr (RSN) {
                // Staged row ty = 4 mt + q4 of this warp holds, per tap (r, s),
                // the products for output row ty - r at column lane - s.  Per
                // r, the lane-shifted sum over s goes to rsum[r][ty - r]; once
                // every epilogue warp's sums are in place (a bounded mbarrier
                // wait: a warp that gave up must not hold the others), each
                // warp adds the three r for its output rows.  rsum holds two
                // tiles, alternating, so tile u's writes never meet tile u - 1's
                // reads (a warp writes tile u only after every warp arrived
                // for tile u - 1, i.e. finished reading tile u - 2).
                float *rb = rsum + (size_t)(u & 1) * (3 * g.TR * 32 * CG);
                for (int mt = set; mt < g.MT; mt += MSTEP) {
                    uint32_t rv[9][CG];
#pragma unroll
                    for (int t = 0; t < 9; ++t) tc::tmem_ld<CG>(tbuf + (uint32_t)(mt * DSTR + t * CG), rv[t]);
                    tc::tmem_wait_ld();
                    if constexpr (X3) {
                        uint32_t cv[9][CG];
#pragma unroll
                        for (int t = 0; t < 9; ++t) tc::tmem_ld<CG>(tbuf + (uint32_t)(mt * DSTR + NB + t * CG), cv[t]);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int t = 0; t < 9; ++t)
#pragma unroll
                            for (int i = 0; i < CG; ++i)
                                rv[t][i] = __float_as_uint(__uint_as_float(rv[t][i]) + __uint_as_float(cv[t][i]));
                    }
                    const int ty = mt * 4 + q4;
#pragma unroll
                    for (int r = 0; r < 3; ++r) {
                        float c[CG];
#pragma unroll
                        for (int i = 0; i < CG; ++i)
                            c[i] = __uint_as_float(rv[3 * r][i]) +
                                   __shfl_down_sync(0xffffffffu, __uint_as_float(rv[3 * r + 1][i]), 1) +
                                   __shfl_down_sync(0xffffffffu, __uint_as_float(rv[3 * r + 2][i]), 2);
                        const int e = ty - r;
                        if (e >= 0 && e < g.TR)
                            *reinterpret_cast<float4 *>(rb + ((r * g.TR + e) * 32 + lane) * CG) =
                                make_float4(c[0], c[1], c[2], c[3]);
                    }
                }
                // every column this warp needs has been read: release the buffer
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
                if (lane == 0) mbar_arrive(smem_u32(&rs_bar[u & 1]));
                const bool all = mbar_wait_bounded(smem_u32(&rs_bar[u & 1]), (uint32_t)((u >> 1) & 1), timeout_ns);
                if (__any_sync(0xffffffffu, !all)) {
                    if (lane == 0) give_up();
                    break;
                }
                constexpr int NEW = X3 ? 4 : 8;                   // epilogue warps
                const int ew = warp < 4 ? warp : warp - 2;        // 0 .. NEW - 1
                for (int e = ew; e < g.TR; e += NEW) {
                    const int oy = y0 + e, ox = x0 + lane;
                    if (lane < tc::TC && oy < H && ox < W) {
                        float o[CG];
#pragma unroll
                        for (int i = 0; i < CG; ++i) o[i] = 0.f;
#pragma unroll
                        for (int r = 0; r < 3; ++r) {
                            const float4 p = *reinterpret_cast<const float4 *>(rb + ((r * g.TR + e) * 32 + lane) * CG);
                            o[0] += p.x;
                            o[1] += p.y;
                            o[2] += p.z;
                            o[3] += p.w;
                        }
#pragma unroll
                        for (int i = 0; i < CG; ++i) o[i] = relu_if(o[i] + bias_r[i], act);
                        unsigned char *yp = reinterpret_cast<unsigned char *>(yv) +
                                            ((((long long)n * H + oy) * W + ox) * Cout + co0) * OSZ;
                        if (co0 < Cout) {
                            if constexpr (YBF16)
                                *reinterpret_cast<uint2 *>(yp) =
                                    make_uint2(tc::pack_bf16(o[0], o[1]), tc::pack_bf16(o[2], o[3]));
                            else
                                *reinterpret_cast<float4 *>(yp) = make_float4(o[0], o[1], o[2], o[3]);
                        }
                    }
                }
                continue;
            }
            const int last_mt = X3 ? g.MT - 1 : set + ((g.MT - 1 - set) & ~1);   // this set's last M-tile (< set: none)
            if (last_mt < set) {
                // nothing of this tile for this warp: release the buffer at once
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
            }
            for (int mt = set; mt < g.MT; mt += MSTEP) {
                // v[i] = sum over s of column (s, i) of lane l + s (X3: heads
                // plus corrections), in the order s = 0, 1, 2, then the bias
                float v[CW];
                if constexpr (X3) {
#pragma unroll
                    for (int blk = 0; blk < 3; ++blk) {
                        uint32_t m[CW], c[CW];
                        tc::tmem_ld<CW>(tbuf + (uint32_t)(mt * DSTR + blk * CG), m);
                        tc::tmem_ld<CW>(tbuf + (uint32_t)(mt * DSTR + NB + blk * CG), c);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < CW; ++i) {
                            float t = __uint_as_float(m[i]) + __uint_as_float(c[i]);
                            if (blk > 0) t = __shfl_down_sync(0xffffffffu, t, blk);
                            v[i] = blk == 0 ? t : v[i] + t;
                        }
                    }
                } else {
                    uint32_t r0[CW], r1[CW], r2[CW];
                    tc::tmem_ld<CW>(tbuf + (uint32_t)(mt * DSTR), r0);
                    tc::tmem_ld<CW>(tbuf + (uint32_t)(mt * DSTR + CG), r1);
                    tc::tmem_ld<CW>(tbuf + (uint32_t)(mt * DSTR + 2 * CG), r2);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < CW; ++i)
                        v[i] = __uint_as_float(r0[i]) + __shfl_down_sync(0xffffffffu, __uint_as_float(r1[i]), 1) +
                               __shfl_down_sync(0xffffffffu, __uint_as_float(r2[i]), 2);
                }
                if (mt == last_mt) {
                    // every column this warp needs is in registers: release the buffer
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
                }
#pragma unroll
                for (int i = 0; i < CW; ++i) v[i] = relu_if(v[i] + bias_r[i], act);
                // the pixel's outputs as 32-bit words: fp32, or bf16 pairs
                constexpr int NWD = CW * OSZ / 4;
                uint32_t o[NWD];
#pragma unroll
                for (int i = 0; i < NWD; ++i) o[i] = YBF16 ? tc::pack_bf16(v[2 * i], v[2 * i + 1]) : __float_as_uint(v[i]);
                const int oy = y0 + mt * 4 + q4;
                if (oy >= H) continue;   // the same for the whole warp
                if constexpr (TMA_OUT) {
                    const uint32_t ob = wst;
                    if (lane == 0) bulk_wait_read<0>();   // the store that last read this buffer is done
                    __syncwarp();
                    if (lane < tc::TC) {
#pragma unroll
                        for (int q = 0; q < OCH; ++q)
                            tc::st_shared_v4(ob + lane * OROWB + ((q ^ tc::stg_key<OROWB>(lane)) << 4), o[4 * q],
                                             o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                    }
                    fence_proxy_async_smem();   // these writes -> visible to the TMA
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_4d(&tmy, ob, co0, x0, oy, n);
                        bulk_commit();
                    }
                } else {
                    // pieces of 4 channels: 16 bytes (fp32) or 8 bytes (bf16)
                    const int ox = x0 + lane;
                    if (lane < tc::TC && ox < W) {
                        unsigned char *yp = reinterpret_cast<unsigned char *>(yv) +
                                            ((((long long)n * H + oy) * W + ox) * Cout + co0) * OSZ;
#pragma unroll
                        for (int q = 0; q < CW / 4; ++q) {
                            if (co0 + 4 * q < Cout) {
                                if constexpr (YBF16)
                                    *reinterpret_cast<uint2 *>(yp + 8 * q) = make_uint2(o[2 * q], o[2 * q + 1]);
                                else
                                    *reinterpret_cast<uint4 *>(yp + 16 * q) =
                                        make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                            }
                        }
                    }
                }
            }
        }
        if (TMA_OUT && lane == 0) bulk_wait_all();   // every store has written global memory
    }

    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) (void)mbar_wait_bounded(smem_u32(&w_bar), 0, timeout_ns);   // the weight copies have landed
    if (aborted() && tid == 0 && status) atomicExch(status, kDeviceTimeout);
    if (warp == 0) tc::tmem_dealloc(tmem, g.tmem_cols);
}

// Largest dynamic shared memory a CTA may use (227 KB less a margin for the
// static barriers), of which 1 KB may go to aligning the stage buffers.
constexpr size_t kTcSmemCap = 227 * 1024 - 1024;

// Tile geometry for output-channel groups of Cg (MMA N = NB): M-tiles of 4
// image rows x 32 padded columns; MT M-tiles per tile so that MT * NB fits one
// accumulator buffer and at least MIN_STAGE stage buffers of (4 MT + 2) rows
// fit in shared memory beside the filters and the epilogue buffers; among
// those, the MT that wastes least work on halo rows, partial tiles and an
// unevenly filled persistent grid.  Leftover shared memory goes to further
// stage buffers (up to MAX_STAGE).  x3 (split TF32): X3_LO more buffers of a
// stage's size hold remainders, the filter bank holds heads and remainders
// (twice the rows), an M-tile takes 2 * NB accumulator columns (heads and
// corrections), and four epilogue warps need four output buffers.
static bool tc_geometry(int Cg, int NB, int kc, int rowb, int groups, int Cin, int RS, int H, int W, int Nimg,
                        bool x3, bool rsn, tc::TcGeom &g)
{
    const int nk = (Cin + kc - 1) / kc;
    // filter bank: (K step, [tap r,] 4-channel block) blocks of NB rows (x3: 2 NB)
    const size_t w_bytes = ((size_t)nk * (rsn ? 1 : 3) * 2 * (x3 ? 2 * NB : NB) * 16 + 1023) & ~(size_t)1023;
    const int cols = x3 ? 2 * NB : NB;   // accumulator columns per M-tile
    const int nlo = x3 ? tc::X3_LO : 0;  // remainder buffers, each the size of a stage
    const size_t stg_base = x3 ? tc::X3_STG_BYTES : tc::STG_BYTES;
    // rsn: output rows per tile = staged rows - 2 (the M rows are the staged
    // rows), and the epilogue's row partial sums for two tiles share the
    // output-buffer region
    auto rows_out = [&](int MT) { return rsn ? 4 * MT - 2 : 4 * MT; };
    auto rows_staged = [&](int MT) { return rsn ? 4 * MT : 4 * MT + 2; };
    auto fixed_of = [&](int MT) {
        size_t stg = stg_base;
        const size_t rs = rsn ? (size_t)2 * 3 * rows_out(MT) * tc::WP * Cg * 4 : 0;
        if (rs > stg) stg = rs;
        return w_bytes + stg + 1024;   // + alignment slack
    };
    if (fixed_of(1) >= kTcSmemCap) return false;
    const int sms = device_sm_count() / groups > 0 ? device_sm_count() / groups : 1;   // CTAs per channel group
    const int tiles_x = (W + tc::TC - 1) / tc::TC;
    int best_mt = 0;
    double best_eff = 0;
    // the OIHW weights are staged in the stage buffers first: an odd pitch
    // of 16-byte units per output channel
    const int raw_pitch = tc::filter_raw_pitch(Cin, RS);
    const size_t raw = (size_t)Cg * raw_pitch * 16;
    for (int MT = 1; MT * cols <= tc::TMEM_BUF && MT <= 16; ++MT) {
        const int TR = rows_out(MT);
        const size_t stage = (size_t)rows_staged(MT) * tc::WP * rowb;
        const size_t fixed = fixed_of(MT);
        if (fixed + (tc::MIN_STAGE + nlo) * stage > kTcSmemCap) break;
        const size_t nfit = (kTcSmemCap - fixed) / stage - nlo;
        if ((nfit < tc::MAX_STAGE ? nfit : tc::MAX_STAGE) * stage < raw) continue;
        const long long tiles = (long long)tiles_x * ((H + TR - 1) / TR) * Nimg;
        const long long rounds = (tiles + sms - 1) / sms;
        const double fill = (double)tiles / ((double)rounds * sms);
        const double edge = (double)H / ((double)((H + TR - 1) / TR) * TR);
        const double halo = (double)TR / rows_staged(MT);
        const double eff = fill * edge * halo;
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best_mt = MT;
        }
    }
    if (best_mt == 0) return false;
    const size_t fixed = fixed_of(best_mt);
    g.MT = best_mt;
    g.TR = rows_out(g.MT);
    g.THh = rows_staged(g.MT);
    g.tiles_x = tiles_x;
    g.tiles_y = (H + g.TR - 1) / g.TR;
    g.ntiles = g.tiles_x * g.tiles_y * Nimg;
    g.nk = nk;
    g.nstg = (Cin + tc::CH - 1) / tc::CH;
    g.stage_bytes = (uint32_t)((size_t)g.THh * tc::WP * rowb);
    g.w_bytes = (uint32_t)w_bytes;
    const int ns = (int)((kTcSmemCap - fixed) / g.stage_bytes) - nlo;
    g.nstage = ns < tc::MAX_STAGE ? ns : tc::MAX_STAGE;
    g.raw_pitch = raw_pitch;
    g.smem_bytes = (uint32_t)(fixed + (size_t)(g.nstage + nlo) * g.stage_bytes);
    g.tmem_cols = 2 * tc::TMEM_BUF;
    return true;
}

static PFN_cuTensorMapEncodeTiled_v12000 tc_tensor_map_encoder()
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

// a.x and a.y point to fp32 or (for OP = OpBF16, YBF16) bf16 NHWC tensors.
template <int CG, class OP, bool YBF16, bool RSN = false>
static cudaError_t launch_tc_cg(const ConvArgs &a, cudaStream_t st)
{
    constexpr int NB = RSN ? (9 * CG + 15) / 16 * 16 : (3 * CG + 15) / 16 * 16;
    constexpr int OSZ = YBF16 ? 2 : 4;
    constexpr int OROWB = CG * OSZ;
    if (RSN && (a.R != 3 || a.S != 3)) return cudaErrorNotSupported;
    tc::TcGeom g;
    const int groups = (a.Cout + CG - 1) / CG;
    if (!tc_geometry(CG, NB, OP::KC, OP::ROWB * OP::SUB, groups, a.Cin, a.R * a.S, a.H, a.W, a.N, OP::X3, RSN, g))
        return cudaErrorNotSupported;
    if ((long long)g.tiles_x * g.tiles_y * a.N > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tc_tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    // NHWC activations as a 4-D tensor (C, W, H, N); box = the channels of
    // one sub-buffer (32 fp32 or 32 bf16: one swizzled row per pixel;
    // channels past Cin read as zero) x 32 padded columns x THh (= TR + 2)
    // rows of one image
    CUtensorMap tm;
    const cuuint64_t dims[4] = {(cuuint64_t)a.Cin, (cuuint64_t)a.W, (cuuint64_t)a.H, (cuuint64_t)a.N};
    const cuuint64_t strides[3] = {(cuuint64_t)a.Cin * OP::ESZ, (cuuint64_t)a.W * a.Cin * OP::ESZ,
                                   (cuuint64_t)a.H * a.W * a.Cin * OP::ESZ};
    const cuuint32_t box[4] = {(cuuint32_t)(tc::CH / OP::SUB), (cuuint32_t)tc::WP, (cuuint32_t)g.THh, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (encode(&tm, OP::ESZ == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<float *>(a.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               OP::ROWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                               : (OP::ROWB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B),
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    // NHWC output as (C, W, H, N); box = the group's CG channels x TC pixels
    // of one row, swizzled like the epilogue's buffers (groups whose outputs
    // take 64 or 128 bytes per pixel; the others store directly and leave
    // this map unused)
    CUtensorMap tmo;
    std::memset(&tmo, 0, sizeof(tmo));
    if (OROWB >= 64) {
        const cuuint64_t odims[4] = {(cuuint64_t)a.Cout, (cuuint64_t)a.W, (cuuint64_t)a.H, (cuuint64_t)a.N};
        const cuuint64_t ostrides[3] = {(cuuint64_t)a.Cout * OSZ, (cuuint64_t)a.W * a.Cout * OSZ,
                                        (cuuint64_t)a.H * a.W * a.Cout * OSZ};
        const cuuint32_t obox[4] = {(cuuint32_t)CG, (cuuint32_t)tc::TC, 1, 1};
        if (encode(&tmo, YBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.y, odims,
                   ostrides, obox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   OROWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorNotSupported;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static KernelCache cache;
    e = ensure_dynamic_smem(cache, dev, conv_tc_kernel<CG, OP, YBF16, RSN>, (int)g.smem_bytes);
    if (e != cudaSuccess) return e;
    const int per_group = device_sm_count() / groups > 0 ? device_sm_count() / groups : 1;
    const int grid = g.ntiles < per_group ? g.ntiles : per_group;
    conv_tc_kernel<CG, OP, YBF16, RSN><<<dim3(grid, groups), tc::NTHREADS, g.smem_bytes, st>>>(
        tm, tmo, a.w, a.b, a.y, a.H, a.W, a.Cin, a.Cout, a.R, a.S, a.act, g, device_status_ptr(), 1000000000ull);
    return cudaGetLastError();
}

// Output channels per CTA: the smallest group that holds Cout, at most 32
// (larger Cout runs as groups on blockIdx.y); where a group's filters do not
// fit in shared memory, smaller groups (a smaller MMA N, lower tensor-core
// efficiency).
template <class OP, bool YBF16>
static cudaError_t launch_tc_groups(const ConvArgs &a, cudaStream_t st)
{
    if (a.R > 3 || a.S > 3) return cudaErrorNotSupported;
    cudaError_t e = cudaErrorNotSupported;
    if (a.Cout > 16) e = launch_tc_cg<32, OP, YBF16>(a, st);
    if (e == cudaErrorNotSupported && a.Cout > 8) e = launch_tc_cg<16, OP, YBF16>(a, st);
    if (e == cudaErrorNotSupported && a.Cout > 4) e = launch_tc_cg<8, OP, YBF16>(a, st);
    // 4 or fewer channels with 3 x 3 filters, TF32 operands: all nine taps in
    // N (with BF16 operands the per-tap form measured faster: 24.6 against
    // 26.6 us on 32 -> 4, 1280 x 720)
    if constexpr (OP::FMT == tc::OpTF32::FMT)
        if (e == cudaErrorNotSupported && a.Cout <= 4) e = launch_tc_cg<4, OP, YBF16, true>(a, st);
    if (e == cudaErrorNotSupported) e = launch_tc_cg<4, OP, YBF16>(a, st);
    return e;
}

cudaError_t launch_conv_tc(const ConvArgs &a, cudaStream_t st) { return launch_tc_groups<tc::OpTF32, false>(a, st); }

cudaError_t launch_conv_tc_x3(const ConvArgs &a, cudaStream_t st)
{
    return launch_tc_groups<tc::OpTF32x3, false>(a, st);
}

cudaError_t launch_conv_tc_bf16(const ConvArgs &a, bool y_bf16, cudaStream_t st)
{
    return y_bf16 ? launch_tc_groups<tc::OpBF16, true>(a, st) : launch_tc_groups<tc::OpBF16, false>(a, st);
}

}  // namespace sc
