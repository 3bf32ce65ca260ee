// Tensor-core variant of the direct convolution: implicit GEMM on the 5th
// generation tensor cores (tcgen05, accumulators in tensor memory), TF32
// operands, fp32 accumulation.  It computes the same operation as
// conv2d_fwd (stride 1, zero "same" padding, bias, ReLU) with TF32 rounding
// of x and w, so it is checked with its own tolerance (5e-3 * sum|x*w|).
//
// GEMM view: D[pixel][co] = sum_{r,s,ci} A[pixel][(r,s,ci)] * B[co][(r,s,ci)],
// A[p][(r,s,ci)] = x at pixel p shifted by (r - R/2, s - S/2), channel ci.
// ("Optimizing Memory Efficiency for Convolution Kernels on Kepler GPUs",
// Section 3.3, compares direct convolution with this GEMM formulation; the
// reuse argument of Section 3.3.2 is kept: each input pixel is staged once
// per tile, and every tap reads it again from shared memory.)
//
// Tile: TR x TC output pixels x N output channels (N = Cout rounded up to
// 16, at most 64; larger Cout runs as channel groups on blockIdx.y).  Shared memory holds the tile's halo as "padded pixels" with row pitch
// WP = TC + K - 1: padded pixel q = ty * WP + tx is image pixel
// (y0 + ty - K/2, x0 + tx - K/2), zero outside the image.  Output pixel
// (ty, tx) of the tile is GEMM row m = ty * WP + tx, and its tap (r, s) reads
// padded pixel m + r * WP + s: the A operand of tap (r, s) is the same
// staged data starting r * WP + s pixels later, so a tap is only a different
// start address in the MMA's shared-memory descriptor.  Rows m with
// tx >= TC are computed and discarded (K - 1 of every WP).
//
// Operand layouts (K-major, no swizzle): the canonical core matrix is 8 rows
// x 16 bytes.  A: a plane of padded pixels per 4-channel block, 16 bytes per
// pixel, so 8 consecutive pixels form a core matrix (SBO = 128 bytes) and the
// next 4 channels are the next plane (LBO = plane stride).  B (filters): per
// tap and 4-channel block, the Cout rows of 16 bytes (SBO 128, LBO N * 16).
// One MMA is M = 128 rows x N x K = 8 (two 4-channel blocks).
//
// Pipeline: persistent CTAs (one per SM), each with its whole filter bank
// resident in shared memory, and warp-specialised roles linked by
// mbarriers:
//  * producer (warp 4, one lane): per stage, two 4-D TMA copies
//    (cp.async.bulk.tensor) of the tile's padded activations, one box of
//    (4 channels, WP pixels, TR+K-1 rows) per channel-block plane; the TMA
//    zero fill outside the image is the convolution's zero padding.  A stage
//    buffer is refilled once the MMAs that read it have completed (`empty`).
//  * MMA issuer (warp 5, one lane): waits for a stage (`full`), issues its
//    K*K*MT MMAs, commits them to the stage's `empty` barrier, and after a
//    tile's last stage commits to the tile's accumulator barrier.
//  * epilogue (warps 0-3, one TMEM lane quadrant each): waits for a tile's
//    accumulators, reads them with tcgen05.ld, adds bias, applies ReLU,
//    writes NHWC, and frees the accumulator buffer.  Accumulators are
//    double-buffered in tensor memory, so a tile's epilogue overlaps the
//    next tile's MMAs.
// Every wait is bounded in time; on expiry the CTA records
// SC_ERR_DEVICE_TIMEOUT, lets its own copies and MMAs land, frees tensor
// memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace sc {

namespace tc {

constexpr int NTHREADS = 192;   // warps 0-3 epilogue (TMEM lane quadrants), 4 producer, 5 MMA
constexpr int NSTAGE = 3;       // activation stages in flight
constexpr int TMEM_BUF = 256;   // tensor-memory columns per accumulator buffer (two buffers)

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    // start address, LBO, SBO in 16-byte units; version 1 (bits 46-47);
    // base offset 0; layout type 0 = no swizzle (bits 61-63)
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::tf32: D = F32, A = B = TF32, both K-major,
// dense, M = 128.
__host__ __device__ constexpr uint32_t idesc_tf32(int n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// 16 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

struct TcGeom {
    int TC, TR, WP, THh, MT, P;  // tile cols/rows, padded pitch, padded rows, M-tiles, pixels per plane
    int tiles_x, tiles_y, ntiles, nk;
    uint32_t a_plane_bytes, a_bytes, box_bytes, w_bytes, smem_bytes, tmem_cols;
};

}  // namespace tc

// N: output channels per CTA (multiple of 16, <= 64), K: kernel size.
template <int K, int N>
__global__ void __launch_bounds__(tc::NTHREADS, 1)
    conv_tc_kernel(const __grid_constant__ CUtensorMap tmx, const float *__restrict__ w,
                   const float *__restrict__ bias, float *__restrict__ y, int Nimg, int H, int W, int Cin, int Cout,
                   int R, int S, int act, tc::TcGeom g, int *status, unsigned long long timeout_ns)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long full_bar[tc::NSTAGE], empty_bar[tc::NSTAGE];
    __shared__ __align__(8) unsigned long long acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int dr = (K - R) / 2, ds = (K - S) / 2;
    const int co0 = blockIdx.y * N;                      // this CTA's output channels co0 .. co0+N-1
    unsigned char *wsm = smem_raw;                       // resident filters
    unsigned char *abuf = smem_raw + g.w_bytes;          // NSTAGE activation stages

    if (warp == 0) tc::tmem_alloc(smem_u32(&tmem_base_sh), g.tmem_cols);
    if (tid == 0) {
        for (int j = 0; j < tc::NSTAGE; ++j) {
            mbar_init(smem_u32(&full_bar[j]), 1);
            mbar_init(smem_u32(&empty_bar[j]), 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(smem_u32(&acc_full[j]), 1);
            mbar_init(smem_u32(&acc_empty[j]), 4);   // one arrive per epilogue warp
        }
        abort_sh = 0;
        fence_mbar_init();
    }
    // Filters, once per CTA, as asynchronous 4-byte copies: element
    // (k, tap, cb, co, j) of the [stage][tap][cb][co][4] bank is input
    // channel 8k + 4cb + j; taps the R x S filter lacks, channels beyond Cin
    // and co beyond Cout read zero.  The overhang of every activation plane
    // (pixels past the TMA box, read only by discarded GEMM rows) is zeroed.
    {
        float *wf = reinterpret_cast<float *>(wsm);
        const int n_e = (int)(g.w_bytes / 4);
        const int RS = R * S;
        for (int e = tid; e < n_e; e += tc::NTHREADS) {
            const int j = e & 3;
            int t2 = e >> 2;
            const int co = t2 % N;
            t2 /= N;
            const int cb = t2 & 1;
            t2 >>= 1;
            const int tap = t2 % (K * K);
            const int k = t2 / (K * K);
            const int ci = 8 * k + 4 * cb + j;
            const int r = tap / K - dr, s = tap % K - ds;
            const bool ok = (k < g.nk) & (ci < Cin) & (co0 + co < Cout) & (r >= 0) & (r < R) & (s >= 0) & (s < S);
            const float *src = ok ? w + ((size_t)(co0 + co) * Cin + ci) * RS + r * S + s : w;
            cp_async4(smem_u32(wf + e), src, ok ? 4 : 0);
        }
        cp_async_commit();
        float4 *af = reinterpret_cast<float4 *>(abuf);
        const int used = g.THh * g.WP;
        for (int e = tid; e < tc::NSTAGE * 2 * g.P; e += tc::NTHREADS) {
            if (e % g.P >= used) af[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        cp_async_wait<0>();
    }
    fence_proxy_async_smem();   // generic-proxy writes above -> visible to the tensor core
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    const int my_tiles = (g.ntiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int total = my_tiles * g.nk;
    auto tile_origin = [&](int u, int &n, int &y0, int &x0) {
        int t = (int)blockIdx.x + u * (int)gridDim.x;
        x0 = (t % g.tiles_x) * g.TC;
        t /= g.tiles_x;
        y0 = (t % g.tiles_y) * g.TR;
        n = t / g.tiles_y;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int *>(&abort_sh) != 0; };
    auto give_up = [&]() { atomicExch(&abort_sh, 1); };

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < total && !aborted(); ++j) {
                const int s = j % tc::NSTAGE;
                if (j >= tc::NSTAGE &&
                    !mbar_wait_bounded(smem_u32(&empty_bar[s]), ((j / tc::NSTAGE) - 1) & 1, timeout_ns)) {
                    give_up();
                    break;
                }
                int n, y0, x0;
                tile_origin(j / g.nk, n, y0, x0);
                const int c = 8 * (j % g.nk);
                unsigned char *st = abuf + s * g.a_bytes;
                mbar_arrive_expect_tx(smem_u32(&full_bar[s]), 2 * g.box_bytes);
                tma_load_4d(smem_u32(st), &tmx, c, x0 - K / 2, y0 - K / 2, n, smem_u32(&full_bar[s]));
                tma_load_4d(smem_u32(st + g.a_plane_bytes), &tmx, c + 4, x0 - K / 2, y0 - K / 2, n,
                            smem_u32(&full_bar[s]));
                issued = j + 1;
            }
            // every copy this lane issued has landed before the CTA may exit
            for (int j = (issued > tc::NSTAGE ? issued - tc::NSTAGE : 0); j < issued; ++j)
                (void)mbar_wait_bounded(smem_u32(&full_bar[j % tc::NSTAGE]), (j / tc::NSTAGE) & 1, timeout_ns);
        }
    } else if (warp == 5) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_tf32(N);
            int j = 0, committed = -1;
            for (int u = 0; u < my_tiles && !aborted(); ++u) {
                const int b = u & 1;
                if (u >= 2 && !mbar_wait_bounded(smem_u32(&acc_empty[b]), ((u >> 1) - 1) & 1, timeout_ns)) {
                    give_up();
                    break;
                }
                tc::fence_after_sync();
                const uint32_t dbase = tmem + (uint32_t)(b * tc::TMEM_BUF);
                bool ok = true;
                for (int k = 0; k < g.nk; ++k, ++j) {
                    const int s = j % tc::NSTAGE;
                    if (!mbar_wait_bounded(smem_u32(&full_bar[s]), (j / tc::NSTAGE) & 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    // descriptors advance by adding 16-byte units to the start-address field
                    const uint64_t a_desc0 = tc::smem_desc(smem_u32(abuf + s * g.a_bytes), g.a_plane_bytes, 128);
                    const uint64_t b_desc0 =
                        tc::smem_desc(smem_u32(wsm + (size_t)k * K * K * 2 * N * 16), N * 16, 128);
#pragma unroll
                    for (int tap = 0; tap < K * K; ++tap) {
                        const int r = tap / K, sx = tap % K;
                        const uint64_t bd = b_desc0 + (uint64_t)(tap * 2 * N);
                        const uint64_t ad_tap = a_desc0 + (uint64_t)(r * g.WP + sx);
#pragma unroll 1
                        for (int mt = 0; mt < g.MT; ++mt)
                            tc::mma_tf32(dbase + (uint32_t)(mt * N), ad_tap + (uint64_t)(mt * 128), bd, idesc,
                                         (k > 0 || tap > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(smem_u32(&empty_bar[s]));
                    committed = j;
                }
                if (!ok) {
                    give_up();
                    break;
                }
                tc::mma_commit(smem_u32(&acc_full[b]));
            }
            // MMAs still executing must finish before tensor memory is freed
            if (committed >= 0)
                (void)mbar_wait_bounded(smem_u32(&empty_bar[committed % tc::NSTAGE]),
                                        (committed / tc::NSTAGE) & 1, timeout_ns);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        for (int u = 0; u < my_tiles; ++u) {
            const int b = u & 1;
            const bool got = mbar_wait_bounded(smem_u32(&acc_full[b]), (u >> 1) & 1, timeout_ns);
            if (__any_sync(0xffffffffu, !got) || aborted()) {
                if (lane == 0) give_up();
                break;
            }
            tc::fence_after_sync();
            int n, y0, x0;
            tile_origin(u, n, y0, x0);
            const uint32_t tbuf = tmem + (uint32_t)(b * tc::TMEM_BUF) + ((uint32_t)(warp * 32) << 16);
            for (int mt = 0; mt < g.MT; ++mt) {
                const int m = mt * 128 + warp * 32 + lane;
                const int ty = m / g.WP, tx = m % g.WP;
                const int oy = y0 + ty, ox = x0 + tx;
                const bool valid = (ty < g.TR) & (tx < g.TC) & (oy < H) & (ox < W);
                float *yp = y + ((((long long)n * H + (valid ? oy : 0)) * W + (valid ? ox : 0)) * Cout + co0);
#pragma unroll 1
                for (int c0 = 0; c0 < N; c0 += 16) {
                    float v[16];
                    tc::tmem_ld16(tbuf + (uint32_t)(mt * N + c0), v);
                    if (valid) {
#pragma unroll
                        for (int q = 0; q < 16; q += 4) {
                            const int co = c0 + q;             // within the group
                            if (co0 + co < Cout) {
                                const float *bq = bias ? bias + co0 + co : nullptr;
                                float4 o;
                                o.x = relu_if(v[q + 0] + (bq ? __ldg(bq + 0) : 0.f), act);
                                o.y = relu_if(v[q + 1] + (bq ? __ldg(bq + 1) : 0.f), act);
                                o.z = relu_if(v[q + 2] + (bq ? __ldg(bq + 2) : 0.f), act);
                                o.w = relu_if(v[q + 3] + (bq ? __ldg(bq + 3) : 0.f), act);
                                *reinterpret_cast<float4 *>(yp + co) = o;
                            }
                        }
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (aborted() && tid == 0 && status) atomicExch(status, kDeviceTimeout);
    if (warp == 0) tc::tmem_dealloc(tmem, g.tmem_cols);
}

// Padded pixels per channel-block plane: every pixel the MMAs read (the
// last GEMM row plus the largest tap offset), rounded to a multiple of 8 so
// each plane starts 128-byte aligned (a TMA destination).
static int tc_plane_pixels(int MT, int K, int WP)
{
    const int need = MT * 128 + (K - 1) * WP + (K - 1);
    return (need + 7) / 8 * 8;
}

// Tile geometry: pitch WP = TC + K - 1; M-tiles of 128 GEMM rows; TR rows
// so that MT * N fits the 512 tensor-memory columns and the resident filters
// plus two activation stages fit in shared memory.
static bool tc_geometry(int K, int N, int groups, int Cin, int H, int W, int Nimg, tc::TcGeom &g)
{
    const int nk = (Cin + 7) / 8;
    const size_t w_bytes = (size_t)nk * K * K * 2 * N * 16;
    if (w_bytes > 160 * 1024) return false;
    int best_tc = -1, best_tr = 0;
    double best_eff = 0;
    const int cands[] = {W, 126, 128, 62, 64};
    for (int TC : cands) {
        // TMA boxes are at most 256 elements per dimension
        if (TC < 1 || TC > W || TC + K - 1 > 256) continue;
        const int WP = TC + K - 1;
        for (int TR = 1; TR <= H && TR + K - 1 <= 256 && TR <= 64; ++TR) {
            const int MT = (TR * WP + 127) / 128;
            if (MT * N > tc::TMEM_BUF) break;
            const int P = tc_plane_pixels(MT, K, WP);
            const size_t total = w_bytes + tc::NSTAGE * (2 * (size_t)P * 16);
            if (total > 220 * 1024) break;
            const long long tiles = (long long)((W + TC - 1) / TC) * ((H + TR - 1) / TR) * Nimg;
            // useful fraction of MMA rows, of the tile area, and of the persistent grid
            const double rows = (double)TR * TC / ((double)MT * 128);
            const double edge = (double)W * H / ((double)((W + TC - 1) / TC) * TC * ((H + TR - 1) / TR) * TR);
            const int sms = (device_sm_count() + groups - 1) / groups;  // SMs per channel group
            const long long rounds = (tiles + sms - 1) / sms;
            const double fill = (double)tiles / ((double)rounds * sms);
            // each tile re-reads K - 1 halo rows of input
            const double halo = (double)TR / (TR + K - 1);
            const double eff = rows * edge * fill * halo;
            if (eff > best_eff + 1e-9) {
                best_eff = eff;
                best_tc = TC;
                best_tr = TR;
            }
        }
    }
    if (best_tc < 0) return false;
    g.TC = best_tc;
    g.TR = best_tr;
    g.WP = g.TC + K - 1;
    g.THh = g.TR + K - 1;
    g.MT = (g.TR * g.WP + 127) / 128;
    g.P = tc_plane_pixels(g.MT, K, g.WP);
    g.tiles_x = (W + g.TC - 1) / g.TC;
    g.tiles_y = (H + g.TR - 1) / g.TR;
    g.ntiles = g.tiles_x * g.tiles_y * Nimg;
    g.nk = nk;
    g.a_plane_bytes = (uint32_t)g.P * 16;
    g.a_bytes = 2 * g.a_plane_bytes;
    g.box_bytes = (uint32_t)(4 * g.WP * g.THh * 4);
    g.w_bytes = (uint32_t)((w_bytes + 1023) & ~(size_t)1023);
    g.smem_bytes = g.w_bytes + tc::NSTAGE * g.a_bytes;
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

template <int K, int N>
static cudaError_t launch_tc_n(const ConvArgs &a, cudaStream_t st)
{
    tc::TcGeom g;
    const int groups = (a.Cout + N - 1) / N;
    if (!tc_geometry(K, N, groups, a.Cin, a.H, a.W, a.N, g)) return cudaErrorNotSupported;
    if ((long long)g.tiles_x * g.tiles_y * a.N > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tc_tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    // NHWC activations as a 4-D tensor (C, W, H, N); box = one 4-channel block
    // of the tile's padded pixels
    CUtensorMap tm;
    const cuuint64_t dims[4] = {(cuuint64_t)a.Cin, (cuuint64_t)a.W, (cuuint64_t)a.H, (cuuint64_t)a.N};
    const cuuint64_t strides[3] = {(cuuint64_t)a.Cin * 4, (cuuint64_t)a.W * a.Cin * 4,
                                   (cuuint64_t)a.H * a.W * a.Cin * 4};
    const cuuint32_t box[4] = {4, (cuuint32_t)g.WP, (cuuint32_t)g.THh, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(a.x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int allowed[64] = {0};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (allowed[dev] < (int)g.smem_bytes) {
        e = cudaFuncSetAttribute(conv_tc_kernel<K, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem_bytes);
        if (e != cudaSuccess) return e;
        allowed[dev] = (int)g.smem_bytes;
    }
    const int per_group = (device_sm_count() + groups - 1) / groups;
    const int grid = g.ntiles < per_group ? g.ntiles : per_group;
    conv_tc_kernel<K, N><<<dim3(grid, groups), tc::NTHREADS, g.smem_bytes, st>>>(
        tm, a.w, a.b, a.y, a.N, a.H, a.W, a.Cin, a.Cout, a.R, a.S, a.act, g, device_status_ptr(), 1000000000ull);
    return cudaGetLastError();
}

cudaError_t launch_conv_tc(const ConvArgs &a, cudaStream_t st)
{
    if (a.R > 3 || a.S > 3) return cudaErrorNotSupported;
    // up to 64 output channels per CTA; more run as groups of 64
    const int n16 = (a.Cout + 15) / 16 * 16;
    switch (n16) {
    case 16: return launch_tc_n<3, 16>(a, st);
    case 32: return launch_tc_n<3, 32>(a, st);
    case 48: return launch_tc_n<3, 48>(a, st);
    default: return launch_tc_n<3, 64>(a, st);
    }
}

}  // namespace sc
