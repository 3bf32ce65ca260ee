// Fused three-stage stencil pipeline: horizontal 5-tap binomial, vertical
// 5-tap binomial, unsharp mask, clamp-to-edge borders, one kernel.
//
// Method: "Model-Based Warp Overlapped Tiling for Image Processing Programs
// on GPUs" (Abstract): the stages are fused into tiles that fit one warp, so
// the only synchronisation is within the warp, and the overlapped (halo)
// part of the tile lives in thread registers rather than in block-shared
// memory (hybrid tiling).  A warp owns a strip 128 columns wide (4
// contiguous pixels per lane) and walks down a band of rows:
//  * the horizontal pass t1 of the last five rows stays in registers (a
//    5-row window), as do the matching input rows for the unsharp step;
//  * the vertical pass and the unsharp mask run on the window, and each
//    output row leaves as one 16-byte store per lane;
//  * the only recomputation is the 4-row vertical overlap at each band's
//    edges; nothing but `in` and `out` touches global memory.
// Clamp-to-edge: a row outside [0, H) is the first or last row, repeated; a
// column outside [0, W) is the first or last column.
//
// Two ways to bring rows in:
//  * stencil_tma_kernel (GB300 path): each warp streams its strip through a
//    ring of 4 shared-memory slots of 5 rows x 136 columns (its 128 columns
//    plus 4 on each side), filled by 2-D TMA copies (cp.async.bulk.tensor)
//    that complete on one mbarrier per slot, so three slots' copies are in
//    flight while the fourth is consumed.  Lanes read their 4 pixels from the
//    slot and the 2 + 2 halo pixels from the neighbour lanes (shuffles).  A
//    slot holds as many rows as the vertical window, so in a band away from
//    the image's top and bottom edges the window's ring index of every row is
//    a compile-time constant of the unrolled slot loop and no register moves.
//    Waits are bounded in time; on expiry the kernel records
//    SC_ERR_DEVICE_TIMEOUT, drains its copies and returns.
//  * stencil_regs_kernel (any size or alignment): each lane loads its 4
//    pixels; the halo pixels come from the neighbour lanes by shuffle.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace sc {

static constexpr int ST_NWARPS = 8;
static constexpr int ST_COLS_PER_WARP = 128;
static constexpr int ST_COLS_PER_CTA = ST_NWARPS * ST_COLS_PER_WARP;

struct Row8 {
    float v[8];  // columns x0-2 .. x0+5 of one input row
};

// Input row `yy` (already clamped to [0, H)) for this lane: own 4 pixels at
// x0..x0+3 (clamped), 2 left and 2 right halo pixels.
__device__ __forceinline__ void st_load_row(Row8 &r, const float *__restrict__ row, int x0, int W,
                                            bool vec, int lane)
{
    float o0, o1, o2, o3;
    if (vec && x0 + 3 < W) {
        const float4 t = ldg_stream(reinterpret_cast<const float4 *>(row + x0));
        o0 = t.x; o1 = t.y; o2 = t.z; o3 = t.w;
    } else {
        const int wm = W - 1;
        o0 = __ldg(row + min(x0 + 0, wm));
        o1 = __ldg(row + min(x0 + 1, wm));
        o2 = __ldg(row + min(x0 + 2, wm));
        o3 = __ldg(row + min(x0 + 3, wm));
    }
    const float l0 = __shfl_up_sync(0xffffffffu, o2, 1);
    const float l1 = __shfl_up_sync(0xffffffffu, o3, 1);
    const float r0 = __shfl_down_sync(0xffffffffu, o0, 1);
    const float r1 = __shfl_down_sync(0xffffffffu, o1, 1);
    r.v[2] = o0; r.v[3] = o1; r.v[4] = o2; r.v[5] = o3;
    r.v[0] = l0; r.v[1] = l1; r.v[6] = r0; r.v[7] = r1;
    if (lane == 0) {
        r.v[0] = __ldg(row + min(max(x0 - 2, 0), W - 1));
        r.v[1] = __ldg(row + min(max(x0 - 1, 0), W - 1));
    }
    if (lane == 31) {
        r.v[6] = __ldg(row + min(x0 + 4, W - 1));
        r.v[7] = __ldg(row + min(x0 + 5, W - 1));
    }
}

// horizontal binomial (1,4,6,4,1)/16 of the 4 own pixels
__device__ __forceinline__ float4 st_hblur(const Row8 &r)
{
    float t[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float s = (r.v[j] + r.v[j + 4]) + 4.0f * (r.v[j + 1] + r.v[j + 3]) + 6.0f * r.v[j + 2];
        t[j] = s * 0.0625f;
    }
    return make_float4(t[0], t[1], t[2], t[3]);
}

__device__ __forceinline__ float st_vblur1(float a, float b, float c, float d, float e)
{
    return ((a + e) + 4.0f * (b + d) + 6.0f * c) * 0.0625f;
}

__device__ __forceinline__ float st_unsharp(float in, float t2)
{
    const float o = in + 1.5f * (in - t2);
    return fminf(fmaxf(o, 0.0f), 1.0f);
}

__global__ void __launch_bounds__(ST_NWARPS * 32)
    stencil_regs_kernel(const float *__restrict__ in, float *__restrict__ out, int H, int W,
                            int rows_per_cta, int col_tiles, int vec)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int ct = blockIdx.x % col_tiles;
    const int rt = blockIdx.x / col_tiles;
    const int x0 = ct * ST_COLS_PER_CTA + warp * ST_COLS_PER_WARP + lane * 4;
    const int y0 = rt * rows_per_cta;
    const int y1 = min(H, y0 + rows_per_cta);
    if (ct * ST_COLS_PER_CTA + warp * ST_COLS_PER_WARP >= W) return;  // whole warp idle

    float4 t1[5];   // ring of horizontal-pass rows, slot = row mod 5 (relative)
    float4 iv[5];   // matching input rows (own pixels)
    // prologue: rows y0-2 .. y0+1 into slots 0..3
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int yy = min(max(y0 - 2 + t, 0), H - 1);
        Row8 r;
        st_load_row(r, in + (long long)yy * W, x0, W, vec, lane);
        t1[t] = st_hblur(r);
        iv[t] = make_float4(r.v[2], r.v[3], r.v[4], r.v[5]);
    }
    // prefetch of the first new row (y0 + 2)
    Row8 nxt;
    st_load_row(nxt, in + (long long)min(y0 + 2, H - 1) * W, x0, W, vec, lane);

    for (int yb = y0; yb < y1; yb += 5) {
#pragma unroll
        for (int u = 0; u < 5; ++u) {
            const int oy = yb + u;
            if (oy >= y1) break;
            // consume the prefetched row oy + 2 into slot (u + 4) % 5, then
            // start the load of row oy + 3
            Row8 cur = nxt;
            if (oy + 1 < y1)
                st_load_row(nxt, in + (long long)min(oy + 3, H - 1) * W, x0, W, vec, lane);
            const int sn = (u + 4) % 5;
            t1[sn] = st_hblur(cur);
            iv[sn] = make_float4(cur.v[2], cur.v[3], cur.v[4], cur.v[5]);
            // output row oy: t1 rows oy-2..oy+2 are slots u..u+4, input row oy is slot u+2
            const float4 a = t1[u % 5], b = t1[(u + 1) % 5], c = t1[(u + 2) % 5],
                         d = t1[(u + 3) % 5], e = t1[(u + 4) % 5];
            const float4 v = iv[(u + 2) % 5];
            float4 o;
            o.x = st_unsharp(v.x, st_vblur1(a.x, b.x, c.x, d.x, e.x));
            o.y = st_unsharp(v.y, st_vblur1(a.y, b.y, c.y, d.y, e.y));
            o.z = st_unsharp(v.z, st_vblur1(a.z, b.z, c.z, d.z, e.z));
            o.w = st_unsharp(v.w, st_vblur1(a.w, b.w, c.w, d.w, e.w));
            float *orow = out + (long long)oy * W;
            if (vec && x0 + 3 < W) {
                stg_stream(reinterpret_cast<float4 *>(orow + x0), o);
            } else {
                if (x0 + 0 < W) orow[x0 + 0] = o.x;
                if (x0 + 1 < W) orow[x0 + 1] = o.y;
                if (x0 + 2 < W) orow[x0 + 2] = o.z;
                if (x0 + 3 < W) orow[x0 + 3] = o.w;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA path
// ---------------------------------------------------------------------------
static constexpr int TS_WARPS = 4;                 // warps per CTA
static constexpr int TS_D = 4;                     // ring slots per warp
static constexpr int TS_RB = 5;                    // rows per slot (TMA box height) = the vertical window
static constexpr int TS_SW = 136;                  // columns per slot row: x0-4 .. x0+131
static constexpr int TS_SLOT = TS_RB * TS_SW;      // floats per slot (one TMA box)
static constexpr unsigned TS_SLOT_BYTES = TS_SLOT * 4;
// slots start 128-byte aligned (a TMA destination): the pitch rounds the box up
static constexpr int TS_SLOT_PITCH = (TS_SLOT * 4 + 127) / 128 * 128 / 4;
static_assert((TS_SLOT_PITCH * 4) % 128 == 0 && TS_SLOT_PITCH >= TS_SLOT, "TMA destinations must be 128-byte aligned");

// Number of times input row yy occurs in the clamped row sequence
// clamp(v, 0, H-1), v = y0-2 .. y1+1, that a band [y0, y1) consumes.
__device__ __forceinline__ int st_row_count(int yy, int y0, int y1, int H)
{
    int a = yy == 0 ? y0 - 2 : yy;
    int b = yy == H - 1 ? y1 + 1 : yy;
    a = max(a, y0 - 2);
    b = min(b, y1 + 1);
    return max(0, b - a + 1);
}

__global__ void __launch_bounds__(TS_WARPS * 32)
    stencil_tma_kernel(const __grid_constant__ CUtensorMap tm, float *__restrict__ out, int H, int W,
                       int band, int nstrips, int *status, unsigned long long timeout_ns, int drop_copy)
{
    __shared__ __align__(128) float ring[TS_WARPS][TS_D][TS_SLOT_PITCH];
    __shared__ __align__(8) unsigned long long bars[TS_WARPS][TS_D];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * TS_WARPS + warp;
    const int strip = gw % nstrips;
    const int y0 = (gw / nstrips) * band;
    if (y0 >= H) return;  // whole warp
    const int y1 = min(H, y0 + band);
    const int xs = strip * ST_COLS_PER_WARP;
    const int ys = max(y0 - 2, 0), ye = min(y1 + 2, H);      // input rows [ys, ye)
    const int nchunks = (ye - ys + TS_RB - 1) / TS_RB;
    float *slots = &ring[warp][0][0];
    const uint32_t bar0 = smem_u32(&bars[warp][0]);

    if (lane == 0) {
#pragma unroll
        for (int d = 0; d < TS_D; ++d) mbar_init(bar0 + 8 * d, 1);
        fence_mbar_init();
    }
    __syncwarp();
    auto issue = [&](int c) {  // lane 0: rows ys + 4c .. ys + 4c + 3 into slot c % D
        const int d = c % TS_D;
        mbar_arrive_expect_tx(bar0 + 8 * d, TS_SLOT_BYTES);
        if (c != drop_copy) tma_load_2d(smem_u32(slots + d * TS_SLOT_PITCH), &tm, xs - 4, ys + c * TS_RB, bar0 + 8 * d);
    };
    if (lane == 0)
        for (int c = 0; c < min(TS_D, nchunks); ++c) issue(c);

    const int x0 = xs + 4 * lane;
    int c = 0;
    bool failed = false;
    if (y0 >= 2 && y1 + 2 <= H) {
        // Interior band (no row is clamped): input row i of the band (image
        // row y0 - 2 + i) is row i % 5 of chunk i / 5, and its horizontal
        // pass goes to ring register t[i % 5]; with 5-row chunks that index
        // is the chunk-row index, a compile-time constant once the chunk is
        // unrolled, so the window never moves.  Output row y0 + i - 4 uses
        // t rows i - 4 .. i and input row i - 2 (iv[(i - 2) % 5]).
        const int nrows = ye - ys;
        float4 t[5], iv[5];
        for (; c < nchunks; ++c) {
            const int d = c % TS_D;
            if (!mbar_wait_bounded(bar0 + 8 * d, (c / TS_D) & 1, timeout_ns)) {
                failed = true;
                break;
            }
            const float *sl = slots + d * TS_SLOT_PITCH;
#pragma unroll
            for (int j = 0; j < TS_RB; ++j) {
                const int i = c * TS_RB + j;
                if (i >= nrows) break;   // the same for the whole warp
                const float *rp = sl + j * TS_SW;
                const float4 own = *reinterpret_cast<const float4 *>(rp + 4 + 4 * lane);
                // halo pixels from the neighbour lanes; the strip's outer two
                // on each side from the slot; clamp at the image's edges
                float l0 = __shfl_up_sync(0xffffffffu, own.z, 1), l1 = __shfl_up_sync(0xffffffffu, own.w, 1);
                float r0 = __shfl_down_sync(0xffffffffu, own.x, 1), r1 = __shfl_down_sync(0xffffffffu, own.y, 1);
                if (lane == 0) {
                    const float2 h = *reinterpret_cast<const float2 *>(rp + 2);
                    l0 = h.x;
                    l1 = h.y;
                }
                if (lane == 31) {
                    const float2 h = *reinterpret_cast<const float2 *>(rp + 4 + 4 * 32);
                    r0 = h.x;
                    r1 = h.y;
                }
                if (x0 == 0) l0 = l1 = own.x;             // columns -2, -1
                if (x0 + 4 >= W) r0 = r1 = own.w;          // columns W, W + 1 (W % 4 == 0)
                Row8 r;
                r.v[0] = l0; r.v[1] = l1; r.v[2] = own.x; r.v[3] = own.y;
                r.v[4] = own.z; r.v[5] = own.w; r.v[6] = r0; r.v[7] = r1;
                t[j] = st_hblur(r);
                iv[j] = own;
                if (i >= 4) {
                    const float4 &a = t[(j + 1) % 5], &b = t[(j + 2) % 5], &cc = t[(j + 3) % 5], &dd = t[(j + 4) % 5],
                                 &e = t[j], &v = iv[(j + 3) % 5];
                    float4 o;
                    o.x = st_unsharp(v.x, st_vblur1(a.x, b.x, cc.x, dd.x, e.x));
                    o.y = st_unsharp(v.y, st_vblur1(a.y, b.y, cc.y, dd.y, e.y));
                    o.z = st_unsharp(v.z, st_vblur1(a.z, b.z, cc.z, dd.z, e.z));
                    o.w = st_unsharp(v.w, st_vblur1(a.w, b.w, cc.w, dd.w, e.w));
                    if (x0 < W) stg_stream(reinterpret_cast<float4 *>(out + (long long)(y0 + i - 4) * W + x0), o);
                }
            }
            // every lane is done reading slot d (its values fed the FMAs above)
            __syncwarp();
            if (lane == 0 && c + TS_D < nchunks) {
                fence_proxy_async_smem();
                issue(c + TS_D);
            }
        }
    } else {
        // A band at the top or bottom edge: clamped rows repeat, so each
        // loaded row is consumed st_row_count times and the window shifts.
        float4 t[5], iv[3];
        int nv = 0;
        for (; c < nchunks; ++c) {
            const int d = c % TS_D;
            if (!mbar_wait_bounded(bar0 + 8 * d, (c / TS_D) & 1, timeout_ns)) {
                failed = true;
                break;
            }
            const float *sl = slots + d * TS_SLOT_PITCH;
            for (int j = 0; j < TS_RB; ++j) {
                const int yy = ys + c * TS_RB + j;
                if (yy >= ye) break;
                const float *rp = sl + j * TS_SW;
                const float4 own = *reinterpret_cast<const float4 *>(rp + 4 + 4 * lane);
                // halo pixels as in the interior bands: from the neighbour
                // lanes, the strip's outer two on each side from the slot
                float2 lh = make_float2(__shfl_up_sync(0xffffffffu, own.z, 1), __shfl_up_sync(0xffffffffu, own.w, 1));
                float2 rh = make_float2(__shfl_down_sync(0xffffffffu, own.x, 1), __shfl_down_sync(0xffffffffu, own.y, 1));
                if (lane == 0) lh = *reinterpret_cast<const float2 *>(rp + 2);
                if (lane == 31) rh = *reinterpret_cast<const float2 *>(rp + 4 + 4 * 32);
                if (x0 == 0) lh = make_float2(own.x, own.x);          // columns -2, -1
                if (x0 + 4 >= W) rh = make_float2(own.w, own.w);      // columns W, W+1 (W % 4 == 0)
                Row8 r;
                r.v[0] = lh.x; r.v[1] = lh.y; r.v[2] = own.x; r.v[3] = own.y;
                r.v[4] = own.z; r.v[5] = own.w; r.v[6] = rh.x; r.v[7] = rh.y;
                const float4 t1 = st_hblur(r);
                for (int k = st_row_count(yy, y0, y1, H); k > 0; --k) {
                    t[0] = t[1]; t[1] = t[2]; t[2] = t[3]; t[3] = t[4]; t[4] = t1;
                    iv[0] = iv[1]; iv[1] = iv[2]; iv[2] = own;
                    if (++nv >= 5) {
                        const int oy = y0 + nv - 5;
                        float4 o;
                        o.x = st_unsharp(iv[0].x, st_vblur1(t[0].x, t[1].x, t[2].x, t[3].x, t[4].x));
                        o.y = st_unsharp(iv[0].y, st_vblur1(t[0].y, t[1].y, t[2].y, t[3].y, t[4].y));
                        o.z = st_unsharp(iv[0].z, st_vblur1(t[0].z, t[1].z, t[2].z, t[3].z, t[4].z));
                        o.w = st_unsharp(iv[0].w, st_vblur1(t[0].w, t[1].w, t[2].w, t[3].w, t[4].w));
                        if (x0 < W) stg_stream(reinterpret_cast<float4 *>(out + (long long)oy * W + x0), o);
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && c + TS_D < nchunks) {
                fence_proxy_async_smem();
                issue(c + TS_D);
            }
        }
    }
    if (failed) {
        if (lane == 0) atomicExch(status, kDeviceTimeout);
        // let this warp's copies still in flight land before the CTA exits
        const int last = min(nchunks, c + TS_D);
        for (int k = c; k < last; ++k)
            (void)mbar_wait_bounded(bar0 + 8 * (k % TS_D), (k / TS_D) & 1, timeout_ns);
    }
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
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

cudaError_t launch_stencil_pipeline(const float *in, float *out, int H, int W, cudaStream_t st,
                                    int drop_copy, unsigned long long timeout_ns)
{
    const bool aligned = ((reinterpret_cast<uintptr_t>(in) & 15) == 0) &&
                         ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    int *status = device_status_ptr();
    if (aligned && (W % 4) == 0 && W >= TS_SW && H >= TS_RB && encode && status) {
        CUtensorMap tm;
        const cuuint64_t dims[2] = {(cuuint64_t)W, (cuuint64_t)H};
        const cuuint64_t strides[1] = {(cuuint64_t)W * sizeof(float)};
        const cuuint32_t box[2] = {TS_SW, TS_RB};
        const cuuint32_t estr[2] = {1, 1};
        CUresult r = encode(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(in), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r == CUDA_SUCCESS) {
            const int nstrips = (W + ST_COLS_PER_WARP - 1) / ST_COLS_PER_WARP;
            // about 16 warps per SM in one wave, bands of at least 16 rows
            const long long want = 16LL * device_sm_count();
            long long bands = (want + nstrips - 1) / nstrips;
            const long long max_bands = (H + 15) / 16;
            if (bands > max_bands) bands = max_bands;
            if (bands < 1) bands = 1;
            const int band = (int)((H + bands - 1) / bands);
            const long long warps = (long long)nstrips * ((H + band - 1) / band);
            const long long ctas = (warps + TS_WARPS - 1) / TS_WARPS;
            if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
            stencil_tma_kernel<<<(unsigned)ctas, TS_WARPS * 32, 0, st>>>(tm, out, H, W, band, nstrips, status,
                                                                         timeout_ns, drop_copy);
            return cudaGetLastError();
        }
    }
    if (drop_copy >= 0) return cudaErrorNotSupported;  // the test hook needs the TMA path
    const int col_tiles = (W + ST_COLS_PER_CTA - 1) / ST_COLS_PER_CTA;
    // Bands of rows: enough CTAs to keep every SM busy with several, but
    // tall enough that the 4 halo rows per band stay a small overhead.
    const long long want = 8LL * device_sm_count();
    long long bands = (want + col_tiles - 1) / col_tiles;
    const long long max_bands = (H + 31) / 32;
    if (bands > max_bands) bands = max_bands;
    if (bands < 1) bands = 1;
    const int rows = (int)((H + bands - 1) / bands);
    const long long nb = (long long)col_tiles * ((H + rows - 1) / rows);
    if (nb > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int vec = ((W & 3) == 0) && aligned;
    stencil_regs_kernel<<<(unsigned)nb, ST_NWARPS * 32, 0, st>>>(in, out, H, W, rows, col_tiles, vec);
    return cudaGetLastError();
}

}  // namespace sc
