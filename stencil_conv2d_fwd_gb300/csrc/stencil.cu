// Fused three-stage stencil pipeline: horizontal 5-tap binomial, vertical
// 5-tap binomial, unsharp mask, clamp-to-edge borders, one kernel.
//
// Method: "Model-Based Warp Overlapped Tiling for Image Processing Programs
// on GPUs" (Abstract): the stages are fused into tiles that fit one warp, so
// the only synchronisation is within the warp, and the overlapped (halo)
// part of the tile lives in thread registers rather than in block-shared
// memory (hybrid tiling).  Here a warp owns a strip 128 columns wide (4
// contiguous pixels per lane, one 16-byte load) and walks down a band of
// rows:
//  * per input row, a lane's 2 + 2 horizontal halo pixels come from its
//    neighbour lanes' registers by shuffle; only lanes 0 and 31 load theirs;
//  * the horizontal pass t1 of the last five rows stays in registers (a
//    5-row ring), as do the matching input rows for the unsharp step;
//  * the vertical pass and the unsharp mask run on the ring, and the output
//    row leaves as one 16-byte store per lane.
// The only recomputation is the 4-row vertical overlap at each band's
// edges.  Nothing but `in` and `out` touches global memory.
// Clamp-to-edge is applied to indices: a lane's pixels beyond the last
// column read in[row][W-1], so neighbour lanes hand out clamped halos for
// free; rows outside [0, H) read row 0 or H-1.
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
    stencil_pipeline_kernel(const float *__restrict__ in, float *__restrict__ out, int H, int W,
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

cudaError_t launch_stencil_pipeline(const float *in, float *out, int H, int W, cudaStream_t st)
{
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
    const int vec = ((W & 3) == 0) && ((reinterpret_cast<uintptr_t>(in) & 15) == 0) &&
                    ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    stencil_pipeline_kernel<<<(unsigned)nb, ST_NWARPS * 32, 0, st>>>(in, out, H, W, rows, col_tiles, vec);
    return cudaGetLastError();
}

}  // namespace sc
