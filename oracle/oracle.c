/*
 * Oracle for the direct 2-D convolution forward pass and the fused
 * blur/unsharp stencil pipeline.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU definition that the CUDA path is checked against.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * Precision: inputs are the same float32 values the GPU sees; every product
 * and sum is formed in double (fp64), in the loop order of the definition.
 *
 * Parity status of each function (what pins it) is stated in its comment and
 * checked by tests/test_oracle_*.py.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of OpenMP threads the oracle uses (<= 0 leaves the default).
 * Returns the count that parallel regions will use. */
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Value of channel plane `plane` (H x W, row-major) at (yy, xx), with zero
 * outside the image: the zero "same" padding of the convolution. */
static double px_zero(const float *plane, long H, long W, long yy, long xx)
{
    if (yy < 0 || yy >= H || xx < 0 || xx >= W) return 0.0;
    return (double)plane[yy * W + xx];
}

/*
 * One output element of the convolution, NCHW activations, OIHW weights.
 *
 * Follows "Optimizing convolution kernels - CNNs in Vulkan Part 2/3",
 * section "Where we left off" (the naive four-loop kernel): for output
 * channel co, sum over input channel ci, kernel row ky, kernel column kx of
 *   input[x + kx - S/2, y + ky - R/2, ci] * weight[co][ci][ky][kx]
 * (weights consumed in co, ci, ky, kx order; no kernel flip, i.e. the CNN
 * cross-correlation), then add the bias after the sum.  Section
 * "Vectorization" applies ReLU to that result when the layer asks for it.
 * Taps outside the image read zero (zero "same" padding, pad = R/2, S/2).
 *
 * Also returns scale = sum |input * weight| + |bias|, the per-element scale
 * of the fp32 error bound.
 */
static void conv_point(const float *x, const float *w, const float *b,
                       long Cin, long H, long W, long R, long S, int act,
                       long n, long co, long h, long xw, double *out, double *scale)
{
    double sum = 0.0, asum = 0.0;
    for (long ci = 0; ci < Cin; ++ci) {
        const float *plane = x + ((n * Cin + ci) * H) * W;
        const float *wk = w + ((co * Cin + ci) * R) * S;
        for (long ky = 0; ky < R; ++ky) {
            for (long kx = 0; kx < S; ++kx) {
                double v = px_zero(plane, H, W, h + ky - R / 2, xw + kx - S / 2);
                double t = v * (double)wk[ky * S + kx];
                sum += t;
                asum += fabs(t);
            }
        }
    }
    double bias = b ? (double)b[co] : 0.0;
    double r = sum + bias;
    if (act == 1 && r < 0.0) r = 0.0;
    *out = r;
    *scale = asum + fabs(bias);
}

/*
 * Rows [h0, h1) of y = act(conv(x, w) + b), NCHW in, NCHW out:
 *   y[n][co][h - h0][w], scale likewise (scale may be NULL).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_conv2d_nchw(const float *x, const float *w, const float *b,
                       int N, int Cin, int H, int W, int Cout, int R, int S, int act,
                       int h0, int h1, double *y, double *scale)
{
    if (!x || !w || !y || N < 1 || Cin < 1 || H < 1 || W < 1 || Cout < 1 || R < 1 || S < 1)
        return -1;
    if (h0 < 0 || h1 > H || h0 > h1) return -1;
    long band = (long)h1 - h0;
#pragma omp parallel for collapse(3) schedule(static)
    for (long n = 0; n < N; ++n)
        for (long co = 0; co < Cout; ++co)
            for (long h = h0; h < h1; ++h)
                for (long xw = 0; xw < W; ++xw) {
                    double o, a;
                    conv_point(x, w, b, Cin, H, W, R, S, act, n, co, h, xw, &o, &a);
                    long idx = ((n * Cout + co) * band + (h - h0)) * W + xw;
                    y[idx] = o;
                    if (scale) scale[idx] = a;
                }
    return 0;
}

/*
 * The same definition at `npts` sampled output coordinates; pts holds
 * (n, co, h, w) quadruples.  Used for parity at sizes where computing every
 * output would take too long on the host.
 */
int oracle_conv2d_points(const float *x, const float *w, const float *b,
                         int N, int Cin, int H, int W, int Cout, int R, int S, int act,
                         long npts, const int32_t *pts, double *y, double *scale)
{
    if (!x || !w || !pts || !y || npts < 0) return -1;
#pragma omp parallel for schedule(static)
    for (long i = 0; i < npts; ++i) {
        long n = pts[4 * i], co = pts[4 * i + 1], h = pts[4 * i + 2], xw = pts[4 * i + 3];
        double o = NAN, a = NAN;
        if (n >= 0 && n < N && co >= 0 && co < Cout && h >= 0 && h < H && xw >= 0 && xw < W)
            conv_point(x, w, b, Cin, H, W, R, S, act, n, co, h, xw, &o, &a);
        y[i] = o;
        if (scale) scale[i] = a;
    }
    return 0;
}

/*
 * Layout change between planar NCHW and channel-interleaved NHWC, by the
 * index definition of the two layouts ("Optimizing convolution kernels -
 * CNNs in Vulkan Part 2/3", section "Vectorization": several channels of one
 * pixel stored next to each other).  to_nhwc != 0: src NCHW -> dst NHWC;
 * otherwise src NHWC -> dst NCHW.  Values are copied, not rounded.
 */
int oracle_repack(const float *src, float *dst, int N, int C, int H, int W, int to_nhwc)
{
    if (!src || !dst || N < 1 || C < 1 || H < 1 || W < 1) return -1;
    for (long n = 0; n < N; ++n)
        for (long c = 0; c < C; ++c)
            for (long h = 0; h < H; ++h)
                for (long xw = 0; xw < W; ++xw) {
                    long nchw = ((n * C + c) * H + h) * W + xw;
                    long nhwc = ((n * H + h) * W + xw) * C + c;
                    if (to_nhwc) dst[nhwc] = src[nchw];
                    else dst[nchw] = src[nhwc];
                }
    return 0;
}

/* ------------------------------------------------------------------------
 * Fused image pipeline: horizontal 5-tap binomial, vertical 5-tap binomial,
 * unsharp mask.  The pipeline is the workload the warp-overlapped tiling of
 * "Model-Based Warp Overlapped Tiling for Image Processing Programs on GPUs"
 * (Abstract) fuses: a chain of stencil stages over one image.  The stages:
 *   t1[y][x] = sum_{k=-2..2} c_k * in[y][clamp(x+k, 0, W-1)]
 *   t2[y][x] = sum_{k=-2..2} c_k * t1[clamp(y+k, 0, H-1)][x]
 *   out      = min(max(in + 1.5 * (in - t2), 0), 1)
 * with c = (1, 4, 6, 4, 1) / 16 and clamp-to-edge at the borders.
 * ------------------------------------------------------------------------ */
static long clampl(long v, long lo, long hi) { return v < lo ? lo : (v > hi ? hi : v); }

static const double BINOM5[5] = {1.0 / 16, 4.0 / 16, 6.0 / 16, 4.0 / 16, 1.0 / 16};

static double stage_hblur(const float *in, long H, long W, long y, long xw)
{
    (void)H;
    double s = 0.0;
    for (long k = -2; k <= 2; ++k) s += BINOM5[k + 2] * (double)in[y * W + clampl(xw + k, 0, W - 1)];
    return s;
}

static double stage_vblur_of_hblur(const float *in, long H, long W, long y, long xw)
{
    double s = 0.0;
    for (long k = -2; k <= 2; ++k) s += BINOM5[k + 2] * stage_hblur(in, H, W, clampl(y + k, 0, H - 1), xw);
    return s;
}

/* Rows [r0, r1) of the pipeline output, out[(y - r0) * W + x]; also the
 * intermediate t2 when t2_out is not NULL. */
int oracle_stencil_pipeline(const float *in, int H, int W, int r0, int r1,
                            double *out, double *t2_out)
{
    if (!in || !out || H < 1 || W < 1 || r0 < 0 || r1 > H || r0 > r1) return -1;
#pragma omp parallel for schedule(static)
    for (long y = r0; y < r1; ++y)
        for (long xw = 0; xw < W; ++xw) {
            double t2 = stage_vblur_of_hblur(in, H, W, y, xw);
            double v = (double)in[y * W + xw];
            double o = v + 1.5 * (v - t2);
            if (o < 0.0) o = 0.0;
            if (o > 1.0) o = 1.0;
            long idx = (y - r0) * (long)W + xw;
            out[idx] = o;
            if (t2_out) t2_out[idx] = t2;
        }
    return 0;
}
