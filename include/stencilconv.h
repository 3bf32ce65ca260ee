/*
 * stencilconv: direct 2-D convolution forward pass and a fused
 * blur/unsharp stencil pipeline on NVIDIA GB300 (sm_103a).
 *
 * C ABI of libstencilconv.so.  Plain pointers and sizes only.
 *
 * Common conventions
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the
 *    library never frees or keeps it past the call's stream work.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *    and return once the work is enqueued.  A nonzero return means nothing
 *    was enqueued (argument errors) or a launch failed (SC_ERR_CUDA).
 *  - Arguments are validated on the host before any launch; there is no CPU
 *    fallback.
 *  - All data is fp32.  Sizes are ints; element offsets are computed in
 *    64-bit, so tensors may exceed 2^31 elements as long as each size fits.
 */
#ifndef STENCILCONV_H
#define STENCILCONV_H

#ifdef __cplusplus
extern "C" {
#endif

/* The library is built with hidden symbol visibility: only the functions
 * declared here are exported, so two copies of the library (or another
 * library with the same internal names) can be loaded in one process. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

struct CUstream_st;                     /* = cudaStream_t's target type */
typedef struct CUstream_st *sc_stream_t;

typedef enum {
    SC_OK = 0,
    SC_ERR_NULL = -1,            /* a required pointer is NULL */
    SC_ERR_SHAPE = -2,           /* a size is < 1, or the sizes overflow */
    SC_ERR_UNSUPPORTED = -3,     /* valid convolution the library does not run */
    SC_ERR_ALIGN = -4,           /* a pointer is not 16-byte aligned */
    SC_ERR_ALIAS = -5,           /* output overlaps an input */
    SC_ERR_CUDA = -6,            /* a CUDA call failed; see sc_last_cuda_error */
    SC_ERR_DEVICE_TIMEOUT = -7   /* a device-side bounded wait gave up */
} sc_status;

typedef enum { SC_NCHW = 0, SC_NHWC = 1 } sc_layout;
typedef enum { SC_ACT_NONE = 0, SC_ACT_RELU = 1 } sc_act;
typedef enum { SC_F32 = 0, SC_BF16 = 1 } sc_dtype;   /* element type of an activation tensor */

/*
 * conv2d_fwd: y = act(conv(x, w) + b), stride 1, zero "same" padding.
 *
 * Operation ("Optimizing convolution kernels - CNNs in Vulkan Part 2/3",
 * section "Where we left off"; "Optimizing Memory Efficiency for
 * Convolution Kernels on Kepler GPUs", Section 3):
 *   y[n][h][w][co] = act( b[co] + sum_{ci<Cin} sum_{r<R} sum_{s<S}
 *                          X(n, h + r - R/2, w + s - S/2, ci) * w[co][ci][r][s] )
 * where X is x inside the image and 0 outside.  This is cross-correlation
 * (weights are not flipped).  act = ReLU is max(v, 0).
 *
 * x : N*H*W*Cin floats, layout `layout` (SC_NHWC: [N][H][W][Cin];
 *     SC_NCHW: [N][Cin][H][W]).
 * w : Cout*Cin*R*S floats, always [Cout][Cin][R][S] (OIHW), row-major.
 * b : Cout floats, or NULL for no bias.
 * y : N*H*W*Cout floats, same layout as x.  Must not overlap x, w or b.
 * R, S : odd, 1..7.
 * Supported: Cin == 1 with Cout == 1 or Cout % 4 == 0; Cin % 4 == 0 with
 *   Cout % 4 == 0.  x and y 16-byte aligned for Cin > 1 (NHWC vectors of 4
 *   channels).  Anything else returns SC_ERR_UNSUPPORTED / SC_ERR_ALIGN.
 * SC_NCHW with more than one channel on either side goes through the
 *   repack kernels and a stream-ordered temporary buffer (allocated on
 *   `stream` from the library's memory pool, freed on `stream` after use;
 *   see sc_release_workspace).
 * Returns SC_OK or a negative sc_status.
 */
int conv2d_fwd(const float *x, const float *w, const float *b, float *y,
               int N, int H, int W, int Cin, int Cout, int R, int S,
               int layout, int act, sc_stream_t stream);

/*
 * One layer of a convolution chain (conv2d_chain_fwd_host): filters w
 * (device memory, [Cout][Cin][R][S] fp32 with Cin the previous layer's
 * output channels), bias b (device memory, Cout floats, or NULL), the
 * filter size R x S and the activation (SC_ACT_NONE or SC_ACT_RELU).
 */
typedef struct {
    const float *w;
    const float *b;
    int Cout, R, S, act;
} sc_conv_layer;

#define SC_CHAIN_MAX_LAYERS 64

/*
 * conv2d_chain_fwd_host: a chain of convolution layers run on an input in
 * host memory, the result returned to host memory, as a network like the
 * upscaling network of "Optimizing convolution kernels - CNNs in Vulkan
 * Part 2/3" (opening paragraphs and "Where we left off": one image through
 * its layers in turn, each layer's output the next one's input):
 *   a_0 = x,  a_l = act_l(conv(a_{l-1}, w_l) + b_l) for l = 1..n_layers,
 *   y = a_{n_layers},
 * each conv exactly conv2d_fwd's (stride 1, zero "same" padding, NHWC).
 * On `stream`, in order: x_host is copied to the device, the layers run
 * with their activations in stream-ordered device buffers from the
 * library's memory pool (freed on `stream` after use; see
 * sc_release_workspace), and the last layer's output is copied to y_host.
 * The call returns once this is enqueued: x_host must stay unchanged and
 * y_host unread until the stream has completed it.  With page-locked
 * (pinned) host buffers both copies are asynchronous DMA transfers; with
 * pageable ones the CUDA runtime stages them and the call may wait for
 * the copies.
 * x_host : N*H*W*Cin floats, NHWC.  y_host : N*H*W*Cout floats of the last
 *   layer, NHWC.  layers : n_layers entries, 1 <= n_layers <=
 *   SC_CHAIN_MAX_LAYERS.
 * Every layer's shape is checked (conv2d_fwd's rules, with its Cin the
 * previous layer's Cout) before anything is enqueued: SC_ERR_NULL for a
 * NULL x_host, y_host, layers or w, SC_ERR_SHAPE / SC_ERR_UNSUPPORTED as
 * conv2d_fwd, SC_ERR_SHAPE for n_layers out of range.  A failed CUDA call
 * returns SC_ERR_CUDA (code in sc_last_cuda_error).
 */
int conv2d_chain_fwd_host(const float *x_host, float *y_host, int N, int H, int W, int Cin,
                          int n_layers, const sc_conv_layer *layers, sc_stream_t stream);

/*
 * conv2d_fwd_tc: the same operation as conv2d_fwd on the tensor cores
 * (tcgen05 MMA, accumulators in tensor memory) as an implicit GEMM
 * (pixels x output channels x (taps, input channels); "Optimizing Memory
 * Efficiency for Convolution Kernels on Kepler GPUs", Section 3.3, sets
 * this GEMM formulation against direct convolution).  x and w enter the
 * MMA as TF32 (10 explicit mantissa bits; the MMA drops the 13 low bits of
 * an fp32 operand, a relative error below 2^-10 per operand), products
 * accumulate in fp32, so results differ from conv2d_fwd by up to about
 * 5e-3 * sum|x * w| per element: a separate variant with its own
 * tolerance, not a replacement.
 * x, y : NHWC, 16-byte aligned.  w : OIHW, 16-byte aligned.  b : Cout
 *   floats or NULL.
 * Supported: Cin % 4 == 0, Cout % 4 == 0, Cout <= 128, R and S odd and <= 3,
 *   and filters small enough to stay resident in shared memory: each CTA
 *   holds the filters of a group of up to 32 output channels (and, while it
 *   starts, a second copy in OIHW order), so the group shrinks to 16, 8 or
 *   4 channels as Cin grows; beyond Cin of about 500, SC_ERR_UNSUPPORTED.
 * Returns SC_OK or a negative sc_status (SC_ERR_UNSUPPORTED outside that,
 *   SC_ERR_ALIGN for unaligned pointers).
 */
int conv2d_fwd_tc(const float *x, const float *w, const float *b, float *y,
                  int N, int H, int W, int Cin, int Cout, int R, int S,
                  int act, sc_stream_t stream);

/*
 * conv2d_fwd_tc_x3: conv2d_fwd_tc with fp32-level accuracy: every operand v
 * is split into a TF32 head hi(v) (v with its 13 low mantissa bits cleared)
 * and a remainder lo(v) = v - hi(v), and each product x * w is computed on
 * the tensor cores as hi(x) hi(w) + hi(x) lo(w) + lo(x) hi(w), the last two
 * in a separate accumulator added once at the end (split or "3xTF32"
 * arithmetic: Ootomo and Yokota, "Recovering single precision accuracy from
 * Tensor Cores while surpassing the FP32 theoretical peak performance",
 * 2022).  The dropped lo(x) lo(w) and the remainders' own TF32 truncation
 * keep every product within about 3 * 2^-20 of exact, so the result meets
 * conv2d_fwd's bound |y - y_ref| <= 1e-5 * (sum|x * w| + |b|).  Three TF32
 * products per product (issued as two MMAs, the filters' heads and
 * remainders side by side in N): a separate variant, not conv2d_fwd's FP32
 * FMA path.
 * Arguments, layouts and errors as for conv2d_fwd_tc.  Both the filters'
 * heads and remainders stay resident in shared memory, so the supported
 * Cin is about half of conv2d_fwd_tc's (about 250).
 */
int conv2d_fwd_tc_x3(const float *x, const float *w, const float *b, float *y,
                     int N, int H, int W, int Cin, int Cout, int R, int S,
                     int act, sc_stream_t stream);

/*
 * conv2d_fwd_tc_bf16: conv2d_fwd_tc with bf16 activation storage and BF16
 * tensor-core operands (tcgen05 kind::f16), fp32 accumulation.  Storing
 * activations in 16-bit floats halves their bytes ("Optimizing convolution
 * kernels - CNNs in Vulkan Part 2/3", the fp16 storage section: the traffic
 * halves at a small loss of precision).  x is bf16, the filters are fp32 and
 * rounded to bf16 (to nearest even) inside, b is fp32, y is bf16 (rounded to
 * nearest even) or fp32.  With x exact in bf16 (8 significant bits, unit
 * roundoff 2^-8), |y - y_ref| <= 2^-8 * sum|x*w| (weight rounding) + fp32
 * accumulation error, within 5e-3 * (sum |x * w| + |b|); a bf16 y adds its
 * own rounding, at most 2^-8 * |y_ref|.
 * x : N*H*W*Cin bf16 (NHWC), 16-byte aligned.  y : N*H*W*Cout elements of
 *   y_dtype (SC_F32 or SC_BF16), NHWC, 16-byte aligned.  w : OIHW fp32,
 *   16-byte aligned.  b : Cout floats or NULL.
 * Supported: Cin % 8 == 0, Cout % 4 == 0, Cout <= 128 (bf16 y with
 *   Cout > 16: Cout % 8 == 0), R and S odd and <= 3, filters that fit in
 *   shared memory as for conv2d_fwd_tc.
 * Returns SC_OK or a negative sc_status.
 */
int conv2d_fwd_tc_bf16(const void *x, const float *w, const float *b, void *y,
                       int N, int H, int W, int Cin, int Cout, int R, int S,
                       int act, int y_dtype, sc_stream_t stream);

/*
 * conv2d_fwd_tc_fused2: two 3 x 3 convolution layers in one pass on the
 * tensor cores, the intermediate activation kept on chip ("Optimizing
 * convolution kernels - CNNs in Vulkan Part 2/3", "Reducing memory traffic";
 * "Model-Based Warp Overlapped Tiling for Image Processing Programs on GPUs",
 * Abstract: overlapped tiles recompute the producer's halo):
 *   t = act1(conv(x, w1) + b1),  y = act2(conv(t, w2) + b2),
 * both "same"-padded with zeros (t is zero outside the image), TF32 operands,
 * fp32 accumulation.  Tolerance: layer 2 of the exact t within
 * 5e-3 * sum|t * w2|, plus layer 1's error (5e-3 * sum|x * w1| per element of
 * t) carried through |w2|.
 * x : N*H*W*C0 NHWC fp32.  w1 : C1*C0*3*3 OIHW.  b1 : C1 floats or NULL.
 * w2 : C2*C1*3*3 OIHW.  b2 : C2 floats or NULL.  y : N*H*W*C2 NHWC fp32.
 * x, y, w1, w2 16-byte aligned.
 * Supported: C0 % 4 == 0 with C0 <= 32 or so (its filters resident in
 *   shared memory beside two input stages), C1 == 32, C2 in {4, 8}.
 * Returns SC_OK or a negative sc_status.
 */
int conv2d_fwd_tc_fused2(const float *x, const float *w1, const float *b1,
                         const float *w2, const float *b2, float *y,
                         int N, int H, int W, int C0, int C1, int C2,
                         int act1, int act2, sc_stream_t stream);

/*
 * stencil_pipeline_fwd: three stencil stages fused in one pass over a
 * single-channel image ("Model-Based Warp Overlapped Tiling for Image
 * Processing Programs on GPUs", Abstract: stages fused into overlapped
 * warp-sized tiles):
 *   t1[y][x] = sum_{k=-2..2} c_k in[y][clamp(x+k, 0, W-1)]
 *   t2[y][x] = sum_{k=-2..2} c_k t1[clamp(y+k, 0, H-1)][x]
 *   out      = min(max(in + 1.5 (in - t2), 0), 1),   c = (1,4,6,4,1)/16.
 * in, out : H*W floats, row-major with pitch W; must not overlap.
 * The intermediates t1 and t2 never leave the chip.
 * Returns SC_OK or a negative sc_status.
 */
int stencil_pipeline_fwd(const float *in, float *out, int H, int W, sc_stream_t stream);

/*
 * sc_repack: change activation layout between NCHW and NHWC
 * ("Optimizing convolution kernels - CNNs in Vulkan Part 2/3", section
 * "Vectorization": the channels of one pixel stored next to each other so
 * a thread moves four of them as one 16-byte vector).
 * src, dst : N*C*H*W floats, device, non-overlapping.
 * src_layout, dst_layout : SC_NCHW or SC_NHWC; equal layouts copy.
 * Returns SC_OK or a negative sc_status.
 */
int sc_repack(const float *src, float *dst, int N, int C, int H, int W,
              int src_layout, int dst_layout, sc_stream_t stream);

/*
 * sc_last_device_status: synchronize `stream`, then return and clear the
 * device-side status word of the current device (SC_OK, or
 * SC_ERR_DEVICE_TIMEOUT when a kernel's bounded wait expired).  Returns
 * SC_ERR_CUDA if the synchronization itself failed.
 */
int sc_last_device_status(sc_stream_t stream);

/* sc_status_string: static English text for a status code (never NULL). */
const char *sc_status_string(int status);

/* sc_last_cuda_error: the cudaError_t value behind the last SC_ERR_CUDA
 * returned on this host thread (0 if none). */
int sc_last_cuda_error(void);

/*
 * sc_measure_ffma_peak: measurement helper, not part of the operation.
 * Runs `blocks` CTAs of 256 threads, each thread doing `iters` iterations
 * of 16 independent fp32 FMA chains (32 FLOP per chain step), and writes
 * one float per thread to `sink` (device, blocks*256 floats) so nothing is
 * optimised away.  Time it on `stream` to measure the FP32 FFMA rate.
 * Returns SC_OK or a negative sc_status.
 */
int sc_measure_ffma_peak(float *sink, int blocks, int iters, sc_stream_t stream);

/*
 * sc_empty_kernel: measurement helper, not part of the operation.  Launches
 * a kernel of `blocks` CTAs of `threads` threads that does nothing, on
 * `stream`; a run of such launches (e.g. replayed from a CUDA graph) gives
 * the cost of one launch, the floor under any kernel of the library.
 * Returns SC_OK, SC_ERR_SHAPE for blocks outside [1, 2^24] or threads
 * outside [1, 1024], or SC_ERR_CUDA.
 */
int sc_empty_kernel(int blocks, int threads, sc_stream_t stream);

/* sc_version: library version as 10000*major + 100*minor + patch. */
int sc_version(void);

/*
 * sc_release_workspace: hand the memory of the library's temporary buffers
 * back to the driver.  Those buffers (the NCHW repack of conv2d_fwd) come
 * from a library-private
 * stream-ordered memory pool per device that otherwise keeps freed memory
 * for the next call.  Memory still in use by queued work is not affected.
 * Returns SC_OK.
 */
int sc_release_workspace(void);

/*
 * sc_set_autotune: first-call autotuning of conv2d_fwd's tile configuration
 * ("Optimizing Memory Efficiency for Convolution Kernels on Kepler GPUs",
 * Table 1: the best configuration differs per filter size and is found by
 * measurement).  With enable != 0, the first conv2d_fwd (NHWC or NCHW, or
 * conv2d_fwd_nchw_noalloc) of each shape with 3 x 3 filters and Cin > 1
 * times every candidate configuration of its output-channel class on the
 * caller's stream and data, which synchronises that stream once; the
 * fastest is cached per device and shape (N, H, W, Cin, Cout, R, S, act,
 * bias present) and used by later calls.  While the stream is being captured
 * into a CUDA graph no timing happens (the default configuration runs and
 * nothing is cached).  Off by default.  Returns the previous setting.
 */
int sc_set_autotune(int enable);

/* sc_autotune_lookup: the cached candidate index (0 = the default
 * configuration) for a shape on the current device, or -1 if not tuned. */
int sc_autotune_lookup(int N, int H, int W, int Cin, int Cout, int R, int S, int act, int has_bias);

/* sc_autotune_clear: forget every cached choice. */
void sc_autotune_clear(void);

/* sc_autotune_candidates: number of candidate configurations for a filter
 * shape (0 if not tuned); if names != NULL, their names, one per line, into
 * names[0 .. names_len-1] (NUL-terminated, truncated to fit). */
int sc_autotune_candidates(int Cin, int Cout, int R, int S, char *names, int names_len);

/*
 * sc_test_conv_candidate: test hook, not part of the operation.  Runs
 * conv2d_fwd (NHWC, 3 x 3) with candidate configuration `candidate` of
 * sc_autotune_candidates; SC_ERR_UNSUPPORTED if it does not exist or does
 * not apply to the shape.
 */
int sc_test_conv_candidate(const float *x, const float *w, const float *b, float *y,
                           int N, int H, int W, int Cin, int Cout, int R, int S,
                           int act, int candidate, sc_stream_t stream);

/*
 * sc_test_conv_wait_expiry: test hook for the device-status path, not part
 * of the operation.  Runs conv2d_fwd's TMA-staged kernel (NHWC, 3 x 3, no
 * activation, the default tile configuration for Cout) with copy
 * `drop_copy` (0-based, in each CTA's issue order) never issued, so the
 * time-bounded waits for it expire after `timeout_us` microseconds (a
 * CTA's consumers on the stage, then its producer on the stage's release).
 * The kernel then records SC_ERR_DEVICE_TIMEOUT (read and cleared by
 * sc_last_device_status), lets its other copies land and returns; the
 * context stays usable.  `y` is left partly written.  Cin % 4 == 0,
 * Cout % 4 == 0, 16-byte aligned x and y; SC_ERR_UNSUPPORTED where the
 * TMA kernel does not apply (a filter bank above its shared-memory limit).
 */
int sc_test_conv_wait_expiry(const float *x, const float *w, const float *b, float *y,
                             int N, int H, int W, int Cin, int Cout, int drop_copy, int timeout_us,
                             sc_stream_t stream);

/*
 * sc_test_stencil_wait_expiry: test hook for the device-status path, not
 * part of the operation.  Runs stencil_pipeline_fwd's TMA kernel with the
 * copy of row chunk `drop_copy` (0-based, per warp) never issued, so each
 * warp's time-bounded wait for it expires after `timeout_us` microseconds.
 * The kernel then records SC_ERR_DEVICE_TIMEOUT (read and cleared by
 * sc_last_device_status), waits for its other copies and returns; the
 * context stays usable.  `out` is left partly written.  Needs the TMA path's
 * conditions (W % 4 == 0, W >= 136, H >= 4, 16-byte aligned in and out),
 * else returns SC_ERR_UNSUPPORTED.
 */
int sc_test_stencil_wait_expiry(const float *in, float *out, int H, int W, int drop_copy,
                                int timeout_us, sc_stream_t stream);

/*
 * sc_test_workspace_allocs: test hook, not part of the operation.  The
 * number of temporary device buffers the library has taken from its memory
 * pool since it was loaded (conv2d_fwd with SC_NCHW takes one per call);
 * lets a test check that an entry point allocates nothing.
 */
long long sc_test_workspace_allocs(void);

/* Floats of device scratch behind conv2d_fwd_nchw_noalloc (32 MiB). */
#define SC_NOALLOC_SCRATCH_FLOATS (8u * 1024u * 1024u)

/*
 * conv2d_fwd_nchw_noalloc: conv2d_fwd with layout SC_NCHW, for callers that
 * must not allocate device memory while they run.  (The pages describe no
 * such entry point; it has no counterpart there.)
 *
 * conv2d_fwd with SC_NCHW and more than one channel repacks through a
 * temporary buffer it allocates on the stream.  Some callers cannot accept
 * that: a service that reserved the GPU's memory for its own pool at
 * start-up and treats any further allocation as a failure, or a per-frame
 * real-time pipeline that cannot risk an allocation's latency or an
 * out-of-memory error in the middle of a frame.  This entry point does the
 * same work (NCHW -> NHWC repack, convolution, NHWC -> NCHW repack) and calls
 * no cudaMalloc, cudaMallocAsync, cudaFree or other allocating routine.
 *
 * Its scratch is one array of SC_NOALLOC_SCRATCH_FLOATS floats in the
 * library's own device memory, present on every device that loads the
 * library until the process exits.  A call needs
 *   (Cin > 1 ? round_up(N*H*W*Cin, 64) : 0) + (Cout > 1 ? N*H*W*Cout : 0)
 * floats of it; a larger problem returns SC_ERR_SHAPE before any work.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current: make that first call
 * before any stream capture starts.  All calls share the one array and
 * nothing is cleared between calls (every scratch element a call reads it
 * has written first), so calls whose GPU work overlaps in time (different
 * streams, or different host threads on one device) race on it and must be
 * ordered by the caller.
 * The device address is cached per device for the life of the process, so
 * a cudaDeviceReset (which unloads the library's device memory) while the
 * library is loaded is not supported.
 * Arguments, layout (x and y NCHW), supported shapes and status codes are
 * those of conv2d_fwd, checked by the same code; a failed CUDA call returns
 * SC_ERR_CUDA and records its error code for sc_last_cuda_error.
 */
int conv2d_fwd_nchw_noalloc(const float *x, const float *w, const float *b, float *y,
                            int N, int H, int W, int Cin, int Cout, int R, int S,
                            int act, sc_stream_t stream);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* STENCILCONV_H */
