// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Not exported.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace sc {

struct ConvArgs {
    const float *x;   // NHWC activations (Cin == 1: [N][H][W])
    const float *w;   // OIHW weights
    const float *b;   // bias or nullptr
    float *y;         // NHWC output
    int N, H, W, Cin, Cout, R, S, act;
};

// General direct convolution, Cin % 4 == 0, Cout % 4 == 0, filters up to
// K x K (conv_general_k*.cu).
cudaError_t launch_conv_general_k1(const ConvArgs &a, cudaStream_t st);
cudaError_t launch_conv_general_k3(const ConvArgs &a, cudaStream_t st);
cudaError_t launch_conv_general_k5(const ConvArgs &a, cudaStream_t st);
cudaError_t launch_conv_general_k7(const ConvArgs &a, cudaStream_t st);

// TMA-staged direct convolution for 3 x 3 filters (conv_tma_k3.cu), 16 or
// fewer output channels (narrow) or more (wide); cudaErrorNotSupported
// where it does not apply.
cudaError_t launch_conv_tma_k3_narrow(const ConvArgs &a, cudaStream_t st);
// Whole-tile-at-once direct convolution for small images (conv_small.cu):
// NHWC, Cin and Cout multiples of 4 up to 16, 3 x 3 filters, at most 64 K
// pixels in all; cudaErrorNotSupported otherwise.
cudaError_t launch_conv_small(const ConvArgs &a, cudaStream_t st);
cudaError_t launch_conv_tma_k3_wide(const ConvArgs &a, cudaStream_t st);
// The same kernel for 5 x 5 filters with 16 or fewer output channels and for
// 1 x 1 filters (conv_tma_k5.cu, conv_tma_k1.cu).
cudaError_t launch_conv_tma_k5_narrow(const ConvArgs &a, cudaStream_t st);
cudaError_t launch_conv_tma_k1_narrow(const ConvArgs &a, cudaStream_t st);
cudaError_t launch_conv_tma_k1_wide(const ConvArgs &a, cudaStream_t st);
// Test hook (sc_test_conv_wait_expiry): the default configuration with
// copy `drop_copy` of every CTA never issued and waits bounded by timeout_ns.
cudaError_t launch_conv_tma_k3_test(const ConvArgs &a, int drop_copy, unsigned long long timeout_ns,
                                    cudaStream_t st);

// NHWC convolution: picks the single-input-channel kernel or the general
// kernel for K = max(R, S) (api.cu).
cudaError_t launch_conv_nhwc(const ConvArgs &a, cudaStream_t st);

// Tensor-core (tcgen05) implicit-GEMM convolution, TF32 operands, NHWC, Cin % 4 == 0,
// Cout <= 128, R, S <= 3 (conv_tc.cu).  cudaErrorNotSupported otherwise.
cudaError_t launch_conv_tc(const ConvArgs &a, cudaStream_t st);
// The same with split-TF32 operands (three MMAs per product, head and
// correction accumulators; conv_tc.cu).
cudaError_t launch_conv_tc_x3(const ConvArgs &a, cudaStream_t st);
// BF16 operands (conv_tc.cu): a.x is a bf16 NHWC tensor, a.y bf16 (y_bf16)
// or fp32; a.w, a.b fp32.
cudaError_t launch_conv_tc_bf16(const ConvArgs &a, bool y_bf16, cudaStream_t st);

// Single-input-channel convolution, Cout == 1 or Cout % 4 == 0 (conv_c1.cu).
cudaError_t launch_conv_c1(const ConvArgs &a, cudaStream_t st);

// Fused blur/unsharp pipeline (stencil.cu).  drop_copy >= 0 leaves that
// TMA copy of every warp un-issued so its bounded wait expires (tests of the
// device-status path); timeout_ns bounds each wait.
cudaError_t launch_stencil_pipeline(const float *in, float *out, int H, int W, cudaStream_t st,
                                    int drop_copy = -1, unsigned long long timeout_ns = 1000000000ull);

// dst[n][b][a] = src[n][a][b] (repack.cu): NCHW->NHWC is (A=C, B=H*W),
// NHWC->NCHW is (A=H*W, B=C).
cudaError_t launch_transpose_batched(const float *src, float *dst, int N, long long A,
                                     long long B, cudaStream_t st);

// FP32 FMA rate probe and launch-cost probe (peak.cu).
cudaError_t launch_ffma_peak(float *sink, int blocks, int iters, cudaStream_t st);
cudaError_t launch_empty(int blocks, int threads, cudaStream_t st);

// Two 3 x 3 layers fused on the tensor cores (conv_tc_fused.cu): x NHWC fp32
// (C0 channels) -> act1(conv(x, w1) + b1) with C1 = 32 channels, kept on
// chip -> y = act2(conv(., w2) + b2) NHWC fp32 with C2 <= 8 channels.
struct FusedArgs {
    const float *x, *w1, *b1, *w2, *b2;
    float *y;
    int N, H, W, C0, C1, C2, act1, act2;
};
cudaError_t launch_conv_tc_fused2(const FusedArgs &a, cudaStream_t st);

// First-call autotuner (autotune.cu): whether sc_set_autotune turned it on,
// and conv2d_fwd for NHWC tensors through it (3 x 3 filters, Cin > 1).
bool autotune_enabled();
cudaError_t launch_conv_tuned(const ConvArgs &a, cudaStream_t st);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Per-device launch caches of one kernel, safe to use from several host
// threads at once: the largest dynamic shared memory the kernel has been
// opted in to (it only grows, so a size below it stays valid), and the
// resident CTAs per SM of the last size queried, as (smem << 32) | CTAs.
// Static storage zero-initialises them.
struct KernelCache {
    std::atomic<int> allowed[64];
    std::atomic<long long> occ[64];
};

// Serialises the cudaFuncSetAttribute calls of every launcher (api.cu).
std::mutex &launch_cache_mutex();

// Opts `kernel` in to `smem` bytes of dynamic shared memory on device dev
// (0 <= dev < 64), once per size increase.  Also below 48 KB: without the
// opt-in, static and dynamic shared memory together are capped at 48 KB.
template <class K>
cudaError_t ensure_dynamic_smem(KernelCache &c, int dev, K kernel, int smem)
{
    if (smem <= 0 || c.allowed[dev].load(std::memory_order_acquire) >= smem) return cudaSuccess;
    std::lock_guard<std::mutex> lock(launch_cache_mutex());
    if (c.allowed[dev].load(std::memory_order_relaxed) >= smem) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) c.allowed[dev].store(smem, std::memory_order_release);
    return e;
}

// Resident CTAs per SM of `kernel` with `threads` threads and `smem` bytes
// of dynamic shared memory on device dev (at least 1).
template <class K>
cudaError_t resident_ctas(KernelCache &c, int dev, K kernel, int threads, int smem, int *ctas)
{
    const long long v = c.occ[dev].load(std::memory_order_acquire);
    if (v != 0 && (int)(v >> 32) == smem) {
        *ctas = (int)(v & 0xffffffffLL);
        return cudaSuccess;
    }
    int b = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, smem);
    if (e != cudaSuccess) return e;
    if (b < 1) b = 1;
    c.occ[dev].store(((long long)smem << 32) | b, std::memory_order_release);
    *ctas = b;
    return cudaSuccess;
}

// Stream-ordered temporary buffers (api.cu) from a library-private memory
// pool of the current device; see sc_release_workspace.
cudaError_t workspace_alloc(void **p, size_t bytes, cudaStream_t st);
cudaError_t workspace_free(void *p, cudaStream_t st);

// conv2d_fwd's argument checks (api.cu), shared by every entry point with
// its contract: SC_OK when the call may launch, else the status to return.
int check_conv_args(const float *x, const float *w, const float *b, const float *y, int N, int H, int W, int Cin,
                    int Cout, int R, int S, int layout, int act);
// The part of those checks that needs no pointers: sizes, filter size,
// layout, activation and the supported channel counts.
int check_conv_shape(int N, int H, int W, int Cin, int Cout, int R, int S, int layout, int act);
// Records e for sc_last_cuda_error (per host thread) and returns SC_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Device address of the current device's status word (api.cu), or nullptr.
int *device_status_ptr();

// Value kernels store in the status word when a bounded wait expires
// (SC_ERR_DEVICE_TIMEOUT of include/stencilconv.h).
constexpr int kDeviceTimeout = -7;

}  // namespace sc
