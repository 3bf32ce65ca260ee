// conv2d_fwd_nchw_noalloc: the NCHW convolution path without any device
// allocation.  conv2d_fwd with SC_NCHW repacks through a temporary buffer it
// allocates on the stream; this entry point uses a fixed array in the
// library's own device memory instead.  Contract: include/stencilconv.h.
#include <mutex>

#include "../../include/stencilconv.h"
#include "launch.h"

namespace {

// Scratch for the NHWC copies of x and y.  It lives in every device that
// loads this library, for the lifetime of the process.
static __device__ __align__(256) float g_noalloc_scratch[SC_NOALLOC_SCRATCH_FLOATS];

// Host code cannot use g_noalloc_scratch as a pointer: on the host the name
// is a stand-in, not a device address.  Resolve the device address once per
// device, with that device current, and hand it to the kernels.
float *scratch_on_current_device(cudaError_t *err)
{
    static std::mutex mu;
    static float *addr[64] = {};
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (*err != cudaSuccess) return nullptr;
        addr[dev] = static_cast<float *>(p);
    }
    return addr[dev];
}

int fail(cudaError_t e) { return sc::record_cuda_error(e); }

}  // namespace

extern "C" int conv2d_fwd_nchw_noalloc(const float *x, const float *w, const float *b, float *y,
                                       int N, int H, int W, int Cin, int Cout, int R, int S, int act,
                                       sc_stream_t stream)
{
    const int chk = sc::check_conv_args(x, w, b, y, N, H, W, Cin, Cout, R, S, SC_NCHW, act);
    if (chk != SC_OK) return chk;
    const long long nx = (long long)N * H * W * Cin, ny = (long long)N * H * W * Cout;

    // Scratch: NHWC x (when Cin > 1), then NHWC y (when Cout > 1), each
    // starting on a 256-byte boundary.
    const long long in_f = Cin > 1 ? nx : 0;
    const long long off = (in_f + 63) & ~63LL;
    const long long out_f = Cout > 1 ? ny : 0;
    if (off + out_f > (long long)SC_NOALLOC_SCRATCH_FLOATS) return SC_ERR_SHAPE;

    cudaError_t e;
    float *scratch = scratch_on_current_device(&e);
    if (!scratch) return fail(e);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    sc::ConvArgs a{x, w, b, y, N, H, W, Cin, Cout, R, S, act};
    if (Cin > 1) {
        e = sc::launch_transpose_batched(x, scratch, N, Cin, (long long)H * W, st);
        if (e != cudaSuccess) return fail(e);
        a.x = scratch;
    }
    if (Cout > 1) a.y = scratch + off;
    e = sc::launch_conv_nhwc(a, st);
    if (e != cudaSuccess) return fail(e);
    if (Cout > 1) {
        e = sc::launch_transpose_batched(scratch + off, y, N, (long long)H * W, Cout, st);
        if (e != cudaSuccess) return fail(e);
    }
    return SC_OK;
}
