// conv2d_fwd_nchw_noalloc: the NCHW convolution path without any device
// allocation.  conv2d_fwd with SC_NCHW repacks through a temporary buffer it
// allocates on the stream; this entry point uses a fixed array in the
// library's own device memory instead.  Contract: include/stencilconv.h.
#include <cstdint>
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

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    if (!a || !b || abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

long long count4(int a, int b, int c, int d)
{
    const int v[4] = {a, b, c, d};
    long long n = 1;
    for (int x : v) {
        if (x < 1 || n > (1LL << 62) / x) return -1;
        n *= x;
    }
    return n;
}

int fail(cudaError_t) { return SC_ERR_CUDA; }

}  // namespace

extern "C" int conv2d_fwd_nchw_noalloc(const float *x, const float *w, const float *b, float *y,
                                       int N, int H, int W, int Cin, int Cout, int R, int S, int act,
                                       sc_stream_t stream)
{
    if (!x || !w || !y) return SC_ERR_NULL;
    const long long nx = count4(N, H, W, Cin), ny = count4(N, H, W, Cout), nw = count4(Cout, Cin, R, S);
    if (nx < 0 || ny < 0 || nw < 0 || H > (1 << 30) || W > (1 << 30)) return SC_ERR_SHAPE;
    if ((R & 1) == 0 || (S & 1) == 0 || R > 7 || S > 7) return SC_ERR_UNSUPPORTED;
    if (act != SC_ACT_NONE && act != SC_ACT_RELU) return SC_ERR_UNSUPPORTED;
    if (Cin == 1) {
        if (Cout != 1 && (Cout % 4) != 0) return SC_ERR_UNSUPPORTED;
    } else if ((Cin % 4) != 0 || (Cout % 4) != 0) {
        return SC_ERR_UNSUPPORTED;
    }
    if (Cin > 1 && !aligned16(x)) return SC_ERR_ALIGN;
    if (Cout > 1 && !aligned16(y)) return SC_ERR_ALIGN;
    const size_t ybytes = (size_t)ny * sizeof(float);
    if (overlaps(y, ybytes, x, (size_t)nx * sizeof(float)) ||
        overlaps(y, ybytes, w, (size_t)nw * sizeof(float)) ||
        overlaps(y, ybytes, b, b ? (size_t)Cout * sizeof(float) : 0))
        return SC_ERR_ALIAS;

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
