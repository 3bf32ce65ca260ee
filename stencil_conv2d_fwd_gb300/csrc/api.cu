// C-ABI of libstencilconv.so: argument validation, dispatch to the kernels,
// the NCHW path through a stream-ordered temporary buffer, and the device
// status word.  Declarations and contracts: include/stencilconv.h.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "../../include/stencilconv.h"
#include "autotune.h"
#include "launch.h"

namespace {

thread_local int g_last_cuda_error = 0;

// Device-side status word (one per device that loads the library).
// Kernels with bounded waits record SC_ERR_DEVICE_TIMEOUT here instead of
// hanging; sc_last_device_status reads and clears it.
__device__ int g_device_status;

int cuda_fail(cudaError_t e) { return sc::record_cuda_error(e); }

// Device allocations made by workspace_alloc (sc_test_workspace_allocs).
std::atomic<long long> g_workspace_allocs{0};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    if (!a || !b || abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// n = product of the sizes, or -1 if any is < 1 or the product would exceed
// 2^62 elements.
long long checked_count(std::initializer_list<int> dims)
{
    long long n = 1;
    for (int d : dims) {
        if (d < 1) return -1;
        if (n > (1LL << 62) / d) return -1;
        n *= d;
    }
    return n;
}

int conv_nhwc_status(const sc::ConvArgs &a, cudaStream_t st)
{
    const cudaError_t e = sc::launch_conv_nhwc(a, st);
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

}  // namespace

namespace sc {

int record_cuda_error(cudaError_t e)
{
    g_last_cuda_error = (int)e;
    return SC_ERR_CUDA;
}

int check_conv_shape(int N, int H, int W, int Cin, int Cout, int R, int S, int layout, int act)
{
    const long long nx = checked_count({N, H, W, Cin});
    const long long ny = checked_count({N, H, W, Cout});
    const long long nw = checked_count({Cout, Cin, R, S});
    if (nx < 0 || ny < 0 || nw < 0) return SC_ERR_SHAPE;
    if (H > (1 << 30) || W > (1 << 30)) return SC_ERR_SHAPE;
    if ((R & 1) == 0 || (S & 1) == 0 || R > 7 || S > 7) return SC_ERR_UNSUPPORTED;
    if (layout != SC_NCHW && layout != SC_NHWC) return SC_ERR_UNSUPPORTED;
    if (act != SC_ACT_NONE && act != SC_ACT_RELU) return SC_ERR_UNSUPPORTED;
    if (Cin == 1) {
        if (Cout != 1 && (Cout % 4) != 0) return SC_ERR_UNSUPPORTED;
    } else {
        if ((Cin % 4) != 0 || (Cout % 4) != 0) return SC_ERR_UNSUPPORTED;
    }
    return SC_OK;
}

int check_conv_args(const float *x, const float *w, const float *b, const float *y, int N, int H, int W, int Cin,
                    int Cout, int R, int S, int layout, int act)
{
    if (!x || !w || !y) return SC_ERR_NULL;
    const int shape = check_conv_shape(N, H, W, Cin, Cout, R, S, layout, act);
    if (shape != SC_OK) return shape;
    const long long nx = (long long)N * H * W * Cin, ny = (long long)N * H * W * Cout;
    const long long nw = (long long)Cout * Cin * R * S;
    if (Cin > 1 && !aligned16(x)) return SC_ERR_ALIGN;
    if (Cout > 1 && !aligned16(y)) return SC_ERR_ALIGN;
    const size_t ybytes = (size_t)ny * sizeof(float);
    if (overlaps(y, ybytes, x, (size_t)nx * sizeof(float)) ||
        overlaps(y, ybytes, w, (size_t)nw * sizeof(float)) ||
        overlaps(y, ybytes, b, b ? (size_t)Cout * sizeof(float) : 0))
        return SC_ERR_ALIAS;
    return SC_OK;
}

cudaError_t launch_conv_nhwc(const ConvArgs &a, cudaStream_t st)
{
    if (autotune_enabled() && a.R == 3 && a.S == 3 && a.Cin > 1) return launch_conv_tuned(a, st);
    if (a.Cin == 1) return launch_conv_c1(a, st);
    switch (a.R > a.S ? a.R : a.S) {
    case 1: return launch_conv_general_k1(a, st);
    case 3: return launch_conv_general_k3(a, st);
    case 5: return launch_conv_general_k5(a, st);
    case 7: return launch_conv_general_k7(a, st);
    default: return cudaErrorInvalidValue;
    }
}

int *device_status_ptr()
{
    static std::atomic<int *> addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    int *a = addr[dev].load(std::memory_order_acquire);
    if (!a) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        a = static_cast<int *>(p);
        addr[dev].store(a, std::memory_order_release);
    }
    return a;
}

std::mutex &launch_cache_mutex()
{
    static std::mutex m;
    return m;
}

// Temporary buffers come from one library-private memory pool per device
// whose release threshold is unlimited: memory freed on a stream stays in
// the pool for the next call, where the default pool would hand it back to
// the driver at the next synchronisation and map it again on the next
// allocation.  sc_release_workspace() trims the pools.
static std::mutex g_pool_mu;
static cudaMemPool_t g_pool[64] = {};

static cudaError_t workspace_pool(cudaMemPool_t *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pool[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = ~0ull;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return e;
        }
        g_pool[dev] = pool;
    }
    *out = g_pool[dev];
    return cudaSuccess;
}

cudaError_t workspace_alloc(void **p, size_t bytes, cudaStream_t st)
{
    cudaMemPool_t pool = nullptr;
    const cudaError_t e = workspace_pool(&pool);
    if (e != cudaSuccess) return e;
    g_workspace_allocs.fetch_add(1, std::memory_order_relaxed);
    return cudaMallocFromPoolAsync(p, bytes, pool, st);
}

cudaError_t workspace_free(void *p, cudaStream_t st) { return cudaFreeAsync(p, st); }

void workspace_trim()
{
    std::lock_guard<std::mutex> lock(g_pool_mu);
    for (cudaMemPool_t pool : g_pool)
        if (pool) cudaMemPoolTrimTo(pool, 0);
}

int device_sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 148;
    if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace sc

extern "C" {

int conv2d_fwd(const float *x, const float *w, const float *b, float *y, int N, int H, int W,
               int Cin, int Cout, int R, int S, int layout, int act, sc_stream_t stream)
{
    const int chk = sc::check_conv_args(x, w, b, y, N, H, W, Cin, Cout, R, S, layout, act);
    if (chk != SC_OK) return chk;
    const long long nx = (long long)N * H * W * Cin, ny = (long long)N * H * W * Cout;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    sc::ConvArgs a{x, w, b, y, N, H, W, Cin, Cout, R, S, act};
    const bool need_in = (layout == SC_NCHW) && Cin > 1;
    const bool need_out = (layout == SC_NCHW) && Cout > 1;
    if (!need_in && !need_out) return conv_nhwc_status(a, st);

    // NCHW with channels: repack to NHWC in a stream-ordered temporary buffer.
    const size_t in_bytes = need_in ? (size_t)nx * sizeof(float) : 0;
    const size_t out_bytes = need_out ? (size_t)ny * sizeof(float) : 0;
    const size_t off = (in_bytes + 255) & ~(size_t)255;
    void *ws = nullptr;
    cudaError_t e = sc::workspace_alloc(&ws, off + out_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e);
    float *x_nhwc = need_in ? static_cast<float *>(ws) : nullptr;
    float *y_nhwc = need_out ? reinterpret_cast<float *>(static_cast<char *>(ws) + off) : y;
    int rc = SC_OK;
    if (need_in) {
        e = sc::launch_transpose_batched(x, x_nhwc, N, Cin, (long long)H * W, st);
        if (e != cudaSuccess) rc = cuda_fail(e);
        a.x = x_nhwc;
    }
    if (rc == SC_OK) {
        a.y = y_nhwc;
        rc = conv_nhwc_status(a, st);
    }
    if (rc == SC_OK && need_out) {
        e = sc::launch_transpose_batched(y_nhwc, y, N, (long long)H * W, Cout, st);
        if (e != cudaSuccess) rc = cuda_fail(e);
    }
    cudaError_t ef = sc::workspace_free(ws, st);
    if (rc == SC_OK && ef != cudaSuccess) rc = cuda_fail(ef);
    return rc;
}

int conv2d_chain_fwd_host(const float *x_host, float *y_host, int N, int H, int W, int Cin, int n_layers,
                          const sc_conv_layer *layers, sc_stream_t stream)
{
    if (!x_host || !y_host || !layers) return SC_ERR_NULL;
    if (n_layers < 1 || n_layers > SC_CHAIN_MAX_LAYERS) return SC_ERR_SHAPE;
    // every layer's shape first: nothing is enqueued for a chain that fails
    int cin = Cin, cmax = 1;
    for (int l = 0; l < n_layers; ++l) {
        const sc_conv_layer &L = layers[l];
        if (!L.w) return SC_ERR_NULL;
        const int rc = sc::check_conv_shape(N, H, W, cin, L.Cout, L.R, L.S, SC_NHWC, L.act);
        if (rc != SC_OK) return rc;
        if (L.Cout > cmax) cmax = L.Cout;
        cin = L.Cout;
    }
    const long long px = (long long)N * H * W;
    const size_t in_bytes = (size_t)(px * Cin) * sizeof(float);
    const size_t out_bytes = (size_t)(px * cin) * sizeof(float);
    const size_t act_bytes = (((size_t)(px * cmax) * sizeof(float)) + 255) & ~(size_t)255;
    const size_t off = (in_bytes + 255) & ~(size_t)255;
    // [input][activation A][activation B]: layer l reads the input (l = 0)
    // or buffer (l - 1) % 2 and writes buffer l % 2
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    cudaError_t e = sc::workspace_alloc(&ws, off + (n_layers > 1 ? 2 : 1) * act_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e);
    char *base = static_cast<char *>(ws);
    float *act_buf[2] = {reinterpret_cast<float *>(base + off), reinterpret_cast<float *>(base + off + act_bytes)};
    int rc = SC_OK;
    e = cudaMemcpyAsync(base, x_host, in_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) rc = cuda_fail(e);
    const float *in = reinterpret_cast<const float *>(base);
    cin = Cin;
    for (int l = 0; l < n_layers && rc == SC_OK; ++l) {
        const sc_conv_layer &L = layers[l];
        const sc::ConvArgs a{in, L.w, L.b, act_buf[l & 1], N, H, W, cin, L.Cout, L.R, L.S, L.act};
        rc = conv_nhwc_status(a, st);
        in = act_buf[l & 1];
        cin = L.Cout;
    }
    if (rc == SC_OK) {
        e = cudaMemcpyAsync(y_host, in, out_bytes, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) rc = cuda_fail(e);
    }
    cudaError_t ef = sc::workspace_free(ws, st);
    if (rc == SC_OK && ef != cudaSuccess) rc = cuda_fail(ef);
    return rc;
}

// The argument checks shared by conv2d_fwd_tc and conv2d_fwd_tc_x3; SC_OK
// when the call may launch.
static int check_tc_args(const float *x, const float *w, const float *b, const float *y, int N, int H, int W,
                         int Cin, int Cout, int R, int S, int act)
{
    if (!x || !w || !y) return SC_ERR_NULL;
    const long long nx = checked_count({N, H, W, Cin});
    const long long ny = checked_count({N, H, W, Cout});
    const long long nw = checked_count({Cout, Cin, R, S});
    if (nx < 0 || ny < 0 || nw < 0) return SC_ERR_SHAPE;
    if (H > (1 << 30) || W > (1 << 30)) return SC_ERR_SHAPE;
    if ((R & 1) == 0 || (S & 1) == 0 || R > 3 || S > 3) return SC_ERR_UNSUPPORTED;
    if (act != SC_ACT_NONE && act != SC_ACT_RELU) return SC_ERR_UNSUPPORTED;
    if ((Cin % 4) != 0 || (Cout % 4) != 0 || Cout > 128) return SC_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(y) || !aligned16(w)) return SC_ERR_ALIGN;
    const size_t ybytes = (size_t)ny * sizeof(float);
    if (overlaps(y, ybytes, x, (size_t)nx * sizeof(float)) ||
        overlaps(y, ybytes, w, (size_t)nw * sizeof(float)) ||
        overlaps(y, ybytes, b, b ? (size_t)Cout * sizeof(float) : 0))
        return SC_ERR_ALIAS;
    return SC_OK;
}

int conv2d_fwd_tc_x3(const float *x, const float *w, const float *b, float *y, int N, int H, int W, int Cin,
                     int Cout, int R, int S, int act, sc_stream_t stream)
{
    const int chk = check_tc_args(x, w, b, y, N, H, W, Cin, Cout, R, S, act);
    if (chk != SC_OK) return chk;
    sc::ConvArgs a{x, w, b, y, N, H, W, Cin, Cout, R, S, act};
    const cudaError_t e = sc::launch_conv_tc_x3(a, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return SC_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

int conv2d_fwd_tc(const float *x, const float *w, const float *b, float *y, int N, int H, int W, int Cin,
                  int Cout, int R, int S, int act, sc_stream_t stream)
{
    const int chk = check_tc_args(x, w, b, y, N, H, W, Cin, Cout, R, S, act);
    if (chk != SC_OK) return chk;
    sc::ConvArgs a{x, w, b, y, N, H, W, Cin, Cout, R, S, act};
    const cudaError_t e = sc::launch_conv_tc(a, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return SC_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

int conv2d_fwd_tc_bf16(const void *x, const float *w, const float *b, void *y, int N, int H, int W, int Cin,
                       int Cout, int R, int S, int act, int y_dtype, sc_stream_t stream)
{
    if (!x || !w || !y) return SC_ERR_NULL;
    const long long nx = checked_count({N, H, W, Cin});
    const long long ny = checked_count({N, H, W, Cout});
    const long long nw = checked_count({Cout, Cin, R, S});
    if (nx < 0 || ny < 0 || nw < 0) return SC_ERR_SHAPE;
    if (H > (1 << 30) || W > (1 << 30)) return SC_ERR_SHAPE;
    if ((R & 1) == 0 || (S & 1) == 0 || R > 3 || S > 3) return SC_ERR_UNSUPPORTED;
    if (act != SC_ACT_NONE && act != SC_ACT_RELU) return SC_ERR_UNSUPPORTED;
    if (y_dtype != SC_F32 && y_dtype != SC_BF16) return SC_ERR_UNSUPPORTED;
    if ((Cin % 8) != 0 || (Cout % 4) != 0 || Cout > 128) return SC_ERR_UNSUPPORTED;
    if (y_dtype == SC_BF16 && Cout > 16 && (Cout % 8) != 0) return SC_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(y) || !aligned16(w)) return SC_ERR_ALIGN;
    const size_t ybytes = (size_t)ny * (y_dtype == SC_BF16 ? 2 : 4);
    if (overlaps(y, ybytes, x, (size_t)nx * 2) || overlaps(y, ybytes, w, (size_t)nw * sizeof(float)) ||
        overlaps(y, ybytes, b, b ? (size_t)Cout * sizeof(float) : 0))
        return SC_ERR_ALIAS;
    // the bf16 tensors travel in ConvArgs' pointer fields; only the kernels read them
    sc::ConvArgs a{static_cast<const float *>(x), w, b, static_cast<float *>(y), N, H, W, Cin, Cout, R, S, act};
    const cudaError_t e = sc::launch_conv_tc_bf16(a, y_dtype == SC_BF16, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return SC_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

int conv2d_fwd_tc_fused2(const float *x, const float *w1, const float *b1, const float *w2, const float *b2,
                         float *y, int N, int H, int W, int C0, int C1, int C2, int act1, int act2, sc_stream_t stream)
{
    if (!x || !w1 || !w2 || !y) return SC_ERR_NULL;
    const long long nx = checked_count({N, H, W, C0});
    const long long ny = checked_count({N, H, W, C2});
    if (nx < 0 || ny < 0 || C1 < 1) return SC_ERR_SHAPE;
    if (H > (1 << 30) || W > (1 << 30)) return SC_ERR_SHAPE;
    if ((act1 != SC_ACT_NONE && act1 != SC_ACT_RELU) || (act2 != SC_ACT_NONE && act2 != SC_ACT_RELU))
        return SC_ERR_UNSUPPORTED;
    if ((C0 % 4) != 0 || C1 != 32 || (C2 % 4) != 0 || C2 > 8) return SC_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(y) || !aligned16(w1) || !aligned16(w2)) return SC_ERR_ALIGN;
    const size_t ybytes = (size_t)ny * sizeof(float);
    if (overlaps(y, ybytes, x, (size_t)nx * sizeof(float)) ||
        overlaps(y, ybytes, w1, (size_t)C1 * C0 * 9 * sizeof(float)) ||
        overlaps(y, ybytes, w2, (size_t)C2 * C1 * 9 * sizeof(float)) ||
        overlaps(y, ybytes, b1, b1 ? (size_t)C1 * sizeof(float) : 0) ||
        overlaps(y, ybytes, b2, b2 ? (size_t)C2 * sizeof(float) : 0))
        return SC_ERR_ALIAS;
    sc::FusedArgs a{x, w1, b1, w2, b2, y, N, H, W, C0, C1, C2, act1, act2};
    const cudaError_t e = sc::launch_conv_tc_fused2(a, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return SC_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

int stencil_pipeline_fwd(const float *in, float *out, int H, int W, sc_stream_t stream)
{
    if (!in || !out) return SC_ERR_NULL;
    const long long n = checked_count({H, W});
    if (n < 0) return SC_ERR_SHAPE;
    if (overlaps(in, (size_t)n * sizeof(float), out, (size_t)n * sizeof(float))) return SC_ERR_ALIAS;
    cudaError_t e = sc::launch_stencil_pipeline(in, out, H, W, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

int sc_repack(const float *src, float *dst, int N, int C, int H, int W, int src_layout,
              int dst_layout, sc_stream_t stream)
{
    if (!src || !dst) return SC_ERR_NULL;
    const long long n = checked_count({N, C, H, W});
    if (n < 0) return SC_ERR_SHAPE;
    if ((src_layout != SC_NCHW && src_layout != SC_NHWC) ||
        (dst_layout != SC_NCHW && dst_layout != SC_NHWC))
        return SC_ERR_UNSUPPORTED;
    if (overlaps(src, (size_t)n * sizeof(float), dst, (size_t)n * sizeof(float))) return SC_ERR_ALIAS;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (src_layout == dst_layout || C == 1)
        e = cudaMemcpyAsync(dst, src, (size_t)n * sizeof(float), cudaMemcpyDeviceToDevice, st);
    else if (src_layout == SC_NCHW)
        e = sc::launch_transpose_batched(src, dst, N, C, (long long)H * W, st);
    else
        e = sc::launch_transpose_batched(src, dst, N, (long long)H * W, C, st);
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

int sc_last_device_status(sc_stream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return v;
}

const char *sc_status_string(int status)
{
    switch (status) {
    case SC_OK: return "ok";
    case SC_ERR_NULL: return "a required pointer is NULL";
    case SC_ERR_SHAPE: return "a size is < 1 or the sizes overflow";
    case SC_ERR_UNSUPPORTED: return "unsupported convolution parameters";
    case SC_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case SC_ERR_ALIAS: return "output overlaps an input";
    case SC_ERR_CUDA: return "a CUDA call failed";
    case SC_ERR_DEVICE_TIMEOUT: return "a device-side bounded wait expired";
    default: return "unknown status";
    }
}

int sc_last_cuda_error(void) { return g_last_cuda_error; }

int sc_measure_ffma_peak(float *sink, int blocks, int iters, sc_stream_t stream)
{
    if (!sink) return SC_ERR_NULL;
    if (blocks < 1 || iters < 1 || blocks > (1 << 24)) return SC_ERR_SHAPE;
    cudaError_t e = sc::launch_ffma_peak(sink, blocks, iters, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

int sc_empty_kernel(int blocks, int threads, sc_stream_t stream)
{
    if (blocks < 1 || blocks > (1 << 24) || threads < 1 || threads > 1024) return SC_ERR_SHAPE;
    cudaError_t e = sc::launch_empty(blocks, threads, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

int sc_version(void) { return 100; }

int sc_test_conv_candidate(const float *x, const float *w, const float *b, float *y, int N, int H, int W, int Cin,
                           int Cout, int R, int S, int act, int candidate, sc_stream_t stream)
{
    if (!x || !w || !y) return SC_ERR_NULL;
    if (checked_count({N, H, W, Cin}) < 0 || checked_count({N, H, W, Cout}) < 0) return SC_ERR_SHAPE;
    if (R != 3 || S != 3 || Cin < 2 || (Cin % 4) != 0 || (Cout % 4) != 0) return SC_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(y)) return SC_ERR_ALIGN;
    sc::ConvArgs a{x, w, b, y, N, H, W, Cin, Cout, R, S, act};
    const sc::TuneCand *c = nullptr;
    const int n = sc::k3_candidates(a, &c);
    if (candidate < 0 || candidate >= n) return SC_ERR_UNSUPPORTED;
    const cudaError_t e = c[candidate].launch(a, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) {
        cudaGetLastError();
        return SC_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

long long sc_test_workspace_allocs(void) { return g_workspace_allocs.load(std::memory_order_relaxed); }

int sc_release_workspace(void)
{
    sc::workspace_trim();
    return SC_OK;
}

int sc_test_stencil_wait_expiry(const float *in, float *out, int H, int W, int drop_copy, int timeout_us,
                                sc_stream_t stream)
{
    if (!in || !out) return SC_ERR_NULL;
    const long long n = checked_count({H, W});
    if (n < 0 || drop_copy < 0 || timeout_us < 1) return SC_ERR_SHAPE;
    if (overlaps(in, (size_t)n * sizeof(float), out, (size_t)n * sizeof(float))) return SC_ERR_ALIAS;
    const cudaError_t e = sc::launch_stencil_pipeline(in, out, H, W, reinterpret_cast<cudaStream_t>(stream),
                                                      drop_copy, 1000ull * (unsigned long long)timeout_us);
    if (e == cudaErrorNotSupported) return SC_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

int sc_test_conv_wait_expiry(const float *x, const float *w, const float *b, float *y, int N, int H, int W, int Cin,
                             int Cout, int drop_copy, int timeout_us, sc_stream_t stream)
{
    if (!x || !w || !y) return SC_ERR_NULL;
    const long long nx = checked_count({N, H, W, Cin});
    const long long ny = checked_count({N, H, W, Cout});
    const long long nw = checked_count({Cout, Cin, 3, 3});
    if (nx < 0 || ny < 0 || nw < 0 || drop_copy < 0 || timeout_us < 1) return SC_ERR_SHAPE;
    if ((Cin % 4) != 0 || (Cout % 4) != 0) return SC_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(y)) return SC_ERR_ALIGN;
    const size_t ybytes = (size_t)ny * sizeof(float);
    if (overlaps(y, ybytes, x, (size_t)nx * sizeof(float)) || overlaps(y, ybytes, w, (size_t)nw * sizeof(float)) ||
        overlaps(y, ybytes, b, b ? (size_t)Cout * sizeof(float) : 0))
        return SC_ERR_ALIAS;
    sc::ConvArgs a{x, w, b, y, N, H, W, Cin, Cout, 3, 3, SC_ACT_NONE};
    const cudaError_t e = sc::launch_conv_tma_k3_test(a, drop_copy, 1000ull * (unsigned long long)timeout_us,
                                                      reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return SC_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SC_OK : cuda_fail(e);
}

}  // extern "C"
