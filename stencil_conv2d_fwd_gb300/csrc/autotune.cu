// First-call autotuning of the general direct convolution's tile
// configuration (F_TB, W_T, tile height x width, CTAs per SM): the pages
// report hand-tuned best configurations per filter size ("Optimizing Memory
// Efficiency for Convolution Kernels on Kepler GPUs", Table 1, and the
// design-space exploration around it); here the library measures the
// candidates on the caller's own call.
//
// When enabled (sc_set_autotune(1)), the first conv2d_fwd of a shape with
// 3 x 3 filters times every candidate of its class on the caller's stream
// and data (one untimed run, then the best of three timed runs each), keeps
// the fastest in a per-device cache, and runs it last so that y holds its
// result.  Later calls of the shape launch the cached choice.  Timing
// synchronises with the stream, so it is skipped (heuristic dispatch, nothing
// cached) while the stream is being captured into a CUDA graph.
#include <array>
#include <map>
#include <mutex>

#include "../../include/stencilconv.h"
#include "autotune.h"

namespace sc {
namespace {

using Key = std::array<int, 10>;   // device, N, H, W, Cin, Cout, R, S, act, bias present
std::mutex g_mu;
std::map<Key, int> g_cache;
int g_enabled = 0;

Key make_key(int dev, const ConvArgs &a)
{
    return Key{dev, a.N, a.H, a.W, a.Cin, a.Cout, a.R, a.S, a.act, a.b != nullptr};
}

bool tunable(const ConvArgs &a) { return a.R == 3 && a.S == 3 && a.Cin > 1; }

// The best of `reps` timed runs of candidate c, in ms; < 0 if it cannot run.
float time_candidate(const TuneCand &c, const ConvArgs &a, cudaStream_t st, cudaEvent_t e0, cudaEvent_t e1,
                     int reps)
{
    if (c.launch(a, st) != cudaSuccess) {
        cudaGetLastError();   // a candidate that does not apply leaves no error behind
        return -1.f;
    }
    float best = -1.f;
    for (int r = 0; r < reps; ++r) {
        if (cudaEventRecord(e0, st) != cudaSuccess) return -1.f;
        if (c.launch(a, st) != cudaSuccess) return -1.f;
        if (cudaEventRecord(e1, st) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess) return -1.f;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) return -1.f;
        if (best < 0.f || ms < best) best = ms;
    }
    return best;
}

}  // namespace

bool autotune_enabled()
{
    std::lock_guard<std::mutex> lock(g_mu);
    return g_enabled != 0;
}

// conv2d_fwd for NHWC tensors through the autotuner (launch_conv_nhwc calls
// this when tuning is on).
cudaError_t launch_conv_tuned(const ConvArgs &a, cudaStream_t st)
{
    if (!tunable(a)) return cudaErrorNotSupported;
    const TuneCand *cands = nullptr;
    const int n = k3_candidates(a, &cands);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const Key key = make_key(dev, a);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_cache.find(key);
        if (it != g_cache.end()) return cands[it->second].launch(a, st);
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(st, &cap);
    if (e != cudaSuccess) return e;
    if (cap != cudaStreamCaptureStatusNone || n < 2) return cands[0].launch(a, st);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if ((e = cudaEventCreate(&e0)) != cudaSuccess) return e;
    if ((e = cudaEventCreate(&e1)) != cudaSuccess) {
        cudaEventDestroy(e0);
        return e;
    }
    int best = 0;
    float best_ms = -1.f;
    for (int i = 0; i < n; ++i) {
        const float ms = time_candidate(cands[i], a, st, e0, e1, 3);
        if (ms >= 0.f && (best_ms < 0.f || ms < best_ms)) {
            best_ms = ms;
            best = i;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        g_cache[key] = best;
    }
    return cands[best].launch(a, st);   // y holds the chosen candidate's result
}

}  // namespace sc

extern "C" {

int sc_set_autotune(int enable)
{
    std::lock_guard<std::mutex> lock(sc::g_mu);
    const int prev = sc::g_enabled;
    sc::g_enabled = enable ? 1 : 0;
    return prev;
}

int sc_autotune_lookup(int N, int H, int W, int Cin, int Cout, int R, int S, int act, int has_bias)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SC_ERR_CUDA;
    sc::ConvArgs a{nullptr, nullptr, has_bias ? reinterpret_cast<const float *>(1) : nullptr, nullptr, N, H, W, Cin, Cout,
                   R, S, act};
    std::lock_guard<std::mutex> lock(sc::g_mu);
    auto it = sc::g_cache.find(sc::make_key(dev, a));
    return it == sc::g_cache.end() ? -1 : it->second;
}

void sc_autotune_clear(void)
{
    std::lock_guard<std::mutex> lock(sc::g_mu);
    sc::g_cache.clear();
}

int sc_autotune_candidates(int Cin, int Cout, int R, int S, char *names, int names_len)
{
    sc::ConvArgs a{nullptr, nullptr, nullptr, nullptr, 1, 1, 1, Cin, Cout, R, S, 0};
    if (!sc::tunable(a)) return 0;
    const sc::TuneCand *c = nullptr;
    const int n = sc::k3_candidates(a, &c);
    if (names && names_len > 0) {
        int pos = 0;
        names[0] = '\0';
        for (int i = 0; i < n; ++i) {
            for (const char *p = c[i].name; *p && pos < names_len - 2; ++p) names[pos++] = *p;
            if (pos < names_len - 1) names[pos++] = '\n';
        }
        names[pos < names_len ? pos : names_len - 1] = '\0';
    }
    return n;
}

}  // extern "C"
