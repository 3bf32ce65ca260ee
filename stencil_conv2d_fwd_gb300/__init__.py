"""Python binding of libstencilconv.so (direct conv2d forward + fused stencil).

Argument marshalling only: every step runs in the library's CUDA kernels.
The functions below carry the C-ABI names of ``include/stencilconv.h`` and
return its status codes.  Tensor arguments may be torch tensors (their
``data_ptr()`` is passed) or raw integer device addresses; ``stream`` may be
a ``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or None for torch's
current stream.

The shared library is built in-tree by ``_build.build()``; if it cannot be
loaded, ``load()`` raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

SC_OK = 0
SC_ERR_NULL = -1
SC_ERR_SHAPE = -2
SC_ERR_UNSUPPORTED = -3
SC_ERR_ALIGN = -4
SC_ERR_ALIAS = -5
SC_ERR_CUDA = -6
SC_ERR_DEVICE_TIMEOUT = -7
SC_NCHW = 0
SC_NHWC = 1
SC_ACT_NONE = 0
SC_ACT_RELU = 1
SC_F32 = 0
SC_BF16 = 1

# Every symbol include/stencilconv.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "conv2d_fwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "conv2d_fwd_tc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "conv2d_fwd_tc_x3": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "conv2d_fwd_tc_bf16": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "conv2d_fwd_tc_fused2": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "stencil_pipeline_fwd": (_I, [_P, _P, _I, _I, _P]),
    "sc_repack": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "sc_last_device_status": (_I, [_P]),
    "sc_status_string": (ctypes.c_char_p, [_I]),
    "sc_last_cuda_error": (_I, []),
    "sc_measure_ffma_peak": (_I, [_P, _I, _I, _P]),
    "sc_version": (_I, []),
    "sc_empty_kernel": (_I, [_I, _I, _P]),
    "sc_release_workspace": (_I, []),
    "sc_set_autotune": (_I, [_I]),
    "sc_autotune_lookup": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "sc_autotune_clear": (None, []),
    "sc_autotune_candidates": (_I, [_I, _I, _I, _I, ctypes.c_char_p, _I]),
    "sc_test_conv_candidate": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "conv2d_fwd_nchw_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "sc_test_stencil_wait_expiry": (_I, [_P, _P, _I, _I, _I, _I, _P]),
    "sc_test_conv_wait_expiry": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "sc_test_workspace_allocs": (ctypes.c_longlong, []),
    "conv2d_chain_fwd_host": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P]),
}
SC_CHAIN_MAX_LAYERS = 64


class ScConvLayer(ctypes.Structure):
    """sc_conv_layer: one layer of conv2d_chain_fwd_host (device filters and bias)."""
    _fields_ = [("w", ctypes.c_void_p), ("b", ctypes.c_void_p), ("Cout", ctypes.c_int), ("R", ctypes.c_int),
                ("S", ctypes.c_int), ("act", ctypes.c_int)]
SC_NOALLOC_SCRATCH_FLOATS = 8 * 1024 * 1024

_lib = None


class StencilConvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = f"{what}: " if what else ""
        super().__init__(f"{msg}status {status} ({status_string(status)})")


def lib_path() -> str:
    return _build.LIB


def load(build_if_stale: bool = True):
    """Load libstencilconv.so (building it first when sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_stale and _build.is_stale():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"libstencilconv.so is missing at {_build.LIB}; run the build first")
    lib = ctypes.CDLL(_build.LIB)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def conv2d_fwd(x, w, b, y, N, H, W, Cin, Cout, R, S, layout=SC_NHWC, act=SC_ACT_NONE, stream=None) -> int:
    return load().conv2d_fwd(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, H, W, Cin, Cout, R, S,
                             layout, act, _stream(stream))


def conv2d_fwd_tc(x, w, b, y, N, H, W, Cin, Cout, R, S, act=SC_ACT_NONE, stream=None) -> int:
    """Tensor-core (TF32) variant of conv2d_fwd, NHWC only (see the header)."""
    return load().conv2d_fwd_tc(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, H, W, Cin, Cout, R, S, act,
                                _stream(stream))


def conv2d_fwd_tc_x3(x, w, b, y, N, H, W, Cin, Cout, R, S, act=SC_ACT_NONE, stream=None) -> int:
    """conv2d_fwd_tc with split-TF32 operands, fp32-level results (see the header)."""
    return load().conv2d_fwd_tc_x3(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, H, W, Cin, Cout, R, S, act,
                                   _stream(stream))


def conv2d_fwd_tc_bf16(x, w, b, y, N, H, W, Cin, Cout, R, S, act=SC_ACT_NONE, y_dtype=SC_BF16,
                       stream=None) -> int:
    """BF16-storage tensor-core variant: x bf16, y bf16 or fp32 (see the header)."""
    return load().conv2d_fwd_tc_bf16(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, H, W, Cin, Cout, R, S, act, y_dtype,
                                     _stream(stream))


def conv2d_fwd_tc_fused2(x, w1, b1, w2, b2, y, N, H, W, C0, C1, C2, act1=SC_ACT_RELU, act2=SC_ACT_NONE,
                         stream=None) -> int:
    """Two 3x3 layers fused on the tensor cores, intermediate on chip (see the header)."""
    return load().conv2d_fwd_tc_fused2(_ptr(x), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2), _ptr(y), N, H, W, C0, C1, C2,
                                       act1, act2, _stream(stream))


def stencil_pipeline_fwd(inp, out, H, W, stream=None) -> int:
    return load().stencil_pipeline_fwd(_ptr(inp), _ptr(out), H, W, _stream(stream))


def sc_repack(src, dst, N, C, H, W, src_layout, dst_layout, stream=None) -> int:
    return load().sc_repack(_ptr(src), _ptr(dst), N, C, H, W, src_layout, dst_layout, _stream(stream))


def sc_last_device_status(stream=None) -> int:
    return load().sc_last_device_status(_stream(stream))


def sc_status_string(status: int) -> str:
    return load().sc_status_string(int(status)).decode()


status_string = sc_status_string


def sc_last_cuda_error() -> int:
    return load().sc_last_cuda_error()


def sc_measure_ffma_peak(sink, blocks, iters, stream=None) -> int:
    return load().sc_measure_ffma_peak(_ptr(sink), blocks, iters, _stream(stream))


def sc_version() -> int:
    return load().sc_version()


def sc_set_autotune(enable) -> int:
    """First-call autotuning of conv2d_fwd's tile configuration on/off (see the header)."""
    return load().sc_set_autotune(1 if enable else 0)


def sc_autotune_lookup(N, H, W, Cin, Cout, R, S, act=SC_ACT_NONE, has_bias=True) -> int:
    return load().sc_autotune_lookup(N, H, W, Cin, Cout, R, S, act, 1 if has_bias else 0)


def sc_autotune_clear() -> None:
    load().sc_autotune_clear()


def sc_autotune_candidates(Cin, Cout, R, S) -> list:
    """Names of the candidate configurations for a filter shape ([] if not tuned)."""
    buf = ctypes.create_string_buffer(4096)
    n = load().sc_autotune_candidates(Cin, Cout, R, S, buf, len(buf))
    names = buf.value.decode().split("\n")
    return [x for x in names if x][:n]


def sc_test_conv_candidate(x, w, b, y, N, H, W, Cin, Cout, R, S, act, candidate, stream=None) -> int:
    """Test hook: conv2d_fwd with one candidate configuration (see the header)."""
    return load().sc_test_conv_candidate(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, H, W, Cin, Cout, R, S, act,
                                         candidate, _stream(stream))


def sc_release_workspace() -> int:
    """Trim the library's pool of temporary device buffers (see the header)."""
    return load().sc_release_workspace()


def conv2d_fwd_nchw_noalloc(x, w, b, y, N, H, W, Cin, Cout, R, S, act=SC_ACT_NONE, stream=None) -> int:
    """NCHW conv2d_fwd that allocates no device memory (see the header)."""
    return load().conv2d_fwd_nchw_noalloc(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, H, W, Cin, Cout, R, S,
                                          act, _stream(stream))


def conv2d_chain_fwd_host(x_host, y_host, N, H, W, Cin, layers, stream=None) -> int:
    """Layers run in turn on a host-resident NHWC input, result to host memory.

    x_host / y_host: host tensors (pinned for asynchronous copies) or raw host
    addresses; layers: sequence of (w, b, Cout, R, S, act) with w and b device
    tensors or addresses (b may be None).  See the header."""
    arr = (ScConvLayer * max(len(layers), 1))()
    for i, (w, b, cout, r, s_, act) in enumerate(layers):
        arr[i] = ScConvLayer(_ptr(w), _ptr(b), cout, r, s_, act)
    return load().conv2d_chain_fwd_host(_ptr(x_host), _ptr(y_host), N, H, W, Cin, len(layers),
                                        ctypes.cast(arr, ctypes.c_void_p), _stream(stream))


def sc_empty_kernel(blocks, threads, stream=None) -> int:
    """Launch a kernel that does nothing (launch-cost probe; see the header)."""
    return load().sc_empty_kernel(blocks, threads, _stream(stream))


def sc_test_workspace_allocs() -> int:
    """Temporary device buffers taken by the library so far (test hook; see the header)."""
    return load().sc_test_workspace_allocs()


def sc_test_conv_wait_expiry(x, w, b, y, N, H, W, Cin, Cout, drop_copy, timeout_us, stream=None) -> int:
    return load().sc_test_conv_wait_expiry(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, H, W, Cin, Cout, drop_copy,
                                           timeout_us, _stream(stream))


def sc_test_stencil_wait_expiry(inp, out, H, W, drop_copy, timeout_us, stream=None) -> int:
    """Test hook: the pipeline with one TMA copy never issued (see the header)."""
    return load().sc_test_stencil_wait_expiry(_ptr(inp), _ptr(out), H, W, drop_copy, timeout_us, _stream(stream))


def check(status: int, what: str = "") -> None:
    """Raise StencilConvError for a nonzero status."""
    if status != SC_OK:
        raise StencilConvError(status, what)
