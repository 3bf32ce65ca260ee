"""Oracle: plain fp64 CPU definitions of the convolution and stencil pipeline.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``stencil_conv2d_fwd_gb300``) never does, and shares no code with it.

``oracle.c`` holds the definitions; this module builds it with gcc (no CUDA),
loads it through ctypes and marshals numpy arrays.  Each wrapper states the
definition it calls; the C file cites the page section it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``src`` (default oracle.c) into a shared library (gcc -O2, OpenMP)."""
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_set_threads.argtypes = [i]
    lib.oracle_set_threads.restype = i
    lib.oracle_conv2d_nchw.argtypes = [dp, dp, dp, i, i, i, i, i, i, i, i, i, i, dp, dp]
    lib.oracle_conv2d_nchw.restype = i
    lib.oracle_conv2d_points.argtypes = [dp, dp, dp, i, i, i, i, i, i, i, i, ctypes.c_long, dp, dp, dp]
    lib.oracle_conv2d_points.restype = i
    lib.oracle_repack.argtypes = [dp, dp, i, i, i, i, i]
    lib.oracle_repack.restype = i
    lib.oracle_stencil_pipeline.argtypes = [dp, i, i, i, i, dp, dp]
    lib.oracle_stencil_pipeline.restype = i
    return lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


class Oracle:
    """The oracle's definitions bound to one build of oracle.c."""

    def __init__(self, path: Optional[str] = None):
        self.path = path or build()
        self._lib = _bind(self.path)

    def set_threads(self, n: int) -> int:
        """Set the OpenMP thread count (n <= 0: keep default); returns the count in use."""
        return int(self._lib.oracle_set_threads(int(n)))

    def conv2d_nchw(self, x, w, b, act: int, rows: Optional[Tuple[int, int]] = None,
                    with_scale: bool = True):
        """y = act(conv(x, w) + b), zero 'same' padding, stride 1, fp64.

        x: float32 [N][Cin][H][W]; w: float32 [Cout][Cin][R][S]; b: [Cout] or None.
        Returns (y, scale) as float64 [N][Cout][rows][W]; scale = sum|x*w| + |b|.
        """
        x, w = _f32(x), _f32(w)
        b = None if b is None else _f32(b)
        N, Cin, H, W = x.shape
        Cout, Cin2, R, S = w.shape
        assert Cin2 == Cin
        h0, h1 = rows if rows is not None else (0, H)
        y = np.empty((N, Cout, h1 - h0, W), dtype=np.float64)
        a = np.empty_like(y) if with_scale else None
        rc = self._lib.oracle_conv2d_nchw(_p(x), _p(w), _p(b), N, Cin, H, W, Cout, R, S, int(act),
                                        h0, h1, _p(y), _p(a))
        if rc != 0:
            raise ValueError("oracle_conv2d_nchw rejected its arguments")
        return y, a

    def conv2d_points(self, x, w, b, act: int, pts: np.ndarray):
        """The same definition at sampled (n, co, h, w) points (int32 [P][4])."""
        x, w = _f32(x), _f32(w)
        b = None if b is None else _f32(b)
        N, Cin, H, W = x.shape
        Cout, _, R, S = w.shape
        pts = np.ascontiguousarray(pts, dtype=np.int32)
        P = pts.shape[0]
        y = np.empty((P,), dtype=np.float64)
        a = np.empty((P,), dtype=np.float64)
        rc = self._lib.oracle_conv2d_points(_p(x), _p(w), _p(b), N, Cin, H, W, Cout, R, S, int(act),
                                          P, _p(pts), _p(y), _p(a))
        if rc != 0:
            raise ValueError("oracle_conv2d_points rejected its arguments")
        return y, a

    def repack(self, src, N: int, C: int, H: int, W: int, to_nhwc: bool) -> np.ndarray:
        """NCHW -> NHWC (to_nhwc) or NHWC -> NCHW, by the index definition."""
        src = _f32(src).reshape(-1)
        dst = np.empty_like(src)
        rc = self._lib.oracle_repack(_p(src), _p(dst), N, C, H, W, 1 if to_nhwc else 0)
        if rc != 0:
            raise ValueError("oracle_repack rejected its arguments")
        return dst.reshape((N, H, W, C) if to_nhwc else (N, C, H, W))

    def stencil_pipeline(self, img, rows: Optional[Tuple[int, int]] = None, with_t2: bool = False):
        """out = clamp(in + 1.5 (in - vblur5(hblur5(in))), 0, 1), clamp-to-edge, fp64."""
        img = _f32(img)
        H, W = img.shape
        r0, r1 = rows if rows is not None else (0, H)
        out = np.empty((r1 - r0, W), dtype=np.float64)
        t2 = np.empty_like(out) if with_t2 else None
        rc = self._lib.oracle_stencil_pipeline(_p(img), H, W, r0, r1, _p(out), _p(t2))
        if rc != 0:
            raise ValueError("oracle_stencil_pipeline rejected its arguments")
        return (out, t2) if with_t2 else out


_default: Optional[Oracle] = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def set_threads(n: int) -> int:
    return default().set_threads(n)


def conv2d_nchw(*a, **k):
    return default().conv2d_nchw(*a, **k)


def conv2d_points(*a, **k):
    return default().conv2d_points(*a, **k)


def repack(*a, **k):
    return default().repack(*a, **k)


def stencil_pipeline(*a, **k):
    return default().stencil_pipeline(*a, **k)
