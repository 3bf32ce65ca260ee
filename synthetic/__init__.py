"""Seeded synthetic inputs for the direct-convolution and stencil workloads.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.
It holds no arithmetic of the method itself: it only draws numbers and lays out
the five workload recipes (shapes, value distributions, seeds).

Generator: a counter-based SplitMix64.  Element ``i`` of sub-stream ``k`` under
seed ``s`` is ``mix64(key(s, k) + (i + 1) * GOLDEN)`` where ``mix64`` is the
SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014).  Uniform doubles use the top 53 bits.  Normals use
the Box-Muller transform on the uniform pair (2i, 2i+1) of the stream, in
float64, then everything is rounded to float32 once.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, stream: int) -> np.uint64:
    """Key of sub-stream ``stream`` under ``seed`` (both non-negative ints)."""
    a = _mix64(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
    b = _mix64(np.array([(stream * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
    return np.uint64(a ^ b)


def raw_u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """The ``n`` 64-bit words ``offset .. offset+n-1`` of one sub-stream."""
    key = stream_key(seed, stream)
    i = np.arange(offset, offset + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = key + (i + np.uint64(1)) * GOLDEN
    return _mix64(z)


def uniform01(seed: int, stream: int, n: int) -> np.ndarray:
    """float64 uniforms in [0, 1) from the top 53 bits."""
    return (raw_u64(seed, stream, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform(seed: int, stream: int, shape, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    u = uniform01(seed, stream, n)
    return (lo + (hi - lo) * u).astype(np.float32).reshape(shape)


def normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """Box-Muller normals, one per uniform pair (2i, 2i+1), untruncated."""
    n = int(np.prod(shape)) if len(shape) else 1
    u = uniform01(seed, stream, 2 * n).reshape(n, 2)
    r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
    z = r * np.cos(2.0 * math.pi * u[:, 1])
    return (std * z).astype(np.float32).reshape(shape)


# --------------------------------------------------------------------------
# Workload recipes.  Activations are generated in NCHW order (the planar
# order of a per-channel image); callers that want NHWC transpose them.
# Weights are OIHW.  Sub-stream ids: x = 0, w = 1, b = 2, plus 16 * layer.
# --------------------------------------------------------------------------


@dataclasses.dataclass
class ConvLayer:
    cin: int
    cout: int
    r: int
    s: int
    act: int          # 0 = none, 1 = ReLU
    w: np.ndarray     # float32 [cout][cin][r][s]
    b: np.ndarray     # float32 [cout]

    @property
    def flops_per_px(self) -> int:
        return 2 * self.cin * self.cout * self.r * self.s


@dataclasses.dataclass
class ConvWorkload:
    name: str
    n: int
    h: int
    w: int
    x: np.ndarray              # float32 NCHW input of layer 0
    layers: List[ConvLayer]

    def flops(self) -> int:
        return sum(self.n * self.h * self.w * L.flops_per_px for L in self.layers)


@dataclasses.dataclass
class PipelineWorkload:
    name: str
    h: int
    w: int
    img: np.ndarray            # float32 [h][w]


def _he_std(fan_in: int) -> float:
    return math.sqrt(2.0 / fan_in)


def config(cid: int, seed: Optional[int] = None, scale: Optional[Dict[str, int]] = None):
    """Build workload ``cid`` (1..5) with seed ``1000 + cid`` unless given.

    ``scale`` may override spatial sizes or batch (keys ``n``, ``h``, ``w``)
    to make a smaller case of the same recipe for quick tests.
    """
    seed = 1000 + cid if seed is None else seed
    sc = scale or {}
    if cid == 1:
        n, h, w = sc.get("n", 1), sc.get("h", 64), sc.get("w", 64)
        x = uniform(seed, 0, (n, 1, h, w), -1.0, 1.0)
        wt = uniform(seed, 1, (1, 1, 3, 3), -1.0, 1.0)
        b = np.full((1,), 0.1, dtype=np.float32)
        return ConvWorkload("single-channel 3x3, 64x64", n, h, w, x, [ConvLayer(1, 1, 3, 3, 0, wt, b)])
    if cid == 2:
        n, h, w = sc.get("n", 1), sc.get("h", 128), sc.get("w", 128)
        x = uniform(seed, 0, (n, 16, h, w), -1.0, 1.0)
        wt = normal(seed, 1, (16, 16, 3, 3), math.sqrt(2.0 / (9 * 16)))
        b = uniform(seed, 2, (16,), -0.1, 0.1)
        return ConvWorkload("16->16 3x3, 128x128", n, h, w, x, [ConvLayer(16, 16, 3, 3, 1, wt, b)])
    if cid == 3:
        n, h, w = sc.get("n", 1), sc.get("h", 720), sc.get("w", 1280)
        x = uniform(seed, 0, (n, 1, h, w), 0.0, 1.0)
        specs = [(1, 32, 5, 1), (32, 32, 3, 1), (32, 4, 3, 0)]
        layers = []
        for li, (ci, co, k, act) in enumerate(specs):
            wt = normal(seed, 16 * li + 1, (co, ci, k, k), _he_std(ci * k * k))
            b = uniform(seed, 16 * li + 2, (co,), -0.05, 0.05)
            layers.append(ConvLayer(ci, co, k, k, act, wt, b))
        return ConvWorkload("3-layer upscaling net, 1280x720", n, h, w, x, layers)
    if cid == 4:
        n, h, w = sc.get("n", 32), sc.get("h", 56), sc.get("w", 56)
        x = np.maximum(normal(seed, 0, (n, 64, h, w), 1.0), np.float32(0.0))
        wt = normal(seed, 1, (64, 64, 3, 3), math.sqrt(2.0 / (9 * 64)))
        b = np.zeros((64,), dtype=np.float32)
        return ConvWorkload("wide layer 64->64 3x3, N=32 56x56", n, h, w, x, [ConvLayer(64, 64, 3, 3, 1, wt, b)])
    if cid == 5:
        h, w = sc.get("h", 4096), sc.get("w", 4096)
        img = uniform(seed, 0, (h, w), 0.0, 1.0)
        return PipelineWorkload("fused blur/unsharp pipeline, 4096x4096", h, w, img)
    raise ValueError(f"unknown workload id {cid}")


def conv_case(seed: int, n: int, cin: int, cout: int, h: int, w: int, r: int, s: int,
              act: int = 1, xlo: float = -1.0, xhi: float = 1.0) -> ConvWorkload:
    """A generic random single-layer case (used for odd shapes in tests)."""
    x = uniform(seed, 0, (n, cin, h, w), xlo, xhi)
    wt = normal(seed, 1, (cout, cin, r, s), math.sqrt(2.0 / (cin * r * s)))
    b = uniform(seed, 2, (cout,), -0.1, 0.1)
    return ConvWorkload(f"case {n}x{cin}x{h}x{w}->{cout} {r}x{s}", n, h, w, x,
                        [ConvLayer(cin, cout, r, s, act, wt, b)])

