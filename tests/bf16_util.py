"""bf16 storage helpers for the tests (host side, numpy): rounding an fp32
array to bf16 bit patterns (round to nearest, ties to even, as the
conversion the kernels use) and widening bf16 bits back to fp32 (exact)."""
import numpy as np


def to_bf16_bits(a) -> np.ndarray:
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_to_bf16(a) -> np.ndarray:
    """fp32 values exactly representable in bf16 (the nearest, ties to even)."""
    return bf16_bits_to_f32(to_bf16_bits(a)).reshape(np.shape(a))
