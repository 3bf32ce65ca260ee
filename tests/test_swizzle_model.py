"""The XOR swizzle formula and its stated properties, as a host-side model.

Page "CUDA共有メモリのスウィズリング" (CUDA shared-memory swizzling), sections
"スウィズリングの公式" (formula) and "スウィズリングのプロパティ" (properties):
for ``T array[][NX]`` with ``NX * sizeof(T) == SW`` (a power of two >= 32),
chunks of ``sizeof(TC)`` bytes are permuted inside each SW-byte row by XOR
with the row index.  Properties: (1) the map is a bijection, (2) NX is a power
of two, (3) a column read over 32 consecutive rows hits as many distinct
swizzled positions as possible.  The worked example is in
tests/golden/swizzle_example.txt.
"""
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "swizzle_example.txt")


def swizzle_x(y, x, nx, t_bytes, tc_bytes):
    """Swizzled column of element [y][x] (the page's formula, integer steps)."""
    sw = nx * t_bytes
    i_chunk = (y * nx + x) * t_bytes // tc_bytes
    y_chunk = i_chunk // (sw // tc_bytes)
    x_chunk = i_chunk % (sw // tc_bytes)
    x_chunk_swz = y_chunk ^ x_chunk
    return (x_chunk_swz * tc_bytes // t_bytes) % nx + x % (tc_bytes // t_bytes)


def ways(byte_addrs, width=4, banks=32):
    """Bank-conflict degree of one warp access: the largest number of distinct
    4-byte words any bank must serve (1 = conflict-free)."""
    per_bank = {}
    for a in byte_addrs:
        for wd in range(a // 4, (a + width) // 4):
            per_bank.setdefault(wd % banks, set()).add(wd)
    return max(len(v) for v in per_bank.values())


def _golden():
    d = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            d[k] = int(v)
    return d


@pytest.mark.parametrize("t_bytes,tc_bytes", [(4, 4), (4, 8), (4, 16), (8, 16), (2, 16)])
@pytest.mark.parametrize("sw", [32, 64, 128, 256])
def test_bijection_per_row(t_bytes, tc_bytes, sw):
    nx = sw // t_bytes
    for y in range(64):
        cols = sorted(swizzle_x(y, x, nx, t_bytes, tc_bytes) for x in range(nx))
        assert cols == list(range(nx))


@pytest.mark.parametrize("sw", [32, 64, 128, 256])
def test_column_spread_over_32_rows(sw):
    """Property 3 with TC = T: a column over 32 rows covers min(32, NX) positions."""
    nx = sw // 4
    for x in range(nx):
        for y0 in (0, 5, 32):
            s = {swizzle_x(y, x, nx, 4, 4) for y in range(y0, y0 + 32)}
            assert len(s) == min(32, nx)


def test_page_example_conflict_counts():
    g = _golden()
    rows, nx, t, tc = g["rows"], g["cols"], g["elem_bytes"], g["chunk_bytes"]
    # write: a warp stores one 32-value matrix row = array rows 2k, 2k+1
    for k in range(rows // 2):
        addrs = [((2 * k + l // nx) * nx + swizzle_x(2 * k + l // nx, l % nx, nx, t, tc)) * t
                 for l in range(32)]
        assert ways(addrs) == g["write_ways_swizzled"]
    for x in range(nx):
        sw_read = [(y * nx + swizzle_x(y, x, nx, t, tc)) * t for y in range(rows)]
        plain = [(y * nx + x) * t for y in range(rows)]
        assert ways(sw_read) == g["read_ways_swizzled"]
        assert ways(plain) == g["read_ways_unswizzled"]
