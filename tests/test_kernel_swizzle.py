"""Shared-memory layouts of the CUDA kernels: the XOR swizzle they use is a
bijection, and the warps' access patterns are bank-conflict-free.

The swizzle functions are compiled from the kernels' own header
(stencil_conv2d_fwd_gb300/csrc/common.cuh) as host C++, so this checks the
code the kernels run.  The per-lane address patterns restate the thread ->
pixel maps of conv_general.cuh and repack.cu.  Properties follow "CUDA共有
メモリのスウィズリング" (section "スウィズリングのプロパティ"): one-to-one, and as
many distinct banks as possible for the warp's access.
"""
import ctypes
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "stencil_conv2d_fwd_gb300", "csrc", "common.cuh")


@pytest.fixture(scope="module")
def swz(tmp_path_factory):
    d = tmp_path_factory.mktemp("swz")
    src = d / "swz.cpp"
    src.write_text(f'#include "{HDR}"\n'
                   'extern "C" int h_swz16(int i, int L) { return sc::swz16(i, L); }\n'
                   'extern "C" int h_swz_col(int r, int c, int L) { return sc::swz_col(r, c, L); }\n'
                   'extern "C" int h_tma_key(int p, int c) { return sc::tma_swz_key(p, c); }\n'
                   'extern "C" int h_c1_band_chunk(int L) { return sc::c1_band_chunk(L); }\n'
                   'extern "C" int h_small_tile_chunk(int p, int cb) { return sc::small_tile_chunk(p, cb); }\n')
    so = d / "libswz.so"
    subprocess.run(["g++", "-std=c++17", "-O1", "-fPIC", "-shared", str(src), "-o", str(so)], check=True)
    lib = ctypes.CDLL(str(so))
    lib.h_swz16.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.h_swz_col.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.h_tma_key.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.h_c1_band_chunk.argtypes = [ctypes.c_int]
    lib.h_small_tile_chunk.argtypes = [ctypes.c_int, ctypes.c_int]
    return lib


def phase_wavefronts(chunks):
    """Wavefronts for one group of lanes served together: its distinct 16-byte
    chunks take one wavefront per chunk that shares a bank group (chunk mod
    8) with another."""
    per_pos = {}
    for c in set(chunks):
        per_pos[c % 8] = per_pos.get(c % 8, 0) + 1
    return max(per_pos.values())


def wavefronts_128bit(chunks_by_lane, ideal=False):
    """Shared-memory wavefronts of one warp-wide 16-byte load on GB300, as
    measured with ncu (l1tex__data_pipe_lsu_wavefronts_mem_shared_op_ld) on
    probe kernels of fixed lane -> chunk patterns: when no quarter-warp (8
    consecutive lanes) asks for more than 2 distinct chunks, each half-warp
    is served in one wavefront (2 in all, also for a pure broadcast);
    otherwise each quarter-warp takes its own (4 in all).  A bank-group
    clash inside the group served together adds wavefronts (ideal=True
    leaves them out)."""
    assert len(chunks_by_lane) == 32
    quarters = [chunks_by_lane[q:q + 8] for q in range(0, 32, 8)]
    if all(len(set(q)) <= 2 for q in quarters):
        groups = [chunks_by_lane[:16], chunks_by_lane[16:]]
    else:
        groups = quarters
    return sum(1 if ideal else phase_wavefronts(g) for g in groups)


def conflict_free_128bit(chunks_by_lane):
    return wavefronts_128bit(chunks_by_lane) == wavefronts_128bit(chunks_by_lane, ideal=True)


def min_wavefronts_128bit(chunks):
    return -(-len(set(chunks)) // 8)


def phases_conflict_free(chunks_by_lane):
    """A 16-byte shared access is served 8 lanes at a time: in each group of 8
    consecutive lanes, distinct chunks must sit in distinct bank groups."""
    for q in range(0, len(chunks_by_lane), 8):
        if phase_wavefronts(chunks_by_lane[q:q + 8]) != 1:
            return False
    return True


@pytest.mark.parametrize("pattern,want", [
    (lambda l: l, 4),                      # 32 distinct contiguous chunks
    (lambda l: 0, 2),                      # one chunk for the whole warp
    (lambda l: l & 3, 4),                  # 4 chunks, lanes interleaved
    (lambda l: l >> 3, 2),                 # one chunk per quarter-warp
    (lambda l: 2 * (l >> 2), 2),           # 8 chunks 2 apart, 4 lanes each
    (lambda l: l >> 2, 2),                 # 8 contiguous chunks, 4 lanes each
    (lambda l: l & 7, 4),                  # 8 contiguous chunks, interleaved
    (lambda l: (l & 3) + 4 * (l >> 4), 4),
    (lambda l: 4 * (l & 1), 2),
    (lambda l: l >> 4, 2),
])
def test_wavefront_model_reproduces_the_measured_probe_counts(pattern, want):
    """The probe kernels' measured wavefronts per load (no bank conflicts in
    any of them)."""
    chunks = [pattern(l) for l in range(32)]
    assert wavefronts_128bit(chunks) == want
    assert conflict_free_128bit(chunks)


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5])
def test_swz16_is_a_bijection_per_row(swz, L):
    n = 1 << L
    for base in range(0, 64 * n, n):
        got = sorted(swz.h_swz16(base + k, L) for k in range(n))
        assert got == list(range(base, base + n))


def test_swz16_matches_the_page_formula(swz):
    """16-byte chunks, 128-byte swizzle rows (T = TC = 16 B, NX = 8):
    x_swz = (y_chunk XOR x_chunk) mod 8 with y_chunk = i / 8, x_chunk = i mod 8."""
    for i in range(4096):
        y, x = divmod(i, 8)
        assert swz.h_swz16(i, 3) == y * 8 + ((y ^ x) % 8)


# (F_TB, W_T, TH, TW, C_SH): the tiles of dispatch_wide / dispatch_narrow
# (C_SH 16 is used for 3x3 with Cin % 16 == 0; 7x7 uses 4)
GEN_TABLE = [(64, 8, 8, 32, 8), (64, 7, 8, 28, 8), (32, 8, 8, 64, 8), (32, 7, 8, 56, 8),
             (64, 8, 8, 32, 16), (64, 7, 8, 28, 16), (32, 8, 8, 64, 16), (32, 7, 8, 56, 16),
             (16, 4, 4, 64, 8), (8, 4, 4, 128, 8), (4, 4, 4, 128, 8)]


def gen_cfg(K, F_TB, W_T, TH, TW, C_SH):
    F_T = 8 if F_TB >= 8 else 4
    T_X = F_TB // F_T
    PXL = 32 // T_X
    WARP_COLS = PXL * W_T
    if K >= 7:
        C_SH = 4
    TWU = TW + K - 1
    return dict(F_T=F_T, T_X=T_X, PXL=PXL, WARP_COLS=WARP_COLS, WPR=TW // WARP_COLS,
                NT=(TW // WARP_COLS) * TH * 32, TWU=TWU, TWP=(TWU + 7) // 8 * 8, CB=C_SH // 4,
                THh=TH + K - 1,
                PLANE=(TH + K - 1) * ((TWU + 7) // 8 * 8) + (1 if C_SH >= 32 else 8 // (C_SH // 4)))


def col_map(swz, W_T, col):
    """phys_col<C>: XOR with the low bits of the 8-chunk group index, as many
    bits as the lane stride W_T needs (GenCfg::SWZ_MASK)."""
    m = 7 if W_T % 8 == 0 else 3 if W_T % 4 == 0 else 1 if W_T % 2 == 0 else 0
    return (col & ~7) | ((col ^ ((col >> 3) & m)) & 7)


@pytest.mark.parametrize("K", [1, 3, 5, 7])
@pytest.mark.parametrize("F_TB,W_T,TH,TW,C_SH", GEN_TABLE)
def test_general_conv_pixel_reads_conflict_free(swz, K, F_TB, W_T, TH, TW, C_SH):
    c = gen_cfg(K, F_TB, W_T, TH, TW, C_SH)
    for warp in range(c["NT"] // 32):
        ry = warp // c["WPR"]
        for cb in range(c["CB"]):
            for r in range(K):
                for j in range(W_T + K - 1):
                    chunks = []
                    for lane in range(32):
                        pl = lane // c["T_X"]
                        cx0 = (warp % c["WPR"]) * c["WARP_COLS"] + pl * W_T
                        chunks.append(cb * c["PLANE"] + (ry + r) * c["TWP"] + col_map(swz, W_T, cx0 + j))
                    assert conflict_free_128bit(chunks), (warp, cb, r, j)
                    assert phases_conflict_free(chunks), (warp, cb, r, j)


@pytest.mark.parametrize("K", [1, 3, 5, 7])
@pytest.mark.parametrize("F_TB,W_T,TH,TW,C_SH", GEN_TABLE)
def test_general_conv_tile_writes_stay_in_tile_and_are_one_to_one(swz, K, F_TB, W_T, TH, TW, C_SH):
    c = gen_cfg(K, F_TB, W_T, TH, TW, C_SH)
    # gen_issue_tile: a warp copies a tile row; lanes over (column, channel block), block fastest
    phys = []
    for yy in range(c["THh"]):
        qs = list(range(c["TWU"] * c["CB"]))
        for it in range(0, len(qs), 32):
            chunks = []
            for q in qs[it:it + 32]:
                cb, xx = q % c["CB"], q // c["CB"]
                chunks.append(cb * c["PLANE"] + yy * c["TWP"] + col_map(swz, W_T, xx))
            # one warp instruction: conflict-free when all 32 lanes copy, and in
            # every 8-lane phase; the partial last instruction of a row may take
            # one extra wavefront
            if len(chunks) == 32:
                assert conflict_free_128bit(chunks)
                assert phases_conflict_free(chunks)
            else:
                assert phase_wavefronts(chunks) <= min_wavefronts_128bit(chunks) + 1
            phys += chunks
    assert len(set(phys)) == len(phys) == c["CB"] * c["THh"] * c["TWU"]   # one-to-one
    assert max(phys) < (c["CB"] * c["PLANE"] + 7) // 8 * 8                 # inside the stage's tile


def test_odd_stride_needs_no_swizzle_and_xor_would_hurt(swz):
    """W_T = 7: plain columns 7k are in 8 different bank groups; XORed ones are not."""
    plain = [7 * k for k in range(8)]
    assert phase_wavefronts(plain) == 1
    assert phase_wavefronts([swz.h_swz16(cc, 3) for cc in plain]) > 1


def test_general_conv_unswizzled_pixel_reads_would_conflict():
    """Without the XOR the same warp read puts its pixel lanes W_T chunks apart,
    so (for W_T = 8) every lane lands on the same bank window position."""
    W_T, PXL = 8, 4
    chunks = [pl * W_T for pl in range(PXL) for _ in range(8)]
    assert phase_wavefronts(chunks) == PXL > min_wavefronts_128bit(chunks)


def bank_ways_32bit(word_addrs):
    per = {}
    for a in set(word_addrs):
        per[a % 32] = per.get(a % 32, 0) + 1
    return max(per.values())


def test_transpose_tile_conflict_free(swz):
    for ra in range(32):  # row write: lanes along the tile row
        words = [ra * 32 + swz.h_swz_col(ra, tx, 5) for tx in range(32)]
        assert bank_ways_32bit(words) == 1
    for rb in range(32):  # swizzled column read: lane = tile row
        words = [tx * 32 + swz.h_swz_col(tx, rb, 5) for tx in range(32)]
        assert bank_ways_32bit(words) == 1
        plain = [tx * 32 + rb for tx in range(32)]
        assert bank_ways_32bit(plain) == 32


# ---------------------------------------------------------------------------
# conv_tma.cuh: stages written by TMA copies with the swizzle of the staged
# pixel's span (32, 64 or 128 bytes).  The copy XORs the 16-byte chunk bits
# (4 and up) of each shared-memory address with the bits 7 and up, as many as
# the span has chunk bits; stage rows are a multiple of 8 pixels and stages
# are 1024-byte aligned.

def tma_swizzled_byte(addr, span):
    """Where a swizzled TMA copy puts the byte that an unswizzled copy would
    put at `addr` (relative to a 1024-byte-aligned stage)."""
    mask = span // 16 - 1
    return addr ^ (((addr >> 7) & mask) << 4)


@pytest.mark.parametrize("c_sh", [8, 16, 32])
def test_tma_key_is_the_copy_swizzle(swz, c_sh):
    span = 4 * c_sh
    for row_pitch_px in (8, 16, 104, 168):            # stage rows: multiples of 8 pixels
        for row in range(3):
            for p in range(row_pitch_px):
                base = (row * row_pitch_px + p) * span
                for q in range(span // 16):
                    want = tma_swizzled_byte(base + 16 * q, span)
                    got = base + 16 * (q ^ swz.h_tma_key(p, c_sh))
                    assert got == want


# (F_TB, W_T, C_SH): the configurations conv_tma_k3.cu instantiates
TMA_CFGS = [(4, 5, 8), (4, 3, 8), (8, 5, 8), (16, 5, 8), (32, 7, 8), (32, 5, 8), (64, 7, 8), (4, 5, 16)]


@pytest.mark.parametrize("cfg", TMA_CFGS, ids=[f"F{a}_W{b}_C{c}" for a, b, c in TMA_CFGS])
def test_tma_stage_pixel_reads_conflict_free(swz, cfg):
    """conv_tma_kernel's pixel loads: lane -> (tx = lane % T_X, pixel lane
    pl = lane / T_X), pixel pl * W_T + j of a tile row, 16-byte chunk cb.
    Every 8-lane phase reads distinct chunks in distinct bank groups, and a
    pixel's chunks are a permutation of its span."""
    F_TB, W_T, C_SH = cfg
    F_T = 8 if F_TB >= 8 else 4
    T_X = F_TB // F_T
    CB, PXB = C_SH // 4, 4 * C_SH
    for j in range(W_T + 6):   # the window of up to 7 x 7 filters
        for cb in range(CB):
            chunks = []
            for lane in range(32):
                p = (lane // T_X) * W_T + j
                chunks.append((p * PXB + 16 * (cb ^ swz.h_tma_key(p, C_SH))) // 16)
            assert phases_conflict_free(chunks)
    for p in range(64):
        assert sorted(cb ^ swz.h_tma_key(p, C_SH) for cb in range(CB)) == list(range(CB))


def test_tma_even_pixel_run_would_conflict(swz):
    """With an even run (W_T = 4) the lanes of a phase read pixels 4 apart,
    which the swizzle cannot separate: the kernel uses odd runs."""
    chunks = [((lane * 4) * 32 + 16 * (0 ^ swz.h_tma_key(lane * 4, 8))) // 16 for lane in range(32)]
    assert not phases_conflict_free(chunks)


# ---------------------------------------------------------------------------
# conv_c1.cu, conv_c1_tile_kernel: lane = 8 * cl + pl (4 channel lanes, one
# per quarter-warp; 8 pixel lanes), 8 pixels 8 * pl + j and 8 output channels
# per thread, staged input rows of 66 16-byte chunks, one 8 KB output buffer
# per warp.

def _c1_lane(lane):
    return lane >> 3, lane & 7          # (cl, pl)


@pytest.mark.parametrize("warp", range(4))
@pytest.mark.parametrize("row", range(3))
def test_c1_tile_band_reads_conflict_free(swz, warp, row):
    """Window chunk q (0..3) of row `row`: logical chunk 16 warp + 2 pl + q,
    stored at c1_band_chunk of it; each quarter-warp asks for its 8 pixel
    lanes' chunks in 8 distinct bank groups."""
    for q in range(4):
        chunks = []
        for lane in range(32):
            cl, pl = _c1_lane(lane)
            chunks.append(66 * row + swz.h_c1_band_chunk(16 * warp + 2 * pl + q))
        assert conflict_free_128bit(chunks), q
        assert wavefronts_128bit(chunks) == 4


def test_c1_tile_band_unswizzled_reads_would_conflict():
    chunks = [2 * _c1_lane(l)[1] for l in range(32)]
    assert not conflict_free_128bit(chunks)


def test_c1_band_chunk_is_one_to_one_on_a_row(swz):
    assert sorted(swz.h_c1_band_chunk(L) for L in range(66)) == list(range(66))


def test_c1_tile_filter_reads_take_two_wavefronts():
    """Filter unit 4 g + cl of a tap: one chunk per quarter-warp.  With the
    channel lane in the low lane bits (cl = lane & 3) every quarter-warp
    would ask for 4 chunks: 4 wavefronts instead of 2."""
    for g in range(2):
        assert wavefronts_128bit([4 * g + _c1_lane(l)[0] for l in range(32)]) == 2
        assert wavefronts_128bit([4 * g + (l & 3) for l in range(32)]) == 4


def _c1_tile_store_chunks(j, g):
    """16-byte chunk of the warp's output buffer that each lane writes at
    step (g, j): pixel 8 pl + j sits in 128-byte row 8 j + pl, its chunk
    q = 4 g + cl at q ^ pl."""
    return [(8 * j + pl) * 8 + ((4 * g + cl) ^ pl) for cl, pl in map(_c1_lane, range(32))]


def test_c1_tile_output_writes_conflict_free_and_one_to_one():
    seen = []
    for g in range(2):
        for j in range(8):
            ch = _c1_tile_store_chunks(j, g)
            assert phases_conflict_free(ch), (g, j)
            seen += ch
    assert sorted(seen) == list(range(64 * 8))


def test_c1_tile_output_buffer_is_the_store_copy_box():
    """The output copy's box is (32 channels, 8 pixel groups, 8 pixels of a
    group), walked channel fastest, then group, then pixel: pixel 8 g + j is
    128-byte row g + 8 j, and the 128-byte TMA swizzle moves its chunk q to
    q ^ (row mod 8) = q ^ g, where the lanes wrote it (g = pl)."""
    for g in range(8):
        for j in range(8):
            row = g + 8 * j
            for q in range(8):
                want = tma_swizzled_byte(row * 128 + 16 * q, 128)
                assert want == row * 128 + 16 * (q ^ g)


# ---------------------------------------------------------------------------
# conv_small.cu, conv_small_kernel: lane = 8 c + q (output-channel quad c, one
# per quarter-warp; pixel run q of 8 pixels), a staged tile row of 66 pixels x
# 4 chunks of 4 channels, filters [ci][tap][16 outputs], exchanged partial
# sums as float4 [row][owner][slot][pair][lane].

def test_small_tile_chunk_is_one_to_one_on_a_row(swz):
    got = sorted(swz.h_small_tile_chunk(p, cb) for p in range(66) for cb in range(4))
    assert got == list(range(264))


@pytest.mark.parametrize("k", range(10))
@pytest.mark.parametrize("grp", range(4))
def test_small_tile_pixel_reads_conflict_free(swz, k, grp):
    """Staged pixel 8 q + k, chunk grp: eight distinct chunks per quarter-warp
    (the four quarter-warps ask for the same eight), in eight bank groups."""
    chunks = [swz.h_small_tile_chunk(8 * (l & 7) + k, grp) for l in range(32)]
    assert conflict_free_128bit(chunks)
    assert wavefronts_128bit(chunks) == 4


def test_small_tile_unswizzled_pixel_reads_would_conflict():
    chunks = [4 * (8 * (l & 7)) for l in range(32)]
    assert wavefronts_128bit(chunks) == 32


def test_small_filter_and_partial_sum_accesses():
    """Filter chunk ((ci 9 + tap) 20 + 4 c) / 4: one chunk per quarter-warp,
    two wavefronts; partial-sum chunk (slot index) 32 + lane: 32 contiguous
    chunks; filter staging stores element e = co 9 Cin + k of the OIHW bank
    to word k 20 + co, lanes along e: at most 4 lanes of a warp per bank."""
    for ci in range(16):
        for tap in range(9):
            chunks = [((ci * 9 + tap) * 20 + 4 * (l >> 3)) // 4 for l in range(32)]
            assert wavefronts_128bit(chunks) == 2 and conflict_free_128bit(chunks)
    for f in range(4):
        chunks = [f * 32 + l for l in range(32)]
        assert phases_conflict_free(chunks) and wavefronts_128bit(chunks) == 4
    for cin in (4, 8, 12, 16):
        KK = 9 * cin
        for warp in range(0, 16 * KK // 32 + 1):
            es = [e for e in range(32 * warp, 32 * warp + 32) if e < 16 * KK]
            if not es:
                continue
            banks = [((e % KK) * 20 + e // KK) % 32 for e in es]
            assert max(banks.count(bk) for bk in set(banks)) <= 4


# ---------------------------------------------------------------------------
# conv_tc.cu: the tensor core reads a K step of A as a 32-byte slice of 8
# consecutive padded-pixel rows.  With the row width equal to the TMA swizzle
# span (TF32: 128-byte rows, 128-byte swizzle; BF16: 64-byte rows, 64-byte
# swizzle), the 16 chunks of a slice fall on every 16-byte bank group exactly
# twice, for every K step and any 8-row-aligned start.

@pytest.mark.parametrize("rowb", [128, 64, 32])
def test_tensor_core_k_slices_spread_over_all_bank_groups(rowb):
    for k in range(rowb // 32):                 # K steps within a row
        for r0 in range(0, 64, 8):
            groups = []
            for r in range(r0, r0 + 8):
                for c in range(2):
                    byte = tma_swizzled_byte(r * rowb + 32 * k + 16 * c, rowb)
                    groups.append((byte // 16) % 8)
            assert sorted(groups) == sorted(list(range(8)) * 2), (rowb, k, r0)
