"""The C-ABI library loads, exports every symbol include/*.h declares, and
rejects bad arguments on the host before any CUDA work (no GPU needed: the
pointers below are never dereferenced)."""
import glob
import os
import re

import pytest

import stencil_conv2d_fwd_gb300 as sc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M):
            if not m.group(0).lstrip().startswith(("typedef", "struct", "#")):
                names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("conv2d_fwd", "stencil_pipeline_fwd", "sc_repack", "sc_last_device_status",
                     "sc_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = sc.load()
    names = declared_functions()
    assert names, "no declarations found"
    for n in sorted(names):
        assert hasattr(lib, n), f"libstencilconv.so does not export {n}"
    assert names <= set(sc.SIGNATURES), "binding lacks a declared function"


def test_status_strings():
    for code in range(-7, 1):
        s = sc.sc_status_string(code)
        assert s and s != "unknown status"
    assert sc.sc_status_string(-99) == "unknown status"


A16 = 1 << 20   # fake, 16-byte aligned addresses: validation only, never dereferenced
B16 = 1 << 24


@pytest.mark.parametrize("args,expect", [
    (dict(x=None), sc.SC_ERR_NULL),
    (dict(w=None), sc.SC_ERR_NULL),
    (dict(y=None), sc.SC_ERR_NULL),
    (dict(N=0), sc.SC_ERR_SHAPE),
    (dict(H=-1), sc.SC_ERR_SHAPE),
    (dict(Cout=0), sc.SC_ERR_SHAPE),
    (dict(R=2), sc.SC_ERR_UNSUPPORTED),
    (dict(S=4), sc.SC_ERR_UNSUPPORTED),
    (dict(R=9, S=9), sc.SC_ERR_UNSUPPORTED),
    (dict(layout=2), sc.SC_ERR_UNSUPPORTED),
    (dict(act=3), sc.SC_ERR_UNSUPPORTED),
    (dict(Cin=6), sc.SC_ERR_UNSUPPORTED),
    (dict(Cout=6), sc.SC_ERR_UNSUPPORTED),
    (dict(Cin=1, Cout=6), sc.SC_ERR_UNSUPPORTED),
    (dict(x=A16 + 4), sc.SC_ERR_ALIGN),
    (dict(y=B16 + 8), sc.SC_ERR_ALIGN),
    (dict(y=A16), sc.SC_ERR_ALIAS),
    (dict(y=A16 + 64), sc.SC_ERR_ALIAS),
    (dict(w=B16 + 128), sc.SC_ERR_ALIAS),
    (dict(b=B16), sc.SC_ERR_ALIAS),
])
def test_conv_argument_errors(args, expect):
    a = dict(x=A16, w=1 << 28, b=None, y=B16, N=1, H=8, W=8, Cin=4, Cout=4, R=3, S=3,
             layout=sc.SC_NHWC, act=0)
    a.update(args)
    rc = sc.conv2d_fwd(a["x"], a["w"], a["b"], a["y"], a["N"], a["H"], a["W"], a["Cin"], a["Cout"],
                       a["R"], a["S"], a["layout"], a["act"], stream=0)
    assert rc == expect, sc.sc_status_string(rc)


@pytest.mark.parametrize("args,expect", [
    (dict(x=None), sc.SC_ERR_NULL),
    (dict(y=None), sc.SC_ERR_NULL),
    (dict(N=0), sc.SC_ERR_SHAPE),
    (dict(W=-3), sc.SC_ERR_SHAPE),
    (dict(R=2), sc.SC_ERR_UNSUPPORTED),
    (dict(R=9, S=9), sc.SC_ERR_UNSUPPORTED),
    (dict(act=3), sc.SC_ERR_UNSUPPORTED),
    (dict(Cin=6), sc.SC_ERR_UNSUPPORTED),
    (dict(Cin=1, Cout=6), sc.SC_ERR_UNSUPPORTED),
    (dict(x=A16 + 4), sc.SC_ERR_ALIGN),
    (dict(y=B16 + 8), sc.SC_ERR_ALIGN),
    (dict(y=A16 + 64), sc.SC_ERR_ALIAS),
    (dict(b=B16), sc.SC_ERR_ALIAS),
])
def test_noalloc_entry_point_rejects_what_conv2d_fwd_rejects(args, expect):
    """conv2d_fwd_nchw_noalloc promises conv2d_fwd's (NCHW) argument rules and status codes."""
    a = dict(x=A16, w=1 << 28, b=None, y=B16, N=1, H=8, W=8, Cin=4, Cout=4, R=3, S=3, act=0)
    a.update(args)
    rc_ref = sc.conv2d_fwd(a["x"], a["w"], a["b"], a["y"], a["N"], a["H"], a["W"], a["Cin"], a["Cout"],
                           a["R"], a["S"], sc.SC_NCHW, a["act"], stream=0)
    rc = sc.conv2d_fwd_nchw_noalloc(a["x"], a["w"], a["b"], a["y"], a["N"], a["H"], a["W"], a["Cin"],
                                    a["Cout"], a["R"], a["S"], a["act"], stream=0)
    assert rc == rc_ref == expect, sc.sc_status_string(rc)


def test_size_overflow_is_a_shape_error():
    rc = sc.conv2d_fwd(A16, 1 << 28, None, B16, 1 << 30, 1 << 30, 1 << 30, 4, 4, 3, 3, 1, 0, stream=0)
    assert rc == sc.SC_ERR_SHAPE


def test_pipeline_and_repack_argument_errors():
    assert sc.stencil_pipeline_fwd(None, B16, 4, 4, stream=0) == sc.SC_ERR_NULL
    assert sc.stencil_pipeline_fwd(A16, B16, 0, 4, stream=0) == sc.SC_ERR_SHAPE
    assert sc.stencil_pipeline_fwd(A16, A16 + 4, 4, 4, stream=0) == sc.SC_ERR_ALIAS
    assert sc.sc_repack(None, B16, 1, 4, 2, 2, 0, 1, stream=0) == sc.SC_ERR_NULL
    assert sc.sc_repack(A16, B16, 1, 4, 2, 2, 0, 5, stream=0) == sc.SC_ERR_UNSUPPORTED
    assert sc.sc_repack(A16, A16 + 16, 1, 4, 2, 2, 0, 1, stream=0) == sc.SC_ERR_ALIAS
    assert sc.sc_measure_ffma_peak(None, 1, 1, stream=0) == sc.SC_ERR_NULL
    assert sc.sc_measure_ffma_peak(A16, 0, 1, stream=0) == sc.SC_ERR_SHAPE


def test_conv_wait_expiry_hook_argument_errors():
    # host-side checks only: nothing is launched
    assert sc.sc_test_conv_wait_expiry(None, A16, None, B16, 1, 4, 4, 4, 4, 0, 10, stream=0) == sc.SC_ERR_NULL
    assert sc.sc_test_conv_wait_expiry(A16, A16, None, B16, 1, 4, 4, 4, 4, -1, 10, stream=0) == sc.SC_ERR_SHAPE
    assert sc.sc_test_conv_wait_expiry(A16, A16, None, B16, 1, 4, 4, 4, 4, 0, 0, stream=0) == sc.SC_ERR_SHAPE
    assert sc.sc_test_conv_wait_expiry(A16, A16, None, B16, 1, 4, 4, 6, 4, 0, 10, stream=0) == sc.SC_ERR_UNSUPPORTED
    assert sc.sc_test_conv_wait_expiry(A16 + 4, A16, None, B16, 1, 4, 4, 4, 4, 0, 10, stream=0) == sc.SC_ERR_ALIGN
    assert sc.sc_test_conv_wait_expiry(A16, A16, None, A16, 1, 4, 4, 4, 4, 0, 10, stream=0) == sc.SC_ERR_ALIAS


NET = [(1 << 28, None, 8, 5, 5, 1), (1 << 28, None, 8, 3, 3, 1), (1 << 28, None, 4, 3, 3, 0)]


@pytest.mark.parametrize("change,expect", [
    (dict(x=None), sc.SC_ERR_NULL),
    (dict(y=None), sc.SC_ERR_NULL),
    (dict(layers=[]), sc.SC_ERR_SHAPE),
    (dict(layers=NET * 22), sc.SC_ERR_SHAPE),                      # more than SC_CHAIN_MAX_LAYERS
    (dict(N=0), sc.SC_ERR_SHAPE),
    (dict(layers=[(None, None, 8, 5, 5, 1)] + NET[1:]), sc.SC_ERR_NULL),
    (dict(layers=[NET[0], (1 << 28, None, 8, 2, 3, 1)]), sc.SC_ERR_UNSUPPORTED),
    (dict(layers=[NET[0], (1 << 28, None, 6, 3, 3, 1)]), sc.SC_ERR_UNSUPPORTED),
    (dict(layers=[(1 << 28, None, 6, 3, 3, 1)]), sc.SC_ERR_UNSUPPORTED),   # Cin 1 -> Cout 6
    (dict(layers=NET[:2] + [(1 << 28, None, 4, 3, 3, 2)]), sc.SC_ERR_UNSUPPORTED),
    (dict(Cin=6, layers=NET[1:]), sc.SC_ERR_UNSUPPORTED),
])
def test_chain_argument_errors(change, expect):
    """conv2d_chain_fwd_host checks every layer (its Cin the previous Cout) by
    conv2d_fwd's rules before it enqueues anything (host-side only)."""
    a = dict(x=A16, y=B16, N=1, H=8, W=8, Cin=1, layers=NET)
    a.update(change)
    rc = sc.conv2d_chain_fwd_host(a["x"], a["y"], a["N"], a["H"], a["W"], a["Cin"], a["layers"], stream=0)
    assert rc == expect, sc.sc_status_string(rc)
