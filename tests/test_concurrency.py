"""Several host threads calling the library at once, each on its own stream.

The worker runs in a fresh process, so every kernel's first call (the
shared-memory opt-in, the occupancy query, the tensor-map encoder, the
workspace pool) happens concurrently.  The threads start together from a
barrier; ctypes releases the interpreter lock during the calls, so they run
in the library at the same time.  Every result is compared with the fp64
oracle at the path's tolerance.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r'''
import sys, threading
sys.path.insert(0, ROOT_DIR)
sys.path.insert(0, ROOT_DIR + "/tests")
import numpy as np, torch
import synthetic as S, oracle
import stencil_conv2d_fwd_gb300 as sc
from parity_util import nchw_to_nhwc, nhwc_to_nchw

dev = torch.device("cuda:0")
torch.cuda.set_device(dev)
sc.load()
CASES = [
    # (name, N, Cin, Cout, H, W, R, layout, entry)
    ("tma narrow", 1, 32, 4, 20, 170, 3, sc.SC_NHWC, "fp32"),
    ("tma wide", 1, 32, 32, 18, 90, 3, sc.SC_NHWC, "fp32"),
    ("tma 64", 1, 64, 64, 9, 60, 3, sc.SC_NHWC, "fp32"),
    ("one channel", 1, 1, 32, 13, 64, 5, sc.SC_NHWC, "fp32"),
    ("nchw workspace", 2, 16, 24, 9, 40, 3, sc.SC_NCHW, "fp32"),
    ("cp.async 5x5", 1, 16, 8, 11, 30, 5, sc.SC_NHWC, "fp32"),
    ("tensor core", 1, 32, 32, 10, 40, 3, sc.SC_NHWC, "tc"),
    ("tensor core split", 1, 32, 32, 10, 40, 3, sc.SC_NHWC, "x3"),
    ("one channel tiled", 1, 1, 32, 9, 300, 5, sc.SC_NHWC, "fp32"),
]
gate = threading.Barrier(len(CASES) + 1)
errors = []

def run_conv(k, name, N, Cin, Cout, H, W, R, layout, entry):
    try:
        c = S.conv_case(600 + k, N, Cin, Cout, H, W, R, R, act=1)
        L = c.layers[0]
        ref, a = oracle.conv2d_nchw(c.x, L.w, L.b, L.act)
        s = torch.cuda.Stream()
        x = c.x if (layout == sc.SC_NCHW or Cin == 1) else nchw_to_nhwc(c.x)
        xd = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        wd, bd = torch.from_numpy(L.w).to(dev), torch.from_numpy(L.b).to(dev)
        yd = torch.empty(N * H * W * Cout, device=dev)
        torch.cuda.synchronize()
        gate.wait(timeout=120)
        for _ in range(4):
            if entry == "tc":
                rc = sc.conv2d_fwd_tc(xd, wd, bd, yd, N, H, W, Cin, Cout, R, R, L.act, stream=s)
            elif entry == "x3":
                rc = sc.conv2d_fwd_tc_x3(xd, wd, bd, yd, N, H, W, Cin, Cout, R, R, L.act, stream=s)
            else:
                rc = sc.conv2d_fwd(xd, wd, bd, yd, N, H, W, Cin, Cout, R, R, layout, L.act, stream=s)
            if rc != 0:
                errors.append(f"{name}: {sc.sc_status_string(rc)}")
                return
        s.synchronize()
        y = yd.cpu().numpy()
        y = y.reshape(N, Cout, H, W) if layout == sc.SC_NCHW else nhwc_to_nchw(y.reshape(N, H, W, Cout))
        tol = 5e-3 if entry == "tc" else 1e-5
        bad = int((np.abs(y - ref) > tol * a).sum())
        if bad:
            errors.append(f"{name}: {bad} elements outside the bound")
    except Exception as e:
        gate.abort()
        errors.append(f"{name}: {e!r}")

def run_stencil():
    try:
        img = S.uniform(61, 0, (40, 300), 0.0, 1.0)
        ref = oracle.stencil_pipeline(img)
        s = torch.cuda.Stream()
        ind = torch.from_numpy(img).to(dev)
        outd = torch.empty_like(ind)
        torch.cuda.synchronize()
        gate.wait(timeout=120)
        for _ in range(4):
            rc = sc.stencil_pipeline_fwd(ind, outd, 40, 300, stream=s)
            if rc != 0:
                errors.append(f"stencil: {sc.sc_status_string(rc)}")
                return
        s.synchronize()
        err = float(np.abs(outd.cpu().numpy() - ref).max())
        if err > 1e-5:
            errors.append(f"stencil: max error {err}")
    except Exception as e:
        gate.abort()
        errors.append(f"stencil: {e!r}")

threads = [threading.Thread(target=run_conv, args=(k, *cs)) for k, cs in enumerate(CASES)]
threads.append(threading.Thread(target=run_stencil))
for t in threads:
    t.start()
for t in threads:
    t.join(timeout=300)
torch.cuda.synchronize()
st = sc.sc_last_device_status()
if st != 0:
    errors.append(f"device status {sc.sc_status_string(st)}")
print("ERRORS: " + " | ".join(errors) if errors else "ALL OK")
'''


def test_concurrent_first_calls_from_several_threads():
    code = WORKER.replace("ROOT_DIR", repr(ROOT))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "ALL OK" in r.stdout, r.stdout[-3000:] + r.stderr[-2000:]
