"""The trace build (MOEFP4_TRACE=1) on the GPU: the single-launch decode
stamps every block's phase boundaries and every expert slot's unit
hand-outs, in order, and computes the same output as the product build.
Runs in a child process (the binding loads one library per process)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import numpy as np, torch
import block_scaled_fp4_router_gb300 as M
from block_scaled_fp4_router_gb300 import build as B, workloads as W
from block_scaled_fp4_router_gb300.device import DeviceLayer
B.build(trace=True)
M.load(M.TRACE_LIB_PATH)
for T in (5, 40):
    wl = W.Workload("tr", T, 512, 256, 16, 4, W.MXFP4, 41, 0.08)
    lay = W.generate(wl)
    dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=T)
    x = torch.from_numpy(lay["x"]).view(torch.int16).cuda()
    M.moe_debug_decode_trace(clear=True)
    out, ids, _ = dev.decode(x)
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    tr, sl = M.moe_debug_decode_trace(slots=True)
    tr = tr.astype(np.int64)
    # per-slot stamps: every assignment in one reached slot; each slot's gate/up
    # handed out, then done, then its h ready, then its down units stored
    info = sl[:, 7].astype(np.int64)
    reached = info > 0
    assert int((info[reached] & 0xFF).sum()) == T * wl.top_k
    st = sl[reached].copy()
    st[:, 0] = np.invert(st[:, 0])
    st[:, 4] = np.invert(st[:, 4])
    st = st.astype(np.int64)
    assert np.all(st[:, 0] <= st[:, 1]) and np.all(st[:, 1] <= st[:, 2]) and np.all(st[:, 2] <= st[:, 3])
    assert np.all(st[:, 4] <= st[:, 5]) and np.all(st[:, 5] <= st[:, 6]) and np.all(st[:, 3] <= st[:, 6])
    blocks = tr[:, 0] > 0
    nb = int(blocks.sum())
    assert nb >= 1 and np.all(tr[nb:, 0] == 0)
    t = tr[:nb]
    for ev in (1, 2, 7, 8, 10):  # router, routing, producer done, units done, end
        assert np.all(t[:, ev] >= t[:, 0]), ev
    assert np.all(t[:, 2] >= t[:, 1]) and np.all(t[:, 10] >= t[:, 8])
    print("OUT", T, out.cpu().numpy().tobytes().hex()[:64], int(out.view(torch.int16).sum()))
"""


def test_trace_build_stamps_phases_and_matches_product_output():
    env = dict(os.environ, PYTHONPATH=ROOT)
    env.pop("MOEFP4_CHECKED", None)
    r = subprocess.run([sys.executable, "-c", "import os\n" + CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    traced = [l for l in r.stdout.splitlines() if l.startswith("OUT")]
    assert len(traced) == 2
    # the same layer through the product build (this process's library)
    import numpy as np
    import torch

    import block_scaled_fp4_router_gb300 as M
    from block_scaled_fp4_router_gb300 import workloads as W
    from block_scaled_fp4_router_gb300.device import DeviceLayer

    M.load()
    for line, T in zip(traced, (5, 40)):
        wl = W.Workload("tr", T, 512, 256, 16, 4, W.MXFP4, 41, 0.08)
        lay = W.generate(wl)
        dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=T)
        out, _, _ = dev.decode(torch.from_numpy(lay["x"]).view(torch.int16).cuda())
        torch.cuda.synchronize()
        want = "OUT %d %s %d" % (T, out.cpu().numpy().tobytes().hex()[:64], int(out.view(torch.int16).sum()))
        assert line == want
