"""The checked build (MOEFP4_CHECKED=1) against the product build, on the GPU.

A caller-given index that is out of range (an expert id passed to
moe_permute, an assignment index in the perm passed to moe_expert_ffn_fp4)
is left out by every build, so nothing is read or written through it; the
checked build also records MOE_ERR_INVALID_ARG in the workspace status word,
and reports nothing on valid inputs.  Each build runs in a child process
(the binding loads one library per process).
"""
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
from oracle import moe as O
import os
B.build(checked=os.environ.get("MOEFP4_CHECKED") == "1")
M.load()
res = []
# moe_permute: one id out of range, the others valid
T, k, E = 40, 4, 16
rng = np.random.default_rng(5)
ids = rng.integers(0, E, (T, k)).astype(np.int32)
ids[7, 2] = E + 3
d = M.desc(T, 128, 128, E, k)
ws = torch.zeros(M.moe_workspace_size(d), dtype=torch.uint8, device="cuda")
counts = torch.empty(E, dtype=torch.int32, device="cuda")
offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
M.moe_permute(d, torch.from_numpy(ids).cuda(), counts, offsets, perm, inv, ws)
torch.cuda.synchronize()
res.append(M.moe_get_status(ws))
valid = ids.ravel()[ids.ravel() < E]
res.append(int(np.array_equal(counts.cpu().numpy(), np.bincount(valid, minlength=E))))
# moe_expert_ffn_fp4 on the tensor-core path (>= 256 assignments): one perm entry out of range
wl = W.Workload("chk", 80, 256, 256, 8, 4, W.MXFP4, 37, 0.05, shared=False)
lay = W.generate(wl)
dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=wl.T)
ref = O.layer_forward(lay, wl.top_k, wl.fmt)
c, o, p, _ = O.permute(ref["ids"], wl.E)
p = p.copy()
p[5] = 10 ** 6
xt = torch.from_numpy(lay["x"]).view(torch.int16).cuda()
xq = torch.empty((wl.T, wl.H // 2), dtype=torch.uint8, device="cuda")
xs = torch.empty((wl.T, wl.H // 32), dtype=torch.uint8, device="cuda")
M.moe_quant_act_mxfp4(wl.T, wl.H, xt, xq, xs)
y = torch.empty((wl.T * wl.top_k, wl.H), dtype=torch.float32, device="cuda")
M.moe_expert_ffn_fp4(dev.desc(wl.T), dev.ex, dev.sh, xt, xq, xs, torch.from_numpy(o).cuda(),
                     torch.from_numpy(p).cuda(), y, None, dev.ws)
torch.cuda.synchronize()
res.append(M.moe_get_status(dev.ws))
# a whole layer on valid inputs: nothing reported
out, i2, _ = dev.forward(xt)
torch.cuda.synchronize()
res.append(M.moe_get_status(dev.ws))
print("RESULT", *res)
"""


def _run(checked):
    env = dict(os.environ, MOEFP4_CHECKED="1" if checked else "0", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT")][-1]
    return [int(v) for v in line.split()[1:]]


def test_checked_build_reports_out_of_range_indices():
    import block_scaled_fp4_router_gb300 as M

    st_perm, counts_ok, st_ffn, st_layer = _run(checked=True)
    assert st_perm == M.MOE_ERR_INVALID_ARG and counts_ok == 1
    assert st_ffn == M.MOE_ERR_INVALID_ARG
    assert st_layer == M.MOE_OK


def test_product_build_leaves_out_of_range_indices_out_silently():
    import block_scaled_fp4_router_gb300 as M

    st_perm, counts_ok, st_ffn, st_layer = _run(checked=False)
    assert (st_perm, counts_ok, st_ffn, st_layer) == (M.MOE_OK, 1, M.MOE_OK, M.MOE_OK)
