"""moe_layer_decode_noalloc against moe_layer_decode.

The no-allocation variant serves callers that cannot give the library device
memory (a plain C host program without a device allocator, or a plugin whose
host framework forbids outside allocations); it runs the same fused decode on
a scratch array built into the library.  Its output must match the workspace
version within the layer tolerance the other tests use, on two calls in a
row (the second call reuses the scratch the first one left behind).  This
file is collected last and needs nothing from the other test files.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp4_router_gb300 as M
from block_scaled_fp4_router_gb300 import build as B
from block_scaled_fp4_router_gb300 import workloads as W
from block_scaled_fp4_router_gb300.device import DeviceLayer

pytestmark = pytest.mark.gpu

LAYER_TOL = 2e-2


def _bf16_to_float(t):
    return (t.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    return M.load()


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode16", "decode1_sfp4"])
def test_noalloc_matches_workspace_decode_twice(lib, name):
    wl = W.WORKLOADS[name]
    lay = W.generate(wl)
    dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=wl.T)
    x = torch.from_numpy(lay["x"]).view(torch.int16).cuda()
    ref_out, ref_ids, ref_w = dev.decode(x)
    torch.cuda.synchronize()
    ref = _bf16_to_float(ref_out)
    for _ in range(2):
        out, ids, w = dev.outputs(wl.T)
        M.moe_layer_decode_noalloc(dev.desc(wl.T), dev.ex, dev.sh, dev.w_router, dev.bias, x, out, ids, w)
        torch.cuda.synchronize()
        got = _bf16_to_float(out)
        err = float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))
        assert err <= LAYER_TOL, err
        assert torch.equal(ids, ref_ids)
        assert torch.allclose(w, ref_w, rtol=1e-6, atol=0)
    assert M.moe_noalloc_get_status() == M.MOE_OK


def test_noalloc_keeps_a_recorded_timeout_until_read(lib):
    """A device-side wait that ran out on the built-in scratch stays recorded
    across later calls (whose per-call clear leaves the status word alone)
    until moe_noalloc_get_status reads it; the timeout is made by the library's
    wait probe (a bounded wait on a counter nothing advances), not by a
    decode."""
    wl = W.WORKLOADS["tiny"]
    lay = W.generate(wl)
    dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=wl.T)
    x = torch.from_numpy(lay["x"]).view(torch.int16).cuda()
    ref_out, _, _ = dev.decode(x)
    M.moe_debug_wait_probe_noalloc(2_000_000)
    out, ids, w = dev.outputs(wl.T)
    M.moe_layer_decode_noalloc(dev.desc(wl.T), dev.ex, dev.sh, dev.w_router, dev.bias, x, out, ids, w)
    torch.cuda.synchronize()
    assert M.moe_noalloc_get_status() == M.MOE_ERR_TIMEOUT
    assert M.moe_noalloc_get_status() == M.MOE_OK  # reading clears it
    assert torch.equal(out, ref_out)


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    # a valid layer whose workspace needs more than the built-in scratch
    big = M.desc(16, 65536, 128, 256, 8)
    assert M.moe_workspace_size(big) > M.NOALLOC_SCRATCH_BYTES
    ex = M.Experts(M.MOE_W_MXFP4, 4096, 4096, 4096, 4096, None)
    sh = M.SharedBF16(None, None)
    with pytest.raises(M.MoeError) as e:
        M.moe_layer_decode_noalloc(big, ex, sh, 4096, None, 4096, 4096, None, None)
    assert e.value.status == M.MOE_ERR_UNSUPPORTED
    with pytest.raises(M.MoeError) as e:
        M.moe_layer_decode_noalloc(M.desc(17, 512, 256, 16, 4), ex, sh, 4096, None, 4096, 4096, None, None)
    assert e.value.status == M.MOE_ERR_UNSUPPORTED
