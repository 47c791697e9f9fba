"""The C ABI without a GPU: the library builds and loads, exports every
entry point the header declares, and rejects invalid calls on the host
before touching device memory (fake pointers are safe here because
validation fails first)."""
import ctypes
import os
import re

import pytest

import block_scaled_fp4_router_gb300 as M
from block_scaled_fp4_router_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return M.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", txt, flags=re.M))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert len(declared) >= 12
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(M.EXPORTED)


def test_checked_build_exports_the_same_entry_points():
    """The checked variant (MOEFP4_CHECKED=1) builds and exports exactly the
    entry points of the header."""
    path = B.build(checked=True)
    assert path == M.CHECKED_LIB_PATH and os.path.exists(path)
    chk = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(chk, name), name


def test_decode_trace_needs_the_trace_build(lib):
    """moe_debug_decode_trace answers only in the trace build."""
    assert lib.moe_debug_decode_trace(None, 0) == M.MOE_ERR_UNSUPPORTED


def test_status_strings(lib):
    for code, name in [(0, "MOE_OK"), (1, "MOE_ERR_INVALID_ARG"), (2, "MOE_ERR_UNSUPPORTED"),
                       (3, "MOE_ERR_CUDA"), (4, "MOE_ERR_TIMEOUT"), (5, "MOE_ERR_WORKSPACE")]:
        assert M.moe_status_string(code) == name


def test_workspace_size_grows_with_tokens(lib):
    a = M.moe_workspace_size(M.desc(1, 4096, 1536, 128, 4))
    b = M.moe_workspace_size(M.desc(16, 4096, 1536, 128, 4))
    c = M.moe_workspace_size(M.desc(8192, 4096, 1536, 128, 4))
    assert 0 < a < b < c and a % 256 == 0
    # y_assign alone is T*k*H*4 bytes
    assert c >= 8192 * 4 * 4096 * 4


@pytest.mark.parametrize("bad,code", [
    (dict(H=100), M.MOE_ERR_INVALID_ARG),
    (dict(I=80), M.MOE_ERR_INVALID_ARG),
    (dict(H=48), M.MOE_ERR_INVALID_ARG),
    (dict(top_k=0), M.MOE_ERR_INVALID_ARG),
    (dict(top_k=9), M.MOE_ERR_INVALID_ARG),
    (dict(E=3), M.MOE_ERR_INVALID_ARG),
    (dict(E=257), M.MOE_ERR_INVALID_ARG),
    (dict(T=-1), M.MOE_ERR_INVALID_ARG),
    (dict(renormalize=0), M.MOE_ERR_UNSUPPORTED),
    (dict(act_quant=0), M.MOE_ERR_UNSUPPORTED),
    (dict(score_func=2), M.MOE_ERR_INVALID_ARG),
    (dict(score_func=-1), M.MOE_ERR_INVALID_ARG),
])
def test_invalid_descriptors_rejected(lib, bad, code):
    d = dict(T=4, H=512, I=256, E=16, top_k=4, renormalize=1, act_quant=1, shared_in_table=0, score_func=0)
    d.update(bad)
    desc = M.LayerDesc(*[d[k] for k in ("T", "H", "I", "E", "top_k", "renormalize", "act_quant",
                                        "shared_in_table", "score_func")])
    out = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(desc), ctypes.byref(out)) == code


@pytest.mark.parametrize("H,I", [(32, 32), (96, 160), (4096, 1536)])
def test_shapes_in_whole_mxfp4_blocks_accepted(lib, H, I):
    """H and I only need whole 32-element blocks (the single-block layer
    H = I = 32 included); shapes the tensor-core tiles do not divide run on
    CUDA cores."""
    out = ctypes.c_size_t(0)
    for T in (1, 16, 300):
        assert lib.moe_workspace_size(ctypes.byref(M.desc(T, H, I, 8, 2)), ctypes.byref(out)) == M.MOE_OK
        assert out.value > 0


def test_decode_range_and_workspace_checks(lib):
    ex = M.Experts(M.MOE_W_MXFP4, 4096, 4096, 4096, 4096, None)
    sh = M.SharedBF16(None, None)
    d129 = M.desc(129, 512, 256, 16, 4)
    # more than 128 tokens is outside the single-launch range
    assert lib.moe_layer_decode(ctypes.byref(d129), ctypes.byref(ex), ctypes.byref(sh), 4096, None, 4096,
                                4096, None, None, 4096, 1 << 30, None) == M.MOE_ERR_UNSUPPORTED
    d4 = M.desc(4, 512, 256, 16, 4)
    need = M.moe_workspace_size(d4)
    # misaligned and undersized workspaces
    assert lib.moe_layer_decode(ctypes.byref(d4), ctypes.byref(ex), ctypes.byref(sh), 4096, None, 4096,
                                4096, None, None, 4096 + 16, need, None) == M.MOE_ERR_WORKSPACE
    assert lib.moe_layer_decode(ctypes.byref(d4), ctypes.byref(ex), ctypes.byref(sh), 4096, None, 4096,
                                4096, None, None, 4096, need - 1, None) == M.MOE_ERR_WORKSPACE
    # MXFP4 experts must not carry a tensor scale; NVFP4 experts must
    bad = M.Experts(M.MOE_W_MXFP4, 4096, 4096, 4096, 4096, 4096)
    assert lib.moe_layer_decode(ctypes.byref(d4), ctypes.byref(bad), ctypes.byref(sh), 4096, None, 4096,
                                4096, None, None, 4096, need, None) == M.MOE_ERR_INVALID_ARG
    bad = M.Experts(M.MOE_W_NVFP4, 4096, 4096, 4096, 4096, None)
    assert lib.moe_layer_decode(ctypes.byref(d4), ctypes.byref(bad), ctypes.byref(sh), 4096, None, 4096,
                                4096, None, None, 4096, need, None) == M.MOE_ERR_INVALID_ARG
    # a half-given shared expert and misaligned weights
    half = M.SharedBF16(4096, None)
    assert lib.moe_layer_decode(ctypes.byref(d4), ctypes.byref(ex), ctypes.byref(half), 4096, None, 4096,
                                4096, None, None, 4096, need, None) == M.MOE_ERR_INVALID_ARG
    mis = M.Experts(M.MOE_W_MXFP4, 4096 + 8, 4096, 4096, 4096, None)
    assert lib.moe_layer_decode(ctypes.byref(d4), ctypes.byref(mis), ctypes.byref(sh), 4096, None, 4096,
                                4096, None, None, 4096, need, None) == M.MOE_ERR_INVALID_ARG
    # T = 0 is a no-op that succeeds without touching anything
    d0 = M.desc(0, 512, 256, 16, 4)
    assert lib.moe_layer_decode(ctypes.byref(d0), ctypes.byref(ex), ctypes.byref(sh), 4096, None, 4096,
                                4096, None, None, 4096, need, None) == M.MOE_OK


def test_shared_in_table_descriptor_checks(lib):
    """The folded shared expert: flag values, the top_k / E limits, the table
    shape in the workspace size, the per-step entry points refusing it and a
    BF16 shared expert given beside it (host checks only)."""
    def dsc(**kw):
        d = dict(T=4, H=512, I=256, E=16, top_k=4, renormalize=1, act_quant=1, shared_in_table=1)
        d.update(kw)
        return M.LayerDesc(*[d[k] for k in ("T", "H", "I", "E", "top_k", "renormalize", "act_quant",
                                            "shared_in_table")])
    out = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(dsc(shared_in_table=2)), ctypes.byref(out)) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_size(ctypes.byref(dsc(top_k=8)), ctypes.byref(out)) == M.MOE_ERR_UNSUPPORTED
    assert lib.moe_workspace_size(ctypes.byref(dsc(E=256)), ctypes.byref(out)) == M.MOE_ERR_UNSUPPORTED
    # the table shape: the same bytes as E + 1 experts and top_k + 1 assignments
    assert M.moe_workspace_size(dsc()) == M.moe_workspace_size(M.desc(4, 512, 256, 17, 5))
    d = dsc()
    need = M.moe_workspace_size(d)
    unsup = M.MOE_ERR_UNSUPPORTED
    assert lib.moe_router_topk(ctypes.byref(d), 4096, 4096, None, 4096, 4096, None, 4096, need, None) == unsup
    assert lib.moe_permute(ctypes.byref(d), 4096, 4096, 4096, 4096, 4096, 4096, need, None) == unsup
    assert lib.moe_combine(ctypes.byref(d), 4096, 4096, 4096, None, 4096, None) == unsup
    ex = M.Experts(M.MOE_W_MXFP4, 4096, 4096, 4096, 4096, None)
    sh = M.SharedBF16(None, None)
    assert lib.moe_expert_ffn_fp4(ctypes.byref(d), ctypes.byref(ex), ctypes.byref(sh), 4096, 4096, 4096, 4096,
                                  4096, 4096, None, 4096, need, None) == unsup
    both = M.SharedBF16(4096, 4096)  # a BF16 shared expert beside the folded one
    assert lib.moe_layer_decode(ctypes.byref(d), ctypes.byref(ex), ctypes.byref(both), 4096, None, 4096,
                                4096, None, None, 4096, need, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward(ctypes.byref(d), ctypes.byref(ex), ctypes.byref(both), 4096, None, 4096,
                                 4096, None, None, 4096, need, None) == M.MOE_ERR_INVALID_ARG


def test_shared_expert_mxfp8_argument_checks(lib):
    d = M.desc(4, 512, 256, 16, 4)
    need = M.moe_workspace_size(d)
    ok = M.SharedMXFP8(4096, 4096, 4096, 4096)
    assert lib.moe_shared_expert_mxfp8(ctypes.byref(d), None, 4096, 4096, 4096, need, None) == M.MOE_ERR_INVALID_ARG
    mis = M.SharedMXFP8(4096 + 8, 4096, 4096, 4096)
    assert lib.moe_shared_expert_mxfp8(ctypes.byref(d), ctypes.byref(mis), 4096, 4096, 4096, need,
                                       None) == M.MOE_ERR_INVALID_ARG
    narrow = M.desc(4, 384, 256, 16, 4)  # H not a multiple of 256
    assert lib.moe_shared_expert_mxfp8(ctypes.byref(narrow), ctypes.byref(ok), 4096, 4096, 4096, need,
                                       None) == M.MOE_ERR_UNSUPPORTED
    assert lib.moe_shared_expert_mxfp8(ctypes.byref(d), ctypes.byref(ok), 4096, 4096, 4096, need - 1,
                                       None) == M.MOE_ERR_WORKSPACE


def test_copy_rows_argument_checks(lib):
    inv = M.MOE_ERR_INVALID_ARG
    assert lib.moe_copy_rows(None, 4096, 64, None) == inv
    assert lib.moe_copy_rows(4096, None, 64, None) == inv
    assert lib.moe_copy_rows(4096 + 8, 4096, 64, None) == inv   # misaligned destination
    assert lib.moe_copy_rows(4096, 4096 + 4, 64, None) == inv   # misaligned source
    assert lib.moe_copy_rows(4096, 8192, 40, None) == inv       # not a multiple of 16 bytes
    assert lib.moe_copy_rows(None, None, 0, None) == M.MOE_OK   # nothing to copy


def test_quant_argument_checks(lib):
    assert lib.moe_quant_act_mxfp4(4, 33, 4096, 4096, 4096, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_act_mxfp4(4, 64, 4096 + 2, 4096, 4096, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_act_mxfp4(0, 64, None, None, None, None) == M.MOE_OK
    assert lib.moe_quant_act_mxfp8(4, 48, 4096, 4096, 4096, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_act_mxfp8(4, 64, 4096, 4096 + 4, 4096, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_act_mxfp8(0, 64, None, None, None, None) == M.MOE_OK


def test_binding_raises_on_error(lib):
    with pytest.raises(M.MoeError) as e:
        M.moe_workspace_size(M.desc(1, 100, 256, 16, 4))
    assert e.value.status == M.MOE_ERR_INVALID_ARG
