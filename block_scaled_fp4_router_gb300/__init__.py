"""Python binding of libmoefp4 (C ABI in include/moefp4.h).

Argument marshalling only: every function here has the name of the C entry
point it calls, takes torch tensors (device memory) or raw integer pointers,
passes the current torch CUDA stream unless one is given, and raises
MoeError on a non-OK status.  Every step of the layer runs in the library's
own CUDA kernels; there is no fallback: if the library is not built, loading
it raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoefp4.so")
# the checked build (out-of-range caller indices recorded in the status word)
CHECKED_LIB_PATH = os.path.join(_HERE, "libmoefp4_checked.so")
TRACE_LIB_PATH = os.path.join(_HERE, "libmoefp4_trace.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_TIMEOUT = 4
MOE_ERR_WORKSPACE = 5
MOE_W_MXFP4 = 1
MOE_W_NVFP4 = 2

EXPORTED = [
    "moe_status_string", "moe_workspace_size", "moe_get_status", "moe_router_topk",
    "moe_quant_act_mxfp4", "moe_permute", "moe_expert_ffn_fp4", "moe_combine",
    "moe_layer_decode", "moe_layer_forward", "moe_set_wait_limit_ns", "moe_debug_wait_probe",
    "moe_layer_decode_noalloc", "moe_debug_requantized_h", "moe_prepare_weights", "moe_convert_nvfp4_to_mxfp4",
    "moe_set_routed_gemm", "moe_copy_rows", "moe_quant_act_mxfp8", "moe_shared_expert_mxfp8",
    "moe_noalloc_get_status", "moe_debug_wait_probe_noalloc", "moe_debug_launch_count", "moe_set_timing_events",
    "moe_debug_decode_trace",
    "moe_dequant_mxfp8_to_bf16", "moe_prepare_shared_mxfp8", "moe_layer_forward_shared_mxfp8",
    "moe_layer_decode_shared_mxfp8",
    "moe_debug_shared_mxfp8_h",
]
NOALLOC_SCRATCH_BYTES = 8 << 20


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s returned %s" % (where, _status_name(status)))


class LayerDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "I", "E", "top_k", "renormalize", "act_quant",
                                              "shared_in_table", "score_func")]


SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1


class SharedMXFP8(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("w13_scale_mma", ctypes.c_void_p), ("w2_scale_mma", ctypes.c_void_p)]


class Experts(ctypes.Structure):
    _fields_ = [
        ("fmt", ctypes.c_int),
        ("w13", ctypes.c_void_p),
        ("w13_scale", ctypes.c_void_p),
        ("w2", ctypes.c_void_p),
        ("w2_scale", ctypes.c_void_p),
        ("tensor_scale", ctypes.c_void_p),
        ("w13_scale_mma", ctypes.c_void_p),
        ("w2_scale_mma", ctypes.c_void_p),
    ]


class SharedBF16(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p)]


_lib = None


def load(path: str = None) -> ctypes.CDLL:
    """Load libmoefp4.so (raises if it has not been built); with
    MOEFP4_CHECKED=1 in the environment, the checked build instead, and with
    MOEFP4_TRACE=1 the trace build."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = (CHECKED_LIB_PATH if os.environ.get("MOEFP4_CHECKED") == "1"
                else TRACE_LIB_PATH if os.environ.get("MOEFP4_TRACE") == "1" else LIB_PATH)
    if not os.path.exists(path):
        raise RuntimeError(
            "libmoefp4.so is not built (expected at %s); run "
            "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
    lib = ctypes.CDLL(path)
    P, S, I32, U64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_uint64
    sig = {
        "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "moe_workspace_size": ([P, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
        "moe_get_status": ([P, ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
        "moe_router_topk": ([P, P, P, P, P, P, P, P, S, P], ctypes.c_int),
        "moe_quant_act_mxfp4": ([I32, I32, P, P, P, P], ctypes.c_int),
        "moe_quant_act_mxfp8": ([I32, I32, P, P, P, P], ctypes.c_int),
        "moe_permute": ([P, P, P, P, P, P, P, S, P], ctypes.c_int),
        "moe_expert_ffn_fp4": ([P, P, P, P, P, P, P, P, P, P, P, S, P], ctypes.c_int),
        "moe_combine": ([P, P, P, P, P, P, P], ctypes.c_int),
        "moe_layer_decode": ([P, P, P, P, P, P, P, P, P, P, S, P], ctypes.c_int),
        "moe_layer_forward": ([P, P, P, P, P, P, P, P, P, P, S, P], ctypes.c_int),
        "moe_set_wait_limit_ns": ([U64], None),
        "moe_set_routed_gemm": ([ctypes.c_int32], ctypes.c_int),
        "moe_copy_rows": ([P, P, S, P], ctypes.c_int),
        "moe_shared_expert_mxfp8": ([P, P, P, P, P, S, P], ctypes.c_int),
        "moe_debug_wait_probe": ([P, S, U64, P], ctypes.c_int),
        "moe_layer_decode_noalloc": ([P, P, P, P, P, P, P, P, P, P], ctypes.c_int),
        "moe_noalloc_get_status": ([ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
        "moe_debug_wait_probe_noalloc": ([U64, P], ctypes.c_int),
        "moe_debug_launch_count": ([ctypes.POINTER(ctypes.c_uint64)], None),
        "moe_debug_decode_trace": ([P, S], ctypes.c_int),
        "moe_dequant_mxfp8_to_bf16": ([I32, I32, P, P, P, P], ctypes.c_int),
        "moe_prepare_shared_mxfp8": ([P, P, P, P, P], ctypes.c_int),
        "moe_layer_forward_shared_mxfp8": ([P, P, P, P, P, P, P, P, P, P, S, P], ctypes.c_int),
        "moe_layer_decode_shared_mxfp8": ([P, P, P, P, P, P, P, P, P, P, S, P], ctypes.c_int),
        "moe_debug_shared_mxfp8_h": ([P, P, S, P, P, P], ctypes.c_int),
        "moe_set_timing_events": ([P, P], None),
        "moe_debug_requantized_h": ([P, P, S, P, P, P], ctypes.c_int),
        "moe_prepare_weights": ([P, P, P, P, P], ctypes.c_int),
        "moe_convert_nvfp4_to_mxfp4": ([P, P, P, P, P, P, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _status_name(st: int) -> str:
    try:
        return load().moe_status_string(st).decode()
    except Exception:  # library not loadable: report the number
        return "status %d" % st


def _p(t):
    """Device pointer of a tensor, an int pointer, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t):
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch

    return torch.cuda.current_stream().cuda_stream


def _check(st: int, where: str):
    if st != MOE_OK:
        raise MoeError(st, where)


def desc(T, H, I, E, top_k, shared_in_table=False, score="softmax") -> LayerDesc:
    return LayerDesc(T, H, I, E, top_k, 1, 1, 1 if shared_in_table else 0,
                     {"softmax": SCORE_SOFTMAX, "sigmoid": SCORE_SIGMOID}[score])


def experts(fmt, w13, w13_scale, w2, w2_scale, tensor_scale=None, w13_scale_mma=None, w2_scale_mma=None) -> Experts:
    return Experts(fmt, _p(w13), _p(w13_scale), _p(w2), _p(w2_scale), _p(tensor_scale), _p(w13_scale_mma),
                   _p(w2_scale_mma))


def shared_bf16(w13=None, w2=None) -> SharedBF16:
    return SharedBF16(_p(w13), _p(w2))


# ---------------------------------------------------------------- entry points


def moe_status_string(st: int) -> str:
    return load().moe_status_string(st).decode()


def moe_workspace_size(d: LayerDesc) -> int:
    out = ctypes.c_size_t(0)
    _check(load().moe_workspace_size(ctypes.byref(d), ctypes.byref(out)), "moe_workspace_size")
    return out.value


def moe_get_status(ws) -> int:
    st = ctypes.c_int(0)
    _check(load().moe_get_status(_p(ws), ctypes.byref(st)), "moe_get_status")
    return st.value


def moe_set_wait_limit_ns(ns: int) -> None:
    load().moe_set_wait_limit_ns(int(ns))


ROUTED_GEMM_AUTO, ROUTED_GEMM_TOKENS_AS_A, ROUTED_GEMM_WEIGHTS_AS_A = 0, 1, 2


def moe_set_routed_gemm(mode: int) -> None:
    _check(load().moe_set_routed_gemm(int(mode)), "moe_set_routed_gemm")


def moe_copy_rows(dst, src, stream=None) -> None:
    """Copies src into dst (same byte size) with the GPU's SMs: device tensors
    or pinned host tensors."""
    nbytes = _nbytes(src)
    if _nbytes(dst) != nbytes:
        raise ValueError("moe_copy_rows: %d bytes into %d" % (nbytes, _nbytes(dst)))
    _check(load().moe_copy_rows(_p(dst), _p(src), nbytes, _stream(stream)), "moe_copy_rows")


def moe_debug_wait_probe(ws, limit_ns: int, stream=None) -> None:
    _check(load().moe_debug_wait_probe(_p(ws), _nbytes(ws), int(limit_ns), _stream(stream)),
           "moe_debug_wait_probe")


def moe_prepare_weights(d, ex, w13_scale_mma, w2_scale_mma, stream=None):
    _check(load().moe_prepare_weights(ctypes.byref(d), ctypes.byref(ex), _p(w13_scale_mma), _p(w2_scale_mma),
                                      _stream(stream)), "moe_prepare_weights")


def moe_convert_nvfp4_to_mxfp4(d, ex, w13_out, w13_scale_out, w2_out, w2_scale_out, stream=None):
    _check(load().moe_convert_nvfp4_to_mxfp4(ctypes.byref(d), ctypes.byref(ex), _p(w13_out), _p(w13_scale_out),
                                             _p(w2_out), _p(w2_scale_out), _stream(stream)),
           "moe_convert_nvfp4_to_mxfp4")


def moe_debug_requantized_h(d, ws, hq, hs, stream=None):
    _check(load().moe_debug_requantized_h(ctypes.byref(d), _p(ws), _nbytes(ws), _p(hq), _p(hs), _stream(stream)),
           "moe_debug_requantized_h")


def moe_router_topk(d, x, w_router, bias, topk_ids, topk_w, logits, ws, stream=None):
    _check(load().moe_router_topk(ctypes.byref(d), _p(x), _p(w_router), _p(bias), _p(topk_ids), _p(topk_w),
                                  _p(logits), _p(ws), _nbytes(ws), _stream(stream)), "moe_router_topk")


def moe_quant_act_mxfp4(rows, K, x, codes, scales, stream=None):
    _check(load().moe_quant_act_mxfp4(int(rows), int(K), _p(x), _p(codes), _p(scales), _stream(stream)),
           "moe_quant_act_mxfp4")


def shared_mxfp8(w13, w13_scale, w2, w2_scale, w13_scale_mma=None, w2_scale_mma=None) -> SharedMXFP8:
    return SharedMXFP8(_p(w13), _p(w13_scale), _p(w2), _p(w2_scale), _p(w13_scale_mma), _p(w2_scale_mma))


def moe_prepare_shared_mxfp8(d, sh8, w13_scale_mma, w2_scale_mma, stream=None):
    _check(load().moe_prepare_shared_mxfp8(ctypes.byref(d), ctypes.byref(sh8), _p(w13_scale_mma), _p(w2_scale_mma),
                                           _stream(stream)), "moe_prepare_shared_mxfp8")


def moe_layer_forward_shared_mxfp8(d, ex, sh8, w_router, bias, x, out, topk_ids, topk_w, ws, stream=None):
    _check(load().moe_layer_forward_shared_mxfp8(ctypes.byref(d), ctypes.byref(ex), ctypes.byref(sh8), _p(w_router),
                                                 _p(bias), _p(x), _p(out), _p(topk_ids), _p(topk_w), _p(ws),
                                                 _nbytes(ws), _stream(stream)), "moe_layer_forward_shared_mxfp8")


def moe_layer_decode_shared_mxfp8(d, ex, sh8, w_router, bias, x, out, topk_ids, topk_w, ws, stream=None):
    _check(load().moe_layer_decode_shared_mxfp8(ctypes.byref(d), ctypes.byref(ex), ctypes.byref(sh8), _p(w_router),
                                                 _p(bias), _p(x), _p(out), _p(topk_ids), _p(topk_w), _p(ws),
                                                 _nbytes(ws), _stream(stream)), "moe_layer_decode_shared_mxfp8")


def moe_debug_shared_mxfp8_h(d, ws, hq, hs, stream=None):
    _check(load().moe_debug_shared_mxfp8_h(ctypes.byref(d), _p(ws), _nbytes(ws), _p(hq), _p(hs), _stream(stream)),
           "moe_debug_shared_mxfp8_h")


def moe_shared_expert_mxfp8(d, sh8, x, y_shared, ws, stream=None):
    _check(load().moe_shared_expert_mxfp8(ctypes.byref(d), ctypes.byref(sh8), _p(x), _p(y_shared), _p(ws),
                                          _nbytes(ws), _stream(stream)), "moe_shared_expert_mxfp8")


def moe_quant_act_mxfp8(rows, K, x, codes, scales, stream=None):
    _check(load().moe_quant_act_mxfp8(int(rows), int(K), _p(x), _p(codes), _p(scales), _stream(stream)),
           "moe_quant_act_mxfp8")


def moe_permute(d, topk_ids, counts, offsets, perm, inv_perm, ws, stream=None):
    _check(load().moe_permute(ctypes.byref(d), _p(topk_ids), _p(counts), _p(offsets), _p(perm), _p(inv_perm),
                              _p(ws), _nbytes(ws), _stream(stream)), "moe_permute")


def moe_expert_ffn_fp4(d, ex, sh, x, xq, xs, offsets, perm, y_assign, y_shared, ws, stream=None):
    _check(load().moe_expert_ffn_fp4(ctypes.byref(d), ctypes.byref(ex), ctypes.byref(sh), _p(x), _p(xq), _p(xs),
                                     _p(offsets), _p(perm), _p(y_assign), _p(y_shared), _p(ws), _nbytes(ws),
                                     _stream(stream)), "moe_expert_ffn_fp4")


def moe_combine(d, y_assign, inv_perm, topk_w, y_shared, out, stream=None):
    _check(load().moe_combine(ctypes.byref(d), _p(y_assign), _p(inv_perm), _p(topk_w), _p(y_shared), _p(out),
                              _stream(stream)), "moe_combine")


def moe_layer_decode(d, ex, sh, w_router, bias, x, out, topk_ids, topk_w, ws, stream=None):
    _check(load().moe_layer_decode(ctypes.byref(d), ctypes.byref(ex), ctypes.byref(sh), _p(w_router), _p(bias),
                                   _p(x), _p(out), _p(topk_ids), _p(topk_w), _p(ws), _nbytes(ws),
                                   _stream(stream)), "moe_layer_decode")


def moe_layer_forward(d, ex, sh, w_router, bias, x, out, topk_ids, topk_w, ws, stream=None):
    _check(load().moe_layer_forward(ctypes.byref(d), ctypes.byref(ex), ctypes.byref(sh), _p(w_router), _p(bias),
                                    _p(x), _p(out), _p(topk_ids), _p(topk_w), _p(ws), _nbytes(ws),
                                    _stream(stream)), "moe_layer_forward")


def moe_layer_decode_noalloc(d, ex, sh, w_router, bias, x, out, topk_ids, topk_w, stream=None):
    """moe_layer_decode with the library's built-in scratch instead of a caller
    workspace, for callers that cannot allocate device memory (see the header)."""
    _check(load().moe_layer_decode_noalloc(ctypes.byref(d), ctypes.byref(ex), ctypes.byref(sh), _p(w_router),
                                           _p(bias), _p(x), _p(out), _p(topk_ids), _p(topk_w), _stream(stream)),
           "moe_layer_decode_noalloc")


def moe_noalloc_get_status() -> int:
    """Reads and clears the status word of the built-in scratch of
    moe_layer_decode_noalloc on the current device."""
    st = ctypes.c_int(0)
    _check(load().moe_noalloc_get_status(ctypes.byref(st)), "moe_noalloc_get_status")
    return st.value


def moe_debug_wait_probe_noalloc(limit_ns: int, stream=None) -> None:
    _check(load().moe_debug_wait_probe_noalloc(int(limit_ns), _stream(stream)), "moe_debug_wait_probe_noalloc")


def moe_debug_launch_count() -> int:
    n = ctypes.c_uint64(0)
    load().moe_debug_launch_count(ctypes.byref(n))
    return n.value


def moe_debug_decode_trace(clear: bool = False, slots: bool = False):
    """Trace builds: the last single-launch decode's per-block %globaltimer
    stamps as a numpy uint64 array [256 blocks, 16 events]; with slots=True
    also the per-slot stamps [320 slots, 8] (a pair).  clear=True zeroes both
    and returns None."""
    import numpy as np
    if clear:
        _check(load().moe_debug_decode_trace(None, 0), "moe_debug_decode_trace")
        return None
    out = np.zeros((256 * 16 + (320 * 8 if slots else 0),), np.uint64)
    _check(load().moe_debug_decode_trace(ctypes.c_void_p(out.ctypes.data), out.nbytes), "moe_debug_decode_trace")
    blocks = out[:256 * 16].reshape(256, 16)
    return (blocks, out[256 * 16:].reshape(320, 8)) if slots else blocks


def moe_set_timing_events(begin=None, end=None) -> None:
    """begin / end: torch.cuda.Event objects (or raw cudaEvent_t ints), None = off."""
    h = lambda e: None if e is None else (e if isinstance(e, int) else e.cuda_event)
    load().moe_set_timing_events(h(begin), h(end))


def moe_dequant_mxfp8_to_bf16(rows, K, codes, scales, out, stream=None):
    _check(load().moe_dequant_mxfp8_to_bf16(int(rows), int(K), _p(codes), _p(scales), _p(out), _stream(stream)),
           "moe_dequant_mxfp8_to_bf16")
