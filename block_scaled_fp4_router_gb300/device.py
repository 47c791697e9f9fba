"""Device-resident layer: the arrays of one MoE layer as torch CUDA tensors,
the C structs that point at them, and a workspace, for calling the C ABI.

Marshalling only -- no layer arithmetic happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (MOE_W_MXFP4, MOE_W_NVFP4, desc, experts, moe_layer_decode, moe_layer_decode_shared_mxfp8,
               moe_layer_forward, moe_layer_forward_shared_mxfp8, moe_prepare_shared_mxfp8, moe_prepare_weights,
               moe_workspace_size, shared_bf16, shared_mxfp8)


def _to_dev(a, device, dtype=None):
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        return a.to(device).contiguous()
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


class DeviceLayer:
    """One layer's weights on the GPU plus a workspace sized for up to T_max tokens.

    Layers also get the tensor-core copy of their scales
    (moe_prepare_weights) unless prepare=False; set_prepared() switches
    between the two descriptions of the same weights."""

    def __init__(self, arrays: dict, H: int, I: int, E: int, top_k: int, fmt: str, T_max: int,
                 device="cuda", shared: bool = True, prepare: bool = True):
        self.H, self.I, self.E, self.k, self.fmt = H, I, E, top_k, fmt
        # the shared expert folded into the FP4 table as expert E (E + 1 experts)
        self.fold = bool(arrays.get("shared_in_table", False))
        self.score = arrays.get("score", "softmax")  # the router's score function
        self.device = torch.device(device)
        d = self.device
        self.w_router = _to_dev(arrays["w_router"], d)
        self.bias = _to_dev(arrays.get("bias"), d)
        self.w13 = _to_dev(arrays["w13"], d)
        self.w13_scale = _to_dev(arrays["w13_scale"], d)
        self.w2 = _to_dev(arrays["w2"], d)
        self.w2_scale = _to_dev(arrays["w2_scale"], d)
        self.tensor_scale = _to_dev(arrays.get("tensor_scale"), d)
        use_shared = shared and arrays.get("ws13") is not None
        self.ws13 = _to_dev(arrays["ws13"], d, torch.int16) if use_shared else None
        self.ws2 = _to_dev(arrays["ws2"], d, torch.int16) if use_shared else None
        wfmt = MOE_W_MXFP4 if fmt == "mxfp4" else MOE_W_NVFP4
        self.ex_plain = experts(wfmt, self.w13, self.w13_scale, self.w2, self.w2_scale, self.tensor_scale)
        self.ex_prepared = None
        # the tensor-core scale layout exists for H and I multiples of 128
        if prepare and H % 128 == 0 and I % 128 == 0:
            self.w13_scale_mma = torch.empty_like(self.w13_scale)
            self.w2_scale_mma = torch.empty_like(self.w2_scale)
            moe_prepare_weights(desc(0, H, I, E, top_k, self.fold), self.ex_plain, self.w13_scale_mma,
                                self.w2_scale_mma)
            self.ex_prepared = experts(wfmt, self.w13, self.w13_scale, self.w2, self.w2_scale, self.tensor_scale,
                                       self.w13_scale_mma, self.w2_scale_mma)
        self.ex = self.ex_prepared if self.ex_prepared is not None else self.ex_plain
        self.sh = shared_bf16(self.ws13, self.ws2)
        # an MXFP8 shared expert (its scales prepared for the tensor cores)
        self.sh8 = None
        if shared and arrays.get("s8_w13") is not None:
            self.s8 = {k: _to_dev(arrays[k], d) for k in ("s8_w13", "s8_w13_scale", "s8_w2", "s8_w2_scale")}
            self.s8_w13_mma = torch.empty_like(self.s8["s8_w13_scale"])
            self.s8_w2_mma = torch.empty_like(self.s8["s8_w2_scale"])
            plain = shared_mxfp8(self.s8["s8_w13"], self.s8["s8_w13_scale"], self.s8["s8_w2"], self.s8["s8_w2_scale"])
            moe_prepare_shared_mxfp8(desc(0, H, I, E, top_k), plain, self.s8_w13_mma, self.s8_w2_mma)
            self.sh8 = shared_mxfp8(self.s8["s8_w13"], self.s8["s8_w13_scale"], self.s8["s8_w2"],
                                    self.s8["s8_w2_scale"], self.s8_w13_mma, self.s8_w2_mma)
        self.T_max = T_max
        nbytes = moe_workspace_size(desc(T_max, H, I, E, top_k, self.fold))
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=d)
        # The zero fill and the scale re-layout ran on the current stream: make
        # them complete before a call on any other stream can read them.
        torch.cuda.synchronize(d)

    @property
    def prepared(self) -> bool:
        return self.ex_prepared is not None and self.ex is self.ex_prepared

    def set_prepared(self, on: bool):
        """Use the prepared scales (tensor-core decode) or only the canonical ones."""
        if on and self.ex_prepared is None:
            raise ValueError("this layer has no prepared scales (prepare=False)")
        self.ex = self.ex_prepared if on else self.ex_plain

    def desc(self, T: int):
        if T > self.T_max:
            raise ValueError("T=%d exceeds the workspace's T_max=%d" % (T, self.T_max))
        return desc(T, self.H, self.I, self.E, self.k, self.fold, self.score)

    def outputs(self, T: int):
        d = self.device
        return (torch.empty((T, self.H), dtype=torch.int16, device=d),
                torch.empty((T, self.k), dtype=torch.int32, device=d),
                torch.empty((T, self.k), dtype=torch.float32, device=d))

    def decode(self, x: torch.Tensor, out=None, ids=None, w=None, stream=None):
        T = x.shape[0]
        if out is None:
            out, ids, w = self.outputs(T)
        if self.sh8 is not None:
            moe_layer_decode_shared_mxfp8(self.desc(T), self.ex, self.sh8, self.w_router, self.bias, x, out, ids, w,
                                          self.ws, stream)
        else:
            moe_layer_decode(self.desc(T), self.ex, self.sh, self.w_router, self.bias, x, out, ids, w, self.ws,
                             stream)
        return out, ids, w

    def forward(self, x: torch.Tensor, out=None, ids=None, w=None, stream=None):
        T = x.shape[0]
        if out is None:
            out, ids, w = self.outputs(T)
        if self.sh8 is not None:
            moe_layer_forward_shared_mxfp8(self.desc(T), self.ex, self.sh8, self.w_router, self.bias, x, out, ids, w,
                                           self.ws, stream)
        else:
            moe_layer_forward(self.desc(T), self.ex, self.sh, self.w_router, self.bias, x, out, ids, w, self.ws,
                              stream)
        return out, ids, w
