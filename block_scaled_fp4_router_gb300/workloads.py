"""Seeded synthetic inputs for the block-scaled FP4 MoE layer.

This module only draws random numbers in the shapes, distributions and
structure of the five layer workloads; it holds none of the layer's
arithmetic (no dequantisation, routing, quantisation or contraction), so
both the CPU oracle and the CUDA path can be fed from it without sharing
any of the method.

Workloads (MiniMax-M3.1 MoE FFN layer: 128 routed experts, 4 active per
token plus a shared expert -- AMD technical article "MiniMax-M3.1 on AMD
Instinct GPUs", section "MiniMax-M3.1 at a glance"):

* ``tiny``       T=16,   H=512,  I=256,  E=16,  k=4, MXFP4, seed 0
* ``decode1``    T=1,    H=4096, I=1536, E=128, k=4, MXFP4, seed 1
* ``decode16``   T=16,   same shape, NVFP4, uniform routing (no bias), seed 2
* ``decode16z``  T=16,   same shape, NVFP4, Zipf(1.2)-skewed router bias, seed 2
* ``batch128``   T=128,  same shape, MXFP4, router logits ~ N(0,1), seed 3
* ``prefill8k``  T=8192, same shape, MXFP4, Zipf(1.1)-skewed expert load, seed 4
* ``*_s8``       128-token batch and 8192-token prefill with the shared
                 expert in MXFP8 (E4M3 + E8M0 per 32) instead of BF16
* ``*_sig``      tiny, 16-token NVFP4 decode and 128-token batch with sigmoid
                 scoring and a Zipf(0.05) correction bias (seeds 14, 15, 16)

Every workload carries an always-on shared expert with BF16 weights, except
the ``*_sfp4`` variants of tiny, decode1 and batch128, whose shared expert is
an MXFP4 expert folded into the expert table as expert E, drawn like the
routed experts (AMD technical article "MiniMax-M3.1 on AMD Instinct GPUs",
section "Performance, mono decode on vs off": folding the shared expert into
the expert table; model card "amd/MiniMax-M3.1-Flash-Quark-MXFP4", section
"Experimental MXFP4 shared experts").

Array conventions (all numpy, C-contiguous, little-endian):

* ``x``            uint16 [T, H]          BF16 bit patterns, values ~ N(0, 1)
* ``w_router``     float32 [E, H]         N(0, wr_std^2)
* ``bias``         float32 [E] or None    Zipf bias  -s * ln(rank_e)
* ``w13``          uint8 [E, 2I, H/2]     E2M1 codes, 2 per byte, low nibble =
                                          even element; rows [0, I) gate,
                                          rows [I, 2I) up
* ``w13_scale``    uint8 [E, 2I, H/32]    E8M0 (MXFP4) or
                   uint8 [E, 2I, H/16]    E4M3 (NVFP4)
* ``w2``           uint8 [E, H, I/2]      E2M1 codes
* ``w2_scale``     uint8 [E, H, I/32] or [E, H, I/16]
* ``tensor_scale`` float32 [E, 3] or None NVFP4 per-(expert, projection)
                                          scale: gate, up, down
* ``ws13``         uint16 [2I, H]         shared expert gate/up, BF16 bits
* ``ws2``          uint16 [H, I]          shared expert down, BF16 bits
* ``score``        str                    router scores: "softmax" (the bias is
                                          part of the logit) or "sigmoid" (the
                                          bias only corrects the top-k choice)
* ``shared_in_table`` bool               the expert arrays hold E + 1 experts,
                                          the last one the shared expert (then
                                          ``ws13`` / ``ws2`` are None)
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

MXFP4 = "mxfp4"
NVFP4 = "nvfp4"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    top_k: int
    fmt: str
    seed: int
    wr_std: float            # router weight standard deviation
    zipf: float = 0.0        # 0 = no router bias
    shared: bool = True
    shared_std: float = 0.02
    shared_fp4: bool = False  # the shared expert as expert E of the FP4 table
    score: str = "softmax"    # router scores: softmax, or sigmoid with a bias-corrected choice
    shared_fmt: str = "bf16"  # the shared expert's weights: BF16, or MXFP8 (E4M3 + E8M0 per 32)
    # E8M0 block-scale exponents drawn uniformly from [lo, hi]
    mx_exp_lo: int = -8
    mx_exp_hi: int = -4

    @property
    def assignments(self) -> int:
        return self.T * self.top_k

    def with_tokens(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 16, 512, 256, 16, 4, MXFP4, 0, 0.02),
        Workload("decode1", 1, 4096, 1536, 128, 4, MXFP4, 1, 0.02),
        Workload("decode16", 16, 4096, 1536, 128, 4, NVFP4, 2, 0.02),
        Workload("decode16z", 16, 4096, 1536, 128, 4, NVFP4, 2, 0.02, zipf=1.2),
        Workload("batch128", 128, 4096, 1536, 128, 4, MXFP4, 3, 1.0 / 64.0),
        Workload("prefill8k", 8192, 4096, 1536, 128, 4, MXFP4, 4, 0.02, zipf=1.1),
        Workload("tiny_sfp4", 16, 512, 256, 16, 4, MXFP4, 10, 0.02, shared=False, shared_fp4=True),
        Workload("decode1_sfp4", 1, 4096, 1536, 128, 4, MXFP4, 11, 0.02, shared=False, shared_fp4=True),
        Workload("batch128_sfp4", 128, 4096, 1536, 128, 4, MXFP4, 13, 1.0 / 64.0, shared=False, shared_fp4=True),
        Workload("batch128_s8", 128, 4096, 1536, 128, 4, MXFP4, 3, 1.0 / 64.0, shared_fmt="mxfp8"),
        Workload("prefill8k_s8", 8192, 4096, 1536, 128, 4, MXFP4, 4, 0.02, zipf=1.1, shared_fmt="mxfp8"),
        Workload("tiny_sig", 16, 512, 256, 16, 4, MXFP4, 14, 0.02, zipf=0.05, score="sigmoid"),
        Workload("decode16_sig", 16, 4096, 1536, 128, 4, NVFP4, 15, 0.02, zipf=0.05, score="sigmoid"),
        Workload("batch128_sig", 128, 4096, 1536, 128, 4, MXFP4, 16, 1.0 / 64.0, zipf=0.05, score="sigmoid"),
    ]
}

# E4M3 codes 0x30 (0.5) .. 0x50 (8.0) are exactly the positive finite E4M3
# encodings whose value lies in [0.5, 8]: exponent fields 6..9 with any
# mantissa, plus exponent field 10 with mantissa 0.
E4M3_CODE_LO = 0x30
E4M3_CODE_HI = 0x50
# NVFP4 per-(expert, projection) FP32 tensor scales: 2^-8 times a factor
# drawn uniformly from [NVFP4_TS_LO, NVFP4_TS_HI), so gate, up and down of
# every expert carry different scales that are (almost surely) not powers of
# two, as the global scale of a real NVFP4 checkpoint (amax / (6 * 448)).
NVFP4_TENSOR_SCALE = 2.0 ** -8
NVFP4_TS_LO, NVFP4_TS_HI = 0.6, 1.7


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 samples to BF16 bit patterns (library conversion)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def generate(w: Workload, layer: int = 0, tokens: Optional[int] = None) -> dict:
    """Draw one layer's inputs on the host from PCG64 seeded by (seed, layer).

    ``tokens`` overrides T (the weights do not depend on T, so a prefix of a
    larger batch draws the same weights).
    """
    T = w.T if tokens is None else tokens
    ss = np.random.SeedSequence([w.seed, layer])
    # the third stream draws only the NVFP4 tensor scales, so the other
    # arrays are the same draws as before those scales existed
    rw, rx, rt = [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(3)]
    H, I, E = w.H, w.I, w.E
    out = {}
    out["w_router"] = rw.normal(0.0, w.wr_std, size=(E, H)).astype(np.float32)
    if w.zipf > 0.0:
        ranks = rw.permutation(E) + 1
        out["bias"] = (-w.zipf * np.log(ranks)).astype(np.float32)
    else:
        out["bias"] = None
    Et = E + 1 if w.shared_fp4 else E  # experts in the table
    out["shared_in_table"] = w.shared_fp4
    out["score"] = w.score
    out["w13"] = rw.integers(0, 256, size=(Et, 2 * I, H // 2), dtype=np.uint8)
    out["w2"] = rw.integers(0, 256, size=(Et, H, I // 2), dtype=np.uint8)
    if w.fmt == MXFP4:
        lo, hi = 127 + w.mx_exp_lo, 127 + w.mx_exp_hi
        out["w13_scale"] = rw.integers(lo, hi + 1, size=(Et, 2 * I, H // 32), dtype=np.uint8)
        out["w2_scale"] = rw.integers(lo, hi + 1, size=(Et, H, I // 32), dtype=np.uint8)
        out["tensor_scale"] = None
    else:
        lo, hi = E4M3_CODE_LO, E4M3_CODE_HI
        out["w13_scale"] = rw.integers(lo, hi + 1, size=(Et, 2 * I, H // 16), dtype=np.uint8)
        out["w2_scale"] = rw.integers(lo, hi + 1, size=(Et, H, I // 16), dtype=np.uint8)
        out["tensor_scale"] = (NVFP4_TENSOR_SCALE * rt.uniform(NVFP4_TS_LO, NVFP4_TS_HI, size=(Et, 3))).astype(
            np.float32)
    if w.shared and w.shared_fmt == "mxfp8":
        out["ws13"] = None
        out["ws2"] = None
        out.update(generate_shared_mxfp8(w, 7919 * w.seed + layer))
    elif w.shared:
        out["ws13"] = _to_bf16_bits(rw.normal(0.0, w.shared_std, size=(2 * I, H)))
        out["ws2"] = _to_bf16_bits(rw.normal(0.0, w.shared_std, size=(H, I)))
    else:
        out["ws13"] = None
        out["ws2"] = None
    out["x"] = _to_bf16_bits(rx.normal(0.0, 1.0, size=(T, H)))
    return out


def generate_shared_mxfp8(w: Workload, seed: int) -> dict:
    """An MXFP8 shared expert for the workload's shape, from PCG64(seed):
    E4M3 codes uniform over the 254 finite non-NaN encodings (either sign),
    E8M0 scale exponents uniform in [-14, -10].  Arrays s8_w13 [2I, H],
    s8_w13_scale [2I, H/32], s8_w2 [H, I], s8_w2_scale [H, I/32] (uint8)."""
    r = np.random.Generator(np.random.PCG64(seed))
    H, I = w.H, w.I

    def codes(shape):
        c = r.integers(0, 0x7F, size=shape, dtype=np.uint8)  # 0x00 .. 0x7E: finite magnitudes
        return c | (r.integers(0, 2, size=shape, dtype=np.uint8) << 7)

    return {
        "s8_w13": codes((2 * I, H)),
        "s8_w13_scale": r.integers(127 - 14, 127 - 10 + 1, size=(2 * I, H // 32), dtype=np.uint8),
        "s8_w2": codes((H, I)),
        "s8_w2_scale": r.integers(127 - 14, 127 - 10 + 1, size=(H, I // 32), dtype=np.uint8),
    }


def generate_tokens(w: Workload, seed: int, T: int) -> np.ndarray:
    """Fresh BF16 token rows ~ N(0, 1) from PCG64(seed): uint16 [T, H]."""
    r = np.random.Generator(np.random.PCG64(seed))
    return _to_bf16_bits(r.normal(0.0, 1.0, size=(T, w.H)))


def generate_device(w: Workload, layer: int, device) -> dict:
    """Draw one layer's weights directly in device memory (torch RNG seeded by
    (seed, layer)); same distributions as :func:`generate`, different bytes.
    Used to fill many distinct layers quickly for timing; parity cases use
    :func:`generate`.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 1_000_003 + layer)
    H, I, E = w.H, w.I, w.E
    u8 = dict(dtype=torch.uint8, device=device, generator=g)
    out = {}
    out["w_router"] = torch.randn((E, H), device=device, generator=g) * w.wr_std
    if w.zipf > 0.0:
        ranks = torch.randperm(E, device=device, generator=g).float() + 1.0
        out["bias"] = -w.zipf * torch.log(ranks)
    else:
        out["bias"] = None
    Et = E + 1 if w.shared_fp4 else E
    out["shared_in_table"] = w.shared_fp4
    out["score"] = w.score
    out["w13"] = torch.randint(0, 256, (Et, 2 * I, H // 2), **u8)
    out["w2"] = torch.randint(0, 256, (Et, H, I // 2), **u8)
    if w.fmt == MXFP4:
        lo, hi = 127 + w.mx_exp_lo, 127 + w.mx_exp_hi
        out["w13_scale"] = torch.randint(lo, hi + 1, (Et, 2 * I, H // 32), **u8)
        out["w2_scale"] = torch.randint(lo, hi + 1, (Et, H, I // 32), **u8)
        out["tensor_scale"] = None
    else:
        lo, hi = E4M3_CODE_LO, E4M3_CODE_HI
        out["w13_scale"] = torch.randint(lo, hi + 1, (Et, 2 * I, H // 16), **u8)
        out["w2_scale"] = torch.randint(lo, hi + 1, (Et, H, I // 16), **u8)
        out["tensor_scale"] = NVFP4_TENSOR_SCALE * (
            NVFP4_TS_LO + (NVFP4_TS_HI - NVFP4_TS_LO) * torch.rand((Et, 3), device=device, generator=g))
    if w.shared and w.shared_fmt == "mxfp8":
        out["ws13"] = None
        out["ws2"] = None
        # E4M3 codes over the finite encodings of either sign, E8M0 exponents in [-14, -10]
        codes = lambda shape: (torch.randint(0, 0x7F, shape, **u8) | (torch.randint(0, 2, shape, **u8) << 7))
        out["s8_w13"] = codes((2 * I, H))
        out["s8_w13_scale"] = torch.randint(127 - 14, 127 - 10 + 1, (2 * I, H // 32), **u8)
        out["s8_w2"] = codes((H, I))
        out["s8_w2_scale"] = torch.randint(127 - 14, 127 - 10 + 1, (H, I // 32), **u8)
    elif w.shared:
        bf = torch.bfloat16
        out["ws13"] = (torch.randn((2 * I, H), device=device, generator=g) * w.shared_std).to(bf)
        out["ws2"] = (torch.randn((H, I), device=device, generator=g) * w.shared_std).to(bf)
    else:
        out["ws13"] = None
        out["ws2"] = None
    return out
