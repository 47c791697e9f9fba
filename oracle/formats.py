"""Number formats of the layer, decoded and encoded from their definitions.

Test infrastructure only (see the package docstring).

Sources:
* OCP MXFP4 = E2M1 elements with one E8M0 scale per 32 contiguous elements:
  model card "amd/MiniMax-M3.1-Flash-Quark-MXFP4", section "Model Overview"
  (routed-expert weights "OCP MXFP4, Static", activations "OCP MXFP4,
  Dynamic").  Element and scale encodings follow the OCP Microscaling (MX)
  v1.0 format definitions: E2M1 has 1 sign, 2 exponent (bias 1) and 1
  mantissa bit, no Inf/NaN; E8M0 is an unsigned power of two 2^(b-127) with
  0xFF = NaN; the shared scale is X = 2^(floor(log2(amax)) - emax_elem) with
  emax_elem = 2 for E2M1, and elements are rounded to nearest-even and
  clamped to the largest E2M1 magnitude.
* NVFP4 = E2M1 elements, one E4M3 scale per 16 elements, one FP32 tensor
  scale: AMD technical article "MiniMax-M3.1 on AMD Instinct GPUs", section
  "MiniMax-M3.1 at a glance" (routed experts are NVFP4).  E4M3 is the OCP
  FP8 E4M3 ("fn") format: bias 7, no Inf, S.1111.111 = NaN, max 448.
* NVFP4 -> MXFP4 re-quantisation of the routed experts: same article,
  section "Enabling the MXFP4 checkpoint with the AMD Quark" (the rounding
  method itself is not given; the plain OCP rule above is used).
* OCP MXFP8 (E4M3 elements, one E8M0 scale per 32): the format of the
  shared expert in the pages' fused decode (same article, section "What we
  Optimized": "the shared expert runs in MXFP8"; section "MiniMax-M3.1 at a
  glance": the shared expert is MXFP8 in the checkpoint).  OCP MX v1.0 with
  emax_elem = 8 for E4M3: X = 2^(floor(log2(amax)) - 8), elements rounded to
  nearest-even E4M3 and saturated to +-448.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------- decoding


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1, mantissa bit 0."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:  # subnormal: 2^(1 - bias) * (m / 2) with bias 1
        mag = man * 0.5
    else:
        mag = 2.0 ** (exp - 1) * (1.0 + man / 2.0)
    return sign * mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E2M1_MAX = 6.0
E2M1_EMAX = 2  # exponent of the largest power of two in E2M1 (4 = 2^2)


def e8m0_value(b: int) -> float:
    """Value of an E8M0 scale byte: 2^(b - 127); 0xFF is NaN."""
    b = int(b) & 0xFF
    if b == 0xFF:
        return float("nan")
    return 2.0 ** (b - 127)


E8M0_TABLE = np.array([e8m0_value(b) for b in range(256)], dtype=np.float64)


def e4m3_value(b: int) -> float:
    """Value of an OCP FP8 E4M3 ("fn") byte."""
    b = int(b) & 0xFF
    sign = -1.0 if b & 0x80 else 1.0
    exp = (b >> 3) & 0xF
    man = b & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:  # subnormal: 2^(1 - 7) * (m / 8)
        mag = man * 2.0 ** -9
    else:
        mag = 2.0 ** (exp - 7) * (1.0 + man / 8.0)
    return sign * mag


E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] (low nibble = even element) -> uint8 codes [..., K]."""
    packed = np.asarray(packed, dtype=np.uint8)
    codes = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    codes[..., 0::2] = packed & 0x0F
    codes[..., 1::2] = packed >> 4
    return codes


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [..., K] -> uint8 [..., K/2] (low nibble = even element)."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] & 0x0F) | ((codes[..., 1::2] & 0x0F) << 4)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact float64 values."""
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest BF16 value, ties to even.

    BF16 keeps 8 significant bits and FP32's exponent range (normal down to
    2^-126, subnormal spacing 2^-133).  Returned as float64 holding the
    exactly-representable BF16 value; magnitudes at or above the overflow
    threshold become +-inf.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    nz = (v != 0) & np.isfinite(v)
    _, p = np.frexp(v[nz])  # v = m * 2^p, 0.5 <= |m| < 1
    # unit in the last place of an 8-bit significand, floored at the
    # subnormal spacing
    ulp_exp = np.maximum(p - 8, -133)
    q = np.rint(np.ldexp(v[nz], -ulp_exp))  # np.rint rounds half to even
    r = np.ldexp(q, ulp_exp)
    r[np.abs(r) >= 2.0 ** 128] = np.inf * np.sign(r[np.abs(r) >= 2.0 ** 128])
    out[nz] = r
    out[~np.isfinite(v)] = v[~np.isfinite(v)]
    return out


def bf16_value_to_bits(v: np.ndarray) -> np.ndarray:
    """Exactly-representable BF16 values (float64) -> uint16 bit patterns."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def round_to_f32(v: np.ndarray) -> np.ndarray:
    """Round float64 values to float32 (nearest-even), returned as float64."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


# ------------------------------------------------------- MXFP4 quantisation

_E2M1_MAGS = E2M1_TABLE[:8]  # codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6


def round_to_e2m1(s: np.ndarray) -> np.ndarray:
    """Round values (already divided by the block scale) to E2M1 codes.

    Nearest E2M1 magnitude, ties to the code with an even mantissa bit,
    magnitudes beyond 6 clamp to 6; the sign goes to bit 3, and a result of
    magnitude zero is always the +0 code 0x0.
    """
    s = np.asarray(s, dtype=np.float64)
    if not np.all(np.isfinite(s)):
        raise ValueError("E2M1 quantisation of a non-finite value")
    mag = np.abs(s)
    dist = np.abs(mag[..., None] - _E2M1_MAGS)  # exact in float64
    best = np.argmin(dist, axis=-1)  # first (lower) code on a tie
    nxt = np.minimum(best + 1, 7)
    dbest = np.take_along_axis(dist, best[..., None], -1)[..., 0]
    dnext = np.take_along_axis(dist, nxt[..., None], -1)[..., 0]
    tie = (nxt != best) & (dnext == dbest)
    best = np.where(tie & (best % 2 == 1), nxt, best)  # prefer even mantissa
    sign = (s < 0) & (best != 0)
    return (best + 8 * sign).astype(np.uint8)


def mx_block_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared-scale exponent floor(log2(amax)) - 2, clamped to E8M0 [-127, 127].

    A block whose amax is 0 takes the smallest scale, 2^-127.
    """
    amax = np.asarray(amax, dtype=np.float64)
    _, p = np.frexp(amax)  # amax = m * 2^p with 0.5 <= m < 1 -> floor(log2) = p - 1
    e = (p - 1) - E2M1_EMAX
    e = np.where(amax > 0, e, -127)
    return np.clip(e, -127, 127).astype(np.int64)


def quantize_mxfp4(v: np.ndarray):
    """OCP MXFP4 quantisation along the last axis (length a multiple of 32).

    Returns (codes uint8 [..., K] unpacked, scale bytes uint8 [..., K/32]).
    """
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    if K % 32:
        raise ValueError("MXFP4 needs the quantised axis to be a multiple of 32")
    blocks = v.reshape(v.shape[:-1] + (K // 32, 32))
    amax = np.max(np.abs(blocks), axis=-1)
    e = mx_block_scale_exponent(amax)
    scaled = np.ldexp(blocks, -e[..., None])  # division by a power of two: exact
    codes = round_to_e2m1(scaled).reshape(v.shape)
    return codes, (e + 127).astype(np.uint8)


def dequantize_mxfp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Unpacked E2M1 codes [..., K] and E8M0 bytes [..., K/32] -> float64."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales)
    K = codes.shape[-1]
    if K % 32 or scales.shape != codes.shape[:-1] + (K // 32,):
        raise ValueError("MXFP4 scales must be [..., K/32] for codes [..., K]")
    vals = E2M1_TABLE[codes].reshape(codes.shape[:-1] + (K // 32, 32))
    return (vals * E8M0_TABLE[np.asarray(scales)][..., None]).reshape(codes.shape)


def dequantize_nvfp4(codes: np.ndarray, scales: np.ndarray, tensor_scale) -> np.ndarray:
    """Unpacked E2M1 codes [..., K], E4M3 bytes [..., K/16] and an FP32 tensor
    scale (scalar or broadcastable to [...]) -> float64 values."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales)
    K = codes.shape[-1]
    if K % 16 or scales.shape != codes.shape[:-1] + (K // 16,):
        raise ValueError("NVFP4 scales must be [..., K/16] for codes [..., K]")
    vals = E2M1_TABLE[codes].reshape(codes.shape[:-1] + (K // 16, 16))
    blk = E4M3_TABLE[np.asarray(scales)][..., None]
    ts = np.asarray(tensor_scale, dtype=np.float64)
    if ts.ndim:
        ts = ts[..., None, None]
    return (vals * blk * ts).reshape(codes.shape)


def requantize_nvfp4_to_mxfp4(codes, scales, tensor_scale):
    """NVFP4 -> MXFP4: dequantise exactly, then the OCP MXFP4 rule per 32."""
    return quantize_mxfp4(dequantize_nvfp4(codes, scales, tensor_scale))


# ------------------------------------------------------- MXFP8 quantisation

E4M3_EMAX = 8  # largest E4M3 binade: 448 = 1.75 * 2^8
# codes 0x00 .. 0x7E: every finite non-negative E4M3 magnitude, increasing
_E4M3_MAGS = E4M3_TABLE[:0x7F]


def round_to_e4m3(s: np.ndarray) -> np.ndarray:
    """Round values (already divided by the block scale) to E4M3 codes.

    Nearest E4M3 magnitude (subnormals included), ties to the code with an
    even mantissa, magnitudes beyond 448 saturate to 448 (code 0x7E); the sign
    goes to bit 7, and a result of magnitude zero is always the +0 code 0x00.
    """
    s = np.asarray(s, dtype=np.float64)
    if not np.all(np.isfinite(s)):
        raise ValueError("E4M3 quantisation of a non-finite value")
    mag = np.minimum(np.abs(s), _E4M3_MAGS[-1])
    dist = np.abs(mag[..., None] - _E4M3_MAGS)  # exact in float64
    best = np.argmin(dist, axis=-1)  # first (lower) code on a tie
    nxt = np.minimum(best + 1, 0x7E)
    dbest = np.take_along_axis(dist, best[..., None], -1)[..., 0]
    dnext = np.take_along_axis(dist, nxt[..., None], -1)[..., 0]
    tie = (nxt != best) & (dnext == dbest)
    best = np.where(tie & (best % 2 == 1), nxt, best)  # prefer the even mantissa
    sign = (s < 0) & (best != 0)
    return (best + 0x80 * sign).astype(np.uint8)


def mx8_block_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared-scale exponent floor(log2(amax)) - 8, clamped to E8M0 [-127, 127];
    a block whose amax is 0 takes 2^-127."""
    amax = np.asarray(amax, dtype=np.float64)
    _, p = np.frexp(amax)
    e = np.where(amax > 0, (p - 1) - E4M3_EMAX, -127)
    return np.clip(e, -127, 127).astype(np.int64)


def quantize_mxfp8(v: np.ndarray):
    """OCP MXFP8 (E4M3) quantisation along the last axis (a multiple of 32).

    Returns (codes uint8 [..., K], scale bytes uint8 [..., K/32])."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    if K % 32:
        raise ValueError("MXFP8 needs the quantised axis to be a multiple of 32")
    blocks = v.reshape(v.shape[:-1] + (K // 32, 32))
    e = mx8_block_scale_exponent(np.max(np.abs(blocks), axis=-1))
    codes = round_to_e4m3(np.ldexp(blocks, -e[..., None])).reshape(v.shape)
    return codes, (e + 127).astype(np.uint8)


def dequantize_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """E4M3 codes [..., K] and E8M0 bytes [..., K/32] -> float64."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales)
    K = codes.shape[-1]
    if K % 32 or scales.shape != codes.shape[:-1] + (K // 32,):
        raise ValueError("MXFP8 scales must be [..., K/32] for codes [..., K]")
    vals = E4M3_TABLE[codes].reshape(codes.shape[:-1] + (K // 32, 32))
    return (vals * E8M0_TABLE[scales][..., None]).reshape(codes.shape)
