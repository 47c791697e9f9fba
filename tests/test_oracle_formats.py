"""Pins of the oracle's number formats against facts fixed outside it.

CPU only.  Each test checks the oracle against something it did not compute
itself: the formats' enumerations (golden files), PyTorch's own FP8 / E8M0 /
BF16 conversions (independent library code), hand-worked quantisation
examples, brute force over all codes, and closed-form invariants.
"""
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ----------------------------------------------------------------- decoding


def test_e2m1_table_matches_format_enumeration():
    rows = _read_golden("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = F.E2M1_TABLE[int(code)]
        assert got == float(val), (code, got, val)
        assert np.signbit(got) == (int(code) >= 8)
    # format parameters: largest normal 6, smallest normal 1, one subnormal 0.5
    mags = sorted(set(np.abs(F.E2M1_TABLE)))
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert F.E2M1_MAX == 6.0 and 2 ** F.E2M1_EMAX == 4.0


def test_e4m3_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = F.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    assert np.nanmax(got) == 448.0 and got[0x01] == 2.0 ** -9


def test_e8m0_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    got = F.E8M0_TABLE
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def test_pack_unpack_nibble_order():
    # low nibble holds the even element: 0x21 -> codes (1, 2) -> (0.5, 1.0)
    codes = F.unpack_e2m1(np.array([0x21, 0xF8], dtype=np.uint8))
    assert codes.tolist() == [1, 2, 8, 15]
    assert F.E2M1_TABLE[codes].tolist() == [0.5, 1.0, -0.0, -6.0]
    rng = np.random.default_rng(5)
    p = rng.integers(0, 256, size=(7, 40), dtype=np.uint8)
    assert np.array_equal(F.pack_e2m1(F.unpack_e2m1(p)), p)


# --------------------------------------------------------------------- BF16


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    f = np.concatenate([
        rng.normal(0, 1, 200_000),
        rng.normal(0, 1e-30, 20_000),
        rng.normal(0, 1e30, 20_000),
    ]).astype(np.float32)
    # exact ties: BF16 values plus half an ulp, both parities
    bits = rng.integers(0, 2 ** 16, size=20_000, dtype=np.uint32)
    ties = ((bits << 16) | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    # subnormal BF16 range
    sub = (rng.integers(0, 2 ** 23, size=20_000, dtype=np.uint32)).view(np.float32)
    f = np.concatenate([f, ties, sub, -sub])
    ref = torch.from_numpy(f).to(torch.bfloat16).double().numpy()
    got = F.round_to_bf16(f.astype(np.float64))
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_bits_round_trip():
    bits = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    v = F.bf16_bits_to_float(bits)
    fin = np.isfinite(v) & (v != 0)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(v[np.isfinite(ref)], ref[np.isfinite(ref)])
    assert np.array_equal(F.bf16_value_to_bits(v[fin]), bits[fin])


def test_e4m3_times_power_of_two_is_exact_in_bf16():
    """vLLM PR #64273, section "Purpose": E4M3 times a power-of-two scale is
    exact in BF16 (an E4M3 value has at most 4 significant bits, BF16 has 8).
    Checked for every finite E4M3 code and every scale 2^s whose product stays
    inside BF16's normal range; the documented edge (subnormal results) is
    checked separately."""
    vals = F.E4M3_TABLE[np.isfinite(F.E4M3_TABLE)]
    vals = vals[vals != 0]
    n_checked = 0
    for s in range(-127, 128):
        p = np.ldexp(vals, s)
        normal = (np.abs(p) >= 2.0 ** -126) & (np.abs(p) < 2.0 ** 128)
        p = p[normal]
        assert np.array_equal(F.round_to_bf16(p), p)
        tp = torch.from_numpy(p.astype(np.float32)).to(torch.bfloat16).double().numpy()
        assert np.array_equal(tp, p)
        n_checked += p.size
    assert n_checked > 50_000
    # edge: the smallest E4M3 subnormal times 2^-127 is far below BF16's
    # smallest subnormal (2^-133) and does not survive
    assert F.round_to_bf16(np.array([2.0 ** -9 * 2.0 ** -127]))[0] == 0.0


def test_e2m1_times_e8m0_is_exact_in_bf16():
    vals = F.E2M1_TABLE[F.E2M1_TABLE != 0]
    for b in range(0, 255):
        p = vals * F.E8M0_TABLE[b]
        normal = (np.abs(p) >= 2.0 ** -126) & (np.abs(p) < 2.0 ** 128)
        assert np.array_equal(F.round_to_bf16(p[normal]), p[normal])


# ------------------------------------------------------------ MXFP4 encoder


def _worked_blocks():
    blocks, cur = [], None
    for row in _read_golden("mxfp4_worked_blocks.txt"):
        if row[0] == "block":
            cur = dict(name=row[1], v=np.zeros(32), code=np.zeros(32, np.uint8))
            blocks.append(cur)
        elif row[0] == "scale":
            cur["scale"] = int(row[1])
        else:
            i = int(row[0])
            cur["v"][i] = float(row[1])
            cur["code"][i] = int(row[2])
    return blocks


@pytest.mark.parametrize("blk", _worked_blocks(), ids=lambda b: b["name"])
def test_mxfp4_hand_worked_blocks(blk):
    codes, scales = F.quantize_mxfp4(blk["v"])
    assert scales.tolist() == [blk["scale"]]
    assert codes.tolist() == blk["code"].tolist()


def _random_blocks(n, seed):
    rng = np.random.default_rng(seed)
    v = rng.normal(0, 1, (n, 32)) * np.exp2(rng.integers(-20, 20, (n, 1)))
    v[rng.random((n, 32)) < 0.05] = 0.0
    # sprinkle exact E2M1 ties relative to the block scale
    return v.astype(np.float32).astype(np.float64)


def test_mxfp4_codes_are_brute_force_nearest_with_even_ties():
    v = _random_blocks(3000, 1)
    codes, scales = F.quantize_mxfp4(v)
    X = F.E8M0_TABLE[scales]  # [n, 1]
    s = v / X
    cand = F.E2M1_TABLE  # all 16 codes
    dist = np.abs(s[..., None] - cand)
    chosen = np.take_along_axis(dist, codes[..., None].astype(np.int64), -1)[..., 0]
    assert np.all(chosen <= dist.min(-1))
    # ties between two magnitudes go to the even mantissa (exact ties are
    # exercised exhaustively by test_mxfp4_ties_at_every_midpoint)
    mags = np.abs(F.E2M1_TABLE[:8])
    dm = np.abs(np.abs(s)[..., None] - mags)
    tie = (dm == dm.min(-1, keepdims=True)).sum(-1) == 2
    assert np.all((codes[tie] & 1) == 0)
    assert np.all(codes[s == 0] == 0)


def test_mxfp4_ties_at_every_midpoint():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    v = np.zeros((len(mags) - 1, 32))
    for i in range(len(mags) - 1):
        v[i, 0] = 4.0  # pins X = 1
        v[i, 1] = (mags[i] + mags[i + 1]) / 2
        v[i, 2] = -(mags[i] + mags[i + 1]) / 2
    codes, scales = F.quantize_mxfp4(v)
    assert np.all(scales == 127)
    for i in range(len(mags) - 1):
        lo, hi = i, i + 1
        want = lo if lo % 2 == 0 else hi
        assert codes[i, 1] == want
        assert codes[i, 2] == (want + 8 if want else 0)


def test_mxfp4_scale_rule_and_error_bound():
    v = _random_blocks(3000, 2)
    codes, scales = F.quantize_mxfp4(v)
    amax = np.abs(v).max(-1)
    X = F.E8M0_TABLE[scales[:, 0]]
    nz = amax > 0
    r = amax[nz] / X[nz]
    assert np.all((r >= 4) & (r < 8))
    assert np.all(scales[~nz] == 0)
    deq = F.dequantize_mxfp4(codes, scales)
    err = np.abs(deq - v)
    inrange = np.abs(v) <= 6 * X[:, None]
    assert np.all(err[inrange] <= (X[:, None] * np.ones_like(v))[inrange])
    assert np.all(err <= 2 * X[:, None])


def test_mxfp4_idempotent_and_round_trip_of_representable_blocks():
    v = _random_blocks(2000, 3)
    c1, s1 = F.quantize_mxfp4(v)
    d1 = F.dequantize_mxfp4(c1, s1)
    c2, s2 = F.quantize_mxfp4(d1)
    assert np.array_equal(F.dequantize_mxfp4(c2, s2), d1)
    # every block of codes with a magnitude-4-or-6 element and any scale
    # reproduces its codes (with -0 written as +0)
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 16, (4000, 32)).astype(np.uint8)
    codes[:, 0] = rng.choice([6, 7, 14, 15], 4000)
    sc = rng.integers(1, 250, (4000, 1)).astype(np.uint8)
    deq = F.dequantize_mxfp4(codes, sc)
    c3, s3 = F.quantize_mxfp4(deq)
    canon = np.where((codes & 7) == 0, 0, codes)
    assert np.array_equal(s3, sc) and np.array_equal(c3, canon)


def test_mxfp4_scale_clamps_at_smallest_e8m0():
    v = np.zeros(32)
    v[0] = 2.0 ** -140  # floor(log2) - 2 = -142 -> clamp to -127
    codes, scales = F.quantize_mxfp4(v)
    assert scales[0] == 0 and codes[0] == 0  # 2^-140 / 2^-127 = 2^-13 -> 0
    v[0] = 2.0 ** -126
    codes, scales = F.quantize_mxfp4(v)
    assert scales[0] == 0 and F.E2M1_TABLE[codes[0]] == 2.0


def test_mxfp4_rejects_non_finite():
    v = np.zeros(32)
    v[3] = np.nan
    with pytest.raises(ValueError):
        F.quantize_mxfp4(v)


# ------------------------------------------------------------------- NVFP4


def test_nvfp4_dequant_closed_form():
    codes = np.zeros((1, 32), np.uint8)
    codes[0, 0] = 7   # 6.0
    codes[0, 16] = 9  # -0.5
    scales = np.array([[0x38, 0x7E]], np.uint8)  # 1.0, 448.0
    v = F.dequantize_nvfp4(codes, scales, 2.0 ** -8)
    assert v[0, 0] == 6.0 * 2 ** -8 and v[0, 16] == -0.5 * 448.0 * 2 ** -8
    assert np.count_nonzero(v) == 2


def test_nvfp4_to_mxfp4_exact_when_halves_share_a_power_of_two_scale():
    rng = np.random.default_rng(6)
    n = 2000
    codes = rng.integers(0, 16, (n, 32)).astype(np.uint8)
    codes[:, 0] = rng.choice([6, 7, 14, 15], n)  # puts amax in the top binade
    k = rng.integers(-6, 8, n)  # E4M3 power of two 2^k: exponent field k + 7
    e4 = ((k + 7) << 3).astype(np.uint8)
    scales = np.stack([e4, e4], axis=1)
    ts = 2.0 ** -8
    deq = F.dequantize_nvfp4(codes, scales, ts)
    mc, ms = F.requantize_nvfp4_to_mxfp4(codes, scales, ts)
    assert np.array_equal(F.dequantize_mxfp4(mc, ms), deq)
    assert np.array_equal(ms.ravel(), (k - 8 + 127).astype(np.uint8))


def test_nvfp4_to_mxfp4_error_bound_and_mx_round_trip():
    rng = np.random.default_rng(7)
    n = 2000
    codes = rng.integers(0, 16, (n, 32)).astype(np.uint8)
    scales = rng.integers(0x30, 0x51, (n, 2)).astype(np.uint8)
    deq = F.dequantize_nvfp4(codes, scales, 2.0 ** -8)
    mc, ms = F.requantize_nvfp4_to_mxfp4(codes, scales, 2.0 ** -8)
    X = F.E8M0_TABLE[ms]  # [n, 1]
    err = np.abs(F.dequantize_mxfp4(mc, ms) - deq)
    assert np.all(err <= 2 * X)
    # MXFP4 -> NVFP4 with power-of-two E4M3 scales -> MXFP4 reproduces values
    c = rng.integers(0, 16, (n, 32)).astype(np.uint8)
    c[:, 0] = 7
    sb = rng.integers(119, 124, (n, 1)).astype(np.uint8)  # 2^-8 .. 2^-4
    mx = F.dequantize_mxfp4(c, sb)
    e4 = ((sb.astype(int) - 127 + 8 + 7) << 3).astype(np.uint8)  # 2^(s+8) in E4M3
    e4 = np.concatenate([e4, e4], 1)
    nv = F.dequantize_nvfp4(c, e4, 2.0 ** -8)
    assert np.array_equal(nv, mx)
    c2, s2 = F.requantize_nvfp4_to_mxfp4(c, e4, 2.0 ** -8)
    assert np.array_equal(F.dequantize_mxfp4(c2, s2), mx)


def test_e2m1_round_exhaustive_over_dyadic_grid():
    """Every multiple of 1/64 in [-8, 8] against the brute-force definition."""
    s = np.arange(-512, 513) / 64.0
    codes = F.round_to_e2m1(s)
    for si, c in zip(s, codes):
        d = [abs(abs(si) - m) for m in F.E2M1_TABLE[:8]]
        best = min(d)
        cands = [i for i in range(8) if d[i] == best]
        want = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        want = want + (8 if (si < 0 and want != 0) else 0)
        assert c == want, (si, c, want)


# ------------------------------------------------------------------ MXFP8


def test_e4m3_rounding_matches_torch_float8():
    """Nearest-even E4M3 against torch's float32 -> float8_e4m3fn cast on
    in-range values of every binade (subnormals included); the only
    difference allowed is the sign of zero (the oracle writes +0)."""
    rng = np.random.default_rng(81)
    mags = np.concatenate([rng.uniform(0, 2.0 ** -6, 4000), 2.0 ** rng.uniform(-9, np.log2(448.0), 20000),
                           F.E4M3_TABLE[:0x7F]])
    v = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = np.where((ref & 0x7F) == 0, 0, ref)
    got = F.round_to_e4m3(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_ties_at_every_midpoint_go_to_even_mantissa():
    mags = F.E4M3_TABLE[:0x7F]
    mid = (mags[:-1] + mags[1:]) / 2  # exact in float64
    lo = np.arange(0x7E)
    even = np.where(lo % 2 == 0, lo, lo + 1)  # of codes lo and lo + 1, the even one
    assert np.array_equal(F.round_to_e4m3(mid), even)
    assert np.array_equal(F.round_to_e4m3(-mid), np.where(even > 0, even | 0x80, 0))


def test_e4m3_saturates_and_zero_is_positive():
    assert F.round_to_e4m3(np.array([448.0, 449.0, 464.0, 511.0, 1e6])).tolist() == [0x7E] * 5
    assert F.round_to_e4m3(np.array([-448.0, -500.0])).tolist() == [0xFE, 0xFE]
    # below half the smallest subnormal (2^-10) the result is +0, whatever the sign
    assert F.round_to_e4m3(np.array([-2.0 ** -11, 2.0 ** -11, -0.0])).tolist() == [0, 0, 0]


def test_mxfp8_scale_rule_and_range():
    """X = 2^(floor(log2 amax) - 8): a block whose amax is 2^k holds it as
    code 0x78 (2^8); every scaled block lies in [-512, 512) and quantises
    within E4M3's range; the error is at most half an E4M3 step of the value
    (or the saturation gap above 448)."""
    blk = np.zeros((1, 32))
    blk[0, 5] = 2.0 ** 3
    c, s = F.quantize_mxfp8(blk)
    assert s[0] == 127 + 3 - 8 and c[0, 5] == 0x78
    rng = np.random.default_rng(82)
    v = rng.normal(0, 1, (64, 256)) * 2.0 ** rng.integers(-20, 20, (64, 1))
    c, s = F.quantize_mxfp8(v)
    X = F.E8M0_TABLE[s]
    amax = np.abs(v.reshape(64, 8, 32)).max(-1)
    assert np.all((amax / X >= 256) & (amax / X < 512))
    d = F.dequantize_mxfp8(c, s).reshape(64, 8, 32)
    sv = np.abs(v.reshape(64, 8, 32)) / X[..., None]
    step = np.where(sv < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(sv, 2.0 ** -6))) - 3))
    err = np.abs(d - v.reshape(64, 8, 32)) / X[..., None]
    assert np.all((err <= step / 2 + 1e-12) | (sv > 448))


def test_mxfp8_idempotent():
    rng = np.random.default_rng(83)
    v = rng.normal(0, 3, (16, 128))
    c, s = F.quantize_mxfp8(v)
    d = F.dequantize_mxfp8(c, s)
    c2, s2 = F.quantize_mxfp8(d)
    assert np.array_equal(F.dequantize_mxfp8(c2, s2), d)


def test_shared_expert_mxfp8_exact_rational():
    """Every contraction of the MXFP8 shared expert on a tiny case, against
    exact rational sums of the dequantised operands rounded once to FP32."""
    from fractions import Fraction
    from oracle import moe as M

    rng = np.random.default_rng(84)
    H, I = 64, 32
    x = F.bf16_bits_to_float(F.bf16_value_to_bits(F.round_to_bf16(rng.normal(0, 1, (1, H)))))
    c13 = rng.integers(0, 0x7F, (2 * I, H)).astype(np.uint8) | (rng.integers(0, 2, (2 * I, H)) * 0x80).astype(np.uint8)
    s13 = rng.integers(115, 119, (2 * I, H // 32)).astype(np.uint8)
    c2 = rng.integers(0, 0x7F, (H, I)).astype(np.uint8)
    s2 = rng.integers(115, 119, (H, I // 32)).astype(np.uint8)
    r = M.shared_expert_mxfp8(x, c13, s13, c2, s2)

    def val(code, sc):
        return Fraction(F.E4M3_TABLE[code]) * Fraction(2) ** (int(sc) - 127)

    xq, xs = r["xq"], r["xs"]
    for i in range(I):
        g = sum(val(xq[0, h], xs[0, h // 32]) * val(c13[i, h], s13[i, h // 32]) for h in range(H))
        u = sum(val(xq[0, h], xs[0, h // 32]) * val(c13[I + i, h], s13[I + i, h // 32]) for h in range(H))
        assert r["G"][0, i] == float(np.float32(float(g)))
        assert r["U"][0, i] == float(np.float32(float(u)))
    for o in range(H):
        y = sum(val(r["hq"][0, i], r["hs"][0, i // 32]) * val(c2[o, i], s2[o, i // 32]) for i in range(I))
        assert r["ys"][0, o] == float(np.float32(float(y)))
