"""Pins of the oracle's layer arithmetic against facts fixed outside it.

CPU only.  Checks: exact rational arithmetic on tiny contractions, brute
force over all top-k subsets, a hand-derived permutation, closed forms of a
structured layer worked out by hand, the MoE identity (sparse dispatch equals
the dense gate-weighted sum over all experts), special cases that reduce to a
known answer, and a cross-format invariant (NVFP4 with power-of-two scales is
the same layer as MXFP4).
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from block_scaled_fp4_router_gb300 import workloads as W
from oracle import formats as F
from oracle import moe as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(vals):
    return F.bf16_value_to_bits(F.round_to_bf16(np.asarray(vals, np.float64)))


# ------------------------------------------------------------------ router


def test_router_logits_exact_rational():
    rng = np.random.default_rng(0)
    T, H, E = 3, 64, 5
    xb = _bf16_bits(rng.normal(0, 1, (T, H)))
    x = F.bf16_bits_to_float(xb)
    wr = rng.normal(0, 0.02, (E, H)).astype(np.float32)
    bias = rng.normal(0, 1, E).astype(np.float32)
    got = M.router_logits(x, wr, bias)
    for t in range(T):
        for e in range(E):
            s = sum(Fraction(float(x[t, h])) * Fraction(float(wr[e, h])) for h in range(H))
            s += Fraction(float(bias[e]))
            assert got[t, e] == float(np.float32(float(s)))


@pytest.mark.parametrize("E,k", [(8, 4), (16, 4), (8, 2), (6, 6)])
def test_topk_is_brute_force_best_subset(E, k):
    rng = np.random.default_rng(E * 10 + k)
    logits = F.round_to_f32(rng.normal(0, 1, (40, E)))
    ids = M.select_topk(logits, k)
    for t in range(logits.shape[0]):
        best = max(itertools.combinations(range(E), k), key=lambda S: sum(logits[t, list(S)]))
        assert set(ids[t].tolist()) == set(best)
        assert np.all(np.diff(logits[t, ids[t]]) <= 0)  # descending


@pytest.mark.parametrize("E,k", [(8, 2), (8, 4), (16, 3)])
def test_sigmoid_topk_is_brute_force_best_subset(E, k):
    """Bias-corrected sigmoid scoring: the selected set maximises the sum of
    sigmoid(l) + b over all C(E, k) subsets (the bias changes the choice), in
    descending order of that key, and the weights are the selected sigmoid
    values (without the bias) over their sum."""
    rng = np.random.default_rng(E * 10 + k)
    for _ in range(20):
        l = rng.normal(0, 2, (1, E))
        b = rng.normal(0, 0.3, E)
        ids, w = M.route(l, k, score="sigmoid", bias=b)
        sig = [1 / (1 + math.exp(-v)) for v in l[0]]
        key = [sig[e] + b[e] for e in range(E)]
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(key[e] for e in c))
        assert set(ids[0].tolist()) == set(best)
        assert all(key[ids[0][j]] >= key[ids[0][j + 1]] for j in range(k - 1))
        tot = sum(sig[e] for e in best)
        for j, e in enumerate(ids[0]):
            assert w[0, j] == float(np.float32(sig[e] / tot))


def test_sigmoid_scoring_closed_form():
    """Worked by hand on the structured layer (logits (1, 3, 2, 0), top-2).
    Softmax picks experts 1, 2.  With sigmoid scoring and bias (0.6, 0, 0,
    0.5) the keys are sigmoid(l) + b = (1.3311, 0.9526, 0.8808, 1.0): experts
    0 and 3 are selected (the bias overrides the larger logits), weighted
    sigmoid(1) / (sigmoid(1) + sigmoid(0)) = 0.5938 and 0.5 / 1.2311 = 0.4062,
    not by their biased keys.  y_e = 1.5 * 2^-e (as in the softmax closed
    form), so out = BF16(1.4609375 + 1.5 w0 + 0.1875 w3) = BF16(2.42786)
    = 2.421875 (155 * 2^-6; the midpoint above it is 2.4296875)."""
    lay = _structured_layer([1.0, 3.0, 2.0, 0.0])
    lay["bias"] = np.array([0.6, 0.0, 0.0, 0.5], np.float32)
    lay["score"] = "sigmoid"
    r = M.layer_forward(lay, 2, "mxfp4", keep=True)
    assert r["logits"].tolist() == [[1.0, 3.0, 2.0, 0.0]]  # raw: the bias stays out of the logits
    assert r["ids"].tolist() == [[0, 3]]
    s1 = 1 / (1 + math.exp(-1))
    w0, w3 = float(np.float32(s1 / (s1 + 0.5))), float(np.float32(0.5 / (s1 + 0.5)))
    assert r["weights"].tolist() == [[w0, w3]]
    assert abs(w0 - 0.5938) < 1e-4 and abs(w3 - 0.4062) < 1e-4
    assert np.all(r["y"][0, 0] == 1.5) and np.all(r["y"][0, 1] == 0.1875)
    acc = 1.4609375 + 1.5 * w0 + 0.1875 * w3
    assert abs(acc - 2.42786) < 1e-5
    assert np.all(r["out"] == 2.421875)
    # the same layer under softmax scoring adds the bias to the logits instead
    lay["score"] = "softmax"
    r2 = M.layer_forward(lay, 2, "mxfp4")
    assert r2["ids"].tolist() == [[1, 2]]


def test_topk_ties_go_to_lower_index():
    logits = np.array([[2.0, 2.0, 1.0, 2.0], [0.0, 0.0, 0.0, 0.0]])
    assert M.select_topk(logits, 2).tolist() == [[0, 1], [0, 1]]
    assert M.select_topk(logits, 3).tolist() == [[0, 1, 3], [0, 1, 2]]


def test_renormalised_weights_equal_softmax_over_selected():
    rng = np.random.default_rng(1)
    logits = F.round_to_f32(rng.normal(0, 2, (50, 16)))
    ids, w = M.route(logits, 4)
    for t in range(50):
        l = logits[t, ids[t]]
        ex = [math.exp(v - l[0]) for v in l]
        ref = [v / sum(ex) for v in ex]
        assert np.allclose(w[t], ref, rtol=2 ** -23, atol=0)
        assert abs(w[t].sum() - 1.0) <= 4 * 2 ** -24
    # a bias shifts logits before the softmax: a large bias forces selection
    wr = np.zeros((4, 32), np.float32)
    x = np.ones((1, 32))
    bias = np.array([0, 0, 30, 0], np.float32)
    ids, w = M.route(M.router_logits(x, wr, bias), 1)
    assert ids.tolist() == [[2]] and w.tolist() == [[1.0]]


# ------------------------------------------------------------- permutation


def test_permutation_hand_example():
    ids = np.array([[2, 0], [0, 2], [1, 2]])
    counts, offsets, perm, inv = M.permute(ids, 3)
    assert counts.tolist() == [2, 1, 3]
    assert offsets.tolist() == [0, 2, 3, 6]
    assert perm.tolist() == [1, 2, 4, 0, 3, 5]
    assert inv.tolist() == [3, 0, 1, 4, 2, 5]


def test_permutation_properties():
    rng = np.random.default_rng(2)
    for E, T, k in [(16, 33, 4), (128, 500, 4), (4, 7, 4)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        counts, offsets, perm, inv = M.permute(ids, E)
        flat = ids.ravel()
        assert sorted(perm.tolist()) == list(range(T * k))
        assert np.array_equal(inv[perm], np.arange(T * k))
        assert np.all(np.diff(flat[perm]) >= 0)
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
        assert counts.sum() == T * k and offsets[-1] == T * k


# ----------------------------------------------------------------- experts


def test_silu_identities():
    g = np.linspace(-30, 30, 1001)
    assert np.allclose(M.silu(g) - M.silu(-g), g, rtol=0, atol=1e-12)
    assert M.silu(np.array([0.0]))[0] == 0.0
    assert abs(M.silu(np.array([1.0]))[0] - 1 / (1 + math.exp(-1))) < 1e-15


def test_routed_contraction_exact_rational():
    rng = np.random.default_rng(3)
    H, I = 64, 32
    x = F.bf16_bits_to_float(_bf16_bits(rng.normal(0, 1, (1, H))))
    xq, xs = M.quantize_activations(x)
    c13 = rng.integers(0, 16, (2 * I, H)).astype(np.uint8)
    s13 = rng.integers(119, 124, (2 * I, H // 32)).astype(np.uint8)
    c2 = rng.integers(0, 16, (H, I)).astype(np.uint8)
    s2 = rng.integers(119, 124, (H, I // 32)).astype(np.uint8)
    w13 = F.dequantize_mxfp4(c13, s13)
    r = M.routed_expert(F.dequantize_mxfp4(xq, xs), w13[:I], w13[I:], F.dequantize_mxfp4(c2, s2))

    def val(code, sc):
        return Fraction(F.E2M1_TABLE[code]) * Fraction(2) ** (int(sc) - 127)

    for i in range(I):
        g = sum(val(xq[0, h], xs[0, h // 32]) * val(c13[i, h], s13[i, h // 32]) for h in range(H))
        u = sum(val(xq[0, h], xs[0, h // 32]) * val(c13[I + i, h], s13[I + i, h // 32]) for h in range(H))
        assert r["G"][0, i] == float(np.float32(float(g)))
        assert r["U"][0, i] == float(np.float32(float(u)))
    for o in range(H):
        y = sum(val(r["hq"][0, i], r["hs"][0, i // 32]) * val(c2[o, i], s2[o, i // 32]) for i in range(I))
        assert r["y"][0, o] == float(np.float32(float(y)))


# ----------------------------------------------- closed-form structured layer


def _structured_layer(c, e2m1_up=4, k=2):
    """H=64, I=32, E=len(c): x = 1, router rows constant c_e / 64 (logit c_e),
    gate codes 1.0 and up codes e2m1_up, both at scale 2^-6, down codes 1.0 at
    scale 2^-(5+e); shared gate 2^-6, up 2^-5, down 2^-5 (BF16)."""
    H, I, E = 64, 32, len(c)
    lay = {}
    lay["x"] = _bf16_bits(np.ones((1, H)))
    lay["w_router"] = np.repeat(np.array(c, np.float32)[:, None] / 64, H, 1).astype(np.float32)
    lay["bias"] = None
    c13 = np.zeros((E, 2 * I, H), np.uint8)
    c13[:, :I] = 2
    c13[:, I:] = e2m1_up
    lay["w13"] = F.pack_e2m1(c13)
    lay["w13_scale"] = np.full((E, 2 * I, H // 32), 127 - 6, np.uint8)
    lay["w2"] = F.pack_e2m1(np.full((E, H, I), 2, np.uint8))
    lay["w2_scale"] = np.stack([np.full((H, I // 32), 127 - 5 - e, np.uint8) for e in range(E)])
    lay["tensor_scale"] = None
    ws13 = np.concatenate([np.full((I, H), 2.0 ** -6), np.full((I, H), 2.0 ** -5)])
    lay["ws13"] = _bf16_bits(ws13)
    lay["ws2"] = _bf16_bits(np.full((H, I), 2.0 ** -5))
    return lay


def test_structured_layer_closed_form():
    """Worked by hand.  Logits (1, 3, 2, 0): top-2 = experts 1, 2 with weights
    1/(1+e^-1) and 1/(1+e).  x = 1 quantises to code 4.0 at scale 2^-2 (exact);
    G = 64 * 2^-6 = 1, U = 64 * 2 * 2^-6 = 2, h = 2 SiLU(1) = 1.46211716; h
    requantises to 6 * 2^-2 = 1.5 (1.4621 / 0.25 = 5.85 -> 6); y_e = 32 * 1.5 *
    2^-(5+e) = 1.5 * 2^-e.  Shared: G = 1, U = 2, h = BF16(1.46211716) =
    1.4609375, ys = 32 * 1.4609375 * 2^-5 = 1.4609375.
    out = BF16(1.4609375 + 0.75 w1 + 0.375 w2) = BF16(2.1100845) = 2.109375."""
    lay = _structured_layer([1.0, 3.0, 2.0, 0.0])
    r = M.layer_forward(lay, 2, "mxfp4", keep=True)
    assert r["logits"].tolist() == [[1.0, 3.0, 2.0, 0.0]]
    assert r["ids"].tolist() == [[1, 2]]
    w1 = float(np.float32(1 / (1 + math.exp(-1))))
    w2 = float(np.float32(1 / (1 + math.exp(1))))
    assert r["weights"].tolist() == [[w1, w2]]
    assert np.all(r["xq"] == 6) and np.all(r["xs"] == 125)
    ex = r["experts"][1]
    assert np.all(ex["G"] == 1.0) and np.all(ex["U"] == 2.0)
    assert np.all(ex["h"] == float(np.float32(2 / (1 + math.exp(-1)))))
    assert np.all(ex["hq"] == 7) and np.all(ex["hs"] == 125)
    assert np.all(r["y"][0, 0] == 0.75) and np.all(r["y"][0, 1] == 0.375)
    assert np.all(r["shared"]["h"] == 1.4609375) and np.all(r["ys"] == 1.4609375)
    assert abs(1.4609375 + 0.75 * w1 + 0.375 * w2 - 2.1100845) < 1e-6
    assert np.all(r["out"] == 2.109375)


def test_structured_layer_closed_form_shared_in_table():
    """The same layer with the shared expert folded into the FP4 table as
    expert E = 4 (gate codes 1.0, up codes 2.0 at 2^-6, down codes 1.0 at
    2^-5, no BF16 shared weights).  It sees the MXFP4 token like a routed
    expert: G = 1, U = 2, h = 2 SiLU(1) requantised to 1.5, y_E = 32 * 1.5 *
    2^-5 = 1.5, weight 1.  out = BF16(1.5 + 0.75 w1 + 0.375 w2) =
    BF16(2.1491470) = 2.15625 (138 * 2^-6; the midpoint below is 2.1484375)."""
    lay = _structured_layer([1.0, 3.0, 2.0, 0.0])
    E, H, I = 4, 64, 32
    c13 = np.zeros((2 * I, H), np.uint8)
    c13[:I] = 2
    c13[I:] = 4
    lay["w13"] = np.concatenate([lay["w13"], F.pack_e2m1(c13)[None]])
    lay["w13_scale"] = np.concatenate([lay["w13_scale"], np.full((1, 2 * I, H // 32), 127 - 6, np.uint8)])
    lay["w2"] = np.concatenate([lay["w2"], F.pack_e2m1(np.full((1, H, I), 2, np.uint8))])
    lay["w2_scale"] = np.concatenate([lay["w2_scale"], np.full((1, H, I // 32), 127 - 5, np.uint8)])
    lay["ws13"] = lay["ws2"] = None
    lay["shared_in_table"] = True
    r = M.layer_forward(lay, 2, "mxfp4", keep=True)
    assert r["ids"].tolist() == [[1, 2]] and int(E) not in r["experts"]
    assert np.all(r["shared"]["hq"] == 7) and np.all(r["shared"]["hs"] == 125)
    assert np.all(r["ys"] == 1.5)
    w1 = float(np.float32(1 / (1 + math.exp(-1))))
    w2 = float(np.float32(1 / (1 + math.exp(1))))
    assert abs(1.5 + 0.75 * w1 + 0.375 * w2 - 2.1491470) < 1e-6
    assert np.all(r["out"] == 2.15625)


def test_structured_layer_closed_form_mxfp8_shared_expert():
    """The structured layer with an MXFP8 shared expert (E4M3 gate codes 1.0,
    up codes 2.0, down codes 1.0; E8M0 scales 2^-6, 2^-6, 2^-5) instead of
    the BF16 one, worked by hand.  x = 1 quantises to MXFP8 exactly (amax 1,
    X = 2^-8, 256 = E4M3 0x78): G = 64 * 2^-6 = 1, U = 64 * 2 * 2^-6 = 2,
    h = 2 SiLU(1) = 1.4621172; h / 2^-8 = 374.30 rounds to the E4M3 value
    384 (neighbours 352 and 384, step 32 in [256, 512)), so hq = 1.5 and
    ys = 32 * 1.5 * 2^-5 = 1.5.  out = BF16(1.5 + 0.75 w1 + 0.375 w2) =
    2.15625, as with the MXFP4 shared expert folded into the table."""
    lay = _structured_layer([1.0, 3.0, 2.0, 0.0])
    H, I = 64, 32
    assert F.E4M3_TABLE[0x38] == 1.0 and F.E4M3_TABLE[0x40] == 2.0 and F.E4M3_TABLE[0x78] == 256.0
    lay["ws13"] = lay["ws2"] = None
    lay["s8_w13"] = np.concatenate([np.full((I, H), 0x38, np.uint8), np.full((I, H), 0x40, np.uint8)])
    lay["s8_w13_scale"] = np.full((2 * I, H // 32), 127 - 6, np.uint8)
    lay["s8_w2"] = np.full((H, I), 0x38, np.uint8)
    lay["s8_w2_scale"] = np.full((H, I // 32), 127 - 5, np.uint8)
    r = M.layer_forward(lay, 2, "mxfp4", keep=True)
    sh = r["shared"]
    assert np.all(sh["xq"] == 0x78) and np.all(sh["xs"] == 127 - 8)
    assert np.all(sh["G"] == 1.0) and np.all(sh["U"] == 2.0)
    assert np.all(F.dequantize_mxfp8(sh["hq"], sh["hs"]) == 1.5)
    assert np.all(r["ys"] == 1.5)
    assert np.all(r["out"] == 2.15625)


def test_structured_layer_routing_ties():
    lay = _structured_layer([2.0, 2.0, 1.0, 2.0])
    r = M.layer_forward(lay, 2, "mxfp4")
    assert r["ids"].tolist() == [[0, 1]] and r["weights"].tolist() == [[0.5, 0.5]]
    # y_0 = 1.5, y_1 = 0.75 -> 0.5 * 2.25 + 1.4609375 = 2.5859375, which sits
    # exactly halfway between the BF16 neighbours 2.578125 (significand
    # 1.0100101b, odd) and 2.59375 (1.0100110b, even): ties-to-even -> 2.59375
    assert np.all(r["out"] == 2.59375)


# ------------------------------------------------------------ MoE identity


@pytest.fixture(scope="module")
def tiny():
    return W.generate(W.WORKLOADS["tiny"])


def test_moe_identity_dense_gate_weighted_sum(tiny):
    """Sparse dispatch == sum over ALL experts of gate_e * FFN_e(x) with gate_e
    the renormalised weight if selected, else 0 (no permutation involved)."""
    wl = W.WORKLOADS["tiny"]
    r = M.layer_forward(tiny, wl.top_k, wl.fmt)
    x = F.bf16_bits_to_float(tiny["x"])
    xq, xs = M.quantize_activations(x)
    xd = F.dequantize_mxfp4(xq, xs)
    acc = M.shared_expert(x, tiny["ws13"], tiny["ws2"])["ys"].copy()
    for e in range(wl.E):
        gate = np.zeros(x.shape[0])
        for t in range(x.shape[0]):
            hit = np.nonzero(r["ids"][t] == e)[0]
            if hit.size:
                gate[t] = r["weights"][t, hit[0]]
        wg, wu, wd = M.expert_matrices(tiny, e, wl.fmt)
        acc += gate[:, None] * M.routed_expert(xd, wg, wu, wd)["y"]
    ref = F.round_to_bf16(acc)
    diff = np.abs(ref - r["out"])
    ulp = np.abs(r["out"]) * 2 ** -7
    assert np.all(diff <= ulp)
    assert np.mean(diff == 0) > 0.99


def test_moe_identity_with_shared_expert_in_table():
    """Folded shared expert: the layer equals the dense gate-weighted sum over
    the E routed experts plus table entry E with gate 1 for every token, each
    computed on the MXFP4 token."""
    wl = W.WORKLOADS["tiny_sfp4"]
    lay = W.generate(wl)
    assert lay["w13"].shape[0] == wl.E + 1 and lay["ws13"] is None
    r = M.layer_forward(lay, wl.top_k, wl.fmt)
    x = F.bf16_bits_to_float(lay["x"])
    xq, xs = M.quantize_activations(x)
    xd = F.dequantize_mxfp4(xq, xs)
    acc = np.zeros((x.shape[0], wl.H))
    for e in range(wl.E + 1):
        gate = np.ones(x.shape[0]) if e == wl.E else np.zeros(x.shape[0])
        for t in range(x.shape[0]):
            hit = np.nonzero(r["ids"][t] == e)[0]
            if hit.size:
                gate[t] = r["weights"][t, hit[0]]
        wg, wu, wd = M.expert_matrices(lay, e, wl.fmt)
        acc += gate[:, None] * M.routed_expert(xd, wg, wu, wd)["y"]
    assert not np.any(r["ids"] == wl.E)  # the router never selects the shared expert
    ref = F.round_to_bf16(acc)
    diff = np.abs(ref - r["out"])
    assert np.all(diff <= np.abs(r["out"]) * 2 ** -7)
    assert np.mean(diff == 0) > 0.99


def test_zero_routed_weights_leave_only_shared_expert(tiny):
    wl = W.WORKLOADS["tiny"]
    lay = dict(tiny)
    lay["w2"] = np.zeros_like(tiny["w2"])
    r = M.layer_forward(lay, wl.top_k, wl.fmt)
    x = F.bf16_bits_to_float(tiny["x"])
    ys = M.shared_expert(x, tiny["ws13"], tiny["ws2"])["ys"]
    assert np.array_equal(r["out"], F.round_to_bf16(ys))


def test_identical_experts_reduce_to_one_dense_ffn(tiny):
    """If every routed expert is the same FFN, the renormalised weights sum to
    1 and the layer is shared + that one FFN."""
    wl = W.WORKLOADS["tiny"]
    lay = dict(tiny)
    for key in ["w13", "w13_scale", "w2", "w2_scale"]:
        lay[key] = np.repeat(tiny[key][:1], wl.E, axis=0)
    r = M.layer_forward(lay, wl.top_k, wl.fmt)
    x = F.bf16_bits_to_float(tiny["x"])
    xq, xs = M.quantize_activations(x)
    wg, wu, wd = M.expert_matrices(lay, 0, wl.fmt)
    y = M.routed_expert(F.dequantize_mxfp4(xq, xs), wg, wu, wd)["y"]
    ys = M.shared_expert(x, tiny["ws13"], tiny["ws2"])["ys"]
    ref = ys + y * r["weights"].sum(1, keepdims=True)
    assert np.allclose(r["out"], F.round_to_bf16(ref), rtol=2 ** -7, atol=0)
    assert np.all(np.abs(r["weights"].sum(1) - 1) < 1e-6)


def test_dense_mixture_when_k_equals_E():
    wl = W.Workload("dense4", 5, 64, 32, 4, 4, W.MXFP4, 11, 0.2)
    lay = W.generate(wl)
    r = M.layer_forward(lay, 4, wl.fmt)
    assert all(sorted(row) == [0, 1, 2, 3] for row in r["ids"].tolist())
    p = M.softmax(r["logits"])
    assert np.allclose(np.take_along_axis(p, r["ids"].astype(int), 1), r["weights"], rtol=1e-6)


def test_one_hot_bias_routes_every_token_to_the_same_experts(tiny):
    wl = W.WORKLOADS["tiny"]
    lay = dict(tiny)
    b = np.zeros(wl.E, np.float32)
    b[[3, 7, 11, 12]] = [40, 39, 38, 37]
    lay["bias"] = b
    r = M.layer_forward(lay, wl.top_k, wl.fmt)
    assert np.all(np.sort(r["ids"], 1) == np.array([3, 7, 11, 12]))
    counts, offsets, perm, inv = M.permute(r["ids"], wl.E)
    assert counts[[3, 7, 11, 12]].tolist() == [wl.T] * 4


def test_single_block_shapes():
    wl = W.Workload("oneblock", 3, 32, 32, 4, 2, W.MXFP4, 12, 0.2)
    lay = W.generate(wl)
    r = M.layer_forward(lay, 2, wl.fmt)
    assert r["xs"].shape == (3, 1) and r["out"].shape == (3, 32)
    assert np.all(np.isfinite(r["out"]))


def test_nvfp4_with_power_of_two_scales_equals_mxfp4_layer():
    """An NVFP4 expert whose E4M3 block scales are 2^(s+8) with tensor scale
    2^-8 dequantises to the same values as the MXFP4 expert with E8M0 2^s, so
    the two layers agree bit for bit."""
    wl = W.Workload("nvmx", 4, 64, 64, 4, 2, W.MXFP4, 13, 0.2)
    mx = W.generate(wl)
    nv = dict(mx)

    def to_e4m3(sb):
        s = sb.astype(int) - 127 + 8
        e4 = ((s + 7) << 3).astype(np.uint8)
        return np.repeat(e4, 2, axis=-1)

    nv["w13_scale"] = to_e4m3(mx["w13_scale"])
    nv["w2_scale"] = to_e4m3(mx["w2_scale"])
    nv["tensor_scale"] = np.full((wl.E, 3), 2.0 ** -8, np.float32)
    a = M.layer_forward(mx, 2, "mxfp4")
    b = M.layer_forward(nv, 2, "nvfp4")
    assert np.array_equal(a["out_bits"], b["out_bits"])


def _e4m3_value(code):
    """E4M3 normal encoding s eeee mmm -> 2^(e - 7) (1 + m / 8), written out."""
    e, m = (code >> 3) & 0xF, code & 7
    return 2.0 ** (e - 7) * (1 + m / 8)


def test_nvfp4_per_projection_tensor_scales_closed_form():
    """NVFP4 experts whose gate, up and down projections carry three
    different FP32 tensor scales (one per (expert, projection), the [E, 3]
    layout gate / up / down), some of them not powers of two, worked by hand.

    The structured layer (x = 1, logits (1, 3, 2, 0), top-2 = experts 1, 2):
    gate codes 1.0 with E4M3 block scale 2.0 (0x40), up codes 2.0 with block
    scale 1.5 (0x3C), down codes 1.0 with block scale 0.75 (0x34).  With
    tensor scales (g, u, d) of the expert, the MXFP4 token is exactly 1, so
      G = 64 * 1.0 * 2.0 * g = 128 g,    U = 64 * 2.0 * 1.5 * u = 192 u,
      h = SiLU(G) U, a constant block that requantises to hq = 4X or 6X with
        X = 2^(floor(log2 h) - 2) (6X when h / X > 5),
      y = 32 * hq * 1.0 * 0.75 * d = 24 hq d,
    each rounded to FP32.  Expert 1 takes (3 * 2^-9, float32(0.0371),
    5 * 2^-10), expert 2 takes (float32(0.0371), 3 * 2^-9, 7 * 2^-10): a
    swapped gate / up index, one scale used for all three projections, or
    another expert's scales change G, U or y."""
    lay = _structured_layer([1.0, 3.0, 2.0, 0.0])
    E, H, I = 4, 64, 32
    lay["w13_scale"] = np.concatenate([np.full((E, I, H // 16), 0x40, np.uint8),
                                       np.full((E, I, H // 16), 0x3C, np.uint8)], axis=1)
    lay["w2_scale"] = np.full((E, H, I // 16), 0x34, np.uint8)
    assert (_e4m3_value(0x40), _e4m3_value(0x3C), _e4m3_value(0x34)) == (2.0, 1.5, 0.75)
    a = float(np.float32(0.0371))
    ts = np.array([[1.0, 1.0, 1.0], [3 * 2.0 ** -9, a, 5 * 2.0 ** -10], [a, 3 * 2.0 ** -9, 7 * 2.0 ** -10],
                   [1.0, 1.0, 1.0]], np.float32)
    lay["tensor_scale"] = ts
    r = M.layer_forward(lay, 2, "nvfp4", keep=True)
    assert r["ids"].tolist() == [[1, 2]]
    f32 = lambda v: float(np.float32(v))
    for slot, e in enumerate((1, 2)):
        g, u, d = (float(v) for v in ts[e])
        G, U = f32(128 * g), f32(192 * u)
        h = f32(G / (1 + math.exp(-G)) * U)
        X = 2.0 ** (math.floor(math.log2(h)) - 2)
        hq = (6 if h / X > 5 else 4) * X
        y = f32(24 * hq * d)
        ex = r["experts"][e]
        assert np.all(ex["G"] == G) and np.all(ex["U"] == U), e
        assert np.all(ex["h"] == h), e
        assert np.all(F.dequantize_mxfp4(ex["hq"], ex["hs"]) == hq), e
        assert np.all(r["y"][0, slot] == y), e
    # the hand values differ between the experts and from a shared scale
    assert f32(128 * ts[1, 0]) != f32(128 * ts[1, 1]) and f32(192 * ts[1, 1]) != f32(192 * ts[1, 0])


def test_forced_routing_matches_free_routing_on_same_ids(tiny):
    wl = W.WORKLOADS["tiny"]
    a = M.layer_forward(tiny, wl.top_k, wl.fmt)
    b = M.layer_forward(tiny, wl.top_k, wl.fmt, forced_ids=a["ids"])
    assert np.array_equal(a["out_bits"], b["out_bits"])
    c = M.layer_forward(tiny, wl.top_k, wl.fmt, tokens=[3, 9])
    assert np.array_equal(c["out_bits"], a["out_bits"][[3, 9]])


# ------------------------------------------------------- regression fixture


def test_tiny_layer_regression_fixture(tiny):
    """tests/golden/tiny_layer.txt was written by tests/golden/make_golden.py,
    which calls only the oracle; it guards the oracle against unintended
    change once its pins above hold."""
    path = os.path.join(GOLDEN, "tiny_layer.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    wl = W.WORKLOADS["tiny"]
    r = M.layer_forward(tiny, wl.top_k, wl.fmt)
    for row in rows:
        t = int(row[1])
        if row[0] == "ids":
            assert r["ids"][t].tolist() == [int(v) for v in row[2:]]
        elif row[0] == "out":
            assert r["out_bits"][t].tolist() == [int(v, 16) for v in row[2:]]
