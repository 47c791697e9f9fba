"""GPU parity: every entry point of the C ABI against the CPU oracle.

Bars (the layer's stated tolerances):
* bit-exact: MXFP4 activation codes and scales, routing ids (on logits with
  an unambiguous top-k), the permutation;
* max normwise relative error <= 1e-3 for single contractions (router
  logits, routed expert outputs, shared expert outputs);
* <= 2e-2 for the whole layer output.
A token whose k-th and (k+1)-th oracle logits lie within 1e-5 (relative) is
"ambiguous": either choice is correct, so its ids are only checked to be a
valid top-k and its output is left out of the element-wise comparison.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp4_router_gb300 as M
from block_scaled_fp4_router_gb300 import workloads as W
from block_scaled_fp4_router_gb300.device import DeviceLayer
from oracle import formats as F
from oracle import moe as O

pytestmark = pytest.mark.gpu

LAYER_TOL = 2e-2
CONTRACTION_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from block_scaled_fp4_router_gb300 import build as B

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    M.load()


def normwise(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def bf16_tensor(bits_np):
    return torch.from_numpy(np.ascontiguousarray(bits_np)).view(torch.int16).cuda()


def bits_to_float(t):
    return F.bf16_bits_to_float(t.cpu().numpy().view(np.uint16))


def ambiguous(logits, k, rel=1e-5):
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)
    gap = s[:, k - 1] - s[:, k] if s.shape[1] > k else np.full(s.shape[0], np.inf)
    return gap <= rel * np.maximum(1.0, np.abs(s[:, 0]))


# ----------------------------------------------------------------- A4 quant


def _quant_gpu(x_bits):
    rows, K = x_bits.shape
    x = bf16_tensor(x_bits)
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
    M.moe_quant_act_mxfp4(rows, K, x, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def test_quant_bitexact_random_rows():
    rng = np.random.default_rng(10)
    x = rng.normal(0, 1, (37, 4096)) * np.exp2(rng.integers(-30, 30, (37, 1)))
    x[3, :64] = 0.0                        # all-zero blocks
    x[5, 32:64] = 1e-40                    # subnormal block
    xb = F.bf16_value_to_bits(F.round_to_bf16(x))
    codes, scales = _quant_gpu(xb)
    rc, rs = F.quantize_mxfp4(F.bf16_bits_to_float(xb))
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, F.pack_e2m1(rc))


def test_quant_bitexact_at_every_rounding_midpoint():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    mids = [(a + b) / 2 for a, b in zip(mags[:-1], mags[1:])]
    rows = []
    for scale_exp in (-20, -3, 0, 7):
        for sign in (1, -1):
            blk = np.zeros(32)
            blk[0] = 4.0  # amax 4 -> X = 1 relative to the block's own scale
            blk[1:1 + len(mids)] = sign * np.array(mids)
            blk[10:17] = sign * np.array(mags[1:])
            blk[20] = 7.0 * sign / 8 * 4  # 3.5
            blk[21] = 5.999
            rows.append(blk * 2.0 ** scale_exp)
    x = np.stack(rows).reshape(-1, 128)  # 4 blocks per row
    xb = F.bf16_value_to_bits(F.round_to_bf16(x))
    codes, scales = _quant_gpu(xb)
    rc, rs = F.quantize_mxfp4(F.bf16_bits_to_float(xb))
    assert np.array_equal(scales, rs) and np.array_equal(codes, F.pack_e2m1(rc))


def _quant8_gpu(x_bits):
    rows, K = x_bits.shape
    codes = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
    M.moe_quant_act_mxfp8(rows, K, bf16_tensor(x_bits), codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def test_mxfp8_quant_bitexact():
    """MXFP8 (E4M3) codes and scales equal the oracle's bit for bit: random
    rows over a wide range of magnitudes, every E4M3 rounding midpoint and
    the saturation band (the block's largest element is scaled into
    [256, 512), above E4M3's 448), and all-zero blocks."""
    rng = np.random.default_rng(31)
    x = rng.normal(0, 1, (37, 512)) * 2.0 ** rng.integers(-30, 30, (37, 1))
    mags = F.E4M3_TABLE[:0x7F]
    mid = (mags[:-1] + mags[1:]) / 2
    blk = np.zeros((8, 512))
    for r in range(8):  # each block: amax 2^8 (so X = 1) and 31 midpoints
        vals = rng.choice(mid, (16, 31)) * rng.choice([-1.0, 1.0], (16, 31))
        b = np.concatenate([np.full((16, 1), 256.0), vals], axis=1)
        blk[r] = b.reshape(-1)
    sat = np.zeros((2, 512))
    sat[:, ::32] = 256.0
    sat[:, 1::32] = rng.uniform(448.0, 511.0, (2, 16))
    sat[0, 2::32] = -rng.uniform(448.0, 511.0, 16)
    xb = F.bf16_value_to_bits(F.round_to_bf16(np.concatenate([x, blk, sat, np.zeros((1, 512))])))
    xv = F.bf16_bits_to_float(xb)
    gc, gs = _quant8_gpu(xb)
    oc, os_ = F.quantize_mxfp8(xv)
    assert np.array_equal(gs, os_)
    assert np.array_equal(gc, oc)


def test_quant_ragged_rows_and_small_K():
    rng = np.random.default_rng(11)
    for rows, K in [(1, 32), (3, 96), (5, 160)]:
        xb = F.bf16_value_to_bits(F.round_to_bf16(rng.normal(0, 3, (rows, K))))
        codes, scales = _quant_gpu(xb)
        rc, rs = F.quantize_mxfp4(F.bf16_bits_to_float(xb))
        assert np.array_equal(scales, rs) and np.array_equal(codes, F.pack_e2m1(rc))


# ------------------------------------------------------------ A1 + A2 router


def _router_gpu(x_bits, wr, bias, k, H, E):
    T = x_bits.shape[0]
    d = M.desc(T, H, 128, E, k)
    ws = torch.zeros(M.moe_workspace_size(d), dtype=torch.uint8, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
    b = None if bias is None else torch.from_numpy(bias).cuda()
    M.moe_router_topk(d, bf16_tensor(x_bits), torch.from_numpy(wr).cuda(), b, ids, w, lg, ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy()


@pytest.mark.parametrize("T,H", [(5, 128), (100, 128), (700, 128), (700, 256)])
def test_topk_bitexact_on_exactly_computed_logits(T, H):
    """x rows are one-hot (1.0 at h_t), so logits[t, e] = Wr[e, h_t] exactly on
    any summation order; the logits include exact ties.  Covers the per-row
    router (up to 512 tokens) and the tiled GEMM."""
    rng = np.random.default_rng(12)
    E, k = 64, 4
    h_t = rng.integers(0, H, T)
    x = np.zeros((T, H))
    x[np.arange(T), h_t] = 1.0
    wr = rng.normal(0, 1, (E, H)).astype(np.float32)
    wr[:8, :] = wr[8:16, :]          # duplicated rows -> tied logits
    wr[20:24, 5] = wr[3, 5]
    xb = F.bf16_value_to_bits(x)
    ids, w, lg = _router_gpu(xb, wr, None, k, H, E)
    ref_logits = O.router_logits(F.bf16_bits_to_float(xb), wr)
    assert np.array_equal(lg, ref_logits.astype(np.float32))
    rid, rw = O.route(ref_logits, k)
    assert np.array_equal(ids, rid)
    assert np.allclose(w, rw, rtol=1e-6, atol=0)


@pytest.mark.parametrize("wl_name,T", [("tiny", 16), ("decode1", 1), ("decode16z", 16), ("prefill8k", 300), ("prefill8k", 600)])
def test_router_topk_random(wl_name, T):
    wl = W.WORKLOADS[wl_name]
    lay = W.generate(wl, tokens=T)
    ids, w, lg = _router_gpu(lay["x"], lay["w_router"], lay["bias"], wl.top_k, wl.H, wl.E)
    ref = O.router_logits(F.bf16_bits_to_float(lay["x"]), lay["w_router"], lay["bias"])
    assert normwise(lg, ref) <= 1e-5
    # element-wise: an FP32-accurate dot product (error within 1e-7 of sum |x w|;
    # a BF16 rounding of the weights, or tensor-core accumulation over H, exceeds it)
    mag = np.abs(F.bf16_bits_to_float(lay["x"])) @ np.abs(lay["w_router"].astype(np.float64)).T
    ratio = np.max(np.abs(lg - ref) / (mag + 1e-30))
    assert ratio <= 1e-7, ratio
    rid, rw = O.route(ref, wl.top_k)
    amb = ambiguous(ref, wl.top_k)
    assert np.array_equal(ids[~amb], rid[~amb])
    assert np.allclose(w[~amb], rw[~amb], rtol=1e-5, atol=1e-7)
    assert amb.sum() <= max(1, T // 100)


# ------------------------------------------------------------- A3 permute


@pytest.mark.parametrize("T,k,E", [(1, 4, 128), (16, 4, 16), (700, 4, 128), (8192, 4, 128), (33, 8, 256),
                                   (5, 1, 4)])
def test_permute_bitexact(T, k, E):
    rng = np.random.default_rng(T * 7 + E)
    # Zipf-skewed ids with repeats allowed: exercises several blocks and ragged tails
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    ids_np = rng.choice(E, size=(T, k), p=p / p.sum()).astype(np.int32)
    d = M.desc(T, 128, 128, E, k)
    ws = torch.zeros(M.moe_workspace_size(d), dtype=torch.uint8, device="cuda")
    n = T * k
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(n, dtype=torch.int32, device="cuda")
    inv = torch.empty(n, dtype=torch.int32, device="cuda")
    M.moe_permute(d, torch.from_numpy(ids_np).cuda(), counts, offsets, perm, inv, ws)
    torch.cuda.synchronize()
    rc, ro, rp, ri = O.permute(ids_np, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(inv.cpu().numpy(), ri)


# ------------------------------------------------------------ layer fixtures

_CACHE = {}


def _workload(name, T=None):
    """(workload, host arrays, device layer, oracle expert cache), cached."""
    key = (name, T)
    if key not in _CACHE:
        wl = W.WORKLOADS[name]
        if T is not None:
            wl = wl.with_tokens(T)
        lay = W.generate(wl)
        dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=wl.T)
        _CACHE.clear()  # keep at most one large layer resident
        _CACHE[key] = (wl, lay, dev, {})
    return _CACHE[key]


def _compare_layer(wl, lay, cache, out, ids, tokens=None, tol=LAYER_TOL, w=None):
    r = O.layer_forward(lay, wl.top_k, wl.fmt, tokens=tokens, cache=cache)
    # ambiguity on the values the selection ranks (logits, or sigmoid + bias)
    amb = ambiguous(O.selection_keys(r["logits"], lay.get("score", "softmax"), lay.get("bias")), wl.top_k)
    tok = r["tokens"]
    g_ids = ids.cpu().numpy()[tok]
    assert np.array_equal(g_ids[~amb], r["ids"][~amb])
    if w is not None:  # the renormalised routing weights of the same tokens
        assert np.allclose(w.cpu().numpy()[tok][~amb], r["weights"][~amb], rtol=1e-5, atol=1e-7)
    g_out = bits_to_float(out)[tok]
    assert np.all(np.isfinite(g_out))
    err = normwise(g_out[~amb], r["out"][~amb])
    assert err <= tol, err
    return err


# ------------------------------------------------------ A5 - A8 expert FFNs

_E2M1_THRESHOLDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _oracle_h_sorted(ref, inv, T, k, I):
    """Oracle's h (float32 values), requantised codes and scales, in sorted order."""
    n = T * k
    h = np.zeros((n, I))
    hq = np.zeros((n, I), np.uint8)
    hs = np.zeros((n, I // 32), np.uint8)
    for e, r in ref["experts"].items():
        p = inv[r["rows"] * k + r["slots"]]
        h[p], hq[p], hs[p] = r["h"], r["hq"], r["hs"]
    return h, hq, hs


def _down_on_gpu_h(lay, fmt, offsets, gq, gs, H):
    """The down projection of every sorted assignment row from the GPU's own
    requantised h (E2M1 codes gq [n, I], E8M0 scales gs [n, I/32]), both
    operands dequantised exactly with the oracle's format routines and
    contracted in float64: the A7 contraction on identically quantised
    inputs.  Row p belongs to the expert e with offsets[e] <= p < offsets[e+1]."""
    hd = F.dequantize_mxfp4(gq, gs)
    y = np.zeros((gq.shape[0], H))
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        c2 = F.unpack_e2m1(lay["w2"][e])
        if fmt == W.MXFP4:
            w2 = F.dequantize_mxfp4(c2, lay["w2_scale"][e])
        else:
            w2 = F.dequantize_nvfp4(c2, lay["w2_scale"][e], float(lay["tensor_scale"][e][2]))
        y[a:b] = hd[a:b] @ w2.T
    return F.round_to_f32(y)


def _check_requant_and_down(dev, d, ref, inv, y_assign, T, k, I, H, lay, fmt, offsets):
    """A6 + A7 on identically quantised inputs.  The GPU's MXFP4 h must equal
    the oracle's block for block, except blocks where the oracle's h lies
    within 1e-5 (relative) of a rounding threshold or of a change of the
    block exponent (G and U are FP32 sums whose order differs).  Every row of
    y must agree within the contraction tolerance with the down projection of
    the GPU's own h (identical quantised inputs), and with the oracle's y
    within the layer tolerance."""
    n = T * k
    ghq = torch.empty((n, I // 2), dtype=torch.uint8, device="cuda")
    ghs = torch.empty((n, I // 32), dtype=torch.uint8, device="cuda")
    M.moe_debug_requantized_h(d, dev.ws, ghq, ghs)
    torch.cuda.synchronize()
    gq = F.unpack_e2m1(ghq.cpu().numpy()).reshape(n, I // 32, 32)
    gs = ghs.cpu().numpy()
    h, oq, os_ = _oracle_h_sorted(ref, inv, T, k, I)
    oq = oq.reshape(n, I // 32, 32)
    same = np.all(gq == oq, axis=2) & (gs == os_)
    hb = h.reshape(n, I // 32, 32)
    amax = np.abs(hb).max(2)
    X = F.E8M0_TABLE[os_]
    near_scale = np.abs(amax / 2.0 ** np.floor(np.log2(np.maximum(amax, 1e-300))) - 1) < 1e-5
    sv = np.abs(hb) / X[..., None]
    near_code = np.any(np.min(np.abs(sv[..., None] / _E2M1_THRESHOLDS - 1), axis=-1) < 1e-5, axis=2)
    assert np.all(same | near_scale | near_code), "requantised h differs away from a rounding boundary"
    assert same.mean() >= 0.999, same.mean()
    y_ref = ref["y"].reshape(n, H)[np.argsort(inv)]
    ya = y_assign.cpu().numpy()
    y_same_h = _down_on_gpu_h(lay, fmt, offsets, gq.reshape(n, I), gs, H)
    assert normwise(ya, y_same_h) <= CONTRACTION_TOL, normwise(ya, y_same_h)
    assert normwise(ya, y_ref) <= LAYER_TOL


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode16", "batch128"])
def test_expert_ffn_contractions(name):
    """Routed expert outputs y (per sorted assignment) and the shared expert
    output ys against the oracle, on the same MXFP4 activations (the GPU's own
    quantiser output, bit-identical to the oracle's by the tests above)."""
    wl, lay, dev, cache = _workload(name)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.top_k
    x = F.bf16_bits_to_float(lay["x"])
    ref = O.layer_forward(lay, k, wl.fmt, cache=cache, keep=True)
    ids_np = ref["ids"]
    counts, offsets, perm, inv = O.permute(ids_np, E)
    d = dev.desc(T)
    xt = bf16_tensor(lay["x"])
    xq = torch.empty((T, H // 2), dtype=torch.uint8, device="cuda")
    xs = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")
    M.moe_quant_act_mxfp4(T, H, xt, xq, xs)
    g_off = torch.from_numpy(offsets).cuda()
    g_perm = torch.from_numpy(perm).cuda()
    y_assign = torch.empty((T * k, H), dtype=torch.float32, device="cuda")
    y_shared = torch.empty((T, H), dtype=torch.float32, device="cuda")
    M.moe_expert_ffn_fp4(d, dev.ex, dev.sh, xt, xq, xs, g_off, g_perm, y_assign, y_shared, dev.ws)
    torch.cuda.synchronize()
    y_ref = ref["y"].reshape(T * k, H)[perm]  # oracle y in sorted-assignment order
    if T * k >= 256:  # the tensor-core path: check that its tiles cover every row
        assert np.all(np.abs(y_assign.cpu().numpy()).max(1) > 0)
    _check_requant_and_down(dev, d, ref, inv, y_assign, T, k, I, H, lay, wl.fmt, offsets)
    assert normwise(y_shared.cpu().numpy(), ref["ys"]) <= CONTRACTION_TOL
    # combine alone on the oracle's expert outputs: out = BF16(ys + sum w y)
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    M.moe_combine(d, torch.from_numpy(y_ref.astype(np.float32)).cuda(), torch.from_numpy(inv).cuda(),
                  torch.from_numpy(ref["weights"].astype(np.float32)).cuda(),
                  torch.from_numpy(ref["ys"].astype(np.float32)).cuda(), out)
    torch.cuda.synchronize()
    g = bits_to_float(out)
    ulp = np.abs(ref["out"]) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(g - ref["out"]) <= ulp)


# ----------------------------------------------------------- whole layer


def _use_prepared(dev, prepared):
    """Selects the tensor-core decode (prepared scales) or the CUDA-core one."""
    dev.set_prepared(prepared)


@pytest.mark.parametrize("prepared", [True, False], ids=["tcgen05", "cudacore"])
@pytest.mark.parametrize("name", ["tiny", "decode1", "decode16", "decode16z", "tiny_sfp4", "decode1_sfp4",
                                  "tiny_sig", "decode16_sig"])
def test_layer_decode_fused(name, prepared):
    wl, lay, dev, cache = _workload(name)
    _use_prepared(dev, prepared)
    out, ids, w = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, cache, out, ids)
    # the fused launch is deterministic and leaves the workspace reusable
    out2, ids2, _ = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(ids, ids2)
    dev.set_prepared(dev.ex_prepared is not None)


def test_prepared_scales_are_the_tensor_core_layout():
    """moe_prepare_weights writes each 128-row x 128-element scale block as
    512 bytes, word 4i + j (little-endian bytes) holding the four scales of
    row 32j + i, blocks ordered [expert][row tile][K group]."""
    wl, lay, dev, cache = _workload("tiny")
    E, H, I = wl.E, wl.H, wl.I

    def relayout(s, R, K):
        s = s.reshape(E, R // 128, 4, 32, K // 128, 4)        # e, rt, j, i, g, byte
        return s.transpose(0, 1, 4, 3, 2, 5).reshape(-1)       # e, rt, g, i, j, byte

    assert np.array_equal(dev.w13_scale_mma.cpu().numpy().reshape(-1), relayout(lay["w13_scale"], 2 * I, H))
    assert np.array_equal(dev.w2_scale_mma.cpu().numpy().reshape(-1), relayout(lay["w2_scale"], H, I))
    # NVFP4: E4M3 per 16, so 4 bytes of a row cover 64 elements (the same map over 2K)
    wl16, lay16, dev16, _ = _workload("decode16")
    E, H, I = wl16.E, wl16.H, wl16.I
    assert np.array_equal(dev16.w2_scale_mma.cpu().numpy().reshape(-1), relayout(lay16["w2_scale"], H, 2 * I))

@pytest.mark.parametrize("name", ["tiny", "decode1", "decode16", "decode1_sfp4", "tiny_sig", "decode16_sig"])
def test_layer_forward_matches_decode(name):
    wl, lay, dev, cache = _workload(name)
    out_f, ids_f, w_f = dev.forward(bf16_tensor(lay["x"]))
    out_d, ids_d, w_d = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    _compare_layer(wl, lay, cache, out_f, ids_f)
    assert torch.equal(ids_f, ids_d)
    assert normwise(bits_to_float(out_f), bits_to_float(out_d)) <= 1e-2


@pytest.mark.parametrize("prepared", [True, False], ids=["tcgen05", "cudacore"])
@pytest.mark.parametrize("T", [1, 2, 7, 13, 16])
def test_decode_token_counts(T, prepared):
    wl, lay, dev, cache = _workload("tiny")
    _use_prepared(dev, prepared)
    sub = dict(lay)
    sub["x"] = lay["x"][:T]
    out, ids, _ = dev.decode(bf16_tensor(sub["x"]))
    torch.cuda.synchronize()
    _compare_layer(wl.with_tokens(T), sub, cache, out, ids)
    dev.set_prepared(True)


@pytest.mark.parametrize("shape", [
    (17, 512, 256, 16, 4, W.MXFP4, {}),
    (33, 512, 512, 32, 4, W.NVFP4, {}),
    (64, 768, 256, 64, 6, W.MXFP4, dict(shared=False)),
    (100, 256, 512, 255, 8, W.MXFP4, {}),
    (128, 512, 256, 16, 7, W.NVFP4, dict(shared=False, shared_fp4=True)),
    (128, 256, 256, 8, 8, W.MXFP4, {}),
    (96, 512, 256, 32, 4, W.MXFP4, dict(score="sigmoid", zipf=0.05)),
    (128, 256, 256, 256, 8, W.MXFP4, dict(shared=False)),
    (100, 512, 256, 64, 4, W.NVFP4, dict(shared_fmt="mxfp8")),
], ids=["T17", "T33_nvfp4", "T64_k6_noshared", "T100_E255_k8", "T128_nvfp4_fold_n1024", "T128_dense",
        "T96_sigmoid", "T128_E256_k8_n1024", "T100_nvfp4_mxfp8_shared"])
def test_wide_single_launch_shapes(shape):
    """Steps of 17-128 tokens through moe_layer_decode, one launch: a ragged
    last 16-token chunk (17, 33, 100), E = 255 with k = 8 (800 assignments),
    the folded shared expert at the largest table step (128 tokens x 8 = 1024
    assignments, every expert split over several 16-row slots), a dense
    mixture (E == k: 128 rows per expert, 8 slots each), 1024 assignments over
    256 experts (up to 320 slots, the shared-memory table's bound), NVFP4
    with distinct tensor scales and an MXFP8 shared expert, sigmoid scoring.
    Every token against the oracle; the launch is bit-reproducible and agrees
    with the batched path."""
    T, H, I, E, k, fmt, kw = shape
    # router weights of std 0.08: logits of std ~1-2 (the workloads' regime),
    # where the FP32 router's rounding stays far below the weights' rtol
    wl = W.Workload("wide", T, H, I, E, k, fmt, 27, 0.08, **kw)
    lay = W.generate(wl)
    dev = DeviceLayer(lay, H, I, E, k, wl.fmt, T_max=T)
    assert dev.prepared
    x = bf16_tensor(lay["x"])
    n0 = M.moe_debug_launch_count()
    out, ids, w = dev.decode(x)
    torch.cuda.synchronize()
    assert M.moe_debug_launch_count() == n0 + 1
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, {}, out, ids, w=w)
    out2, ids2, _ = dev.decode(x)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(ids, ids2)
    out_f, ids_f, _ = dev.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_f)
    assert normwise(bits_to_float(out), bits_to_float(out_f)) <= 1e-2


@pytest.mark.parametrize("name", ["batch128", "batch128_sfp4", "batch128_sig"])
def test_batch128_single_launch_every_token(name):
    """The 128-token step at full size (H = 4096, I = 1536, E = 128, top-4)
    in one launch of the tensor-core decode, every token against the oracle."""
    wl, lay, dev, cache = _workload(name)
    n0 = M.moe_debug_launch_count()
    out, ids, w = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_debug_launch_count() == n0 + 1
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, cache, out, ids, w=w)


@pytest.fixture
def routed_gemm():
    """Sets the routed GEMM orientation for one test, automatic afterwards."""
    yield M.moe_set_routed_gemm
    M.moe_set_routed_gemm(M.ROUTED_GEMM_AUTO)


@pytest.mark.parametrize("gemm", [M.ROUTED_GEMM_AUTO, M.ROUTED_GEMM_TOKENS_AS_A], ids=["auto", "tokens_as_A"])
def test_batch128_forward_every_token(gemm, routed_gemm):
    """The 128-token batched decode layer through moe_layer_forward, every
    token against the oracle (ids, weights, output), in both orientations of
    the routed tensor-core GEMMs."""
    routed_gemm(gemm)
    wl, lay, dev, cache = _workload("batch128")
    out, ids, w = dev.forward(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, cache, out, ids, w=w)


@pytest.mark.parametrize("name,T", [("tiny_sfp4", 16), ("batch128_sfp4", 128), ("decode1_sfp4", 1)])
def test_layer_forward_shared_in_table(name, T):
    """The shared expert folded into the FP4 table (expert E, weight 1) through
    the batched path: CUDA-core routed experts for a few assignments,
    weights-as-A tensor-core GEMMs for batch128 (a 128-token window of the
    shared expert next to ~4-token windows of the routed ones)."""
    wl, lay, dev, cache = _workload(name, T if T != W.WORKLOADS[name].T else None)
    out, ids, w = dev.forward(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    assert ids.shape == (T, wl.top_k) and int(ids.max()) < wl.E  # the router's top-k only
    tokens = None if T <= 16 else np.sort(np.random.default_rng(15).choice(T, 24, replace=False))
    _compare_layer(wl, lay, cache, out, ids, tokens=tokens)


def test_batch128_sigmoid_scoring_every_token():
    """Sigmoid scores with a bias-corrected top-k choice (the bias moves the
    choice, not the weights) through the batched path, every token against the
    oracle (ids, weights, output), and the router entry point on the same
    tokens: its logits are the raw products, without the bias."""
    wl, lay, dev, cache = _workload("batch128_sig")
    out, ids, w = dev.forward(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, cache, out, ids, w=w)
    # the bias changes the choice for a good share of the tokens
    x = F.bf16_bits_to_float(lay["x"])
    raw = O.router_logits(x, lay["w_router"])
    sel_sig, _ = O.route(raw, wl.top_k, score="sigmoid", bias=lay["bias"])
    sel_nob, _ = O.route(raw, wl.top_k, score="sigmoid")
    assert np.mean(np.any(sel_sig != sel_nob, axis=1)) > 0.2
    d = dev.desc(wl.T)
    g_ids = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device="cuda")
    g_w = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device="cuda")
    g_lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    M.moe_router_topk(d, bf16_tensor(lay["x"]), dev.w_router, dev.bias, g_ids, g_w, g_lg, dev.ws)
    torch.cuda.synchronize()
    mag = np.abs(x) @ np.abs(lay["w_router"].astype(np.float64)).T
    assert np.max(np.abs(g_lg.cpu().numpy() - raw) / (mag + 1e-30)) <= 1e-7
    keys = O.selection_keys(raw, "sigmoid", lay["bias"])
    amb = ambiguous(keys, wl.top_k)
    assert np.array_equal(g_ids.cpu().numpy()[~amb], sel_sig[~amb])


def test_prefill8k_forward_every_token():
    """The 8192-token prefill layer (Zipf(1.1) expert load) through
    moe_layer_forward in the launch configuration the benchmark times: every
    token's ids, weights and output against the oracle run over the whole
    batch (one pass over the 128 experts, dequantised one at a time)."""
    wl, lay, dev, _ = _workload("prefill8k")
    out, ids, w = dev.forward(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    # Zipf(1.1) load: the realised per-expert histogram is skewed
    counts = np.bincount(ids.cpu().numpy().ravel(), minlength=wl.E)
    assert counts.sum() == wl.T * wl.top_k and counts.max() > 4 * counts.mean()
    _compare_layer(wl, lay, None, out, ids, w=w)


# ---------------------------------------------------- tensor-core path shapes


@pytest.mark.parametrize("gemm", [M.ROUTED_GEMM_TOKENS_AS_A, M.ROUTED_GEMM_WEIGHTS_AS_A],
                         ids=["tokens_as_A", "weights_as_A"])
@pytest.mark.parametrize("shape", [(64, 256, 256, 8, 4), (160, 512, 256, 16, 4), (130, 256, 512, 4, 2),
                                   (300, 512, 512, 32, 8), (90, 256, 256, 64, 3)])
def test_tensor_core_path_shapes(shape, gemm, routed_gemm):
    """From 256 assignments the MXFP4 experts run on tcgen05 tensor cores
    (and the shared expert from 128 tokens), in either orientation of the
    routed GEMMs: ragged per-expert tiles and token windows (experts with
    1-15, 16-64 and more than 64 assignments), several K stages, both entry
    points."""
    T, H, I, E, k = shape
    routed_gemm(gemm)
    wl = W.Workload("tc", T, H, I, E, k, W.MXFP4, 23, 0.05)
    lay = W.generate(wl)
    dev = DeviceLayer(lay, H, I, E, k, wl.fmt, T_max=T)
    cache = {}
    out, ids, _ = dev.forward(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, cache, out, ids)
    ref = O.layer_forward(lay, k, wl.fmt, cache=cache, keep=True)
    counts, offsets, perm, inv = O.permute(ref["ids"], E)
    d = dev.desc(T)
    xt = bf16_tensor(lay["x"])
    xq = torch.empty((T, H // 2), dtype=torch.uint8, device="cuda")
    xs = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")
    M.moe_quant_act_mxfp4(T, H, xt, xq, xs)
    y_assign = torch.full((T * k, H), float("nan"), dtype=torch.float32, device="cuda")
    y_shared = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    M.moe_expert_ffn_fp4(d, dev.ex, dev.sh, xt, xq, xs, torch.from_numpy(offsets).cuda(),
                         torch.from_numpy(perm).cuda(), y_assign, y_shared, dev.ws)
    torch.cuda.synchronize()
    ya = y_assign.cpu().numpy()
    assert np.all(np.isfinite(ya)) and np.all(np.isfinite(y_shared.cpu().numpy()))
    _check_requant_and_down(dev, d, ref, inv, y_assign, T, k, I, H, lay, wl.fmt, offsets)
    assert normwise(y_shared.cpu().numpy(), ref["ys"]) <= CONTRACTION_TOL


# ------------------------------------------------- NVFP4 -> MXFP4 conversion


def _random_nvfp4_layer(rng, E, H, I, scale_codes):
    def mat(R, K):
        codes = rng.integers(0, 16, (E, R, K)).astype(np.uint8)
        return F.pack_e2m1(codes), codes, rng.choice(scale_codes, (E, R, K // 16)).astype(np.uint8)
    w13p, w13c, w13s = mat(2 * I, H)
    w2p, w2c, w2s = mat(H, I)
    # non-power-of-two FP32 tensor scales, one per (expert, gate / up / down)
    ts = rng.uniform(1e-3, 3e-2, (E, 3)).astype(np.float32)
    return w13p, w13c, w13s, w2p, w2c, w2s, ts


def test_nvfp4_to_mxfp4_conversion_bitexact():
    """Every code and scale byte equals the oracle's exact requantisation,
    for random codes, E4M3 scales over normal and subnormal encodings, and
    non-power-of-two tensor scales."""
    rng = np.random.default_rng(31)
    E, H, I = 6, 512, 256
    scale_codes = np.concatenate([np.arange(0x01, 0x08), np.arange(0x20, 0x60)])
    w13p, w13c, w13s, w2p, w2c, w2s, ts = _random_nvfp4_layer(rng, E, H, I, scale_codes)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    d13p, d13s, d2p, d2s, dts = dev(w13p), dev(w13s), dev(w2p), dev(w2s), dev(ts)
    ex = M.experts(M.MOE_W_NVFP4, d13p, d13s, d2p, d2s, dts)
    o13 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device="cuda")
    o13s = torch.empty((E, 2 * I, H // 32), dtype=torch.uint8, device="cuda")
    o2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device="cuda")
    o2s = torch.empty((E, H, I // 32), dtype=torch.uint8, device="cuda")
    M.moe_convert_nvfp4_to_mxfp4(M.desc(1, H, I, E, 4), ex, o13, o13s, o2, o2s)
    torch.cuda.synchronize()
    for e in range(E):
        tsr = np.where(np.arange(2 * I) < I, ts[e, 0], ts[e, 1])  # per row: gate, then up
        rc, rs = F.requantize_nvfp4_to_mxfp4(w13c[e], w13s[e], tsr)
        assert np.array_equal(o13[e].cpu().numpy(), F.pack_e2m1(rc))
        assert np.array_equal(o13s[e].cpu().numpy(), rs)
        rc, rs = F.requantize_nvfp4_to_mxfp4(w2c[e], w2s[e], ts[e, 2])
        assert np.array_equal(o2[e].cpu().numpy(), F.pack_e2m1(rc))
        assert np.array_equal(o2s[e].cpu().numpy(), rs)
    with pytest.raises(M.MoeError):  # the source must be NVFP4
        M.moe_convert_nvfp4_to_mxfp4(M.desc(1, H, I, E, 4), M.experts(M.MOE_W_MXFP4, d13p, o13s, d2p, o2s), o13,
                                     o13s, o2, o2s)


def test_decode_on_converted_weights():
    """An NVFP4 layer converted on the GPU runs as an MXFP4 layer: the decode
    matches the oracle on the oracle's own conversion of the same weights."""
    wl = W.WORKLOADS["tiny"]
    nv = W.Workload("tiny_nv", wl.T, wl.H, wl.I, wl.E, wl.top_k, W.NVFP4, 27, wl.wr_std)
    lay = W.generate(nv)
    E, H, I = nv.E, nv.H, nv.I
    src = DeviceLayer(lay, H, I, E, nv.top_k, nv.fmt, T_max=nv.T, prepare=False)
    o13 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device="cuda")
    o13s = torch.empty((E, 2 * I, H // 32), dtype=torch.uint8, device="cuda")
    o2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device="cuda")
    o2s = torch.empty((E, H, I // 32), dtype=torch.uint8, device="cuda")
    M.moe_convert_nvfp4_to_mxfp4(src.desc(nv.T), src.ex, o13, o13s, o2, o2s)
    torch.cuda.synchronize()
    mx = dict(lay)
    ts = lay["tensor_scale"]
    ts13 = np.where(np.arange(2 * I)[None, :] < I, ts[:, 0:1], ts[:, 1:2])  # [E, 2I]: gate rows, up rows
    c13, s13 = F.requantize_nvfp4_to_mxfp4(F.unpack_e2m1(lay["w13"]), lay["w13_scale"], ts13)
    c2, s2 = F.requantize_nvfp4_to_mxfp4(F.unpack_e2m1(lay["w2"]), lay["w2_scale"], ts[:, 2:3])
    mx.update(w13=F.pack_e2m1(c13), w13_scale=s13, w2=F.pack_e2m1(c2), w2_scale=s2, tensor_scale=None)
    assert np.array_equal(o13.cpu().numpy(), mx["w13"]) and np.array_equal(o2s.cpu().numpy(), mx["w2_scale"])
    mxw = W.Workload("tiny_conv", nv.T, H, I, E, nv.top_k, W.MXFP4, 27, wl.wr_std)
    dev = DeviceLayer(mx, H, I, E, nv.top_k, W.MXFP4, T_max=nv.T)
    out, ids, _ = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    _compare_layer(mxw, mx, {}, out, ids)


# --------------------------------------------------------------- edge cases


@pytest.mark.parametrize("shape", [(4, 128, 128, 4, 4, W.MXFP4), (9, 256, 128, 8, 2, W.MXFP4),
                                   (3, 128, 256, 256, 8, W.MXFP4), (3, 32, 32, 4, 2, W.MXFP4),
                                   (5, 32, 32, 4, 2, W.NVFP4), (13, 96, 160, 8, 4, W.MXFP4),
                                   (70, 160, 96, 8, 4, W.NVFP4), (140, 96, 224, 16, 2, W.MXFP4),
                                   (6, 192, 320, 8, 4, W.NVFP4), (16, 320, 192, 8, 3, W.MXFP4)])
def test_small_and_degenerate_shapes(shape):
    """Dense mixture (E == k), E = 256 with k = 8, and H, I that only hold
    whole 32-element blocks: the single-block layer H = I = 32 (one MXFP4
    block along each), and shapes no tensor-core tile divides (CUDA-core
    paths: the single-launch decode where H and I are multiples of 64, the
    per-step kernels otherwise; 70 and 140 tokens take the batched path with
    >= 256 assignments)."""
    T, H, I, E, k, fmt = shape
    wl = W.Workload("edge", T, H, I, E, k, fmt, 21, 0.5)
    lay = W.generate(wl)
    dev = DeviceLayer(lay, H, I, E, k, wl.fmt, T_max=T)
    cache = {}
    if T <= 16:
        out, ids, _ = dev.decode(bf16_tensor(lay["x"]))
        torch.cuda.synchronize()
        _compare_layer(wl, lay, cache, out, ids)
    out, ids, _ = dev.forward(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    _compare_layer(wl, lay, cache, out, ids)


@pytest.mark.parametrize("shape", [(5, 256, 256, 256, 8, W.MXFP4), (16, 256, 512, 4, 4, W.MXFP4),
                                   (1, 768, 768, 8, 2, W.MXFP4), (11, 1024, 256, 64, 6, W.MXFP4),
                                   (6, 768, 512, 24, 4, W.NVFP4), (16, 256, 256, 256, 8, W.NVFP4),
                                   (3, 512, 2560, 8, 4, W.NVFP4)])
def test_tensor_core_decode_shapes(shape):
    """The tcgen05 decode on E = 256 with k = 8, a dense mixture (E == k) at
    16 tokens, odd numbers of K chunks (H = I = 768), a mid-size case and
    three NVFP4 layers, one with I = 2560 (h's UE4M3 scale blocks converted
    in two chunks of 32); the CUDA-core decode on the same layer agrees."""
    T, H, I, E, k, fmt = shape
    wl = W.Workload("dcedge", T, H, I, E, k, fmt, 24, 0.5)
    lay = W.generate(wl)
    dev = DeviceLayer(lay, H, I, E, k, wl.fmt, T_max=T)
    cache = {}
    out, ids, _ = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, cache, out, ids)
    dev.set_prepared(False)
    out_c, ids_c, _ = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_c)
    assert normwise(bits_to_float(out), bits_to_float(out_c)) <= 1e-2


def test_decode_after_large_forward_on_one_workspace():
    """A workspace sized for a 300-token forward also serves single-launch steps:
    the forward's scratch never lands where the decode expects its zeroed
    tickets and launch-tagged logits."""
    H, I, E, k = 512, 256, 16, 4
    wl = W.Workload("mixed", 300, H, I, E, k, W.MXFP4, 26, 0.05)
    lay = W.generate(wl)
    dev = DeviceLayer(lay, H, I, E, k, wl.fmt, T_max=300)
    cache = {}
    for _ in range(2):
        out, ids, _ = dev.forward(bf16_tensor(lay["x"]))
        torch.cuda.synchronize()
        for T in (1, 5, 16, 40):
            sub = dict(lay)
            sub["x"] = lay["x"][:T]
            o, i, _ = dev.decode(bf16_tensor(sub["x"]))
            torch.cuda.synchronize()
            assert M.moe_get_status(dev.ws) == M.MOE_OK
            _compare_layer(wl.with_tokens(T), sub, cache, o, i)


def test_nvfp4_decode_across_launch_number_wrap():
    """The tensor-core NVFP4 decode tags its router logits and its per-row h
    exponents (combined by atomicMax) with a 32-bit launch number kept in the
    workspace.  Seeded two launches below the wrap, three launches whose
    tokens differ in magnitude by 2^6 (so their h row exponents differ) each
    match the oracle: nothing left by the launch before the wrap survives into
    the launches after it."""
    wl = W.Workload("wrap_nv", 16, 512, 256, 16, 4, W.NVFP4, 33, 0.05)
    lay = W.generate(wl)
    dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=wl.T)
    assert dev.prepared
    C_DC_EPOCH = 12
    dev.ws[:64].view(torch.int32)[C_DC_EPOCH] = -2  # the next launch is number 0xFFFFFFFF
    cache = {}
    for i, mag in enumerate((2.0 ** 6, 1.0, 2.0 ** 3)):
        x = F.bf16_bits_to_float(W.generate_tokens(wl, 40 + i, wl.T)) * mag
        sub = dict(lay)
        sub["x"] = F.bf16_value_to_bits(F.round_to_bf16(x))
        out, ids, _ = dev.decode(bf16_tensor(sub["x"]))
        torch.cuda.synchronize()
        assert M.moe_get_status(dev.ws) == M.MOE_OK
        _compare_layer(wl, sub, cache, out, ids)
    assert int(dev.ws[:64].view(torch.int32)[C_DC_EPOCH]) == 2  # 0xFFFFFFFF, then 1 and 2 (0 is skipped)


def test_tensor_core_decode_without_shared_expert():
    wl = W.Workload("noshared_mx", 3, 512, 512, 16, 4, W.MXFP4, 25, 0.05, shared=False)
    lay = W.generate(wl)
    dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=wl.T)
    assert dev.prepared
    out, ids, _ = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, {}, out, ids)


def test_layer_without_shared_expert():
    wl = W.Workload("noshared", 6, 512, 256, 16, 4, W.NVFP4, 22, 0.05, shared=False)
    lay = W.generate(wl)
    dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=wl.T)
    cache = {}
    for fn in (dev.decode, dev.forward):
        out, ids, _ = fn(bf16_tensor(lay["x"]))
        torch.cuda.synchronize()
        _compare_layer(wl, lay, cache, out, ids)


@pytest.mark.parametrize("nbytes", [16, 8192, (1 << 20) + 16])
def test_copy_rows_pinned_host_and_device(nbytes):
    """moe_copy_rows moves bytes exactly: pinned host -> device -> pinned host,
    eagerly and replayed from a CUDA graph; pageable host memory is refused."""
    rng = np.random.default_rng(nbytes)
    src = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    M.moe_copy_rows(dev, src)
    M.moe_copy_rows(back, dev)
    torch.cuda.synchronize()
    assert torch.equal(back, src) and torch.equal(dev.cpu(), src)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    back.zero_()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        M.moe_copy_rows(dev, src, stream=s)
        M.moe_copy_rows(back, dev, stream=s)
    src.copy_(torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    pageable = torch.zeros(nbytes, dtype=torch.uint8)
    with pytest.raises(M.MoeError) as e:
        M.moe_copy_rows(dev, pageable)
    assert e.value.status == M.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("T,H,I", [(16, 512, 256), (130, 512, 512), (1, 4096, 1536)])
def test_shared_expert_mxfp8(T, H, I):
    """The MXFP8 shared expert on kind::mxf8f6f4 tensor cores against the
    oracle: the same MXFP8 token (bit-exact quantiser), FP32 G / U, MXFP8 h;
    ragged token tiles (130 = 128 + 2) and a decode shape (K = 4096)."""
    wl = W.Workload("s8", T, H, I, 16, 4, W.MXFP4, 29, 0.02)
    arr = W.generate_shared_mxfp8(wl, 29 + T)
    xb = W.generate_tokens(wl, 31 + T, T)
    d = M.desc(T, H, I, 16, 4)
    ws = torch.zeros(M.moe_workspace_size(d), dtype=torch.uint8, device="cuda")
    dev = {k: torch.from_numpy(v).cuda() for k, v in arr.items()}
    sh8 = M.shared_mxfp8(dev["s8_w13"], dev["s8_w13_scale"], dev["s8_w2"], dev["s8_w2_scale"])
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    M.moe_shared_expert_mxfp8(d, sh8, bf16_tensor(xb), y, ws)
    torch.cuda.synchronize()
    assert M.moe_get_status(ws) == M.MOE_OK
    ref = O.shared_expert_mxfp8(F.bf16_bits_to_float(xb), arr["s8_w13"], arr["s8_w13_scale"], arr["s8_w2"],
                                arr["s8_w2_scale"])
    got = y.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert normwise(got, ref["ys"]) <= CONTRACTION_TOL
    _check_mxfp8_h(d, ws, T, I, ref, F.dequantize_mxfp8(ref["xq"], ref["xs"]),
                   F.dequantize_mxfp8(arr["s8_w13"], arr["s8_w13_scale"]))


_E4M3_MIDS = (F.E4M3_TABLE[:0x7E] + F.E4M3_TABLE[1:0x7F]) / 2  # between neighbouring positive E4M3 values


def _check_mxfp8_h(d, ws, T, I, ref, xq_deq, w13):
    """The MXFP8-requantised h of the shared expert (codes and the E8M0 scale
    bytes in their tensor-core layout) equals the oracle's block for block,
    except blocks where the oracle's h lies within the FP32 contraction's
    error of an E4M3 rounding midpoint or of a change of the block exponent.
    G and U are FP32 tensor-core sums over K = H products: their error is
    bounded here by 2^-19 sum |xq w| (an FP32 accumulation of K terms in any
    order, with room), and carried to h through dh = |SiLU'(G) U| dG +
    |SiLU(G)| dU; E4M3's midpoints are dense enough (every 1/16 of a binade)
    that a fixed relative margin would not hold."""
    tp = (T + 127) // 128 * 128
    ghq = torch.empty((T, I), dtype=torch.uint8, device="cuda")
    ghs = torch.empty(tp * I // 32, dtype=torch.uint8, device="cuda")
    M.moe_debug_shared_mxfp8_h(d, ws, ghq, ghs)
    torch.cuda.synchronize()
    # word (i, j) of block (row tile, 128-column group) holds rows 32 j + i
    raw = ghs.cpu().numpy().reshape(tp // 128, I // 128, 32, 4, 4)   # tile, group, i, j, byte
    gs = raw.transpose(0, 3, 2, 1, 4).reshape(tp, I // 32)[:T]       # tile, j, i -> row; group, byte -> block
    gq = ghq.cpu().numpy().reshape(T, I // 32, 32)
    oq = ref["hq"].reshape(T, I // 32, 32)
    same = np.all(gq == oq, axis=2) & (gs == ref["hs"])
    G, U = ref["G"], ref["U"]
    mag = np.abs(xq_deq) @ np.abs(w13).T                           # [T, 2I]: sum |xq w|
    dG, dU = 2.0 ** -19 * mag[:, :I], 2.0 ** -19 * mag[:, I:]
    sg = 1.0 / (1.0 + np.exp(-G))
    dh = np.abs(sg * (1 + G * (1 - sg)) * U) * dG + np.abs(G * sg) * dU + 2.0 ** -23 * np.abs(ref["h"])
    hb = ref["h"].reshape(T, I // 32, 32)
    db = dh.reshape(T, I // 32, 32)
    amax = np.abs(hb).max(2)
    p2 = 2.0 ** np.floor(np.log2(np.maximum(amax, 1e-300)))
    near_scale = (np.abs(amax - p2) <= db.max(2)) | (np.abs(amax - 2 * p2) <= db.max(2))
    X = F.E8M0_TABLE[ref["hs"]][..., None]
    sv, sd = np.abs(hb) / X, db / X
    near_code = np.any(np.min(np.abs(sv[..., None] - _E4M3_MIDS), axis=-1) <= sd, axis=2)
    assert np.all(same | near_scale | near_code), "MXFP8 h differs away from a rounding boundary"
    assert same.mean() >= 0.99, same.mean()


@pytest.mark.parametrize("name,T,gemm", [("batch128_s8", None, M.ROUTED_GEMM_AUTO),
                                         ("batch128_s8", 300, M.ROUTED_GEMM_TOKENS_AS_A)])
def test_layer_forward_with_mxfp8_shared_expert(name, T, gemm, routed_gemm):
    """The layer with the shared expert in MXFP8 (moe_layer_forward_shared_mxfp8,
    scales prepared at load time) against the oracle on every token: 128
    tokens (weights-as-A routed GEMMs, separate combine) and 300 tokens
    (128-token routed tiles, the combine fused into the down GEMM, the MXFP8
    shared expert writing the accumulator first)."""
    routed_gemm(gemm)
    wl, lay, dev, cache = _workload(name, T)
    assert dev.sh8 is not None
    out, ids, w = dev.forward(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, cache, out, ids, w=w)
    ref = O.shared_expert_mxfp8(F.bf16_bits_to_float(lay["x"]), lay["s8_w13"], lay["s8_w13_scale"], lay["s8_w2"],
                                lay["s8_w2_scale"])
    _check_mxfp8_h(dev.desc(wl.T), dev.ws, wl.T, wl.I, ref, F.dequantize_mxfp8(ref["xq"], ref["xs"]),
                   F.dequantize_mxfp8(lay["s8_w13"], lay["s8_w13_scale"]))


@pytest.mark.parametrize("T", [1, 16, 40, None], ids=["T1", "T16", "T40", "T128"])
def test_layer_decode_with_mxfp8_shared_expert(T):
    """moe_layer_decode_shared_mxfp8 in one launch (the tensor-core decode
    with kind::mxf8f6f4 shared units: x quantised to MXFP8 in the launch, h
    requantised to MXFP8 by the shared gate/up finisher) on the full-size
    layer: 1 token, one 16-token chunk, a ragged third chunk (40) and 128
    tokens.  Every token against the oracle; the launch is bit-reproducible
    and agrees with the batched moe_layer_forward_shared_mxfp8."""
    wl, lay, dev, cache = _workload("batch128_s8", T)
    assert dev.sh8 is not None and dev.prepared
    x = bf16_tensor(lay["x"])
    n0 = M.moe_debug_launch_count()
    out, ids, w = dev.decode(x)
    torch.cuda.synchronize()
    assert M.moe_debug_launch_count() == n0 + 1
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, cache, out, ids, w=w)
    out2, _, _ = dev.decode(x)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    out_f, ids_f, _ = dev.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_f)
    assert normwise(bits_to_float(out), bits_to_float(out_f)) <= 1e-2


@pytest.mark.parametrize("T", [5, 33])
def test_layer_decode_mxfp8_shared_nvfp4_experts(T):
    """The MXFP8 shared expert beside NVFP4 routed experts (distinct tensor
    scales), one launch, small shape (H = 512, I = 256), every token."""
    wl = W.Workload("s8nv", T, 512, 256, 16, 4, W.NVFP4, 28, 0.08, shared_fmt="mxfp8")
    lay = W.generate(wl)
    dev = DeviceLayer(lay, wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=T)
    n0 = M.moe_debug_launch_count()
    out, ids, w = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    assert M.moe_debug_launch_count() == n0 + 1
    assert M.moe_get_status(dev.ws) == M.MOE_OK
    _compare_layer(wl, lay, {}, out, ids, w=w)


def test_mxfp8_to_bf16_dequant_bitexact():
    """The MXFP8 -> BF16 copy against the oracle's exact dequantisation
    rounded once to BF16: every E4M3 code under scales across the E8M0 range
    (the BF16 subnormal band, overflow to inf and the NaN byte included), and
    a random tensor.  Where the value lies in BF16's normal range the copy is
    lossless: the BF16 result equals the exact product."""
    codes = np.tile(np.arange(256, dtype=np.uint8), 32).reshape(-1, 256)       # 32 rows, every code 8 x per row
    sexp = np.array([0, 1, 5, 9, 100, 118, 127, 135, 200, 247, 248, 253, 254, 255], dtype=np.uint8)
    rng = np.random.default_rng(41)
    scales = rng.choice(sexp, (32, 8)).astype(np.uint8)
    scales[0] = sexp[:8]
    scales[1] = sexp[6:]
    rc = rng.integers(0, 256, (300, 1024), dtype=np.uint8)
    rs = rng.integers(100, 150, (300, 32), dtype=np.uint8)
    for c, sc in ((codes, scales), (rc, rs)):
        rows, K = c.shape
        out = torch.empty((rows, K), dtype=torch.int16, device="cuda")
        M.moe_dequant_mxfp8_to_bf16(rows, K, torch.from_numpy(c).cuda(), torch.from_numpy(sc).cuda(), out)
        torch.cuda.synchronize()
        got = out.cpu().numpy().view(np.uint16)
        exact = F.dequantize_mxfp8(c, sc)
        ref = F.round_to_bf16(exact)
        nan = np.isnan(exact)
        gv = F.bf16_bits_to_float(got)
        assert np.array_equal(np.isnan(gv), nan)
        want = F.bf16_value_to_bits(np.where(nan, 0.0, ref))
        zero = exact == 0  # E4M3 -0 (0x80) times a scale is -0, kept as the BF16 sign bit
        want[zero] = np.where(np.signbit(exact[zero]), 0x8000, 0)
        assert np.array_equal(got[~nan], want[~nan])
        normal = ~nan & (np.abs(exact) >= 2.0 ** -126) & (np.abs(exact) < 2.0 ** 128)
        assert np.array_equal(gv[normal], exact[normal])  # lossless in BF16's normal range
        assert normal.sum() > 0.5 * exact.size


def test_zero_tokens_is_a_no_op():
    wl, lay, dev, cache = _workload("tiny")
    x = torch.empty((0, wl.H), dtype=torch.int16, device="cuda")
    out, ids, w = dev.decode(x)
    out, ids, w = dev.forward(x)
    torch.cuda.synchronize()
    assert out.shape == (0, wl.H)


# ------------------------------------------------------------ failure path


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait on a counter nothing advances runs out after ~2 ms, records
    MOE_ERR_TIMEOUT in the workspace status word, and the GPU stays usable."""
    wl, lay, dev, cache = _workload("tiny")
    ws = torch.zeros(M.moe_workspace_size(dev.desc(wl.T)), dtype=torch.uint8, device="cuda")
    M.moe_debug_wait_probe(ws, 2_000_000)
    torch.cuda.synchronize()
    assert M.moe_get_status(ws) == M.MOE_ERR_TIMEOUT
    assert M.moe_get_status(ws) == M.MOE_OK  # reading clears it
    out, ids, _ = dev.decode(bf16_tensor(lay["x"]))
    torch.cuda.synchronize()
    _compare_layer(wl, lay, cache, out, ids)
