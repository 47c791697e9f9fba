"""The sparse MoE FFN layer, step by step, in float64.

Test infrastructure only (see the package docstring).

What the layer computes (AMD technical article "MiniMax-M3.1 on AMD Instinct
GPUs: Day-0 support and optimization"):
* section "MiniMax-M3.1 at a glance": 128 routed experts with 4 active per
  token plus a shared expert every token passes through; routers are high
  precision;
* section "What we Optimized": a stacked router GEMM, then the MXFP4 fused MoE
  with the shared expert, fused for decode steps of at most 16 tokens;
* model card "amd/MiniMax-M3.1-Flash-Quark-MXFP4", section "Model Overview":
  routed-expert weights OCP MXFP4 (static), routed-expert activations OCP
  MXFP4 (dynamic).

Readings where the pages are silent:
* scores are softmax over the E router logits (the bias, when present, is
  part of the logit); the top-k experts are those with the k largest logits,
  ties to the lower expert index, emitted in that order; their probabilities
  are renormalised to sum to 1;
* the sigmoid variant (layer["score"] == "sigmoid"): scores are sigmoid of
  the raw router logits, the bias only corrects the selection (the k largest
  sigmoid + bias, ties to the lower index, in that order), and the weights
  are the selected sigmoid scores renormalised to sum to 1;
* an expert is a SwiGLU FFN: h = SiLU(x W_gate^T) * (x W_up^T), y = h W_down^T,
  with SiLU(g) = g / (1 + exp(-g));
* a routed expert sees the token quantised to MXFP4 (per 32 along H), and its
  intermediate h is re-quantised to MXFP4 (per 32 along I) before the down
  projection;
* the shared expert has BF16 weights, takes the BF16 token as is, and rounds
  its intermediate h to BF16 before its down projection; its weight in the
  combine is 1;
* an MXFP8 shared expert (layer["s8_w13"] ...) follows shared_expert_mxfp8:
  the token and h quantised to MXFP8 per 32, weight 1;
* folded into the expert table (model card "amd/MiniMax-M3.1-Flash-Quark-MXFP4",
  section "Experimental MXFP4 shared experts"; AMD article, section
  "Performance, mono decode on vs off"), the shared expert is expert E of the
  FP4 table (E = the router's rows): every token passes through it exactly
  as through a routed expert (MXFP4 token, MXFP4-requantised h), weight 1;
* out = BF16(ys + sum_j w_j * y_j), rounded once, to nearest-even.

Precision: every contraction accumulates in float64 and is rounded to float32
where the result is materialised (logits, G, U, h, y, ys); routing weights are
rounded to float32.
"""
from __future__ import annotations

import numpy as np

from . import formats as F

# ------------------------------------------------------------------ router


def router_logits(x: np.ndarray, w_router: np.ndarray, bias=None) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * Wr[e, h] (+ bias[e]), rounded to float32.

    x: float64 [T, H] (BF16 values); w_router: float32 [E, H]; bias: [E] or None.
    """
    acc = np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T
    if bias is not None:
        acc = acc + np.asarray(bias, dtype=np.float64)[None, :]
    return F.round_to_f32(acc)


def softmax(logits: np.ndarray) -> np.ndarray:
    """p = exp(l - max l) / sum exp(l - max l) over the expert axis, float64."""
    l = np.asarray(logits, dtype=np.float64)
    z = np.exp(l - l.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """ids [T, k]: the k largest logits per row, descending, ties -> lower index."""
    l = np.asarray(logits, dtype=np.float64)
    T, E = l.shape
    ids = np.empty((T, k), dtype=np.int32)
    idx = np.arange(E)
    for t in range(T):
        order = np.lexsort((idx, -l[t]))  # primary key -logit, secondary index
        ids[t] = order[:k]
    return ids


def sigmoid(l: np.ndarray) -> np.ndarray:
    """1 / (1 + exp(-l)) in float64."""
    return 1.0 / (1.0 + np.exp(-np.asarray(l, dtype=np.float64)))


def route(logits: np.ndarray, k: int, forced_ids=None, score: str = "softmax", bias=None):
    """Scores, top-k and renormalisation over the selected k.

    score "softmax": ``logits`` already hold the bias; p = softmax over all
    experts, the top-k logits are selected, weights p_sel / sum p_sel.
    score "sigmoid" (bias-corrected selection): ``logits`` are the raw router
    products x . Wr^T; s = sigmoid(logits), the experts with the k largest
    s_e + bias_e are selected (bias 0 when None), weights s_sel / sum s_sel.
    Returns (ids int32 [T, k], weights float64 [T, k] holding float32 values).
    ``forced_ids`` replaces the selection (weights still come from ``logits``).
    """
    if score == "softmax":
        p = softmax(logits)
        key = logits
    elif score == "sigmoid":
        p = sigmoid(logits)
        key = p + (0.0 if bias is None else np.asarray(bias, dtype=np.float64)[None, :])
    else:
        raise ValueError(score)
    ids = select_topk(key, k) if forced_ids is None else np.asarray(forced_ids, np.int32)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=-1)
    w = sel / sel.sum(axis=-1, keepdims=True)
    return ids, F.round_to_f32(w)


def selection_keys(logits: np.ndarray, score: str = "softmax", bias=None) -> np.ndarray:
    """The values top-k selection ranks: the logits (softmax scoring) or
    sigmoid(logits) + bias (bias-corrected sigmoid scoring), float64."""
    if score == "softmax":
        return np.asarray(logits, dtype=np.float64)
    return sigmoid(logits) + (0.0 if bias is None else np.asarray(bias, dtype=np.float64)[None, :])


# ------------------------------------------------------------- permutation


def permute(ids: np.ndarray, E: int):
    """Counting sort of the T*k assignments by expert, stable.

    Returns counts int32 [E], offsets int32 [E+1] (exclusive prefix sum),
    perm int32 [T*k] (sorted position -> flat assignment index t*k + j, sorted
    by expert, then token, then slot) and inv_perm int32 [T*k] (flat
    assignment index -> sorted position).
    """
    flat = np.asarray(ids, dtype=np.int64).ravel()
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    inv_perm = np.empty_like(perm)
    inv_perm[perm] = np.arange(perm.size, dtype=np.int32)
    return counts, offsets, perm, inv_perm


# ----------------------------------------------------------------- experts


def silu(g: np.ndarray) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """SiLU(g) * u in float64."""
    return silu(g) * np.asarray(u, dtype=np.float64)


def quantize_activations(x: np.ndarray):
    """Dynamic MXFP4 quantisation of token rows: (codes [T, H], scales [T, H/32])."""
    return F.quantize_mxfp4(x)


def expert_matrices(layer: dict, e: int, fmt: str):
    """Dequantised float64 (W_gate [I, H], W_up [I, H], W_down [H, I]) of expert e."""
    c13 = F.unpack_e2m1(layer["w13"][e])
    c2 = F.unpack_e2m1(layer["w2"][e])
    if fmt == "mxfp4":
        w13 = F.dequantize_mxfp4(c13, layer["w13_scale"][e])
        w2 = F.dequantize_mxfp4(c2, layer["w2_scale"][e])
    elif fmt == "nvfp4":
        ts = layer["tensor_scale"][e].astype(np.float64)
        I = c13.shape[0] // 2
        w13 = np.concatenate(
            [
                F.dequantize_nvfp4(c13[:I], layer["w13_scale"][e][:I], ts[0]),
                F.dequantize_nvfp4(c13[I:], layer["w13_scale"][e][I:], ts[1]),
            ]
        )
        w2 = F.dequantize_nvfp4(c2, layer["w2_scale"][e], ts[2])
    else:
        raise ValueError(fmt)
    I = w13.shape[0] // 2
    return w13[:I], w13[I:], w2


def routed_expert(xq_deq: np.ndarray, wg, wu, wd):
    """One routed expert on MXFP4-dequantised token rows xq_deq [n, H].

    Returns dict(G, U, h, hq codes, hs scales, y) with G, U, h, y float32 values.
    """
    G = F.round_to_f32(xq_deq @ wg.T)
    U = F.round_to_f32(xq_deq @ wu.T)
    h = F.round_to_f32(swiglu(G, U))
    hq, hs = F.quantize_mxfp4(h)
    y = F.round_to_f32(F.dequantize_mxfp4(hq, hs) @ wd.T)
    return dict(G=G, U=U, h=h, hq=hq, hs=hs, y=y)


def shared_expert(x: np.ndarray, ws13_bits: np.ndarray, ws2_bits: np.ndarray):
    """BF16 shared expert on BF16 token rows x [n, H] (float64 values).

    Returns dict(G, U, h, ys): G, U, ys float32 values, h BF16 values.
    """
    ws13 = F.bf16_bits_to_float(ws13_bits)
    ws2 = F.bf16_bits_to_float(ws2_bits)
    I = ws13.shape[0] // 2
    G = F.round_to_f32(x @ ws13[:I].T)
    U = F.round_to_f32(x @ ws13[I:].T)
    h = F.round_to_bf16(swiglu(G, U))
    ys = F.round_to_f32(h @ ws2.T)
    return dict(G=G, U=U, h=h, ys=ys)


def shared_expert_mxfp8(x: np.ndarray, w13_codes, w13_scales, w2_codes, w2_scales):
    """MXFP8 shared expert on token rows x [n, H] (float64 values).

    The pages' fused decode runs the shared expert in MXFP8 (AMD article,
    section "What we Optimized"); reading: the token is quantised to MXFP8 per
    32 along H and the intermediate h re-quantised to MXFP8 per 32 along I,
    as the routed experts do with MXFP4 (an MXFP8 datapath takes FP8 on both
    operands).  Weights: E4M3 codes [2I, H] / [H, I] with E8M0 scales per 32.
    Returns dict(xq, xs, G, U, h, hq, hs, ys): G, U, h, ys float32 values.
    """
    xq, xs = F.quantize_mxfp8(x)
    xd = F.dequantize_mxfp8(xq, xs)
    w13 = F.dequantize_mxfp8(w13_codes, w13_scales)
    w2 = F.dequantize_mxfp8(w2_codes, w2_scales)
    I = w13.shape[0] // 2
    G = F.round_to_f32(xd @ w13[:I].T)
    U = F.round_to_f32(xd @ w13[I:].T)
    h = F.round_to_f32(swiglu(G, U))
    hq, hs = F.quantize_mxfp8(h)
    ys = F.round_to_f32(F.dequantize_mxfp8(hq, hs) @ w2.T)
    return dict(xq=xq, xs=xs, G=G, U=U, h=h, hq=hq, hs=hs, ys=ys)


# ------------------------------------------------------------------- layer


def layer_forward(layer: dict, top_k: int, fmt: str, tokens=None, forced_ids=None,
                  keep=False, cache=None) -> dict:
    """The whole layer for the token rows ``tokens`` (default: all rows of x).

    ``layer`` holds the arrays described in the workload module (x as BF16
    bits, weights as codes / scale bytes).  ``forced_ids`` [len(tokens), k]
    overrides the top-k selection.  ``cache`` (a dict owned by the caller, one
    per layer) memoises the dequantised expert matrices across calls.  Returns
    float64 arrays holding exact
    float32 / BF16 values: logits, ids, weights, ys (or None), y [n, k, H],
    out [n, H] (BF16 values) and out_bits (uint16); with ``keep`` also the
    per-assignment intermediates.
    """
    xb = np.asarray(layer["x"])
    if tokens is None:
        tokens = np.arange(xb.shape[0])
    tokens = np.asarray(tokens)
    x = F.bf16_bits_to_float(xb[tokens])
    n, H = x.shape
    E = layer["w_router"].shape[0]

    score = layer.get("score", "softmax")
    if score == "softmax":  # the bias is part of the logit
        logits = router_logits(x, layer["w_router"], layer.get("bias"))
        ids, w = route(logits, top_k, forced_ids)
    else:  # the bias only corrects the selection
        logits = router_logits(x, layer["w_router"])
        ids, w = route(logits, top_k, forced_ids, score, layer.get("bias"))

    xq, xs = quantize_activations(x)
    xq_deq = F.dequantize_mxfp4(xq, xs)

    y = np.zeros((n, top_k, H), dtype=np.float64)
    inter = {}
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        if cache is not None:
            if int(e) not in cache:
                cache[int(e)] = expert_matrices(layer, int(e), fmt)
            wg, wu, wd = cache[int(e)]
        else:
            wg, wu, wd = expert_matrices(layer, int(e), fmt)
        r = routed_expert(xq_deq[rows], wg, wu, wd)
        y[rows, slots] = r["y"]
        if keep:
            inter[int(e)] = dict(rows=rows, slots=slots, **r)

    ys = None
    if layer.get("shared_in_table"):
        # the shared expert is table entry E, applied to every token like a
        # routed expert
        if cache is not None:
            if E not in cache:
                cache[E] = expert_matrices(layer, E, fmt)
            wg, wu, wd = cache[E]
        else:
            wg, wu, wd = expert_matrices(layer, E, fmt)
        sh = routed_expert(xq_deq, wg, wu, wd)
        ys = sh["y"]
    elif layer.get("s8_w13") is not None:
        # the MXFP8 shared expert the pages' fused decode runs (AMD article,
        # section "What we Optimized")
        sh = shared_expert_mxfp8(x, layer["s8_w13"], layer["s8_w13_scale"], layer["s8_w2"], layer["s8_w2_scale"])
        ys = sh["ys"]
    elif layer.get("ws13") is not None:
        sh = shared_expert(x, layer["ws13"], layer["ws2"])
        ys = sh["ys"]
    acc = np.einsum("nk,nkh->nh", w, y)
    if ys is not None:
        acc = acc + ys
    out = F.round_to_bf16(acc)
    res = dict(logits=logits, ids=ids, weights=w, xq=xq, xs=xs, y=y, ys=ys, out=out,
               out_bits=F.bf16_value_to_bits(out), tokens=tokens)
    if keep:
        res["experts"] = inter
        if ys is not None:
            res["shared"] = sh
    return res
