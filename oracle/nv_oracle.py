"""NVFP4 definition for the expert GEMMs.

TEST INFRASTRUCTURE, like the rest of ``oracle``: only the tests, the smoke
check and the benchmark's CPU-baseline leg use it.

The report lists NVFP4 among its supported precisions (summary page,
"Modeling" and "Key Terms": NVIDIA's 4-bit floating point) without defining
it. The reading here is
NVIDIA's published NVFP4 format, two-level scaled:

* elements are FP4 E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit):
  magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; rounding to nearest, ties to even;
  magnitudes above 6 saturate to 6;
* a block is 16 consecutive elements along the GEMM operand's K and shares one
  positive FP8 E4M3 scale s_b;
* the tensor shares one fp32 scale g = amax(tensor) / (6 * 448) (g = 1 for an
  all-zero tensor), so that the largest block scale lands on the largest E4M3
  value;
* encoding, in fp32 arithmetic (each operation rounded to nearest even, the
  order fixed so that the quantised codes are a function of the inputs alone):
      s_b = E4M3(fp32(fp32(amax_b / 6) / g))      (round to nearest even)
      t   = fp32(s_b * g)
      q   = E2M1(fp32(v / t))   (q = 0 where t == 0)
  and the value of a code is q * s_b * g.

A GEMM on NVFP4 operands sums the products of the decoded values: with per
block scales inside the tensor cores and the product of the two tensor scales
applied once to each output.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import (CONTRACT, aux_loss, bf16_rne, permute_plan, route, router_backward, silu, silu_grad,
                         softmax)
from .mx_oracle import e4m3_encode, e4m3_round

__all__ = ["E2M1_MAX", "e2m1_round", "e2m1_encode", "e2m1_decode", "nv_tensor_scale", "nv_quantize",
           "nv_dequantize", "nv_roundtrip", "nv_grouped_gemm", "routed_rows_roundtrip", "gate_up_store",
           "activation_roundtrip", "nv_layer_fwd", "output_grad_roundtrip", "swiglu_grad_roundtrip",
           "dgrad_weight_roundtrip", "nv_layer_bwd", "nv_expert_weight_grads"]

E2M1_MAX = 6.0
NV_BLOCK = 16
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_round(v):
    """Nearest E2M1 value of each v (ties to even), saturating at +-6.

    Quantum: 0.5 below 2 (the subnormal 0.5 and the binade [1, 2)), 1 in
    [2, 4), 2 in [4, 8); a / q is exact and numpy's round is half-even, so
    ties go to the value with an even mantissa bit."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    q = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.minimum(np.round(a / q) * q, E2M1_MAX)
    return np.where(v < 0, -r, r)


def e2m1_encode(r):
    """4-bit codes (S EE M) of E2M1 values."""
    r = np.asarray(r, np.float64)
    idx = np.searchsorted(_E2M1_MAG, np.abs(r))
    if not np.all(_E2M1_MAG[np.minimum(idx, 7)] == np.abs(r)):
        raise ValueError("not an E2M1 value")
    return (idx | (np.signbit(r).astype(np.int64) << 3)).astype(np.uint8)


def e2m1_decode(c):
    c = np.asarray(c, np.uint8).astype(np.int64)
    mag = _E2M1_MAG[c & 7]
    return np.where(c & 8, -mag, mag)


def nv_tensor_scale(amax):
    """fp32 tensor scale amax / (6 * 448); 1 for amax == 0."""
    g = np.float32(np.float32(amax) / np.float32(6.0 * 448.0))
    return np.float32(1.0) if g == 0 else g


def nv_quantize(v, axis=-1, g=None):
    """NVFP4 quantisation of v along ``axis`` (a multiple of 16).

    v is taken as fp32 (exactly, for bf16 inputs). Returns (codes uint8 of
    4-bit values, same shape as v; block scales uint8 E4M3 codes, the axis
    shortened 16-fold; tensor scale g, fp32; computed from v unless given)."""
    v = np.moveaxis(np.asarray(v, np.float32), axis, -1)
    K = v.shape[-1]
    if K % NV_BLOCK:
        raise ValueError("quantised axis must be a multiple of 16")
    if g is None:
        g = nv_tensor_scale(np.abs(v).max() if v.size else 0.0)
    g = np.float32(g)
    blk = v.reshape(*v.shape[:-1], K // NV_BLOCK, NV_BLOCK)
    amax = np.abs(blk).max(axis=-1).astype(np.float32)
    s = (amax / np.float32(6.0)).astype(np.float32)
    s = (s / g).astype(np.float32)
    sb = e4m3_round(s.astype(np.float64)).astype(np.float32)          # exact in fp32
    t = (sb * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        x = np.where(t[..., None] > 0, (blk / t[..., None]).astype(np.float32), np.float32(0.0))
    q = e2m1_round(x.astype(np.float64))
    codes = e2m1_encode(q).reshape(v.shape)
    return np.moveaxis(codes, -1, axis), np.moveaxis(e4m3_encode(sb.astype(np.float64)), -1, axis), g


def nv_dequantize(codes, scales, g, axis=-1):
    from .mx_oracle import e4m3_decode
    c = np.moveaxis(np.asarray(codes), axis, -1)
    sc = np.moveaxis(np.asarray(scales), axis, -1)
    K = c.shape[-1]
    val = e2m1_decode(c).reshape(*c.shape[:-1], K // NV_BLOCK, NV_BLOCK) * e4m3_decode(sc)[..., None]
    return np.moveaxis(val.reshape(c.shape) * np.float64(g), -1, axis)


def nv_roundtrip(v, axis=-1, g=None):
    codes, scales, g = nv_quantize(v, axis, g)
    return nv_dequantize(codes, scales, g, axis)


def nv_grouped_gemm(x, offsets, W, out_bf16=True):
    """Grouped NVFP4 GEMM: rows offsets[e]..offsets[e+1] of x [R,K] times
    expert e's W[e] [K,N]. x is one tensor (one tensor scale over all rows, its
    blocks along K); each W[e] is a tensor of its own (blocks along K). The
    products of decoded values are summed in fp64; the output is rounded to
    bf16 if ``out_bf16``."""
    x = np.asarray(x, np.float32)
    R, K = x.shape
    xq = nv_roundtrip(x, axis=1)
    E = len(offsets) - 1
    N = np.asarray(W[0]).shape[1]
    y = np.zeros((R, N))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        We = nv_roundtrip(np.asarray(W[e], np.float32), axis=0)
        y[lo:hi] = xq[lo:hi] @ We
    return bf16_rne(y) if out_bf16 else y


def routed_rows_roundtrip(rows, offsets):
    """NVFP4 round trip of the routed rows x_perm [R,H] as ONE tensor: one fp32
    tensor scale from the maximum over every routed row (whatever its expert),
    16-element blocks along H (the gate/up GEMM's K)."""
    rows = np.asarray(rows, np.float32)
    g = nv_tensor_scale(np.abs(rows).max() if rows.size else 0.0)
    return nv_roundtrip(rows, axis=1, g=g)


def gate_up_store(h):
    """The gate/up GEMM's output as the layer stores it: bf16 (round to nearest
    even), before the activation is formed from it."""
    return bf16_rne(h)


def activation_roundtrip(a, offsets):
    """NVFP4 round trip of the SwiGLU activation a [R,F] as ONE tensor over all
    routed rows (one tensor scale), 16-element blocks along F (the down GEMM's
    K)."""
    a = np.asarray(a, np.float32)
    g = nv_tensor_scale(np.abs(a).max() if a.size else 0.0)
    return nv_roundtrip(a, axis=1, g=g)


def nv_layer_fwd(x, w_r, W1, W3, W2, k, score="softmax", expert_bias=None, logit_bias=None, n_groups=1,
                 topk_groups=1, gate_scale=1.0, tokens=None, force_balanced=False):
    """Forward of the layer with NVFP4 expert GEMMs.

    Routing and combine as in the bf16 layer (fp64). The routed rows x_perm
    form one tensor; expert e's [W1_e | W3_e] (H x 2F, blocks along H) one
    tensor and W2_e (blocks along F) another. Per expert:
      h  = bf16(Q(x_e) Q([W1_e | W3_e]))        (the gate/up GEMM, stored bf16)
      a  = bf16(SiLU(h1) h3)                    (from the stored h; stored bf16)
      out = bf16(Q(a_e) Q(W2_e))                (a quantised as one tensor over all rows)
    with Q = ``nv_roundtrip`` (steps: ``routed_rows_roundtrip``,
    ``gate_up_store``, ``activation_roundtrip``). The tensor scale of a comes
    from the maximum of a over every routed row, so a is formed for all rows;
    ``tokens`` restricts the combine."""
    x = np.asarray(x, np.float64)
    T, H = x.shape
    rt = route(x, w_r, k, score, expert_bias, logit_bias, n_groups, topk_groups, gate_scale, force_balanced)
    E = np.asarray(w_r).shape[0]
    counts, offsets, row = permute_plan(rt["topk_idx"], E)
    R = T * k
    x_perm = np.zeros((R, H), np.float32)
    x_perm[row.reshape(-1)] = np.repeat(x.astype(np.float32), k, axis=0)
    xq = routed_rows_roundtrip(x_perm, offsets)
    F = np.asarray(W1[0]).shape[1]
    a = np.zeros((R, F))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        W13 = np.concatenate([np.asarray(W1[e], np.float32), np.asarray(W3[e], np.float32)], axis=1)
        h = gate_up_store(xq[lo:hi] @ nv_roundtrip(W13, axis=0))
        a[lo:hi] = bf16_rne(silu(h[:, :F]) * h[:, F:])
    aq = activation_roundtrip(a, offsets)
    y_perm = np.zeros((R, H))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        y_perm[lo:hi] = bf16_rne(aq[lo:hi] @ nv_roundtrip(np.asarray(W2[e], np.float32), axis=0))
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    y = np.full((T, H), np.nan)
    acc = np.zeros((len(tok), H))
    for i in range(k):
        acc = acc + rt["topk_gate"][tok, i:i + 1] * y_perm[row[tok, i]]
    y[tok] = acc
    return {**rt, "counts": counts, "offsets": offsets, "row_id_map": row, "y": y}


# ----------------------------------------------------------------------------
# Training step with NVFP4 data-gradient GEMMs
# ----------------------------------------------------------------------------
def output_grad_roundtrip(dy, offsets):
    """NVFP4 round trip of dy_perm [R,H] (the down data gradient's activation
    operand) as ONE tensor over all routed rows, 16-element blocks along H."""
    dy = np.asarray(dy, np.float32)
    g = nv_tensor_scale(np.abs(dy).max() if dy.size else 0.0)
    return nv_roundtrip(dy, axis=1, g=g)


def swiglu_grad_roundtrip(dh, offsets):
    """NVFP4 round trip of [dh1 | dh3] [R,2F] (the gate/up data gradient's
    activation operand) as ONE tensor over all routed rows, 16-element blocks
    along 2F."""
    dh = np.asarray(dh, np.float32)
    g = nv_tensor_scale(np.abs(dh).max() if dh.size else 0.0)
    return nv_roundtrip(dh, axis=1, g=g)


def dgrad_weight_roundtrip(W):
    """NVFP4 round trip of one expert's weight as the data-gradient GEMM reads
    it: W [N, K] row-wise (16-element blocks along K, the GEMM's contraction
    axis), the expert's matrix a tensor of its own (W2_e [F, H] along H;
    [W1_e | W3_e] [H, 2F] along 2F)."""
    return nv_roundtrip(np.asarray(W, np.float32), axis=1)


def nv_layer_bwd(x, w_r, W1, W3, W2, dO, k, score="softmax", expert_bias=None, logit_bias=None, n_groups=1,
                 topk_groups=1, gate_scale=1.0, aux_coeff=0.0, prec=CONTRACT, force_balanced=False, quant=True):
    """Forward and backward of the layer with NVFP4 expert GEMMs, for the loss
    <dO, y> + L_aux.

    The report trains in NVFP4 (summary page, "Modeling"; Key Terms) without
    giving a recipe. The reading here follows the NVFP4 forward
    (``nv_layer_fwd``): each data-gradient GEMM quantises both operands along
    its own contraction axis, the operand made of routed rows as ONE tensor
    over all of them (one fp32 tensor scale), each expert's weight as a tensor
    of its own; the weight gradients stay bf16 x bf16 (fp32 out). In row space
    (rows ordered by expert as the permute lays them out):

      forward  h = Q(x_perm) Q([W1_e | W3_e])         (Q along H; stored per prec.h13)
               a = SiLU(h1) h3                          (from the stored h; per prec.a)
               y_perm = Q(a) Q(W2_e)                    (Q along F; per prec.y_perm)
      backward dy_perm = g dO (per prec.dy_perm); dg = <dO, y_perm>
               da = Q(dy_perm) Q(W2_e)^T                (Q along H, W2_e [F,H] row-wise; not rounded)
               dh1 = da h3 SiLU'(h1), dh3 = da SiLU(h1) (stored h; per prec.dh13)
               dx_perm = Q([dh1 | dh3]) Q([W1_e | W3_e])^T   (Q along 2F; per prec.dx_perm)
               dW2_e = a_e^T dy_perm_e, dW1_e = x_e^T dh1_e, dW3_e = x_e^T dh3_e (fp64 sums)
               router backward, aux loss and dx = sum of the token's dx_perm rows + dL W_r as in
               the bf16 layer

    Round trips: ``routed_rows_roundtrip`` (x_perm), ``activation_roundtrip``
    (a), ``output_grad_roundtrip`` (dy_perm), ``swiglu_grad_roundtrip``
    ([dh1 | dh3]), ``nv_roundtrip`` along axis 0 for the forward weights and
    ``dgrad_weight_roundtrip`` for the backward ones. ``quant=False`` makes
    every round trip the identity: the bf16 layer's backward on the same
    stored tensors. No shared expert. Returns the keys of the bf16 oracle's
    ``layer_bwd`` for the whole layer (dW1, dW3, dW2 as dicts over every
    expert) and, for the pins and tolerances, the row-space tensors "h13",
    "dy_perm", "da", "dh13" and "dx_perm"."""
    x = np.asarray(x, np.float64)
    dO = np.asarray(dO, np.float64)
    T, H = x.shape
    w_r = np.asarray(w_r, np.float64)
    E = w_r.shape[0]
    F = np.asarray(W1[0]).shape[1]
    rt = route(x, w_r, k, score, expert_bias, logit_bias, n_groups, topk_groups, gate_scale, force_balanced)
    idx, gate = rt["topk_idx"], rt["topk_gate"]
    counts, offsets, row = permute_plan(idx, E)
    R = T * k
    flat = row.reshape(-1)
    x_perm = np.zeros((R, H))
    x_perm[flat] = np.repeat(x, k, axis=0)
    g_perm = np.zeros(R)
    g_perm[flat] = gate.reshape(-1)
    dO_perm = np.zeros((R, H))
    dO_perm[flat] = np.repeat(dO, k, axis=0)
    ident = lambda v, *a: np.asarray(v, np.float64)  # noqa: E731
    rows_q = routed_rows_roundtrip if quant else ident
    act_q = activation_roundtrip if quant else ident
    dy_q = output_grad_roundtrip if quant else ident
    dh_q = swiglu_grad_roundtrip if quant else ident
    fw_q = (lambda W: nv_roundtrip(np.asarray(W, np.float32), axis=0)) if quant else ident
    bw_q = dgrad_weight_roundtrip if quant else ident
    segs = [(e, int(offsets[e]), int(offsets[e + 1])) for e in range(E) if offsets[e + 1] > offsets[e]]
    W13 = {e: np.concatenate([np.asarray(W1[e], np.float64), np.asarray(W3[e], np.float64)], axis=1)
           for e, _, _ in segs}
    # forward
    xq = rows_q(x_perm, offsets)
    h = np.zeros((R, 2 * F))
    for e, lo, hi in segs:
        h[lo:hi] = prec.r("h13", xq[lo:hi] @ fw_q(W13[e]))
    h1, h3 = h[:, :F], h[:, F:]
    a = prec.r("a", silu(h1) * h3)
    aq = act_q(a, offsets)
    y_perm = np.zeros((R, H))
    for e, lo, hi in segs:
        y_perm[lo:hi] = prec.r("y_perm", aq[lo:hi] @ fw_q(np.asarray(W2[e], np.float64)))
    y = np.zeros((T, H))
    for i in range(k):
        y += gate[:, i:i + 1] * y_perm[row[:, i]]
    # backward
    dy = prec.r("dy_perm", g_perm[:, None] * dO_perm)
    dgate = np.einsum("th,tih->ti", dO, y_perm[row])
    dyq = dy_q(dy, offsets)
    da = np.zeros((R, F))
    for e, lo, hi in segs:
        da[lo:hi] = dyq[lo:hi] @ bw_q(np.asarray(W2[e], np.float64)).T
    dh1 = prec.r("dh13", da * h3 * silu_grad(h1))
    dh3 = prec.r("dh13", da * silu(h1))
    dh = np.concatenate([dh1, dh3], axis=1)
    dhq = dh_q(dh, offsets)
    dx_perm = np.zeros((R, H))
    for e, lo, hi in segs:
        dx_perm[lo:hi] = prec.r("dx_perm", dhq[lo:hi] @ bw_q(W13[e]).T)
    dW1 = {e: np.zeros((H, F)) for e in range(E)}
    dW3 = {e: np.zeros((H, F)) for e in range(E)}
    dW2 = {e: np.zeros((F, H)) for e in range(E)}
    for e, lo, hi in segs:
        dW1[e] = x_perm[lo:hi].T @ dh1[lo:hi]
        dW3[e] = x_perm[lo:hi].T @ dh3[lo:hi]
        dW2[e] = a[lo:hi].T @ dy[lo:hi]
    aux = aux_coeff if score == "softmax" else 0.0
    dL = router_backward(rt["logits"], idx, gate, dgate, score, gate_scale, counts, k, aux, T_total=T)
    dx = dL @ w_r
    for i in range(k):
        dx += dx_perm[row[:, i]]
    res = {**rt, "counts": counts, "offsets": offsets, "row_id_map": row, "y": prec.r("y", y), "dgate": dgate,
           "dW1": dW1, "dW3": dW3, "dW2": dW2, "dlogits": dL, "dx": prec.r("dx", dx), "dW_r": dL.T @ x,
           "h13": h, "dy_perm": dy, "da": da, "dh13": dh, "dx_perm": dx_perm}
    if aux:
        res["aux_loss"] = aux_loss(softmax(rt["logits"]), counts, k, aux)
    return res


def nv_expert_weight_grads(x, w_r, W1, W3, W2, dO, k, experts, score="softmax", expert_bias=None, logit_bias=None,
                           n_groups=1, topk_groups=1, gate_scale=1.0, prec=CONTRACT, force_balanced=False):
    """dW1_e, dW3_e, dW2_e of ``nv_layer_bwd`` for the listed experts, from
    those experts' rows alone (for layers too large for the whole step).

    Of the tensor scales, the weight gradients depend on two, and both follow
    from per-token maxima: x_perm's (every token is routed, so its maximum is
    x's) and dy_perm's (the largest |g dO| is the largest gate of a token
    times the largest |dO| of that token, maximised over tokens, then stored
    per prec.dy_perm; rounding is monotone). Per expert e, on its rows:
      h = Q(x_e) Q([W1_e | W3_e]) (per prec.h13), a = SiLU(h1) h3 (per prec.a),
      dy = g dO (per prec.dy_perm), da = Q(dy) Q(W2_e)^T,
      dh1 = da h3 SiLU'(h1), dh3 = da SiLU(h1) (per prec.dh13),
      dW1_e = x_e^T dh1, dW3_e = x_e^T dh3, dW2_e = a^T dy.
    Returns {"dW1": {e: ..}, "dW3": .., "dW2": .., "counts": counts}."""
    x = np.asarray(x, np.float64)
    dO = np.asarray(dO, np.float64)
    w_r = np.asarray(w_r, np.float64)
    E = w_r.shape[0]
    rt = route(x, w_r, k, score, expert_bias, logit_bias, n_groups, topk_groups, gate_scale, force_balanced)
    idx, gate = rt["topk_idx"], rt["topk_gate"]
    counts = np.bincount(idx.ravel(), minlength=E)
    g_x = nv_tensor_scale(np.abs(x).max() if x.size else 0.0)
    dy_max = prec.r("dy_perm", np.max(np.abs(gate).max(axis=1) * np.abs(dO).max(axis=1)) if x.size else 0.0)
    g_dy = nv_tensor_scale(dy_max)
    out = {"dW1": {}, "dW3": {}, "dW2": {}, "counts": counts}
    for e in experts:
        e = int(e)
        tt, ii = np.nonzero(idx == e)                       # the expert's rows, ascending t
        F = np.asarray(W1[e]).shape[1]
        if len(tt) == 0:
            H = x.shape[1]
            out["dW1"][e], out["dW3"][e], out["dW2"][e] = np.zeros((H, F)), np.zeros((H, F)), np.zeros((F, H))
            continue
        xr = x[tt]
        W13 = np.concatenate([np.asarray(W1[e], np.float64), np.asarray(W3[e], np.float64)], axis=1)
        h = prec.r("h13", nv_roundtrip(np.asarray(xr, np.float32), axis=1, g=g_x)
                   @ nv_roundtrip(np.asarray(W13, np.float32), axis=0))
        h1, h3 = h[:, :F], h[:, F:]
        a = prec.r("a", silu(h1) * h3)
        dy = prec.r("dy_perm", gate[tt, ii][:, None] * dO[tt])
        da = nv_roundtrip(np.asarray(dy, np.float32), axis=1, g=g_dy) @ dgrad_weight_roundtrip(W2[e]).T
        dh1 = prec.r("dh13", da * h3 * silu_grad(h1))
        dh3 = prec.r("dh13", da * silu(h1))
        out["dW1"][e] = xr.T @ dh1
        out["dW3"][e] = xr.T @ dh3
        out["dW2"][e] = a.T @ dy
    return out
