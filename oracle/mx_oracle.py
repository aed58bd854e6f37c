"""MXFP8 (microscaling FP8) definition for the expert GEMMs, in fp64.

TEST INFRASTRUCTURE, like the rest of ``oracle``: only the tests, the smoke
check and the benchmark's CPU-baseline leg use it.

The report names MXFP8 as the Blackwell FP8 recipe of its benchmarks (captions
page, Table 11: "MXFP8 denotes microscaling FP8 on Blackwell"; Fig. 30: the
FP8 recipes, MXFP8 among them) but does not define the format. The reading
here is the published OCP Microscaling Formats (MX) v1.0 definition of MXFP8:

* a block is 32 consecutive elements along the contraction (K) dimension of a
  GEMM operand, so every operand is quantised along its own K;
* each block shares one E8M0 scale X = 2^s (an unsigned byte e = s + 127,
  s in [-127, 127]; 255 would be NaN and is never produced), with
  s = floor(log2(max |v|)) - 8, 8 being the exponent of the largest E4M3
  normal (448 = 1.75 * 2^8); an all-zero block takes s = -127;
* each element is v / X rounded to E4M3 (1 sign, 4 exponent bits with bias 7,
  3 mantissa bits, subnormals below 2^-6, no infinities) to nearest with ties
  to even; magnitudes above 448 saturate to 448 (the format has no infinity).
  v / X < 2^9, so saturation only touches values in [448, 512) * X.

The MXFP8 forward of the MoE layer quantises x (along H) and W1, W3 (along H)
for the gate/up GEMM, the SwiGLU activation a (along F) and W2 (along F) for
the down GEMM; products of dequantised values are summed exactly (fp64 here),
the expert outputs are stored in bf16 as in the bf16 layer, and routing and
combine are unchanged.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import (CONTRACT, aux_loss, permute_plan, route, router_backward, silu, silu_grad,
                         softmax, swiglu_expert)

__all__ = ["E4M3_MAX", "e4m3_round", "e4m3_encode", "e4m3_decode", "e8m0_exponent", "mx_quantize",
           "mx_dequantize", "mx_roundtrip", "mx_layer_fwd", "mx_matmul_nt", "mx_matmul_tn", "mx_layer_bwd"]

E4M3_MAX = 448.0
MX_BLOCK = 32


def e4m3_round(v):
    """Nearest E4M3 value of each fp64 v (ties to even), saturating at +-448.

    The quantum of a magnitude a in [2^e, 2^(e+1)) is 2^(e-3) (3 mantissa
    bits); below the smallest normal 2^-6 it stays 2^-9 (subnormals). a / q is
    exact (q is a power of two) and numpy's round is round-half-even."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))  # a = f 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    e = np.maximum(ex - 1, -6)
    q = np.ldexp(1.0, e - 3)
    r = np.minimum(np.round(a / q) * q, E4M3_MAX)
    return np.where(v < 0, -r, r)


def e4m3_encode(r):
    """Byte codes of E4M3 values (outputs of ``e4m3_round``)."""
    r = np.asarray(r, np.float64)
    a = np.abs(r)
    sign = (np.signbit(r)).astype(np.uint8) << 7
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = ex - 1
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e + 7, 0)
    mant = np.where(normal, a / np.ldexp(1.0, e) * 8 - 8, a / 2.0 ** -9)
    code = (exp_field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    return (sign | code.astype(np.uint8)).astype(np.uint8)


def e4m3_decode(c):
    """fp64 value of E4M3 byte codes (S.1111.111, the NaN codes, are rejected)."""
    c = np.asarray(c, np.uint8).astype(np.int64)
    if np.any((c & 0x7F) == 0x7F):
        raise ValueError("E4M3 NaN code")
    s = (c >> 7) & 1
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    return np.where(s == 1, -mag, mag)


def e8m0_exponent(amax):
    """Shared scale exponent s of blocks with maximum magnitude amax:
    floor(log2 amax) - 8, clamped to [-127, 127]; -127 for amax == 0."""
    amax = np.asarray(amax, np.float64)
    _, ex = np.frexp(np.where(amax > 0, amax, 1.0))
    s = np.clip(ex - 1 - 8, -127, 127)
    return np.where(amax > 0, s, -127).astype(np.int64)


def mx_quantize(v, axis=-1):
    """MXFP8 quantisation of v along ``axis`` (its length a multiple of 32).

    Returns (codes uint8, same shape as v; scales uint8 = s + 127, the axis
    shortened 32-fold)."""
    v = np.moveaxis(np.asarray(v, np.float64), axis, -1)
    K = v.shape[-1]
    if K % MX_BLOCK:
        raise ValueError("quantised axis must be a multiple of 32")
    blk = v.reshape(*v.shape[:-1], K // MX_BLOCK, MX_BLOCK)
    s = e8m0_exponent(np.abs(blk).max(axis=-1))
    q = e4m3_round(blk / np.ldexp(1.0, s)[..., None])
    codes = e4m3_encode(q).reshape(v.shape)
    scales = (s + 127).astype(np.uint8)
    return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis)


def mx_dequantize(codes, scales, axis=-1):
    """Values of MXFP8 data: code value * 2^(scale - 127), blockwise along axis."""
    c = np.moveaxis(np.asarray(codes), axis, -1)
    sc = np.moveaxis(np.asarray(scales), axis, -1).astype(np.int64)
    K = c.shape[-1]
    val = e4m3_decode(c).reshape(*c.shape[:-1], K // MX_BLOCK, MX_BLOCK)
    val = val * np.ldexp(1.0, sc - 127)[..., None]
    return np.moveaxis(val.reshape(c.shape), -1, axis)


def mx_roundtrip(v, axis=-1):
    """dequantize(quantize(v)): the value an MXFP8 GEMM multiplies."""
    return mx_dequantize(*mx_quantize(v, axis), axis=axis)


def mx_layer_fwd(x, w_r, W1, W3, W2, k, score="softmax", expert_bias=None, logit_bias=None, n_groups=1,
                 topk_groups=1, gate_scale=1.0, Ws=None, prec=CONTRACT, tokens=None, force_balanced=False):
    """Forward of the layer with MXFP8 expert GEMMs.

    Routing and combine are those of the bf16 layer (fp64). Per expert e on its
    rows xr: h1 = Q(xr) Q(W1e), h3 = Q(xr) Q(W3e) with Q = ``mx_roundtrip``
    along H; a = SiLU(h1) h3; out = Q(a) Q(W2e) along F, stored per
    ``prec.y_perm``. W1/W3 [E,H,F] and W2 [E,F,H] are the bf16 layer's
    weights; ``tokens`` restricts the expert and combine stages as in
    ``layer_fwd``. The optional shared expert ``Ws`` runs unquantised, as in
    ``layer_fwd``."""
    x = np.asarray(x, np.float64)
    T, H = x.shape
    rt = route(x, w_r, k, score, expert_bias, logit_bias, n_groups, topk_groups, gate_scale, force_balanced)
    E = np.asarray(w_r).shape[0]
    counts, offsets, row = permute_plan(rt["topk_idx"], E)
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    idx = rt["topk_idx"]
    yp = {}
    for e in range(E):
        sel_t, sel_i = np.nonzero(idx[tok] == e)
        if len(sel_t) == 0:
            continue
        t_e = tok[sel_t]
        xq = mx_roundtrip(x[t_e], axis=1)
        W1q = mx_roundtrip(np.asarray(W1[e], np.float64), axis=0)
        W3q = mx_roundtrip(np.asarray(W3[e], np.float64), axis=0)
        W2q = mx_roundtrip(np.asarray(W2[e], np.float64), axis=0)
        a = silu(xq @ W1q) * (xq @ W3q)
        out = prec.r("y_perm", mx_roundtrip(a, axis=1) @ W2q)
        for j in range(len(t_e)):
            yp[(int(t_e[j]), int(sel_i[j]))] = out[j]
    y = np.full((T, H), np.nan)
    acc = np.zeros((len(tok), H))
    if Ws is not None:
        Ws1, Ws3, Ws2 = (np.asarray(w, np.float64) for w in Ws)
        acc = acc + prec.r("shared", swiglu_expert(x[tok], Ws1, Ws3, Ws2, prec)[3])
    for i in range(k):
        rows = np.stack([yp[(int(t), i)] for t in tok]) if len(tok) else np.zeros((0, H))
        acc = acc + rt["topk_gate"][tok, i:i + 1] * rows
    y[tok] = prec.r("y", acc)
    return {**rt, "counts": counts, "offsets": offsets, "row_id_map": row, "y": y, "y_perm_rows": yp}


def mx_matmul_nt(A, B, quant=True):
    """A [M, K] times B [N, K] transposed, both operands MXFP8 along their
    shared K (the GEMM's contraction axis), products summed in fp64.
    ``quant=False`` replaces the round trips by the identity."""
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    if quant:
        A, B = mx_roundtrip(A, axis=1), mx_roundtrip(B, axis=1)
    return A @ B.T


def mx_matmul_tn(A, B, quant=True):
    """A [K, M] transposed times B [K, N], both operands MXFP8 along their
    shared K (axis 0, the GEMM's contraction axis) in blocks of 32 from row 0;
    a last partial block is quantised as if zero-padded to 32 rows (zeros
    change neither a block's maximum nor the products). Products summed in
    fp64. ``quant=False`` replaces the round trips by the identity."""
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    if quant:
        K = A.shape[0]
        pad = (-K) % MX_BLOCK
        A = mx_roundtrip(np.concatenate([A, np.zeros((pad, A.shape[1]))]), axis=0)[:K]
        B = mx_roundtrip(np.concatenate([B, np.zeros((pad, B.shape[1]))]), axis=0)[:K]
    return A.T @ B


def mx_layer_bwd(x, w_r, W1, W3, W2, dO, k, score="softmax", expert_bias=None, logit_bias=None, n_groups=1,
                 topk_groups=1, gate_scale=1.0, aux_coeff=0.0, prec=CONTRACT, experts=None, tokens=None,
                 force_balanced=False, quant=True, wgrad="bf16"):
    """Forward and backward of the layer with MXFP8 expert GEMMs, for the
    loss <dO, y> + L_aux.

    The report trains its Blackwell runs in MXFP8 without spelling out the
    recipe; the reading here quantises both operands of each MXFP8 GEMM
    along that GEMM's own contraction axis, as the forward does: along H or
    F for the data gradients, along the expert's tokens for the weight
    gradients, which are bf16 unless ``wgrad="mxfp8"``:

    forward, per expert e on its rows (as ``mx_layer_fwd``):
      h1 = Q(x) Q(W1_e), h3 = Q(x) Q(W3_e)       (Q along H)
      a = SiLU(h1) h3;  y_perm = Q(a) Q(W2_e)    (Q along F; stored per prec.y_perm)
      saved: h1, h3 stored per prec.h13
    backward:
      dy_perm = g dO (per prec.dy_perm); dg = <dO, y_perm>
      da  = Q(dy_perm) Q(W2_e)^T                 (Q along H: W2_e [F, H] row-wise; not
                                                  stored, so not rounded, as in the bf16 layer)
      dh1 = da h3 SiLU'(h1), dh3 = da SiLU(h1)   (saved h13; stored per prec.dh13)
      a'  = SiLU(h1) h3 from the saved h13       (stored per prec.a)
      dW2_e = Q(a')^T Q(dy_perm)                 (Q along the expert's tokens; wgrad="mxfp8")
      dx_perm = Q([dh1 | dh3]) Q([W1_e | W3_e])^T  (Q along 2F; per prec.dx_perm)
      dW1_e = Q(x)^T Q(dh1), dW3_e = Q(x)^T Q(dh3)  (Q along the expert's tokens, wgrad="mxfp8";
                                                 x = the bf16 rows of x_perm; Q = identity for "bf16")
      router backward, aux loss and dx = sum of dx_perm rows + dL W_r as in
      the bf16 layer.
    No shared expert. ``quant=False`` replaces every MXFP8 round trip by the
    identity, which is the bf16 layer's backward on the same stored tensors. Returns the same keys as the bf16 oracle's
    ``layer_bwd`` (plus ``y``, and ``wg_amax``: per expert the largest magnitude of each weight-gradient operand)."""
    x = np.asarray(x, np.float64)
    dO = np.asarray(dO, np.float64)
    T, H = x.shape
    w_r = np.asarray(w_r, np.float64)
    E = w_r.shape[0]
    rt = route(x, w_r, k, score, expert_bias, logit_bias, n_groups, topk_groups, gate_scale, force_balanced)
    idx, gate = rt["topk_idx"], rt["topk_gate"]
    counts, offsets, row = permute_plan(idx, E)
    Q = (lambda v, axis: mx_roundtrip(v, axis=axis)) if quant else (lambda v, axis: np.asarray(v, np.float64))
    need_tok = np.zeros(T, bool)
    if tokens is None:
        need_tok[:] = True
    else:
        need_tok[np.asarray(tokens)] = True
    exp_set = set(range(E)) if experts is None else set(int(e) for e in experts)
    F = np.asarray(W1[0]).shape[1]
    dgate = np.full((T, k), np.nan)
    dx = np.zeros((T, H))
    y = np.zeros((T, H))
    dW1 = {e: np.zeros((H, F)) for e in exp_set}
    dW3 = {e: np.zeros((H, F)) for e in exp_set}
    dW2 = {e: np.zeros((F, H)) for e in exp_set}
    wg_amax = {}  # per expert: the largest magnitude of each weight-gradient operand
    for e in range(E):
        tt, ii = np.nonzero(idx == e)                 # rows of expert e, ascending t
        if len(tt) == 0:
            continue
        want = need_tok[tt] if e not in exp_set else np.ones(len(tt), bool)
        if not want.any():
            continue
        tt, ii = tt[want], ii[want]
        W1e, W3e, W2e = (np.asarray(W[e], np.float64) for W in (W1, W3, W2))
        xr = x[tt]
        xq = Q(xr, 1)
        h1 = xq @ Q(W1e, 0)
        h3 = xq @ Q(W3e, 0)
        out = prec.r("y_perm", Q(silu(h1) * h3, 1) @ Q(W2e, 0))
        gsel = gate[tt, ii]
        y[tt] += gsel[:, None] * out
        h1s, h3s = prec.r("h13", h1), prec.r("h13", h3)
        dyr = prec.r("dy_perm", gsel[:, None] * dO[tt])
        dgate[tt, ii] = np.sum(dO[tt] * out, axis=1)
        da = mx_matmul_nt(dyr, W2e, quant)            # contraction over H
        dh1 = prec.r("dh13", da * h3s * silu_grad(h1s))
        dh3 = prec.r("dh13", da * silu(h1s))
        a_w = prec.r("a", silu(h1s) * h3s)
        dxr = prec.r("dx_perm", mx_matmul_nt(np.concatenate([dh1, dh3], axis=1),
                                             np.concatenate([W1e, W3e], axis=1), quant))  # over 2F
        np.add.at(dx, tt, dxr)
        if e in exp_set:
            wq = quant and wgrad == "mxfp8"
            dW1[e] += mx_matmul_tn(xr, dh1, wq)
            dW3[e] += mx_matmul_tn(xr, dh3, wq)
            dW2[e] += mx_matmul_tn(a_w, dyr, wq)
            wg_amax[e] = {n: float(np.abs(v).max()) for n, v in (("x", xr), ("dh1", dh1), ("dh3", dh3), ("a", a_w),
                                                                    ("dy", dyr))}
    res = {**rt, "counts": counts, "offsets": offsets, "row_id_map": row, "y": y,
           "dgate": dgate, "dW1": dW1, "dW3": dW3, "dW2": dW2, "wg_amax": wg_amax}
    lg = rt["logits"][need_tok]
    aux = aux_coeff if score == "softmax" else 0.0
    dL = router_backward(lg, idx[need_tok], gate[need_tok], dgate[need_tok], score, gate_scale, counts, k, aux,
                         T_total=T)
    if aux:
        res["aux_loss"] = aux_loss(softmax(rt["logits"]), counts, k, aux)
    dx[need_tok] += dL @ w_r
    res["dlogits"] = dL
    res["dx"] = np.where(need_tok[:, None], prec.r("dx", dx), np.nan)
    if tokens is None:
        res["dW_r"] = dL.T @ x
    return res
