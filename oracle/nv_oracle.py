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

from .moe_oracle import bf16_rne, permute_plan, route, silu
from .mx_oracle import e4m3_encode, e4m3_round

__all__ = ["E2M1_MAX", "e2m1_round", "e2m1_encode", "e2m1_decode", "nv_tensor_scale", "nv_quantize",
           "nv_dequantize", "nv_roundtrip", "nv_grouped_gemm", "routed_rows_roundtrip", "gate_up_store",
           "activation_roundtrip", "nv_layer_fwd"]

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
