"""Pins of the NVFP4 oracle (CPU): the E2M1 code table and its ties, the
E4M3 block-scale and fp32 tensor-scale rules on hand-computed blocks, the
quantisation error bound, the grouped GEMM on inputs where quantisation is
exact, the layer forward on inputs where every NVFP4 quantisation is exact
(it then reduces to the plain bf16 layer), and planted mistakes that the pins
must catch."""
import numpy as np
import pytest

import oracle as O


def test_e2m1_code_table_and_ties():
    vals = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c, v in enumerate(vals):
        assert O.e2m1_decode(np.uint8(c)) == v and O.e2m1_decode(np.uint8(c | 8)) == -v
        assert int(O.e2m1_encode(np.float64(v))) == c
    assert int(O.e2m1_encode(np.float64(-3.0))) == 0b1101
    # ties go to the even mantissa bit: 0 (0.25), 1 (0.75, 1.25), 2 (1.75, 2.5), 4 (3.5, 5)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -1.25])
    assert np.array_equal(O.e2m1_round(ties), [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -1.0])
    # off-tie values round to the nearest; saturation at 6
    assert np.array_equal(O.e2m1_round([0.26, 0.74, 2.49, 2.51, 4.99, 5.01, 6.5, 100.0]),
                          [0.5, 0.5, 2.0, 3.0, 4.0, 6.0, 6.0, 6.0])


def test_tensor_and_block_scales_hand_blocks():
    v = np.zeros((3, 16), np.float32)
    v[0, 3] = 2688.0          # tensor amax: g = 2688 / 2688 = 1
    v[1, :] = 6.0             # block amax 6: s_b = 6 / 6 / 1 = 1 -> E4M3 0x38; codes 6 -> 0b0111
    v[2, 0] = -0.75           # s_b = 0.125 = 2^-3 (0x20); -0.75 / 0.125 = -6 -> 0b1111
    codes, scales, g = O.nv_quantize(v)
    assert g == np.float32(1.0)
    assert list(scales) == [0x7E, 0x38, 0x20]      # 2688 / 6 = 448 -> 0x7E
    assert codes[0, 3] == 0b0111 and np.all(codes[1] == 0b0111) and codes[2, 0] == 0b1111
    assert np.all(codes[0, np.arange(16) != 3] == 0)
    # an all-zero tensor takes g = 1 and zero codes
    c0, s0, g0 = O.nv_quantize(np.zeros((2, 32), np.float32))
    assert g0 == 1.0 and not c0.any() and not s0.any()
    # the tensor scale moves every block scale by the same factor
    _, s2, g2 = O.nv_quantize(v * np.float32(0.5))
    assert g2 == np.float32(0.5) and list(s2) == list(scales)


def test_nv_error_bound():
    rng = np.random.default_rng(4)
    v = (rng.normal(0, 1, (8, 128)) * np.exp(rng.normal(0, 1, (8, 1)))).astype(np.float32)
    codes, scales, g = O.nv_quantize(v, axis=1)
    back = O.nv_dequantize(codes, scales, g, axis=1)
    # per block: the error is at most half a quantum of E2M1 (2 at the top
    # binade, i.e. 1/6 of the block maximum) plus the block scale's own E4M3
    # rounding (relative 2^-4)
    blk = np.abs(v.reshape(8, 8, 16)).max(axis=2)
    bound = np.repeat(blk, 16, axis=1) * (1.0 / 6.0 + 2.0 ** -4) * (1 + 1e-6)
    assert np.all(np.abs(back - v) <= bound)
    # axis handling: quantising v.T along axis 0 gives the transposed result
    c2, s2, g2 = O.nv_quantize(v.T, axis=0)
    assert np.array_equal(c2, codes.T) and np.array_equal(s2, scales.T) and g2 == g


def test_grouped_gemm_exact_inputs():
    # every block's maximum is 6 * 2^j and every element an E2M1 value times
    # the same 2^j, and the tensor maxima make g a power of two: the block
    # scales are powers of two (or 448 for the block holding the tensor
    # maximum, which holds nothing else), so quantisation is exact and the
    # grouped GEMM is the plain product
    rng = np.random.default_rng(8)
    E, K, N = 3, 64, 24
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    x = (rng.choice(vals, (40, K)) * rng.choice([-1, 1], (40, K))).astype(np.float32)
    x[:, ::16] = 6.0                           # block maximum 6 -> scale 6 / 6 / g
    x[0, :16] = 0.0
    x[0, 0] = 6.0 * 448 * 2.0 ** -8           # tensor amax 10.5: g = 2^-8, this block's scale 448
    W = (rng.choice(vals, (E, K, N)) * 2.0 ** -4).astype(np.float32)
    W[:, ::16, :] = 6.0 * 2.0 ** -4
    for e in range(E):
        W[e, :16, 0] = 0.0
        W[e, 0, 0] = 6.0 * 448 * 2.0 ** -12   # g_e = 2^-12
    offsets = np.array([0, 10, 10, 40])
    y = O.nv_grouped_gemm(x, offsets, W, out_bf16=False)
    assert np.array_equal(O.nv_roundtrip(x, axis=1), x.astype(np.float64))
    for e in range(E):
        assert np.array_equal(O.nv_roundtrip(W[e], axis=0), W[e].astype(np.float64))
    ref = np.zeros((40, N))
    for e in range(E):
        ref[offsets[e]:offsets[e + 1]] = x[offsets[e]:offsets[e + 1]].astype(np.float64) @ W[e]
    np.testing.assert_allclose(y, ref, rtol=0, atol=0)


def _round_half_away(v):
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    q = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.minimum(np.floor(a / q + 0.5) * q, 6.0)
    return np.where(v < 0, -r, r)


def _scale_no_tensor_level(amax):
    return np.float32(1.0)


@pytest.mark.parametrize("name,fn,pins", [
    ("e2m1_round", _round_half_away, ["test_e2m1_code_table_and_ties"]),
    ("nv_tensor_scale", _scale_no_tensor_level, ["test_tensor_and_block_scales_hand_blocks"]),
], ids=["half_away", "no_tensor_scale"])
def test_planted_nv_mistake_is_caught(monkeypatch, name, fn, pins):
    import oracle.nv_oracle as NV
    monkeypatch.setattr(NV, name, fn)
    monkeypatch.setattr(O, name, fn)
    caught = 0
    for pin in pins:
        try:
            globals()[pin]()
        except AssertionError:
            caught += 1
    assert caught > 0


def test_nv_layer_routing_and_fp4_closeness():
    # routing, counts and the permutation are the bf16 layer's; the output
    # differs from the exact layer by FP4 rounding (present, and of FP4 size)
    rng = np.random.default_rng(12)
    T, H, E, k, F = 64, 256, 4, 2, 256
    x = rng.normal(size=(T, H))
    w_r = rng.normal(size=(E, H)) / 16
    W1 = rng.normal(size=(E, H, F)) / 16
    W3 = rng.normal(size=(E, H, F)) / 16
    W2 = rng.normal(size=(E, F, H)) / 16
    out = O.nv_layer_fwd(x, w_r, W1, W3, W2, k)
    ref = O.layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT)
    assert np.array_equal(out["topk_idx"], ref["topk_idx"]) and np.array_equal(out["row_id_map"], ref["row_id_map"])
    rel = np.linalg.norm(out["y"] - ref["y"]) / np.linalg.norm(ref["y"])
    assert 0.02 < rel < 0.5, rel
    # the tokens argument restricts the combine only
    sub = O.nv_layer_fwd(x, w_r, W1, W3, W2, k, tokens=np.array([3, 7]))
    np.testing.assert_array_equal(sub["y"][[3, 7]], out["y"][[3, 7]])


# ---------------------------------------------------------------------------
# The NVFP4 layer on exact inputs.
#
# Every operand below is an E2M1 value times a power of two per 16-element
# block (the block's largest magnitude being 6 or 7.5 times that power), and
# each tensor's maximum sits alone in its block with 2688 = 6 * 448 times a
# power of two, so every tensor scale is a power of two and every block scale
# an E4M3 value: quantising x_perm, [W1_e | W3_e], a and W2_e changes nothing.
# The gate pre-activation of one entry carries a part below half a bf16 ulp
# (64 + 7/32), which the stored bf16 h drops. The NVFP4 layer must then equal
# the plain bf16 layer (a and y_perm rounded to bf16) run on weights without
# that part.
#
# Layout: T = 32 tokens, H = 80 (blocks of 16: 0..3 signal, 4 routing), F = 32,
# E = 2, k = 1; tokens 0..15 go to expert 0, 16..31 to expert 1.
# ---------------------------------------------------------------------------
def _exact_layer():
    T, H, F, E = 32, 80, 32, 2
    A, B, D, C, Z, C2 = 0, 1, 2, 16, 17, 18
    x = np.zeros((T, H))
    x[:, 0] = 4.0                      # shared feature: h1 = 4 * 16 = 64 everywhere
    x[:, 14] = 6.0                     # block-0 maximum of every row (its weight rows are zero)
    x[:16, 64] = 6.0                   # routing feature of expert 0
    x[16:, 65] = 6.0                   # routing feature of expert 1
    x[A, 1] = 6.0                      # private features
    x[A, 16], x[A, 30] = 0.5, 6.0
    x[A, 32], x[A, 46] = -1.0, 6.0
    x[B, 2] = 1.0
    x[B, 20] = 7.5                     # alone in its block: a block of the 1.25 * 2^j family
    x[D, 4] = 6.0
    x[C, 3] = 1.0
    x[C2, 5] = 1.0
    x[Z, 48] = 10.5                    # the tensor maximum of x: 2688 * 2^-8, alone in its block
    w_r = np.zeros((E, H))
    w_r[0, 64] = 1.0
    w_r[1, 65] = 1.0
    W1 = np.zeros((E, H, F))
    W3 = np.zeros((E, H, F))
    W2 = np.zeros((E, F, H))
    for e in range(E):
        W1[e, 0, :] = 16.0             # x feature 0 (4) * 16 = 64
        W1[e, 15, :] = 24.0            # block maximum 6 * 4 (x is 0 on row 15)
        W1[e, 49, 1] = 42.0            # tensor maximum of [W1_e | W3_e]: 2688 * 2^-6, alone
        W2[e, 15, :79] = 0.375         # block maxima of W2 (a is 0 on columns 15 and 31)
        W2[e, 31, :79] = 0.375
        W2[e, 14, 79] = 2.625          # tensor maximum of W2_e: 2688 * 2^-10, alone
    rng = np.random.default_rng(21)
    vals = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]) * 2.0 ** -4
    for e in range(E):
        for rows in (slice(0, 14), slice(16, 30)):
            W2[e, rows, :79] = rng.choice(vals, (14, 79)) * rng.choice([-1.0, 1.0], (14, 79))
    # the entry (A, f=0): h1 = 64 + 0.5 * 0.5 - 1 * 2^-5 = 64.21875, stored as 64
    W1[0, 16, 0], W1[0, 31, 0] = 0.5, 6.0
    W1[0, 32, 0], W1[0, 47, 0] = 2.0 ** -5, 6.0 * 2.0 ** -5
    # expert 0's up projection: h3(A,0) = 6 * 0.25 - 0.5 * 0.375 = 1.3125 (a = 84,
    # the tensor maximum of a: 2688 * 2^-5); h3(B,0) = 0.25 (a = 16), h3(B,1) =
    # 0.375 (a = 24); token D: h3 = 6 * 2^-6 +- 0.5 * 2^-11, the two bf16 ties
    # around 0.09375, both stored as 0.09375 (a = 6)
    W3[0, 1, 0], W3[0, 2, 0], W3[0, 15, 0] = 0.25, 0.25, 3.0
    W3[0, 16, 0], W3[0, 31, 0] = -0.375, 1.5
    W3[0, 2, 1], W3[0, 15, 1] = 0.375, 1.5
    for f, sgn in ((16, 1.0), (17, -1.0)):
        W3[0, 4, f], W3[0, 15, f] = 2.0 ** -6, 6.0 * 2.0 ** -6
        W3[0, 17, f], W3[0, 31, f] = sgn * 2.0 ** -11, 6.0 * 2.0 ** -11
    # expert 1: h3(C,0) = 0.09375 (a = 6); h3(C2,2) = 0.1171875 (a = 7.5, alone
    # in its block: the 1.25 * 2^j family)
    W3[1, 3, 0], W3[1, 15, 0] = 0.09375, 0.375
    W3[1, 5, 2], W3[1, 15, 2] = 0.1171875, 0.46875
    plain_W1 = W1.copy()
    plain_W1[0, 16, 0] = 0.0           # the part of h1(A,0) below half a bf16 ulp
    plain_W1[0, 32, 0] = 0.0
    return x, w_r, W1, W3, W2, plain_W1


def test_nv_layer_exact_inputs_reduce_to_plain_layer():
    x, w_r, W1, W3, W2, plain_W1 = _exact_layer()
    out = O.nv_layer_fwd(x, w_r, W1, W3, W2, 1)
    # the quantisations are exact: x_perm, [W1_e | W3_e] and W2_e round-trip unchanged
    xp = np.zeros_like(x)
    xp[out["row_id_map"][:, 0]] = x
    assert np.array_equal(O.routed_rows_roundtrip(xp, out["offsets"]), xp)
    for e in range(2):
        W13 = np.concatenate([W1[e], W3[e]], axis=1)
        assert np.array_equal(O.nv_roundtrip(W13, axis=0), W13)
        assert np.array_equal(O.nv_roundtrip(W2[e], axis=0), W2[e])
    ref = O.layer_fwd(x, w_r, plain_W1, W3, W2, 1, prec=O.CONTRACT)
    assert np.array_equal(out["topk_idx"], ref["topk_idx"]) and np.array_equal(out["row_id_map"], ref["row_id_map"])
    assert np.array_equal(out["counts"], [16, 16])
    np.testing.assert_allclose(out["y"], ref["y"], rtol=1e-12, atol=1e-12)
    # the output is not trivially zero and carries every designed activation
    assert np.count_nonzero(np.abs(ref["y"]) > 1.0) > 100


def _per_expert_rows(rows, offsets):
    out = np.zeros(np.shape(rows))
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            out[lo:hi] = O.nv_roundtrip(np.asarray(rows[lo:hi], np.float32), axis=1)
    return out


def _act_wrong_axis(a, offsets):
    return O.nv_roundtrip(np.asarray(a, np.float32), axis=0)


@pytest.mark.parametrize("name,fn", [
    ("routed_rows_roundtrip", _per_expert_rows),     # a tensor scale per expert for x_perm
    ("gate_up_store", lambda h: np.asarray(h)),      # h not rounded to bf16 before SiLU
    ("activation_roundtrip", _per_expert_rows),      # a tensor scale per expert for a
    ("activation_roundtrip", _act_wrong_axis),       # a quantised along the rows, not along F
], ids=["x_scale_per_expert", "h_unrounded", "a_scale_per_expert", "a_wrong_axis"])
def test_planted_nv_layer_mistake_is_caught(monkeypatch, name, fn):
    import oracle.nv_oracle as NV
    monkeypatch.setattr(NV, name, fn)
    with pytest.raises(AssertionError):
        test_nv_layer_exact_inputs_reduce_to_plain_layer()


# ---------------------------------------------------------------------------
# The NVFP4 training step (forward and backward with NVFP4 data gradients).
# ---------------------------------------------------------------------------
def _nv_train_case(seed, T=48, H=64, E=4, k=2, F=32):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (T, H))
    w_r = rng.normal(0, 0.4, (E, H))
    W1 = rng.normal(0, H ** -0.5, (E, H, F))
    W3 = rng.normal(0, H ** -0.5, (E, H, F))
    W2 = rng.normal(0, F ** -0.5, (E, F, H))
    dO = rng.normal(0, 1, (T, H))
    return x, w_r, W1, W3, W2, dO, k


def test_nv_layer_bwd_without_quantisation_is_the_bf16_backward():
    # every round trip the identity: the plain backward (terms, signs, transposes)
    x, w_r, W1, W3, W2, dO, k = _nv_train_case(3)
    got = O.nv_layer_bwd(x, w_r, W1, W3, W2, dO, k, aux_coeff=1e-2, prec=O.EXACT, quant=False)
    ref = O.layer_bwd(x, w_r, W1, W3, W2, dO, k, aux_coeff=1e-2, prec=O.EXACT)
    for key in ("dx", "dW_r", "dgate"):
        np.testing.assert_allclose(got[key], ref[key], rtol=1e-11, atol=1e-12, err_msg=key)
    y = O.layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT)["y"]
    np.testing.assert_allclose(got["y"], y, rtol=1e-11, atol=1e-12)
    for key in ("dW1", "dW3", "dW2"):
        for e in ref[key]:
            np.testing.assert_allclose(got[key][e], ref[key][e], rtol=1e-11, atol=1e-12, err_msg=f"{key}[{e}]")
    assert got["aux_loss"] == pytest.approx(ref["aux_loss"], rel=1e-14)


def test_nv_layer_bwd_forward_is_the_nv_forward():
    x, w_r, W1, W3, W2, dO, k = _nv_train_case(4)
    got = O.nv_layer_bwd(x, w_r, W1, W3, W2, dO, k)
    ref = O.nv_layer_fwd(x, w_r, W1, W3, W2, k)
    np.testing.assert_array_equal(got["y"], ref["y"])


def test_nv_data_gradients_are_the_pinned_grouped_gemm():
    # each data-gradient GEMM is the (exact-input pinned) grouped NVFP4 GEMM
    # on the operands the backward defines: dy_perm against W2_e^T [H, F]
    # (blocks along H), [dh1 | dh3] against [W1_e | W3_e]^T [2F, H] (blocks
    # along 2F); the routed-row operand one tensor over all rows
    x, w_r, W1, W3, W2, dO, k = _nv_train_case(5)
    W2 = W2 * np.array([1.0, 8.0, 0.125, 1.0])[:, None, None]      # experts of different magnitudes
    dO = dO * np.exp(np.random.default_rng(6).normal(0, 1, (dO.shape[0], 1)))
    out = O.nv_layer_bwd(x, w_r, W1, W3, W2, dO, k)
    off = out["offsets"]
    E = len(off) - 1
    da = O.nv_grouped_gemm(out["dy_perm"], off, [W2[e].T for e in range(E)], out_bf16=False)
    np.testing.assert_allclose(out["da"], da, rtol=1e-12, atol=1e-12)
    W13t = [np.concatenate([W1[e], W3[e]], axis=1).T for e in range(E)]
    dxp = O.nv_grouped_gemm(out["dh13"], off, W13t)
    np.testing.assert_allclose(out["dx_perm"], dxp, rtol=1e-12, atol=1e-12)
    # and quantisation is present: the data gradients are not the plain products
    plain = np.zeros_like(out["da"])
    for e in range(E):
        plain[off[e]:off[e + 1]] = out["dy_perm"][off[e]:off[e + 1]] @ W2[e].T
    assert np.linalg.norm(out["da"] - plain) > 1e-2 * np.linalg.norm(plain)


def test_nv_backward_tensor_scales_span_all_rows():
    # one tensor scale over every routed row: an expert whose rows are 2^-24
    # times the others' sits below the smallest E4M3 block scale and its
    # quantised rows are zero (a scale per expert would keep them)
    x, w_r, W1, W3, W2, dO, k = _nv_train_case(7, k=1)
    rt = O.route(x, w_r, 1)
    e_small = int(rt["topk_idx"][0, 0])
    tok = rt["topk_idx"][:, 0] == e_small
    # (a) dO of the expert's tokens tiny: dy_perm's blocks vanish, so does da
    # (and dh13, dx_perm), while the bf16 weight gradient dW2 = a^T dy is not zero
    dO_s = dO.copy()
    dO_s[tok] *= 2.0 ** -24
    out = O.nv_layer_bwd(x, w_r, W1, W3, W2, dO_s, 1)
    lo, hi = int(out["offsets"][e_small]), int(out["offsets"][e_small + 1])
    assert hi > lo
    assert not out["da"][lo:hi].any() and not out["dx_perm"][lo:hi].any()
    assert np.abs(out["dW2"][e_small]).max() > 0
    assert np.abs(np.delete(out["da"], np.s_[lo:hi], axis=0)).max() > 0.1
    # (b) the expert's W2_e tiny: dy_perm is as usual (its own weight tensor
    # scale keeps Q(W2_e)), da is 2^-24 small, [dh1 | dh3]'s global scale zeroes
    # those rows: dx_perm vanishes, the bf16 weight gradient dW1 does not
    W2_s = W2.copy()
    W2_s[e_small] *= 2.0 ** -24
    out = O.nv_layer_bwd(x, w_r, W1, W3, W2_s, dO, 1)
    assert np.abs(out["da"][lo:hi]).max() > 0
    assert not out["dx_perm"][lo:hi].any()
    assert np.abs(out["dW1"][e_small]).max() > 0


def _rows_per_expert(v, offsets):
    out = np.zeros(np.shape(v))
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            out[lo:hi] = O.nv_roundtrip(np.asarray(v[lo:hi], np.float32), axis=1)
    return out


@pytest.mark.parametrize("name,fn", [
    ("output_grad_roundtrip", _rows_per_expert),                      # dy_perm: a scale per expert
    ("swiglu_grad_roundtrip", _rows_per_expert),                      # dh13: a scale per expert
    ("dgrad_weight_roundtrip", lambda W: O.nv_roundtrip(np.asarray(W, np.float32), axis=0)),  # weight along N
    ("output_grad_roundtrip", lambda v, off: O.nv_roundtrip(np.asarray(v, np.float32), axis=0)),  # along rows
], ids=["dy_scale_per_expert", "dh_scale_per_expert", "weight_wrong_axis", "dy_wrong_axis"])
def test_planted_nv_bwd_mistake_is_caught(monkeypatch, name, fn):
    import oracle.nv_oracle as NV
    monkeypatch.setattr(NV, name, fn)
    with pytest.raises(AssertionError):
        test_nv_data_gradients_are_the_pinned_grouped_gemm()
        test_nv_backward_tensor_scales_span_all_rows()


@pytest.mark.parametrize("seed,k", [(8, 2), (9, 4)])
def test_nv_expert_weight_grads_are_the_layer_backward(seed, k):
    # the per-expert evaluation (tensor scales from per-token maxima) equals the
    # whole backward on every expert
    x, w_r, W1, W3, W2, dO, _ = _nv_train_case(seed, T=40, k=k)
    dO = dO * np.exp(np.random.default_rng(seed).normal(0, 1, (dO.shape[0], 1)))
    full = O.nv_layer_bwd(x, w_r, W1, W3, W2, dO, k)
    part = O.nv_expert_weight_grads(x, w_r, W1, W3, W2, dO, k, experts=range(4))
    assert np.array_equal(part["counts"], full["counts"])
    for key in ("dW1", "dW3", "dW2"):
        for e in range(4):
            np.testing.assert_allclose(part[key][e], full[key][e], rtol=1e-12, atol=1e-12, err_msg=f"{key}[{e}]")
