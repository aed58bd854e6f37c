"""Pins of the MXFP8 oracle (CPU): the E4M3 code table, round-to-nearest-even
checked against torch's float8_e4m3fn conversion, saturation, the E8M0 scale
rule on hand-computed blocks, the quantisation error bound, the MXFP8
layer forward against its definitions on inputs where quantisation is exact,
and the MXFP8 training backward: its GEMM helper exact on operands that are
representable along the contraction axis only, and with the quantisers
replaced by the identity the bf16 layer's backward (itself pinned by finite
differences)."""
import numpy as np
import pytest
import torch

import oracle as O


def test_e4m3_code_table():
    # hand-derived codes: S EEEE MMM with exponent bias 7, subnormals m 2^-9
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x78: 256.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in table.items():
        assert O.e4m3_decode(np.uint8(c)) == v, hex(c)
        if v != 0.0:
            assert int(O.e4m3_encode(np.float64(v))) == c, hex(c)
    # every finite code decodes to an E4M3 value that encodes back to it
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F and c != 0x80], np.uint8)
    vals = O.e4m3_decode(codes)
    assert np.array_equal(O.e4m3_round(vals), vals)
    assert np.array_equal(O.e4m3_encode(vals), codes)
    with pytest.raises(ValueError):
        O.e4m3_decode(np.uint8(0x7F))


def test_e4m3_rounding_matches_torch():
    rng = np.random.default_rng(3)
    finite = O.e4m3_decode(np.array([c for c in range(128) if c != 0x7F], np.uint8))
    mids = (finite[:-1] + finite[1:]) / 2  # exact ties between neighbours
    v = np.concatenate([rng.uniform(-448, 448, 4000), rng.normal(0, 1, 4000), rng.normal(0, 0.01, 2000),
                        mids, -mids, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)])
    v = v.astype(np.float32).astype(np.float64)  # float32-exact, so torch sees the same value
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_round(v), ref)


def test_e4m3_saturation():
    v = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 511.0, 1e6, -500.0])
    assert np.array_equal(O.e4m3_round(v), [448, 448, 448, 448, 448, 448, 448, -448])


def test_e8m0_scale_rule_hand_blocks():
    blk = np.zeros((5, 32))
    blk[0, 3] = 448.0           # floor(log2 448) = 8 -> s = 0, code 127, elements kept
    blk[1, 0] = 1.0             # s = -8, code 119: 1.0 -> 256 = 0x78
    blk[2, 7] = -500.0          # s = 0: 500 saturates to 448
    blk[3, :] = 3.0             # floor(log2 3) = 1 -> s = -7: 3 * 128 = 384 = 1.5 * 2^8 = 0x7C
    codes, scales = O.mx_quantize(blk)
    assert list(scales) == [127, 119, 127, 120, 0]   # all-zero block: s = -127 -> 0
    assert codes[0, 3] == 0x7E and codes[1, 0] == 0x78 and codes[2, 7] == 0xFE
    assert np.all(codes[3] == 0x7C) and np.all(codes[4] == 0)
    assert O.e8m0_exponent(2.0 ** -140) == -127 and O.e8m0_exponent(2.0 ** 140) == 127


def test_mx_quantize_axis_and_error_bound():
    rng = np.random.default_rng(5)
    v = rng.normal(0, 1, (6, 128)) * np.exp(rng.normal(0, 2, (6, 1)))
    c_row, s_row = O.mx_quantize(v, axis=1)
    c_col, s_col = O.mx_quantize(v.T, axis=0)
    assert np.array_equal(c_row, c_col.T) and np.array_equal(s_row, s_col.T)
    assert s_row.shape == (6, 4)
    back = O.mx_dequantize(c_row, s_row, axis=1)
    X = np.repeat(np.ldexp(1.0, s_row.astype(np.int64) - 127), 32, axis=1)
    normal = np.abs(v) >= X * 2.0 ** -6
    unsat = np.abs(v) < 448 * X
    ok = normal & unsat
    assert np.all(np.abs(back - v)[ok] <= 2.0 ** -4 * np.abs(v)[ok] * (1 + 1e-12))
    assert np.all(np.abs(back - v)[~normal] <= 2.0 ** -10 * X[~normal])
    # the block maximum never exceeds its E4M3 range after scaling
    assert np.all(np.abs(back) <= 448 * X)


def test_mx_layer_exact_inputs_reduce_to_plain_gemm():
    # x and weights are small integers times powers of two (E4M3-exact in
    # every block), so the gate/up GEMMs are exact; a is then quantised by the
    # definition, which this test applies by hand
    rng = np.random.default_rng(9)
    T, H, E, k, F = 20, 64, 4, 2, 64
    x = rng.integers(-4, 5, (T, H)) * 0.25
    w_r = rng.normal(0, 0.3, (E, H))
    W1 = rng.integers(-3, 4, (E, H, F)) * 0.125
    W3 = rng.integers(-3, 4, (E, H, F)) * 0.125
    W2 = rng.integers(-3, 4, (E, F, H)) * 0.0625
    for W in (W1, W3):
        assert np.array_equal(O.mx_roundtrip(W, axis=1), W)
    assert np.array_equal(O.mx_roundtrip(x, axis=1), x)
    out = O.mx_layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT)
    ref_rt = O.route(x, w_r, k)
    y = np.zeros((T, H))
    for t in range(T):
        for i in range(k):
            e = ref_rt["topk_idx"][t, i]
            a = O.silu(x[t] @ W1[e]) * (x[t] @ W3[e])
            y[t] += ref_rt["topk_gate"][t, i] * (O.mx_roundtrip(a[None], axis=1)[0] @ W2[e])
    np.testing.assert_allclose(out["y"], y, rtol=1e-12, atol=1e-12)
    # the a-quantisation is not the identity here: dropping it changes y
    y_noq = O.layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT)["y"]
    assert np.max(np.abs(y_noq - y)) > 1e-3


def test_mx_layer_close_to_bf16_layer():
    rng = np.random.default_rng(11)
    T, H, E, k, F = 64, 128, 8, 2, 96
    x = rng.normal(0, 1, (T, H))
    w_r = rng.normal(0, H ** -0.5, (E, H))
    W1 = rng.normal(0, H ** -0.5, (E, H, F))
    W3 = rng.normal(0, H ** -0.5, (E, H, F))
    W2 = rng.normal(0, F ** -0.5, (E, F, H))
    ymx = O.mx_layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT)["y"]
    y = O.layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT)["y"]
    rel = np.linalg.norm(ymx - y) / np.linalg.norm(y)
    assert 1e-3 < rel < 0.1  # FP8 error: present, and of FP8 size


def _k_exact_operand(rng, M, K):
    """[M, K]: integers in [-7, 7] times a power of two that is constant over
    each 32-element block of a row but differs by 2^20 between neighbouring
    rows, so every block along K is MXFP8-exact while blocks along M are not."""
    ints = rng.integers(-7, 8, (M, K)).astype(np.float64)
    ints[:, ::32] = 7.0                                      # every block holds its maximum
    row_exp = np.where(np.arange(M) % 2 == 0, 0, -20)[:, None]
    blk_exp = rng.integers(-3, 4, (M, K // 32)).repeat(32, axis=1)
    return ints * np.ldexp(1.0, row_exp + blk_exp)


def test_mx_matmul_nt_exact_along_the_contraction_axis():
    rng = np.random.default_rng(31)
    A = _k_exact_operand(rng, 64, 128)
    B = _k_exact_operand(rng, 96, 128)
    for V in (A, B):
        assert np.array_equal(O.mx_roundtrip(V, axis=1), V)
        assert not np.array_equal(O.mx_roundtrip(V, axis=0), V)  # the other axis would round
    np.testing.assert_array_equal(O.mx_matmul_nt(A, B), A @ B.T)
    np.testing.assert_array_equal(O.mx_matmul_nt(A, B, quant=False), A @ B.T)


def _token_exact_operand(rng, K, M):
    """[K, M]: integers in [-7, 7] times 2^(b + c), b alternating 0 / -16 over
    the 32-row blocks counted from row 0 and c alternating 0 / -20 over the
    columns, each block's first row holding its maximum: exact in MXFP8 along
    axis 0 in blocks aligned at row 0 (a misaligned block mixes exponents 16
    apart and rounds the small ones), not along axis 1."""
    ints = rng.integers(-7, 8, (K, M)).astype(np.float64)
    ints[::32] = 7.0
    blk = np.where((np.arange(K) // 32) % 2 == 0, 0, -16)[:, None]
    col = np.where(np.arange(M) % 2 == 0, 0, -20)[None, :]
    return ints * np.ldexp(1.0, blk + col)


def test_mx_matmul_tn_exact_along_tokens_with_a_ragged_last_block():
    # [K, M] operands exact along axis 0 in blocks of 32 from row 0 (the last
    # block has 16 rows), not along axis 1
    rng = np.random.default_rng(32)
    A = _token_exact_operand(rng, 80, 64)
    B = _token_exact_operand(rng, 80, 96)
    for V in (A, B):
        pad = np.concatenate([V, np.zeros((16, V.shape[1]))])
        assert np.array_equal(O.mx_roundtrip(pad, axis=0)[:80], V)
        assert not np.array_equal(O.mx_roundtrip(V, axis=1), V)
    np.testing.assert_array_equal(O.mx_matmul_tn(A, B), A.T @ B)
    np.testing.assert_array_equal(O.mx_matmul_tn(A, B, quant=False), A.T @ B)


def test_mx_weight_gradients_quantised_along_tokens():
    x, w_r, W1, W3, W2, dO, k = _train_case(6, T=64, H=128, E=4, F=96)
    q = O.mx_layer_bwd(x, w_r, W1, W3, W2, dO, k, wgrad="mxfp8")
    b = O.mx_layer_bwd(x, w_r, W1, W3, W2, dO, k, wgrad="bf16")
    np.testing.assert_array_equal(q["dx"], b["dx"])          # the switch touches the weight gradients only
    np.testing.assert_array_equal(q["dW_r"], b["dW_r"])
    for key in ("dW1", "dW3", "dW2"):
        num = sum(np.sum((q[key][e] - b[key][e]) ** 2) for e in b[key])
        den = sum(np.sum(b[key][e] ** 2) for e in b[key])
        assert 1e-3 < np.sqrt(num / den) < 0.1, key          # FP8 error: present, and of FP8 size


def _train_case(seed, T=24, H=64, E=4, k=2, F=64):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (T, H))
    w_r = rng.normal(0, 0.4, (E, H))
    W1 = rng.normal(0, H ** -0.5, (E, H, F))
    W3 = rng.normal(0, H ** -0.5, (E, H, F))
    W2 = rng.normal(0, F ** -0.5, (E, F, H))
    dO = rng.normal(0, 1, (T, H))
    return x, w_r, W1, W3, W2, dO, k


def test_mx_layer_bwd_without_quantisation_is_the_bf16_backward():
    x, w_r, W1, W3, W2, dO, k = _train_case(3)
    got = O.mx_layer_bwd(x, w_r, W1, W3, W2, dO, k, aux_coeff=1e-2, prec=O.EXACT, quant=False)
    ref = O.layer_bwd(x, w_r, W1, W3, W2, dO, k, aux_coeff=1e-2, prec=O.EXACT)
    for key in ("dx", "dW_r", "dgate"):
        np.testing.assert_allclose(got[key], ref[key], rtol=1e-11, atol=1e-12, err_msg=key)
    for key in ("dW1", "dW3", "dW2"):
        for e in ref[key]:
            np.testing.assert_allclose(got[key][e], ref[key][e], rtol=1e-11, atol=1e-12, err_msg=f"{key}[{e}]")
    assert got["aux_loss"] == pytest.approx(ref["aux_loss"], rel=1e-14)
    y = O.layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT)["y"]
    np.testing.assert_allclose(got["y"], y, rtol=1e-11, atol=1e-12)


def test_mx_layer_bwd_forward_is_the_mx_forward():
    x, w_r, W1, W3, W2, dO, k = _train_case(4, H=128, F=96)
    got = O.mx_layer_bwd(x, w_r, W1, W3, W2, dO, k)
    ref = O.mx_layer_fwd(x, w_r, W1, W3, W2, k)
    np.testing.assert_allclose(got["y"], ref["y"], rtol=1e-12, atol=1e-12)


def test_mx_layer_bwd_close_to_bf16_backward():
    x, w_r, W1, W3, W2, dO, k = _train_case(5, T=64, H=128, E=8, F=96)
    got = O.mx_layer_bwd(x, w_r, W1, W3, W2, dO, k)
    ref = O.layer_bwd(x, w_r, W1, W3, W2, dO, k)
    for key in ("dx", "dW_r"):
        rel = np.linalg.norm(got[key] - ref[key]) / np.linalg.norm(ref[key])
        assert 1e-3 < rel < 0.1, (key, rel)  # FP8 error: present, and of FP8 size
    num = sum(np.sum((got["dW1"][e] - ref["dW1"][e]) ** 2) for e in ref["dW1"])
    den = sum(np.sum(ref["dW1"][e] ** 2) for e in ref["dW1"])
    assert 1e-3 < np.sqrt(num / den) < 0.1


# planted mistakes: each must fail at least one pin above
def _round_half_away(v):
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    r = np.minimum(np.floor(a / q + 0.5) * q, 448.0)
    return np.where(v < 0, -r, r)


def _no_saturation(v):
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    r = np.round(a / q) * q
    return np.where(v < 0, -r, r)


def _scale_ceil(amax):
    amax = np.asarray(amax, np.float64)
    s = np.clip(np.ceil(np.log2(np.where(amax > 0, amax, 1.0))) - 8, -127, 127)
    return np.where(amax > 0, s, -127).astype(np.int64)


def _matmul_wrong_axis(A, B, quant=True):
    import oracle.mx_oracle as MX
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    if quant:
        A, B = MX.mx_roundtrip(A, axis=0), MX.mx_roundtrip(B, axis=0)
    return A @ B.T


def _matmul_transposed_operand(A, B, quant=True):
    import oracle.mx_oracle as MX
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    if quant:
        A, B = MX.mx_roundtrip(A, axis=1), MX.mx_roundtrip(B, axis=1)
    return A @ B[::-1].T if B.shape[0] > 1 else A @ B.T


def _matmul_tn_wrong_axis(A, B, quant=True):
    import oracle.mx_oracle as MX
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    if quant:
        A, B = MX.mx_roundtrip(A, axis=1), MX.mx_roundtrip(B, axis=1)
    return A.T @ B


def _matmul_tn_pad_in_front(A, B, quant=True):
    import oracle.mx_oracle as MX
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    if quant:
        K = A.shape[0]
        pad = (-K) % 32
        A = MX.mx_roundtrip(np.concatenate([np.zeros((pad, A.shape[1])), A]), axis=0)[pad:]
        B = MX.mx_roundtrip(np.concatenate([np.zeros((pad, B.shape[1])), B]), axis=0)[pad:]
    return A.T @ B


MX_MUTATIONS = [
    ("e4m3_round", _round_half_away, [test_e4m3_rounding_matches_torch]),
    ("e4m3_round", _no_saturation, [test_e4m3_saturation]),
    ("e8m0_exponent", _scale_ceil, [test_e8m0_scale_rule_hand_blocks]),
    ("mx_matmul_nt", _matmul_wrong_axis, [test_mx_matmul_nt_exact_along_the_contraction_axis]),
    ("mx_matmul_nt", _matmul_transposed_operand,
     [test_mx_matmul_nt_exact_along_the_contraction_axis, test_mx_layer_bwd_without_quantisation_is_the_bf16_backward]),
    ("mx_matmul_tn", _matmul_tn_wrong_axis, [test_mx_matmul_tn_exact_along_tokens_with_a_ragged_last_block]),
    ("mx_matmul_tn", _matmul_tn_pad_in_front, [test_mx_matmul_tn_exact_along_tokens_with_a_ragged_last_block]),
]


@pytest.mark.parametrize("name,fn,pins", MX_MUTATIONS,
                         ids=["half_away", "no_saturation", "scale_ceil", "matmul_wrong_axis", "matmul_row_order",
                              "matmul_tn_wrong_axis", "matmul_tn_pad_in_front"])
def test_planted_mx_mistake_is_caught(monkeypatch, name, fn, pins):
    import oracle.mx_oracle as MX
    monkeypatch.setattr(MX, name, fn)
    monkeypatch.setattr(O, name, fn)
    caught = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0
