"""Pins of the NVFP4 oracle (CPU): the E2M1 code table and its ties, the
E4M3 block-scale and fp32 tensor-scale rules on hand-computed blocks, the
quantisation error bound, the grouped GEMM on inputs where quantisation is
exact, and planted mistakes that the pins must catch."""
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
