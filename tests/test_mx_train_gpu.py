"""MXFP8 training step (GPU) against the MXFP8 oracle: the weights of the two
data-gradient GEMMs quantised bit for bit (codes and tile-ready scales), and
the forward output and every gradient (dx, dW_router, dW1, dW3, dW2, aux
loss) of the training step within the layer's tolerance, with bf16 and with
MXFP8 weight gradients, on shapes with several tiles, ragged N tiles of the
data-gradient GEMMs, experts whose token count is not a multiple of 32 and
zero-token experts."""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth
from tests._util import assert_close, f64, mx_wgrad_atol, rel_l2, wgrad_atol
from tests.test_mx_gpu import _decode_tile_scales

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


@pytest.mark.parametrize("E,H,F", [(3, 256, 384), (2, 384, 640)])
def test_mx_bwd_weight_quantization_bit_exact(E, H, F):
    ls = synth.shape("tiny", T=64, H=H, E=E, k=2, F=F)
    d = synth.make_layer(ls, seed=6, device="cuda", training=False)
    cfg = ops.config_from_shape(ls)
    w = ops.mx_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
    torch.cuda.synchronize()
    W1, W3, W2 = f64(d["W1"]), f64(d["W3"]), f64(d["W2"])
    w2h = w["w2h"].cpu().numpy()
    w13f = w["w13f"].cpu().numpy()
    ntf, nth = -(-F // 192), -(-H // 192)
    s2 = _decode_tile_scales(w["sf2h"].cpu().numpy(), E, ntf, H // 128,
                             lambda j, b: 192 * j + b if b < 192 and 192 * j + b < F else None)
    s13 = _decode_tile_scales(w["sf13f"].cpu().numpy(), E, nth, 2 * F // 128,
                              lambda j, b: 192 * j + b if b < 192 and 192 * j + b < H else None)
    for e in range(E):
        rq, rs = O.mx_quantize(W2[e], axis=1)  # [F, H], blocks along H
        assert np.array_equal(w2h[e], rq), e
        assert np.array_equal(np.stack([s2[f][e] for f in range(F)]), rs), e
        q1, s1 = O.mx_quantize(W1[e], axis=1)  # [H, F], blocks along F
        q3, s3 = O.mx_quantize(W3[e], axis=1)
        assert np.array_equal(w13f[e], np.concatenate([q1, q3], axis=1)), e
        assert np.array_equal(np.stack([s13[h][e] for h in range(H)]), np.concatenate([s1, s3], axis=1)), e


TRAIN_SHAPES = {
    "tiny": synth.shape("tiny", T=300, H=256, E=8, k=2, F=384),
    # ragged N tiles in both data-gradient GEMMs (F = 640 = 3 x 192 + 64,
    # H = 384 = 2 x 192), several m tiles per expert
    "ragged": synth.shape("tiny", T=1000, H=384, E=8, k=4, F=640),
    "e128_k8": synth.shape("tiny", T=777, H=256, E=128, k=8, F=256, w_std=0.05),
    # zero-token experts: their weight gradients are zero
    "skew": synth.shape("tiny", T=900, H=256, E=32, k=4, F=128, skew=1.2),
    # the sigmoid router with an expert bias and a group limit (its backward
    # through the sigmoid scores), gates scaled
    "sigmoid_groups": synth.shape("tiny", T=333, H=256, E=64, k=8, F=256, score="sigmoid", n_groups=8, topk_groups=4,
                                  gate_scale=2.5, expert_bias_range=0.1),
}


def _train(ls, d, cfg, mx_wgrad=False):
    mxw = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
    mxbw = ops.mx_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
    ws = ops.mx_train_workspace(cfg)
    saved = ops.alloc_saved_mxfp8(cfg)
    y = ops.layer_fwd_mxfp8_train(cfg, d["x"], d["router_w"], mxw, saved, d["expert_bias"], d["logit_bias"], ws=ws)
    g = ops.layer_bwd_mxfp8(cfg, d["dO"], d["x"], d["router_w"], mxbw, saved, ws=ws, mx_wgrad=mx_wgrad)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    return y, g, saved


@pytest.mark.parametrize("wgrad", ["bf16", "mxfp8"])
@pytest.mark.parametrize("name", list(TRAIN_SHAPES))
def test_layer_train_mxfp8(name, wgrad):
    ls = TRAIN_SHAPES[name]
    d = synth.make_layer(ls, seed=1234, device="cuda", training=True)
    aux = 1e-2 if ls.score == "softmax" else 0.0  # the aux loss applies to the softmax router
    cfg = ops.config_from_shape(ls, aux_coeff=aux, out_fp32=True)
    y, g, saved = _train(ls, d, cfg, mx_wgrad=wgrad == "mxfp8")
    n = {k_: (None if v is None else f64(v)) for k_, v in d.items()}
    ref = O.mx_layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score,
                         n["expert_bias"], n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale,
                         aux_coeff=aux, prec=O.Precision(y=False, dx=False), wgrad=wgrad)
    assert np.array_equal(saved["topk_idx"].cpu().numpy(), ref["topk_idx"]), "routing differs (tie)"
    assert np.array_equal(saved["counts"].cpu().numpy(), ref["counts"])
    assert_close("y", f64(y), ref["y"])
    E = ls.E
    pairs = {"dx": (f64(g["dx"]), ref["dx"]), "dW_r": (f64(g["dW_r"]), ref["dW_r"]),
             "dW1": (f64(g["dW1"]), np.stack([ref["dW1"][e] for e in range(E)])),
             "dW3": (f64(g["dW3"]), np.stack([ref["dW3"][e] for e in range(E)])),
             "dW2": (f64(g["dW2"]), np.stack([ref["dW2"][e] for e in range(E)]))}
    # MXFP8 weight gradients (operands quantised along the tokens): the bound
    # of a flipped code, from the largest operand magnitudes over the experts
    ops_of = {"dW1": ("x", "dh1"), "dW3": ("x", "dh3"), "dW2": ("a", "dy")}
    for key, (got, want) in pairs.items():
        if key in ops_of and wgrad == "mxfp8":
            am = ref["wg_amax"]
            a_max = max(am[e][ops_of[key][0]] for e in am)
            b_max = max(am[e][ops_of[key][1]] for e in am)
            atol = mx_wgrad_atol(want, a_max, b_max)
        else:
            # bf16-stored activations (dh13, a, dy_perm) can round to the other
            # neighbour where fp32 and fp64 accumulation straddle a boundary
            atol = wgrad_atol(want)
        assert_close(key, got, want, atol=atol)
    if ls.skew:
        empty = np.nonzero(ref["counts"] == 0)[0]
        assert len(empty) > 0
        assert not np.any(f64(g["dW1"])[empty]) and not np.any(f64(g["dW2"])[empty])
    if aux:
        assert abs(float(g["aux_loss"].item()) - ref["aux_loss"]) <= 1e-5 * max(1.0, abs(ref["aux_loss"]))
    # the MXFP8 step differs from the bf16 step by FP8 rounding, not more
    ref16 = O.layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score,
                        n["expert_bias"], n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale,
                        aux_coeff=aux, prec=O.Precision(y=False, dx=False))
    assert 1e-3 < rel_l2(f64(g["dx"]), ref16["dx"]) < 0.2  # two chained FP8 GEMMs: ~8%


def test_mx_train_saved_buffers_required():
    ls = TRAIN_SHAPES["tiny"]
    d = synth.make_layer(ls, seed=2, device="cuda", training=True)
    cfg = ops.config_from_shape(ls)
    mxw = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
    saved = ops.alloc_saved_mxfp8(cfg)
    saved["h13"] = None
    with pytest.raises(ops.MoeError):
        ops.layer_fwd_mxfp8_train(cfg, d["x"], d["router_w"], mxw, saved)
