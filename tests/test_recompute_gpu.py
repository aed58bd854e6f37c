"""Memory-saving backward (captions page, Fig. 7 and Table 4 SwiGLU recompute)
through the C ABI against the oracle's recompute variant (GPU): the training
forward keeps neither a nor y_perm; the backward recomputes a from h13 and
takes the gate gradient from the down-projection dgrad. Every output within
the layer tolerances; the forward output equals the standard mode's bit for
bit (only where a and y_perm live changes)."""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth
from tests._util import MAX_ABS, assert_close, f64, wgrad_atol

pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny": synth.shape("tiny"),
    "ragged": synth.shape("tiny", T=1000, H=320, E=8, k=2, F=192),
    "e128_k8": synth.shape("tiny", T=777, H=256, E=128, k=8, F=256, w_std=0.05),
    "skew": synth.shape("tiny", T=900, H=256, E=32, k=4, F=128, skew=1.2),
    "sigmoid_fb": synth.shape("dsv3", T=333, H=256, E=64, k=8, F=128, F_shared=0, force_balanced=True),
}
FLIP_BOUND = {"ragged", "e128_k8", "skew"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


@pytest.mark.parametrize("name", list(SHAPES))
def test_memory_saving_backward(name):
    ls = SHAPES[name]
    d = synth.make_layer(ls, seed=91, device="cuda", training=True)
    aux = 1e-2 if ls.score == "softmax" else 0.0
    cfg = ops.config_from_shape(ls, aux_coeff=aux, out_fp32=True)
    ws = ops.workspace(cfg, True)
    args = (d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"])
    saved_std = ops.alloc_saved(cfg)
    y_std = ops.layer_fwd(cfg, *args, saved=saved_std, ws=ws)
    saved = ops.alloc_saved(cfg, recompute=True)
    assert saved["a"] is None and saved["y_perm"] is None
    y = ops.layer_fwd(cfg, *args, saved=saved, ws=ws)
    g = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    assert torch.equal(y, y_std)
    n = {k: (None if v is None else f64(v)) for k, v in d.items()}
    ref = O.layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score, n["expert_bias"],
                      n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale, aux_coeff=aux,
                      prec=O.Precision(y=False, dx=False), force_balanced=ls.force_balanced, recompute=True)
    assert np.array_equal(saved["topk_idx"].cpu().numpy(), ref["topk_idx"]), "routing differs (tie)"
    E = ls.E
    pairs = {"dx": (f64(g["dx"]), ref["dx"]), "dW_r": (f64(g["dW_r"]), ref["dW_r"]),
             "dW1": (f64(g["dW1"]), np.stack([ref["dW1"][e] for e in range(E)])),
             "dW3": (f64(g["dW3"]), np.stack([ref["dW3"][e] for e in range(E)])),
             "dW2": (f64(g["dW2"]), np.stack([ref["dW2"][e] for e in range(E)]))}
    for key, (got, want) in pairs.items():
        atol = wgrad_atol(want) if (key != "dx" or name in FLIP_BOUND) else MAX_ABS
        assert_close(key, got, want, atol=atol)
    if aux:
        assert abs(float(g["aux_loss"].item()) - ref["aux_loss"]) <= 1e-5 * max(1.0, abs(ref["aux_loss"]))


def test_one_of_a_and_y_perm_null_is_rejected():
    ls = SHAPES["tiny"]
    d = synth.make_layer(ls, seed=92, device="cuda", training=True)
    cfg = ops.config_from_shape(ls)
    saved = ops.alloc_saved(cfg)
    saved["a"] = None
    with pytest.raises(ops.MoeError):
        ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved=saved)
