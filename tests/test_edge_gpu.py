"""Edge cases of the layer through the C ABI against the oracle (GPU): the
largest supported router (E = 256 experts, k = 16, 8-wide per-lane candidate
lists, the 16-slot combine paths), a single token, and the smallest dimensions
(H = F = 64, E = 2, k = 1). Forward and backward, every output compared in
full (no sampling); tokens within the tie margin are excused as elsewhere."""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth
from tests._util import assert_close, compare_topk, f64, topk_margin, wgrad_atol

pytestmark = pytest.mark.gpu

SHAPES = {
    "max_e_k": synth.shape("tiny", T=300, H=128, E=256, k=16, F=128),
    "one_token": synth.shape("tiny", T=1, H=64, E=4, k=2, F=64),
    "min_dims": synth.shape("tiny", T=129, H=64, E=2, k=1, F=64),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


@pytest.mark.parametrize("name", list(SHAPES))
def test_edge_layer(name):
    ls = SHAPES[name]
    d = synth.make_layer(ls, seed=321, device="cuda", training=True)
    aux = 1e-2
    cfg = ops.config_from_shape(ls, aux_coeff=aux, out_fp32=True)
    ws = ops.workspace(cfg, True)
    saved = ops.alloc_saved(cfg)
    y = ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"],
                      saved=saved, ws=ws)
    g = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    n = {k: (None if v is None else f64(v)) for k, v in d.items()}
    ref = O.layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, aux_coeff=aux,
                      prec=O.Precision(y=False, dx=False))
    fw = O.layer_fwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], ls.k, prec=O.Precision(y=False))
    idx = saved["topk_idx"].cpu().numpy()
    excused = compare_topk(idx, ref["topk_idx"], ref["z"], ls.k)
    counts = saved["counts"].cpu().numpy()
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=ls.E))
    keep = topk_margin(ref["z"], ls.k) >= 1e-6
    assert_close("y", f64(y)[keep], fw["y"][keep])
    if excused:
        return  # a tie changes the expert rows, so the gradients are not comparable
    E = ls.E
    pairs = {"dx": (f64(g["dx"]), ref["dx"]), "dW_r": (f64(g["dW_r"]), ref["dW_r"]),
             "dW1": (f64(g["dW1"]), np.stack([ref["dW1"][e] for e in range(E)])),
             "dW3": (f64(g["dW3"]), np.stack([ref["dW3"][e] for e in range(E)])),
             "dW2": (f64(g["dW2"]), np.stack([ref["dW2"][e] for e in range(E)]))}
    for key, (got, want) in pairs.items():
        assert_close(key, got, want, atol=wgrad_atol(want))
    assert abs(float(g["aux_loss"].item()) - ref["aux_loss"]) <= 1e-5 * max(1.0, abs(ref["aux_loss"]))
