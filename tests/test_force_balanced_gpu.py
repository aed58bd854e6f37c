"""Force-balanced routing (throughput page, Table 11) through the C ABI against
the oracle (GPU): the assignment and the counts bit for bit; gates, the layer
output and every gradient within the layer tolerances. The assignment does not
depend on the scores, so no token is excused for a near tie."""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth
from tests._util import MAX_ABS, assert_close, f64, wgrad_atol

pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny": synth.shape("tiny"),
    "e128_k8": synth.shape("tiny", T=777, H=256, E=128, k=8, F=256, w_std=0.05),
    "dsv3_small": synth.shape("dsv3", T=333, H=256, E=64, k=8, F=128, F_shared=192),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


def _np(d):
    return {k: (None if v is None else f64(v)) for k, v in d.items()}


@pytest.mark.parametrize("name", list(SHAPES))
def test_router_and_counts(name):
    ls = SHAPES[name]
    d = synth.make_layer(ls, seed=77, device="cuda", training=True)
    cfg = ops.config_from_shape(ls, force_balanced=True)
    idx, gate, logits, _ = ops.router_topk(cfg, d["x"], d["router_w"], d["expert_bias"], d["logit_bias"],
                                           want_logits=True)
    torch.cuda.synchronize()
    n = _np(d)
    ref = O.route(n["x"], n["router_w"], ls.k, ls.score, n["expert_bias"], n["logit_bias"], ls.n_groups,
                  ls.topk_groups, ls.gate_scale, force_balanced=True)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    assert_close("gate", f64(gate), ref["topk_gate"])
    _, _, counts, offsets = ops.permute(cfg, d["x"], idx)
    c = counts.cpu().numpy()
    assert c.min() == (ls.T * ls.k) // ls.E and c.max() <= -(-(ls.T * ls.k) // ls.E)
    assert np.array_equal(c, np.bincount(ref["topk_idx"].ravel(), minlength=ls.E))


@pytest.mark.parametrize("name", list(SHAPES))
def test_layer_fwd_bwd(name):
    ls = SHAPES[name]
    d = synth.make_layer(ls, seed=78, device="cuda", training=True)
    aux = 1e-2 if ls.score == "softmax" else 0.0
    cfg = ops.config_from_shape(ls, force_balanced=True, aux_coeff=aux, out_fp32=True)
    ws = ops.workspace(cfg, True)
    saved = ops.alloc_saved(cfg)
    Ws = (d["Ws1"], d["Ws3"], d["Ws2"]) if ls.F_shared else None
    y = ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"], Ws,
                      saved=saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    n = _np(d)
    kw = dict(force_balanced=True)
    nWs = (n["Ws1"], n["Ws3"], n["Ws2"]) if ls.F_shared else None
    prec_f = O.Precision(y_perm=not ls.inter_fp32, shared=not ls.inter_fp32, y=False)
    fw = O.layer_fwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], ls.k, ls.score, n["expert_bias"],
                     n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale, Ws=nWs, prec=prec_f, **kw)
    assert np.array_equal(saved["topk_idx"].cpu().numpy(), fw["topk_idx"])
    assert_close("y", f64(y), fw["y"])
    if ls.F_shared:
        return  # the backward does not take a shared expert
    g = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    ref = O.layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score, n["expert_bias"],
                      n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale, aux_coeff=aux,
                      prec=O.Precision(y=False, dx=False), **kw)
    E = ls.E
    pairs = {"dx": (f64(g["dx"]), ref["dx"]), "dW_r": (f64(g["dW_r"]), ref["dW_r"]),
             "dW1": (f64(g["dW1"]), np.stack([ref["dW1"][e] for e in range(E)])),
             "dW3": (f64(g["dW3"]), np.stack([ref["dW3"][e] for e in range(E)])),
             "dW2": (f64(g["dW2"]), np.stack([ref["dW2"][e] for e in range(E)]))}
    for key, (got, want) in pairs.items():
        atol = wgrad_atol(want) if (key != "dx" or name == "e128_k8") else MAX_ABS
        assert_close(key, got, want, atol=atol)
    if aux:
        assert abs(float(g["aux_loss"].item()) - ref["aux_loss"]) <= 1e-5 * max(1.0, abs(ref["aux_loss"]))
