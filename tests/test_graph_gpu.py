"""Whole-layer CUDA Graph capture (GPU). The forward and the backward keep the
per-expert offsets on the device and never synchronise with the host, so one
training step (router, permute, expert GEMMs, combine and the whole backward)
captures into a single graph. Replays must reproduce the eager results bit for
bit (every kernel of the path is deterministic), and a replay after new inputs
are copied into the captured buffers must match an eager step on them."""
import pytest
import torch

from route_permute_grouped_gb300 import ops, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


def _step(cfg, d, saved, ws, y, grads):
    ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"],
                  saved=saved, ws=ws, y=y)
    ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws, grads=grads)


def _snapshot(y, grads):
    return [y.clone()] + [grads[k].clone() for k in ("dx", "dW_r", "dW1", "dW3", "dW2", "aux_loss")]


@pytest.mark.parametrize("name,force", [("tiny", False), ("e128", False), ("e128", True)])
def test_training_step_graph_replay(name, force):
    ls = synth.shape("tiny") if name == "tiny" else synth.shape("tiny", T=777, H=256, E=128, k=8, F=256, w_std=0.05)
    d = synth.make_layer(ls, seed=5, device="cuda", training=True)
    cfg = ops.config_from_shape(ls, aux_coeff=1e-2, force_balanced=force)
    ws = ops.workspace(cfg, True)
    saved = ops.alloc_saved(cfg)
    grads = ops.alloc_grads(cfg)
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _step(cfg, d, saved, ws, y, grads)  # eager: also does the one-time per-device set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = _snapshot(y, grads)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _step(cfg, d, saved, ws, y, grads)
    for a in (y, *grads.values()):
        a.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    for a, b in zip(eager, _snapshot(y, grads)):
        assert torch.equal(a, b)
    # new inputs through the captured buffers
    d2 = synth.make_layer(ls, seed=6, device="cuda", training=True)
    for key in ("x", "dO"):
        d[key].copy_(d2[key])
    g.replay()
    torch.cuda.synchronize()
    replayed = _snapshot(y, grads)
    _step(cfg, d, saved, ws, y, grads)
    torch.cuda.synchronize()
    for a, b in zip(replayed, _snapshot(y, grads)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("prec", ["mxfp8", "nvfp4"])
def test_low_precision_training_step_graph_replay(prec):
    # the MXFP8 and NVFP4 training steps keep their scales and tensor maxima
    # on the device too: one step captures and replays bit for bit
    ls = synth.shape("tiny", T=300, H=256, E=8, k=2, F=256)
    d = synth.make_layer(ls, seed=5, device="cuda", training=True)
    cfg = ops.config_from_shape(ls, aux_coeff=1e-2)
    grads = ops.alloc_grads(cfg)
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    if prec == "mxfp8":
        wf = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
        wb = ops.mx_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
        ws, saved = ops.mx_train_workspace(cfg), ops.alloc_saved_mxfp8(cfg)
        fwd, bwd = ops.layer_fwd_mxfp8_train, ops.layer_bwd_mxfp8
    else:
        wf = ops.nv_quantize_layer_weights(cfg, d["W1"], d["W3"], d["W2"])
        wb = ops.nv_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
        ws, saved = ops.nv_train_workspace(cfg), ops.alloc_saved(cfg)
        fwd, bwd = ops.layer_fwd_nvfp4_train, ops.layer_bwd_nvfp4

    def step():
        fwd(cfg, d["x"], d["router_w"], wf, saved, d["expert_bias"], d["logit_bias"], ws=ws, y=y)
        bwd(cfg, d["dO"], d["x"], d["router_w"], wb, saved, ws=ws, grads=grads)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = _snapshot(y, grads)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for a in (y, *grads.values()):
        a.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    for a, b in zip(eager, _snapshot(y, grads)):
        assert torch.equal(a, b)
