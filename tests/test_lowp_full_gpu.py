"""MXFP8 forward and NVFP4 grouped GEMM at full sizes (GPU), in the kernel
configuration the benchmark times, checked on sampled outputs the oracle
computes one by one: the MXFP8 layer on the Qwen3 expert shape (H=4096,
F=1536, top-8; 32 experts, T=4096) for 48 sampled tokens, and the NVFP4
grouped GEMM on the down projection's full shape (131072 x 1536 x 4096, 128
experts) for the rows of three experts, and the MXFP8 training step on the
full Qwen3 training workload (T=16384, E=128), with bf16 and with MXFP8
weight gradients, for one token's output and input gradient and one expert's
weight gradients; and the NVFP4 training step on the same workload for two
experts' weight gradients (its input gradient as a property against the bf16
step)."""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth
from tests._util import (TIE_MARGIN, assert_close, assert_close_but_flips, compare_topk, f64, mx_wgrad_atol,
                         wgrad_atol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


def test_mxfp8_layer_qwen3_expert_shape_sampled():
    ls = synth.shape("qwen3_e32")
    d = synth.make_layer(ls, seed=1234, device="cuda", training=False)
    cfg = ops.config_from_shape(ls)
    w = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
    ws = ops.mx_workspace(cfg)
    y = ops.layer_fwd_mxfp8(cfg, d["x"], d["router_w"], w, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    tok = np.random.default_rng(3).choice(ls.T, 48, replace=False)
    n = {k: (None if v is None else f64(v)) for k, v in d.items() if k in ("x", "router_w", "W1", "W3", "W2")}
    ref = O.mx_layer_fwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], ls.k, tokens=tok)
    assert_close("y (sampled tokens)", f64(y)[tok], ref["y"][tok])


def test_nvfp4_grouped_gemm_full_shape_sampled():
    E, R, K, N = 128, 131072, 1536, 4096
    offsets = np.arange(0, R + 1, R // E, dtype=np.int32)
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn((R, K), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((E, K, N), generator=g, device="cuda") * K ** -0.5).to(torch.bfloat16)
    w = ops.nv_quantize_weights(W)
    ws = ops.nv_workspace(E, R, K)
    y = ops.nv_grouped_gemm(x, torch.from_numpy(offsets).cuda(), w, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    # the tensor maximum from a host copy of the input (exact on bf16 values)
    gx = O.nv_tensor_scale(float(x.cpu().abs().max().float().item()))
    for e in (0, 63, 127):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        xe = f64(x[lo:hi]).astype(np.float32)
        xq = O.nv_roundtrip(xe, axis=1, g=gx)
        We = O.nv_roundtrip(f64(W[e]).astype(np.float32), axis=0)
        ref = O.bf16_rne(xq @ We)
        assert_close(f"y rows of expert {e}", f64(y[lo:hi]), ref, atol=max(2e-2, 2.0 ** -7 * float(np.abs(ref).max())))


class _PerExpert:
    """W[e] as an fp64 array, converted from the device tensor on demand."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return f64(self.t[e])


@pytest.mark.parametrize("wgrad", ["bf16", "mxfp8"])
def test_mxfp8_train_qwen3_full_sampled(wgrad):
    ls = synth.shape("qwen3_train")
    d = synth.make_layer(ls, seed=1234, device="cuda", training=True)
    cfg = ops.config_from_shape(ls, out_fp32=True)
    mxw = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
    mxbw = ops.mx_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
    ws = ops.mx_train_workspace(cfg)
    saved = ops.alloc_saved_mxfp8(cfg)
    y = ops.layer_fwd_mxfp8_train(cfg, d["x"], d["router_w"], mxw, saved, ws=ws)
    g = ops.layer_bwd_mxfp8(cfg, d["dO"], d["x"], d["router_w"], mxbw, saved, ws=ws, mx_wgrad=wgrad == "mxfp8")
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    x, w_r, dO = f64(d["x"]), f64(d["router_w"]), f64(d["dO"])
    k = ls.k
    rt = O.route(x, w_r, k)
    zs = -np.sort(-rt["z"], axis=1)
    ties = np.nonzero(zs[:, k - 1] - zs[:, k] < TIE_MARGIN)[0]
    ok = np.ones(ls.T, bool)
    ok[ties] = False
    # selected sets exact outside near-ties (slot order where the scores are separated)
    compare_topk(saved["topk_idx"].cpu().numpy(), rt["topk_idx"], rt["z"], k)
    # experts a near-tie token could move to or from are not sampled
    near = set()
    for t in ties:
        near.update(int(e) for e in np.argsort(-rt["z"][t], kind="stable")[k - 1:k + 1])
    counts = np.bincount(rt["topk_idx"].reshape(-1), minlength=ls.E)
    cand = [e for e in np.argsort(counts, kind="stable") if int(e) not in near]
    e0 = int(cand[len(cand) // 2])
    t0 = int(np.random.default_rng(7).choice(np.nonzero(ok)[0]))
    ref = O.mx_layer_bwd(x, w_r, _PerExpert(d["W1"]), _PerExpert(d["W3"]), _PerExpert(d["W2"]), dO, k,
                         aux_coeff=ls.aux_coeff, prec=O.Precision(y=False, dx=False), experts=[e0], tokens=[t0],
                         wgrad=wgrad)
    assert_close("y (sampled token)", f64(y)[t0], ref["y"][t0])
    assert_close("dx (sampled token)", f64(g["dx"])[t0], ref["dx"][t0], atol=wgrad_atol(ref["dx"][t0]))
    am = ref["wg_amax"][e0]
    for key, (oa, ob) in (("dW1", ("x", "dh1")), ("dW3", ("x", "dh3")), ("dW2", ("a", "dy"))):
        want = ref[key][e0]
        atol = mx_wgrad_atol(want, am[oa], am[ob]) if wgrad == "mxfp8" else wgrad_atol(want)
        assert_close(f"{key} (expert {e0}, {counts[e0]} rows)", f64(g[key][e0]), want, atol=atol)
    assert abs(float(g["aux_loss"].item()) - ref["aux_loss"]) <= 1e-5 * max(1.0, abs(ref["aux_loss"]))


def test_nvfp4_train_qwen3_full_sampled():
    # the NVFP4 training step on the full Qwen3 training workload: two experts'
    # weight gradients (the median and the largest row count among experts no
    # near-tie token can enter or leave) against the per-expert NVFP4 oracle,
    # whose tensor scales come from per-token maxima; the input gradient (whose
    # dh13 tensor scale needs every row) against the bf16 step as a property:
    # FP4-sized, not more
    ls = synth.shape("qwen3_train")
    d = synth.make_layer(ls, seed=1234, device="cuda", training=True)
    cfg = ops.config_from_shape(ls, out_fp32=True)
    nvw = ops.nv_quantize_layer_weights(cfg, d["W1"], d["W3"], d["W2"])
    nvbw = ops.nv_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
    ws = ops.nv_train_workspace(cfg)
    saved = ops.alloc_saved(cfg)
    ops.layer_fwd_nvfp4_train(cfg, d["x"], d["router_w"], nvw, saved, ws=ws)
    g = ops.layer_bwd_nvfp4(cfg, d["dO"], d["x"], d["router_w"], nvbw, saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    del nvw, nvbw, ws
    x, w_r, dO = f64(d["x"]), f64(d["router_w"]), f64(d["dO"])
    k = ls.k
    rt = O.route(x, w_r, k)
    zs = -np.sort(-rt["z"], axis=1)
    ties = np.nonzero(zs[:, k - 1] - zs[:, k] < TIE_MARGIN)[0]
    compare_topk(saved["topk_idx"].cpu().numpy(), rt["topk_idx"], rt["z"], k)
    near = set()
    for t in ties:
        near.update(int(e) for e in np.argsort(-rt["z"][t], kind="stable")[k - 1:k + 1])
    counts = np.bincount(rt["topk_idx"].reshape(-1), minlength=ls.E)
    cand = [int(e) for e in np.argsort(counts, kind="stable") if int(e) not in near]
    sample = [cand[len(cand) // 2], cand[-1]]
    ref = O.nv_expert_weight_grads(x, w_r, _PerExpert(d["W1"]), _PerExpert(d["W3"]), _PerExpert(d["W2"]), dO, k,
                                   experts=sample, prec=O.Precision(y=False, dx=False))
    for e in sample:
        for key in ("dW1", "dW3", "dW2"):
            want = ref[key][e]
            # flipped E2M1 codes of dy_perm (see assert_close_but_flips): an
            # expert of ~1000 rows x 4096 columns can see a few, each a rank-one
            # error; a GEMM error would not be of low rank
            assert_close_but_flips(f"{key} (expert {e}, {counts[e]} rows)", f64(g[key][e]), want,
                                   atol=wgrad_atol(want), rank=4)
    # the bf16 step on the same inputs (GPU): the NVFP4 input gradient differs
    # from it by FP4 rounding of two chained GEMMs
    ws16, sv16 = ops.workspace(cfg, True), ops.alloc_saved(cfg)
    ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved=sv16, ws=ws16)
    g16 = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], sv16, ws=ws16)
    torch.cuda.synchronize()
    dx, dx16 = g["dx"].float(), g16["dx"].float()
    assert torch.isfinite(dx).all()
    r = float((dx - dx16).norm() / dx16.norm())
    assert 1e-2 < r < 0.5, r
