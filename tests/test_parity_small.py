"""Parity of every C-ABI entry point against the fp64 oracle on small layers
that still span several tiles and a ragged tail (GPU). Integer outputs are
compared bit for bit; floating-point outputs to relative L2 <= 5e-3 and
max-abs <= 2e-2."""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth
from tests._util import MAX_ABS, assert_close, compare_topk, f64, rel_l2, report_exact, wgrad_atol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


SHAPES = {
    "tiny": synth.shape("tiny"),
    # ragged: T not a multiple of 128, H not a multiple of 256, F not of 128
    "ragged": synth.shape("tiny", T=1000, H=320, E=8, k=2, F=192),
    "e128_k8": synth.shape("tiny", T=777, H=256, E=128, k=8, F=256, w_std=0.05),
    "skew": synth.shape("tiny", T=900, H=256, E=32, k=4, F=128, skew=1.2),
    "dsv3_small": synth.shape("dsv3", T=333, H=256, E=64, k=8, F=128, F_shared=192),
    "e_eq_k": synth.shape("tiny", T=200, H=128, E=4, k=4, F=128),
    "k1": synth.shape("tiny", T=300, H=192, E=3, k=1, F=64),
    # softmax scores with a group limit and no expert bias: groups are ranked
    # by sums of probabilities (not of logits)
    "softmax_groups": synth.shape("tiny", T=450, H=256, E=64, k=6, F=128, n_groups=8, topk_groups=3, w_std=0.1),
}


# shapes outside the layer configurations (fan-in scaled weights, larger
# activations): gradients use the one-bf16-ulp max-abs allowance
FLIP_BOUND_SHAPES = {"ragged", "e128_k8", "skew", "k1"}


def _inputs(name, device="cuda", seed=1234):
    ls = SHAPES[name]
    d = synth.make_layer(ls, seed=seed, device=device, training=True)
    return ls, d


def _np(d):
    return {k: (None if v is None else f64(v)) for k, v in d.items()}


def _oracle_route(ls, n):
    return O.route(n["x"], n["router_w"], ls.k, ls.score, n["expert_bias"], n["logit_bias"], ls.n_groups,
                   ls.topk_groups, ls.gate_scale)


@pytest.mark.parametrize("name", list(SHAPES))
def test_router(name):
    ls, d = _inputs(name)
    cfg = ops.config_from_shape(ls)
    ws = ops.workspace(cfg)
    idx, gate, logits, aux = ops.router_topk(cfg, d["x"], d["router_w"], d["expert_bias"], d["logit_bias"],
                                             want_logits=True, want_aux=ls.score == "softmax", ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    n = _np(d)
    rt = _oracle_route(ls, n)
    assert rel_l2(f64(logits), rt["logits"]) < 1e-5
    assert np.max(np.abs(f64(logits) - rt["logits"])) < 1e-4
    excluded = compare_topk(idx.cpu().numpy(), rt["topk_idx"], rt["z"], ls.k)
    assert excluded <= max(2, ls.T // 100)
    # gates: compare where the selection matches the oracle
    same = np.all(idx.cpu().numpy() == rt["topk_idx"], axis=1)
    assert_close("gates", f64(gate)[same], rt["topk_gate"][same])
    np.testing.assert_allclose(f64(gate).sum(1), ls.gate_scale, rtol=1e-5)
    if aux is not None:
        p = rt["scores"]
        nsl = 4 * ((ls.T + 127) // 128)
        ref = np.stack([p[32 * i:32 * (i + 1)].sum(0) if 32 * i < ls.T else np.zeros(ls.E) for i in range(nsl)])
        assert_close("aux_partials", f64(aux), ref, rel=1e-5, atol=1e-4)


@pytest.mark.parametrize("T,E,k,skew", [(1000, 8, 2, 0.0), (777, 128, 8, 0.0), (4097, 128, 8, 1.2),
                                        (65, 256, 8, 1.5), (1, 4, 3, 0.0), (3000, 3, 1, 0.0)])
def test_permute_bit_exact(T, E, k, skew):
    H = 192
    cfg = ops.make_config(T, H, E, k, 64)
    idx = synth.synthetic_topk(T, E, k, seed=7, skew=skew, device="cuda")
    x = synth.make_layer(synth.shape("tiny", T=T, H=H, E=E, k=k, F=64), device="cuda")["x"]
    ws = ops.workspace(cfg)
    xp, rows, counts, offs = ops.permute(cfg, x, idx, ws)
    assert ops.device_status(ws) == 0
    c_ref, o_ref, r_ref = O.permute_plan(idx.cpu().numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), c_ref)
    assert np.array_equal(offs.cpu().numpy(), o_ref)
    assert np.array_equal(rows.cpu().numpy(), r_ref)
    xp_ref = O.permute_rows(x.cpu().view(torch.int16).numpy(), r_ref)  # bytes move unchanged
    assert np.array_equal(xp.cpu().view(torch.int16).numpy(), xp_ref)
    if skew > 0:  # the skewed draws are far from balanced
        assert c_ref.max() > 4 * c_ref.mean()


def _ffn_inputs(ls, d):
    n = _np(d)
    rt = _oracle_route(ls, n)
    counts, offs, rows = O.permute_plan(rt["topk_idx"], ls.E)
    # bf16 rows moved as raw 16-bit patterns
    xp = torch.from_numpy(O.permute_rows(d["x"].cpu().view(torch.int16).numpy(), rows)).view(torch.bfloat16)
    return n, rt, counts, offs, rows, xp


@pytest.mark.parametrize("name", ["tiny", "ragged", "e128_k8", "skew", "k1"])
def test_grouped_swiglu_ffn(name):
    ls, d = _inputs(name)
    cfg = ops.config_from_shape(ls)
    n, rt, counts, offs, rows, xp = _ffn_inputs(ls, d)
    xp_d = xp.cuda()
    offs_d = torch.from_numpy(offs.astype(np.int32)).cuda()
    ws = ops.workspace(cfg)
    y_perm, h13, a = ops.grouped_swiglu_ffn(cfg, xp_d, offs_d, d["W1"], d["W3"], d["W2"], save=True, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    h13_ref, a_ref, y_ref = O.grouped_swiglu(f64(xp), offs, n["W1"], n["W3"], n["W2"])
    assert_close("h13", f64(h13), h13_ref)
    assert_close("a", f64(a), a_ref)
    assert_close("y_perm", f64(y_perm), y_ref)


def test_grouped_swiglu_ffn_tile_boundaries():
    # expert row counts on every side of the tile boundaries: an expert's last
    # m tile holding 1, 63, 64, 65, 127 or 128 rows runs as a half-height
    # (M = 128) pair tile, 129..256 rows as a whole tile; an empty expert; F and
    # H ragged against the 128- and 256-column tiles
    counts = [1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 384, 385, 0, 512, 640]
    E, H, F = len(counts), 384, 320
    R = int(sum(counts))
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    g = torch.Generator().manual_seed(17)
    xp = torch.randn((R, H), generator=g).to(torch.bfloat16)
    W1 = (torch.randn((E, H, F), generator=g) * H ** -0.5).to(torch.bfloat16)
    W3 = (torch.randn((E, H, F), generator=g) * H ** -0.5).to(torch.bfloat16)
    W2 = (torch.randn((E, F, H), generator=g) * F ** -0.5).to(torch.bfloat16)
    cfg = ops.make_config(R, H, E, 1, F)
    y_perm, h13, a = ops.grouped_swiglu_ffn(cfg, xp.cuda(), torch.from_numpy(offs.astype(np.int32)).cuda(),
                                            W1.cuda(), W3.cuda(), W2.cuda(), save=True)
    torch.cuda.synchronize()
    h13_ref, a_ref, y_ref = O.grouped_swiglu(f64(xp), offs, f64(W1), f64(W3), f64(W2))
    assert_close("h13", f64(h13), h13_ref)
    assert_close("a", f64(a), a_ref)
    assert_close("y_perm", f64(y_perm), y_ref)


@pytest.mark.parametrize("name", ["tiny", "e128_k8", "dsv3_small"])
def test_unpermute_combine(name):
    ls, d = _inputs(name)
    cfg = ops.config_from_shape(ls, out_fp32=True)
    R = ls.T * ls.k
    g = torch.Generator(device="cuda").manual_seed(5)
    y_perm = torch.randn((R, ls.H), generator=g, device="cuda").to(torch.float32 if ls.inter_fp32 else torch.bfloat16)
    idx = synth.synthetic_topk(ls.T, ls.E, ls.k, seed=3, device="cuda")
    _, _, rows = O.permute_plan(idx.cpu().numpy(), ls.E)
    gate = torch.rand((ls.T, ls.k), generator=g, device="cuda")
    shared = None
    if ls.F_shared:
        shared = torch.randn((ls.T, ls.H), generator=g, device="cuda").to(y_perm.dtype)
    y = ops.unpermute_combine(cfg, y_perm, torch.from_numpy(rows.astype(np.int32)).cuda(), gate, shared)
    ref = O.combine(f64(y_perm), rows, f64(gate), None if shared is None else f64(shared))
    # fp32 reduction of k terms: a few fp32 ulps
    assert_close("y", f64(y), ref, rel=1e-6, atol=1e-5)


def _layer_ref(ls, n, prec):
    Ws = (n["Ws1"], n["Ws3"], n["Ws2"]) if ls.F_shared else None
    return O.layer_fwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], ls.k, ls.score, n["expert_bias"],
                       n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale, Ws=Ws, prec=prec)


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("out_fp32", [True, False])
def test_layer_fwd(name, out_fp32):
    ls, d = _inputs(name)
    cfg = ops.config_from_shape(ls, out_fp32=out_fp32)
    ws = ops.workspace(cfg)
    Ws = (d["Ws1"], d["Ws3"], d["Ws2"]) if ls.F_shared else None
    y = ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"], Ws,
                      ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    n = _np(d)
    prec = O.Precision(y_perm=not ls.inter_fp32, shared=not ls.inter_fp32, y=not out_fp32)
    ref = _layer_ref(ls, n, prec)
    rt = ref
    # tokens near a selection tie may route differently; compare the others
    from tests._util import topk_margin
    keep = topk_margin(rt["z"], ls.k) >= 1e-6
    assert keep.sum() >= 0.99 * ls.T
    assert_close("y", f64(y)[keep], ref["y"][keep])
    report_exact(f"layer_fwd[{name}, out_fp32={out_fp32}] y", f64(y)[keep], _layer_ref(ls, n, O.EXACT)["y"][keep])


@pytest.mark.parametrize("name", ["tiny", "ragged", "e128_k8", "skew", "k1"])
def test_layer_bwd(name):
    ls, d = _inputs(name)
    aux = 1e-2
    cfg = ops.config_from_shape(ls, aux_coeff=aux, out_fp32=True)
    ws = ops.workspace(cfg, True)
    saved = ops.alloc_saved(cfg)
    y = ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"],
                      saved=saved, ws=ws)
    g = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    n = _np(d)
    ref = O.layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score, n["expert_bias"],
                      n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale, aux_coeff=aux,
                      prec=O.Precision(y=False, dx=False))
    # the selection must agree for the gradient comparison to be meaningful
    assert np.array_equal(saved["topk_idx"].cpu().numpy(), ref["topk_idx"]), "routing differs (tie)"
    E = ls.E
    pairs = {"dx": (f64(g["dx"]), ref["dx"]), "dW_r": (f64(g["dW_r"]), ref["dW_r"]),
             "dW1": (f64(g["dW1"]), np.stack([ref["dW1"][e] for e in range(E)])),
             "dW3": (f64(g["dW3"]), np.stack([ref["dW3"][e] for e in range(E)])),
             "dW2": (f64(g["dW2"]), np.stack([ref["dW2"][e] for e in range(E)]))}
    for key, (got, want) in pairs.items():
        # weight gradients: the bf16-storage flip bound (see wgrad_atol); dx
        # keeps the layer's 2e-2 on the layer configurations and takes the same
        # flip bound on the fan-in-scaled robustness shapes, whose activations
        # are larger
        atol = wgrad_atol(want) if (key != "dx" or name in FLIP_BOUND_SHAPES) else MAX_ABS
        assert_close(key, got, want, atol=atol)
    ex = O.layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score, n["expert_bias"],
                     n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale, aux_coeff=aux, prec=O.EXACT)
    for key in ("dx", "dW_r"):
        report_exact(f"layer_bwd[{name}] {key}", pairs[key][0], ex[key])
    for key in ("dW1", "dW3", "dW2"):
        report_exact(f"layer_bwd[{name}] {key}", pairs[key][0], np.stack([ex[key][e] for e in range(E)]))
    assert abs(float(g["aux_loss"].item()) - ref["aux_loss"]) <= 1e-5 * max(1.0, abs(ref["aux_loss"]))


SHARED_SHAPES = {
    "dsv3_small": SHAPES["dsv3_small"],
    "softmax_shared": synth.shape("tiny", T=300, H=192, E=8, k=2, F=128, F_shared=128),
}


@pytest.mark.parametrize("name", list(SHARED_SHAPES))
def test_layer_bwd_shared_expert(name):
    """The backward of a layer with a shared expert (figures & tables page,
    Fig. 40): the shared expert's weight gradients (independent of routing)
    in full, and the routed gradients and dx where the routing agrees with
    the oracle's (tokens within the selection tie margin may differ)."""
    ls = SHARED_SHAPES[name]
    d = synth.make_layer(ls, seed=1234, device="cuda", training=True)
    cfg = ops.config_from_shape(ls, out_fp32=True)
    ws = ops.workspace(cfg, True)
    saved = ops.alloc_saved(cfg)
    Ws = (d["Ws1"], d["Ws3"], d["Ws2"])
    ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"], Ws,
                  saved=saved, ws=ws)
    g = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws, Ws=Ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    n = _np(d)
    Wsn = (n["Ws1"], n["Ws3"], n["Ws2"])
    prec = O.Precision(y_perm=not ls.inter_fp32, shared=not ls.inter_fp32, dx_perm=not ls.inter_fp32, y=False,
                       dx=False)
    ref = O.layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score, n["expert_bias"],
                      n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale, Ws=Wsn, prec=prec)
    ex = O.layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score, n["expert_bias"],
                     n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale, Ws=Wsn, prec=O.EXACT)
    for key in ("dWs1", "dWs3", "dWs2"):
        assert_close(key, f64(g[key]), ref[key], atol=wgrad_atol(ref[key]))
        report_exact(f"layer_bwd_shared[{name}] {key}", f64(g[key]), ex[key])
    idx = saved["topk_idx"].cpu().numpy()
    excused = compare_topk(idx, ref["topk_idx"], ref["z"], ls.k)
    same_tok = np.all(np.sort(idx, 1) == np.sort(ref["topk_idx"], 1), axis=1)
    assert same_tok.sum() >= ls.T - excused
    atol_dx = wgrad_atol(ref["dx"]) if name in FLIP_BOUND_SHAPES else MAX_ABS
    assert_close("dx", f64(g["dx"])[same_tok], ref["dx"][same_tok], atol=atol_dx)
    report_exact(f"layer_bwd_shared[{name}] dx", f64(g["dx"])[same_tok], ex["dx"][same_tok])
    same_e = [e for e in range(ls.E)
              if np.array_equal(np.nonzero((idx == e).any(1))[0], np.nonzero((ref["topk_idx"] == e).any(1))[0])]
    assert len(same_e) >= ls.E // 2
    for key in ("dW1", "dW3", "dW2"):
        want = np.stack([ref[key][e] for e in same_e])
        assert_close(key, f64(g[key])[same_e], want, atol=wgrad_atol(want))
