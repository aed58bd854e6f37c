"""Parity at the full layer sizes (GPU, slow): the Qwen3-235B-shaped layer
(balanced and Zipf-skewed routing), the Mixtral-8x7B-shaped and the
DeepSeek-V3-shaped layers (forward), and the Qwen3 training step (forward +
backward, balanced and skewed), in the launch configuration the benchmark
times. Routing, counts, offsets and the permutation are checked in full;
floating-point outputs on seeded samples the fp64 oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth
from tests._util import assert_close, compare_topk, f64, report_exact, topk_margin, wgrad_atol

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


def _getter(d):
    def get(e):
        return f64(d["W1"][e]), f64(d["W3"][e]), f64(d["W2"][e])
    return get


def _check_routing(ls, d, saved):
    """Full routing check. Returns (oracle route dict, tokens away from ties)."""
    x = f64(d["x"])
    rt = O.route(x, f64(d["router_w"]), ls.k, ls.score,
                 None if d["expert_bias"] is None else f64(d["expert_bias"]),
                 None if d["logit_bias"] is None else f64(d["logit_bias"]),
                 ls.n_groups, ls.topk_groups, ls.gate_scale)
    idx = saved["topk_idx"].cpu().numpy()
    excluded = compare_topk(idx, rt["topk_idx"], rt["z"], ls.k)
    assert excluded <= ls.T // 200, f"{excluded} tokens within the tie margin"
    counts = saved["counts"].cpu().numpy()
    offs = saved["offsets"].cpu().numpy()
    rows = saved["row_id_map"].cpu().numpy()
    if excluded == 0:
        c_ref, o_ref, r_ref = O.permute_plan(rt["topk_idx"], ls.E)
        assert np.array_equal(counts, c_ref) and np.array_equal(offs, o_ref) and np.array_equal(rows, r_ref)
    # properties that hold for any valid selection: counts are the histogram of
    # the selection, offsets its prefix sum, rows a bijection grouped by expert
    # in token order
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=ls.E))
    assert offs[0] == 0 and np.array_equal(np.diff(offs), counts) and offs[-1] == ls.T * ls.k
    flat = rows.ravel()
    assert np.array_equal(np.sort(flat), np.arange(ls.T * ls.k))
    e_of_row = np.empty(ls.T * ls.k, np.int64)
    t_of_row = np.empty(ls.T * ls.k, np.int64)
    e_of_row[flat] = idx.ravel()
    t_of_row[flat] = np.repeat(np.arange(ls.T), ls.k)
    key = e_of_row * ls.T + t_of_row
    assert np.all(np.diff(key) > 0)
    keep = topk_margin(rt["z"], ls.k) >= 1e-6
    return rt, keep


def _sample(rng, keep, n):
    cand = np.nonzero(keep)[0]
    return np.sort(rng.choice(cand, size=min(n, len(cand)), replace=False))


# The Qwen3 shapes run as the benchmark does (bf16 y). The Mixtral and
# DeepSeek-V3 shapes reach |y| ~ 10-15, where one bf16 ulp of y (0.03-0.06)
# is above the 2e-2 bar by itself, so their parity reads the fp32 output.
@pytest.mark.parametrize("name,ntok,out_fp32", [("qwen3", 384, False), ("qwen3_skew", 384, False),
                                               ("mixtral", 256, True), ("dsv3", 64, True)])
def test_full_forward(name, ntok, out_fp32):
    ls = synth.shape(name)
    d = synth.make_layer(ls, seed=1234, device="cuda", training=False)
    cfg = ops.config_from_shape(ls, out_fp32=out_fp32)
    ws = ops.workspace(cfg, True)
    saved = ops.alloc_saved(cfg)
    Ws = (d["Ws1"], d["Ws3"], d["Ws2"]) if ls.F_shared else None
    y = ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"], Ws,
                      saved=saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    rt, keep = _check_routing(ls, d, saved)
    if ls.skew:
        # Zipf-skewed popularity: a dominant expert and experts with no token
        counts = saved["counts"].cpu().numpy()
        assert counts.max() > 8 * counts.mean()
        assert (counts == 0).sum() >= 1
    rng = np.random.default_rng(7)
    tok = _sample(rng, keep, ntok)
    prec = O.Precision(y_perm=not ls.inter_fp32, shared=not ls.inter_fp32, y=not out_fp32)
    Wsn = tuple(f64(w) for w in Ws) if Ws is not None else None
    ref = O.layer_fwd(f64(d["x"]), f64(d["router_w"]), _getter(d), None, None, ls.k, ls.score,
                      None if d["expert_bias"] is None else f64(d["expert_bias"]),
                      None if d["logit_bias"] is None else f64(d["logit_bias"]),
                      ls.n_groups, ls.topk_groups, ls.gate_scale, Ws=Wsn, prec=prec, tokens=tok)
    assert_close("y", f64(y[torch.from_numpy(tok).cuda()]), ref["y"][tok])
    ex = O.layer_fwd(f64(d["x"]), f64(d["router_w"]), _getter(d), None, None, ls.k, ls.score,
                     None if d["expert_bias"] is None else f64(d["expert_bias"]),
                     None if d["logit_bias"] is None else f64(d["logit_bias"]),
                     ls.n_groups, ls.topk_groups, ls.gate_scale, Ws=Wsn, prec=O.EXACT, tokens=tok)
    report_exact(f"full_forward[{name}] y ({len(tok)} tokens)", f64(y[torch.from_numpy(tok).cuda()]), ex["y"][tok])
    # gates of the sampled tokens
    assert_close("gates", f64(saved["topk_gate"])[tok], ref["topk_gate"][tok])


@pytest.mark.parametrize("name", ["qwen3_train", "qwen3_skew_train"])
def test_full_training_step(name):
    ls = synth.shape(name)
    d = synth.make_layer(ls, seed=1234, device="cuda", training=True)
    cfg = ops.config_from_shape(ls)  # bf16 y and dx, as the benchmark
    ws = ops.workspace(cfg, True)
    saved = ops.alloc_saved(cfg)
    ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"],
                  saved=saved, ws=ws)
    g = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    rt, keep = _check_routing(ls, d, saved)
    counts = saved["counts"].cpu().numpy()
    if ls.skew:
        assert counts.max() > 8 * counts.mean() and (counts == 0).sum() >= 1
    rng = np.random.default_rng(11)
    gidx = saved["topk_idx"].cpu().numpy()
    # an expert's weight gradient is comparable when the GPU and the oracle route
    # the same tokens to it (a token near a selection tie may go either way)
    same = [e for e in range(ls.E)
            if np.array_equal(np.nonzero((gidx == e).any(1))[0], np.nonzero((rt["topk_idx"] == e).any(1))[0])]
    assert len(same) >= ls.E // 2
    if ls.skew:
        nz = np.array([e for e in np.nonzero(counts)[0] if e in same])
        order = nz[np.argsort(counts[nz])]
        experts = sorted({int(order[-1]), int(order[len(order) // 2]), int(order[0])})
    else:
        experts = sorted(rng.choice(same, size=3, replace=False).tolist())
    # dx on tokens sampled away from selection ties
    tok = _sample(rng, keep, 128)
    x = f64(d["x"])
    lb = None if d["logit_bias"] is None else f64(d["logit_bias"])
    prec = O.Precision(y=True, dx=True)
    ref = O.layer_bwd(x, f64(d["router_w"]), _getter(d), None, None, f64(d["dO"]), ls.k, ls.score, None, lb,
                      aux_coeff=ls.aux_coeff, prec=prec, experts=experts, tokens=tok)
    assert_close("dx", f64(g["dx"][torch.from_numpy(tok).cuda()]), ref["dx"][tok])
    for e in experts:
        for key in ("dW1", "dW3", "dW2"):
            want = ref[key][e]
            assert_close(f"{key}[{e}]", f64(g[key][e]), want, atol=wgrad_atol(want))
    ex = O.layer_bwd(x, f64(d["router_w"]), _getter(d), None, None, f64(d["dO"]), ls.k, ls.score, None, lb,
                     aux_coeff=ls.aux_coeff, prec=O.EXACT, experts=experts, tokens=tok)
    report_exact(f"full_training_step[{name}] dx ({len(tok)} tokens)", f64(g["dx"][torch.from_numpy(tok).cuda()]),
                 ex["dx"][tok])
    for e in experts:
        for key in ("dW1", "dW3", "dW2"):
            report_exact(f"full_training_step[{name}] {key}[{e}] ({int(counts[e])} rows)", f64(g[key][e]), ex[key][e])
    # router weight gradient, row of one expert: dL[t,e] for every token. Tokens
    # routed to e need their gate gradients (all k expert outputs); the others
    # only carry the aux-loss part, which depends on their softmax and the counts.
    e = experts[0]
    te = np.nonzero(rt["topk_idx"] == e)[0]
    part = O.layer_bwd(x, f64(d["router_w"]), _getter(d), None, None, f64(d["dO"]), ls.k, ls.score, None, lb,
                       aux_coeff=ls.aux_coeff, prec=prec, experts=[], tokens=te)
    others = np.setdiff1d(np.arange(ls.T), te)
    dL_aux = O.router_backward(rt["logits"][others], rt["topk_idx"][others], rt["topk_gate"][others],
                               np.zeros((len(others), ls.k)), ls.score, ls.gate_scale, rt_counts(rt, ls), ls.k,
                               ls.aux_coeff, T_total=ls.T)
    dwr_e = part["dlogits"][:, e] @ x[te] + dL_aux[:, e] @ x[others]
    assert_close(f"dW_r[{e}]", f64(g["dW_r"][e]), dwr_e, atol=wgrad_atol(dwr_e))
    assert abs(float(g["aux_loss"].item()) - ref["aux_loss"]) <= 1e-4 * abs(ref["aux_loss"])


def rt_counts(rt, ls):
    return np.bincount(rt["topk_idx"].ravel(), minlength=ls.E)


@pytest.mark.parametrize("skew", [0.0, 1.2])
def test_full_permute_bit_exact(skew):
    T, H, E, k = 16384, 4096, 128, 8
    cfg = ops.make_config(T, H, E, k, 1536)
    idx = synth.synthetic_topk(T, E, k, seed=3, skew=skew, device="cuda")
    x = synth.make_layer(synth.shape("qwen3"), seed=3, device="cuda")["x"]
    ws = ops.workspace(cfg)
    xp, rows, counts, offs = ops.permute(cfg, x, idx, ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    c_ref, o_ref, r_ref = O.permute_plan(idx.cpu().numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), c_ref)
    assert np.array_equal(offs.cpu().numpy(), o_ref)
    assert np.array_equal(rows.cpu().numpy(), r_ref)
    # x_perm rows of a seeded sample of (t, i) pairs, bytes unchanged
    rng = np.random.default_rng(1)
    ts = rng.choice(T, size=512, replace=False)
    xb = x.view(torch.int16)
    xpb = xp.view(torch.int16)
    for i in range(k):
        r = torch.from_numpy(r_ref[ts, i]).cuda()
        assert torch.equal(xpb[r], xb[torch.from_numpy(ts).cuda()])


@pytest.mark.parametrize("mode", ["memory_saving", "force_balanced"])
def test_full_training_step_modes(mode):
    """The two optional training modes at the full Qwen3 size, as
    `bench.py --recompute` / `--force-balanced` time them: the memory-saving
    backward (a and y_perm not kept) against the oracle's recompute variant,
    and force-balanced routing (assignment and counts bit for bit)."""
    force = mode == "force_balanced"
    rec = mode == "memory_saving"
    ls = synth.shape("qwen3_train", force_balanced=force)
    d = synth.make_layer(ls, seed=1234, device="cuda", training=True)
    cfg = ops.config_from_shape(ls)
    ws = ops.workspace(cfg, True)
    saved = ops.alloc_saved(cfg, recompute=rec)
    ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"],
                  saved=saved, ws=ws)
    g = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    x = f64(d["x"])
    rt = O.route(x, f64(d["router_w"]), ls.k, ls.score, None, None, ls.n_groups, ls.topk_groups, ls.gate_scale,
                 force_balanced=force)
    gidx = saved["topk_idx"].cpu().numpy()
    counts = saved["counts"].cpu().numpy()
    if force:
        assert np.array_equal(gidx, rt["topk_idx"])
        assert np.all(counts == ls.T * ls.k // ls.E)
        keep = np.ones(ls.T, bool)
    else:
        assert compare_topk(gidx, rt["topk_idx"], rt["z"], ls.k) <= ls.T // 200
        keep = topk_margin(rt["z"], ls.k) >= 1e-6
    same = [e for e in range(ls.E)
            if np.array_equal(np.nonzero((gidx == e).any(1))[0], np.nonzero((rt["topk_idx"] == e).any(1))[0])]
    assert len(same) >= ls.E // 2
    rng = np.random.default_rng(13)
    experts = sorted(rng.choice(same, size=3, replace=False).tolist())
    tok = _sample(rng, keep, 128)
    prec = O.Precision(y=True, dx=True)
    kw = dict(force_balanced=force, recompute=rec)
    ref = O.layer_bwd(x, f64(d["router_w"]), _getter(d), None, None, f64(d["dO"]), ls.k, ls.score, None, None,
                      aux_coeff=ls.aux_coeff, prec=prec, experts=experts, tokens=tok, **kw)
    assert_close("dx", f64(g["dx"][torch.from_numpy(tok).cuda()]), ref["dx"][tok])
    for e in experts:
        for key in ("dW1", "dW3", "dW2"):
            want = ref[key][e]
            assert_close(f"{key}[{e}]", f64(g[key][e]), want, atol=wgrad_atol(want))
    e = experts[0]
    te = np.nonzero(rt["topk_idx"] == e)[0]
    part = O.layer_bwd(x, f64(d["router_w"]), _getter(d), None, None, f64(d["dO"]), ls.k, ls.score, None, None,
                       aux_coeff=ls.aux_coeff, prec=prec, experts=[], tokens=te, **kw)
    others = np.setdiff1d(np.arange(ls.T), te)
    dL_aux = O.router_backward(rt["logits"][others], rt["topk_idx"][others], rt["topk_gate"][others],
                               np.zeros((len(others), ls.k)), ls.score, ls.gate_scale, rt_counts(rt, ls), ls.k,
                               ls.aux_coeff, T_total=ls.T)
    dwr_e = part["dlogits"][:, e] @ x[te] + dL_aux[:, e] @ x[others]
    assert_close(f"dW_r[{e}]", f64(g["dW_r"][e]), dwr_e, atol=wgrad_atol(dwr_e))


def test_full_training_step_shared_expert():
    """The DeepSeek-V3-shaped layer (256 experts, sigmoid with group limit,
    one shared expert F=2048) through forward and backward: the shared
    expert's weight gradients (they depend on every token, not on routing) on
    sampled rows, dx on sampled tokens, two routed experts' weight
    gradients."""
    ls = synth.shape("dsv3")
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
    rt, keep = _check_routing(ls, d, saved)
    gidx = saved["topk_idx"].cpu().numpy()
    rng = np.random.default_rng(17)
    same = [e for e in range(ls.E)
            if np.array_equal(np.nonzero((gidx == e).any(1))[0], np.nonzero((rt["topk_idx"] == e).any(1))[0])]
    experts = sorted(rng.choice(same, size=2, replace=False).tolist())
    tok = _sample(rng, keep, 64)
    x = f64(d["x"])
    Wsn = tuple(f64(w) for w in Ws)
    prec = O.Precision(y_perm=False, shared=False, dx_perm=False, y=False, dx=False)
    ref = O.layer_bwd(x, f64(d["router_w"]), _getter(d), None, None, f64(d["dO"]), ls.k, ls.score,
                      f64(d["expert_bias"]), None, ls.n_groups, ls.topk_groups, ls.gate_scale, Ws=Wsn, prec=prec,
                      experts=experts, tokens=tok)
    assert_close("dx", f64(g["dx"][torch.from_numpy(tok).cuda()]), ref["dx"][tok])
    for e in experts:
        for key in ("dW1", "dW3", "dW2"):
            want = ref[key][e]
            assert_close(f"{key}[{e}]", f64(g[key][e]), want, atol=wgrad_atol(want))
    rows_h = np.sort(rng.choice(ls.H, size=256, replace=False))
    rows_f = np.sort(rng.choice(ls.F_shared, size=128, replace=False))
    for key, rows in (("dWs1", rows_h), ("dWs3", rows_h), ("dWs2", rows_f)):
        want = ref[key][rows]
        assert_close(f"{key} ({len(rows)} rows)", f64(g[key][torch.from_numpy(rows).cuda()]), want,
                     atol=wgrad_atol(ref[key]))
