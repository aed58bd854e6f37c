"""Pins of the fp64 oracle against what the report and the mathematics fix.

None of these tests compares the oracle with itself: each pin is a closed form,
a brute-force evaluation written independently here, a library routine, an
invariant, or a central finite difference. CPU only.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _ev(s):
    """Evaluate a golden-file expression: integers, fractions, lnN, and
    products like '-9/7*ln3'."""
    if isinstance(s, (int, float)):
        return float(s)
    s = s.strip()
    sign = -1.0 if s.startswith("-") else 1.0
    s = s.lstrip("-")
    val = 1.0
    for part in s.split("*"):
        if part.startswith("ln"):
            val *= math.log(float(part[2:]))
        else:
            val *= float(Fraction(part))
    return sign * val


def _arr(x):
    return np.array(x, dtype=object) if False else np.vectorize(_ev, otypes=[float])(np.array(x, dtype=object))


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_rne_matches_torch_on_fp32_values():
    # library routine: torch's float32 -> bfloat16 conversion (RNE). For values
    # that are exactly float32 no double rounding is possible, so the direct
    # fp64 rounding must agree bit for bit.
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 1, 37, 1e4)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_rne(v.astype(np.float64))
    assert np.array_equal(ref, got)


def test_bf16_rne_ties_to_even():
    ulp = 2.0 ** -7
    assert O.bf16_rne(np.array([1 + ulp / 2]))[0] == 1.0            # tie -> even (1.0)
    assert O.bf16_rne(np.array([1 + ulp + ulp / 2]))[0] == 1 + 2 * ulp  # tie -> even
    assert O.bf16_rne(np.array([1 + ulp / 2 + 1e-12]))[0] == 1 + ulp  # above the tie
    assert O.bf16_rne(np.array([-3.0]))[0] == -3.0


# ---------------------------------------------------------------- golden cases
def test_golden_softmax_top2_single_token():
    c = json.load(open(os.path.join(GOLD, "closed_form_cases.json")))["softmax_top2_single_token"]
    x = _arr(c["x"]); w_r = _arr(c["router_w"])
    W1 = _arr(c["W1"]); W3 = _arr(c["W3"]); W2 = _arr(c["W2"])
    ex = c["expected"]
    out = O.layer_fwd(x, w_r, W1, W3, W2, c["k"], prec=O.EXACT)
    np.testing.assert_allclose(out["scores"], _arr(ex["scores"]), rtol=0, atol=1e-15)
    assert out["topk_idx"].tolist() == ex["topk_idx"]
    np.testing.assert_allclose(out["topk_gate"], _arr(ex["topk_gate"]), rtol=0, atol=1e-15)
    assert out["counts"].tolist() == ex["counts"]
    assert out["offsets"].tolist() == ex["offsets"]
    assert out["row_id_map"].tolist() == ex["row_id_map"]
    np.testing.assert_allclose(out["y"], _arr(ex["y"]), rtol=0, atol=1e-14)


def test_golden_sigmoid_group_limited_single_token():
    c = json.load(open(os.path.join(GOLD, "closed_form_cases.json")))["sigmoid_group_limited_single_token"]
    x = _arr(c["x"]); w_r = _arr(c["router_w"])
    rt = O.route(x, w_r, c["k"], "sigmoid", expert_bias=_arr(c["expert_bias"]),
                 n_groups=c["n_groups"], topk_groups=c["topk_groups"], gate_scale=_ev(c["gate_scale"]))
    ex = c["expected"]
    np.testing.assert_allclose(rt["scores"], _arr(ex["scores"]), rtol=0, atol=1e-15)
    assert rt["topk_idx"].tolist() == ex["topk_idx"]
    np.testing.assert_allclose(rt["topk_gate"], _arr(ex["topk_gate"]), rtol=0, atol=1e-15)


# ---------------------------------------------------------------- router
def _brute_topk_set(z, k):
    """max-sum k-subset by enumeration (distinct values)."""
    best = None
    for sub in itertools.combinations(range(len(z)), k):
        s = sum(z[j] for j in sub)
        if best is None or s > best[0]:
            best = (s, sub)
    return set(best[1])


def test_topk_against_subset_enumeration():
    rng = np.random.default_rng(1)
    for E, k in [(6, 1), (6, 3), (7, 7), (8, 2), (9, 4)]:
        z = rng.standard_normal((40, E))
        idx = O.topk_select(z, k)
        for t in range(40):
            assert len(set(idx[t].tolist())) == k
            assert set(idx[t].tolist()) == _brute_topk_set(z[t], k)
            # slot order: descending z
            assert all(z[t, idx[t, i]] >= z[t, idx[t, i + 1]] for i in range(k - 1))
            # every selected value >= every unselected value
            un = [e for e in range(E) if e not in idx[t]]
            if un:
                assert z[t, idx[t]].min() >= z[t, un].max()


def test_topk_tie_rule():
    z = np.array([[1.0, 2.0, 2.0, 0.5, 2.0]])
    assert O.topk_select(z, 2).tolist() == [[1, 2]]
    assert O.topk_select(z, 4).tolist() == [[1, 2, 4, 0]]


def _brute_group_limited(z, G, Gt, k):
    E = len(z)
    gs = E // G
    gscore = [sum(sorted(z[g * gs:(g + 1) * gs], reverse=True)[:min(2, gs)]) for g in range(G)]
    # best set of Gt groups by enumeration (distinct sums)
    best = max(itertools.combinations(range(G), Gt), key=lambda sub: sum(gscore[g] for g in sub))
    allowed = [e for e in range(E) if e // gs in best]
    return set(sorted(allowed, key=lambda e: -z[e])[:k])


def test_group_limit_against_enumeration():
    rng = np.random.default_rng(2)
    for E, G, Gt, k in [(8, 4, 2, 3), (12, 3, 2, 4), (16, 8, 4, 8), (8, 2, 1, 2)]:
        z = rng.standard_normal((30, E))
        idx = O.topk_select(O.group_limit_mask(z, G, Gt), k)
        for t in range(30):
            assert set(idx[t].tolist()) == _brute_group_limited(z[t], G, Gt, k)
            assert len({e // (E // G) for e in idx[t]}) <= Gt


def test_group_limit_reduces_to_plain_topk():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((50, 16))
    plain = O.topk_select(z, 4)
    assert np.array_equal(O.topk_select(O.group_limit_mask(z, 1, 1), 4), plain)
    assert np.array_equal(O.topk_select(O.group_limit_mask(z, 4, 4), 4), plain)


def test_gates_sum_and_closed_form():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 32)); w = rng.standard_normal((16, 32)) / 6
    rt = O.route(x, w, 4)
    np.testing.assert_allclose(rt["topk_gate"].sum(1), 1.0, rtol=0, atol=1e-15)
    # renormalised softmax == softmax over the selected logits (closed form)
    Lsel = np.take_along_axis(rt["logits"], rt["topk_idx"], 1)
    q = np.exp(Lsel - Lsel.max(1, keepdims=True)); q /= q.sum(1, keepdims=True)
    np.testing.assert_allclose(rt["topk_gate"], q, rtol=1e-14, atol=0)
    rs = O.route(x, w, 4, "sigmoid", expert_bias=rng.uniform(-.1, .1, 16), n_groups=4,
                 topk_groups=2, gate_scale=2.5)
    np.testing.assert_allclose(rs["topk_gate"].sum(1), 2.5, rtol=0, atol=1e-14)


def test_force_balanced_assignment():
    """Force-balanced routing: the T k assignments cycle through the experts
    (counted here with a running counter, one assignment at a time), every
    expert gets floor(T k / E) or one more, a token's experts are distinct, and
    the gates are the renormalised scores of the assigned experts."""
    rng = np.random.default_rng(21)
    for T, E, k in ((37, 8, 3), (64, 16, 4), (5, 4, 4), (9, 7, 1)):
        idx = O.balanced_assignment(T, E, k)
        c = 0
        for t in range(T):
            for i in range(k):
                assert idx[t, i] == c % E
                c += 1
        counts = np.bincount(idx.ravel(), minlength=E)
        assert counts.min() == (T * k) // E and counts.max() <= (T * k + E - 1) // E
        assert all(len(set(row)) == k for row in idx.tolist())
        x = rng.standard_normal((T, 8)); w = rng.standard_normal((E, 8)) / 3
        rt = O.route(x, w, k, force_balanced=True)
        assert np.array_equal(rt["topk_idx"], idx)
        Lsel = np.take_along_axis(rt["logits"], idx, 1)
        q = np.exp(Lsel - Lsel.max(1, keepdims=True)); q /= q.sum(1, keepdims=True)
        np.testing.assert_allclose(rt["topk_gate"], q, rtol=1e-13, atol=0)
        rs = O.route(x, w, k, "sigmoid", gate_scale=2.5, force_balanced=True)
        ssel = 1.0 / (1.0 + np.exp(-np.take_along_axis(rs["logits"], idx, 1)))
        np.testing.assert_allclose(rs["topk_gate"], 2.5 * ssel / ssel.sum(1, keepdims=True), rtol=1e-13, atol=0)
        if (T * k) % E == 0:
            # every f_e = 1/E, and the mean probabilities sum to one: L_aux = alpha
            assert abs(O.aux_loss(rt["scores"], counts, k, 0.01) - 0.01) < 1e-15


def test_recompute_variant_equals_standard_in_exact_arithmetic():
    """The memory-saving backward (a recomputed from h1, h3; gate gradient
    <da, a> / g instead of <dO, y_perm>) is the same function as the standard
    backward when nothing is rounded."""
    rng = np.random.default_rng(22)
    T, H, E, k, F = 40, 12, 6, 3, 10
    x = rng.standard_normal((T, H)); w_r = rng.standard_normal((E, H)) / 2
    W1, W3, W2 = _experts(rng, E, H, F)
    dO = rng.standard_normal((T, H))
    for kw in (dict(aux_coeff=0.05), dict(score="sigmoid", gate_scale=2.5, n_groups=3, topk_groups=2),
               dict(force_balanced=True, aux_coeff=0.05)):
        a = O.layer_bwd(x, w_r, W1, W3, W2, dO, k, prec=O.EXACT, **kw)
        b = O.layer_bwd(x, w_r, W1, W3, W2, dO, k, prec=O.EXACT, recompute=True, **kw)
        np.testing.assert_allclose(b["dgate"], a["dgate"], rtol=1e-11, atol=1e-12)
        for key in ("dx", "dW_r"):
            np.testing.assert_allclose(b[key], a[key], rtol=1e-11, atol=1e-12)
        for key in ("dW1", "dW3", "dW2"):
            for e in range(E):
                np.testing.assert_allclose(b[key][e], a[key][e], rtol=1e-11, atol=1e-12)


def test_router_logits_against_python_loop():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 5)); w = rng.standard_normal((4, 5)); b = rng.standard_normal(4)
    L = O.router_logits(x, w, b)
    for t in range(3):
        for e in range(4):
            assert abs(L[t, e] - (sum(x[t, h] * w[e, h] for h in range(5)) + b[e])) < 1e-13


def test_softmax_sigmoid_library():
    L = np.random.default_rng(6).standard_normal((10, 7)) * 3
    np.testing.assert_allclose(O.softmax(L), torch.softmax(torch.from_numpy(L), 1).numpy(), rtol=1e-14)
    np.testing.assert_allclose(O.sigmoid(L), torch.sigmoid(torch.from_numpy(L)).numpy(), rtol=1e-14)


# ---------------------------------------------------------------- permute
def test_permute_invariants_and_brute_force():
    rng = np.random.default_rng(7)
    T, E, k = 200, 9, 3
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    idx[:, :] = np.where(idx == 4, 5, idx) if False else idx
    counts, offsets, row = O.permute_plan(idx, E)
    assert counts.sum() == T * k and offsets[-1] == T * k and np.all(np.diff(offsets) >= 0)
    assert sorted(row.ravel().tolist()) == list(range(T * k))          # bijection
    # brute force: walk tokens in order, hand out the next row of each expert
    nxt = offsets[:-1].copy()
    for t in range(T):
        for i in range(k):
            e = idx[t, i]
            assert row[t, i] == nxt[e]
            nxt[e] += 1
    # rows sorted by (expert, token)
    key = np.empty((T * k, 2), int)
    for t in range(T):
        for i in range(k):
            key[row[t, i]] = (idx[t, i], t)
    assert all(tuple(key[r]) < tuple(key[r + 1]) for r in range(T * k - 1))


def test_permute_zero_token_experts():
    idx = np.array([[3, 1], [3, 1], [1, 3]])
    counts, offsets, row = O.permute_plan(idx, 6)
    assert counts.tolist() == [0, 3, 0, 3, 0, 0]
    assert offsets.tolist() == [0, 0, 3, 3, 6, 6, 6]
    assert row.tolist() == [[3, 0], [4, 1], [2, 5]]


def test_combine_of_permute_is_scaled_identity():
    rng = np.random.default_rng(8)
    T, H, E, k = 50, 12, 8, 3
    x = rng.standard_normal((T, H))
    rt = O.route(x[:, :12], rng.standard_normal((E, 12)), k)
    _, _, row = O.permute_plan(rt["topk_idx"], E)
    xp = O.permute_rows(x, row)
    np.testing.assert_allclose(O.combine(xp, row, rt["topk_gate"]), x, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(O.combine(xp, row, np.ones((T, k))), k * x, rtol=1e-14)
    np.testing.assert_allclose(O.combine(xp, row, 2.5 * rt["topk_gate"]), 2.5 * x, rtol=1e-14)


# ---------------------------------------------------------------- experts / layer
def _experts(rng, E, H, F):
    return (rng.standard_normal((E, H, F)) / math.sqrt(H), rng.standard_normal((E, H, F)) / math.sqrt(H),
            rng.standard_normal((E, F, H)) / math.sqrt(F))


def _dense_reference(x, w_r, W1, W3, W2, k, score, bias, G, Gt, scale, Ws=None):
    """Brute-force dense evaluation, written independently of the oracle: run
    every expert on every token and weight by a dense gate vector that is zero
    off the selected set. Membership is decided by counting how many experts beat
    an expert (ties: lower index wins), after the group mask."""
    T, H = x.shape
    E = W1.shape[0]
    L = x @ w_r.T
    if score == "softmax":
        s = np.exp(L - L.max(1, keepdims=True)); s /= s.sum(1, keepdims=True)
    else:
        s = 1 / (1 + np.exp(-L))
    z = s + (0 if bias is None else bias)
    gs = E // G
    y = np.zeros((T, H))
    for t in range(T):
        allowed = set(range(E))
        if G > 1 and Gt < G:
            gsc = [sum(sorted(z[t, g * gs:(g + 1) * gs], reverse=True)[:min(2, gs)]) for g in range(G)]
            beat = [sum(1 for h in range(G) if gsc[h] > gsc[g] or (gsc[h] == gsc[g] and h < g)) for g in range(G)]
            allowed = {e for e in range(E) if beat[e // gs] < Gt}
        sel = []
        for e in allowed:
            nb = sum(1 for f in allowed if z[t, f] > z[t, e] or (z[t, f] == z[t, e] and f < e))
            if nb < k:
                sel.append(e)
        gv = np.zeros(E)
        tot = sum(s[t, e] for e in sel)
        for e in sel:
            gv[e] = scale * s[t, e] / tot
        for e in range(E):
            h1 = x[t] @ W1[e]; h3 = x[t] @ W3[e]
            a = h1 / (1 + np.exp(-h1)) * h3
            y[t] += gv[e] * (a @ W2[e])
        if Ws is not None:
            h1 = x[t] @ Ws[0]; h3 = x[t] @ Ws[1]
            y[t] += (h1 / (1 + np.exp(-h1)) * h3) @ Ws[2]
    return y


@pytest.mark.parametrize("case", [
    dict(T=16, H=24, E=8, k=2, F=16, score="softmax", G=1, Gt=1, scale=1.0, bias=False, shared=False),
    dict(T=12, H=16, E=8, k=3, F=8, score="sigmoid", G=4, Gt=2, scale=2.5, bias=True, shared=True),
    dict(T=10, H=8, E=6, k=6, F=8, score="softmax", G=1, Gt=1, scale=1.0, bias=False, shared=False),
])
def test_layer_against_dense_bruteforce(case):
    rng = np.random.default_rng(9)
    T, H, E, k, F = case["T"], case["H"], case["E"], case["k"], case["F"]
    x = rng.standard_normal((T, H)); w_r = rng.standard_normal((E, H)) / math.sqrt(H)
    W1, W3, W2 = _experts(rng, E, H, F)
    bias = rng.uniform(-.1, .1, E) if case["bias"] else None
    Ws = (rng.standard_normal((H, 8)) / 4, rng.standard_normal((H, 8)) / 4,
          rng.standard_normal((8, H)) / 3) if case["shared"] else None
    out = O.layer_fwd(x, w_r, W1, W3, W2, k, case["score"], expert_bias=bias,
                      n_groups=case["G"], topk_groups=case["Gt"], gate_scale=case["scale"],
                      Ws=Ws, prec=O.EXACT)
    ref = _dense_reference(x, w_r, W1, W3, W2, k, case["score"], bias, case["G"], case["Gt"],
                           case["scale"], Ws)
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def test_identical_experts_give_scaled_ffn():
    # All experts equal => y = (sum g) * FFN(x) for any routing (the report's
    # upcycling figure: copies of one MLP reproduce the dense model).
    rng = np.random.default_rng(10)
    T, H, E, k, F = 20, 16, 6, 3, 12
    x = rng.standard_normal((T, H)); w_r = rng.standard_normal((E, H))
    w1, w3, w2 = rng.standard_normal((H, F)), rng.standard_normal((H, F)), rng.standard_normal((F, H))
    W1, W3, W2 = np.stack([w1] * E), np.stack([w3] * E), np.stack([w2] * E)
    h1 = x @ w1
    ffn = (h1 / (1 + np.exp(-h1)) * (x @ w3)) @ w2
    out = O.layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT)
    np.testing.assert_allclose(out["y"], ffn, rtol=1e-12, atol=1e-12)
    out = O.layer_fwd(x, w_r, W1, W3, W2, k, "sigmoid", gate_scale=2.5, prec=O.EXACT)
    np.testing.assert_allclose(out["y"], 2.5 * ffn, rtol=1e-12, atol=1e-12)


def test_e_equals_k_is_dense_softmax_moe():
    rng = np.random.default_rng(11)
    T, H, E, F = 15, 10, 4, 6
    x = rng.standard_normal((T, H)); w_r = rng.standard_normal((E, H))
    W1, W3, W2 = _experts(rng, E, H, F)
    xt = torch.from_numpy(x)
    p = torch.softmax(xt @ torch.from_numpy(w_r).T, 1)
    ref = sum(p[:, e:e + 1] * ((torch.nn.functional.silu(xt @ torch.from_numpy(W1[e])) *
                                (xt @ torch.from_numpy(W3[e]))) @ torch.from_numpy(W2[e])) for e in range(E))
    out = O.layer_fwd(x, w_r, W1, W3, W2, E, prec=O.EXACT)
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_single_expert_is_textbook_swiglu_mlp():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((9, 8)); W1, W3, W2 = _experts(rng, 1, 8, 5)
    xt = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(xt @ torch.from_numpy(W1[0])) * (xt @ torch.from_numpy(W3[0]))) \
        @ torch.from_numpy(W2[0])
    out = O.layer_fwd(x, rng.standard_normal((1, 8)), W1, W3, W2, 1, prec=O.EXACT)
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-13, atol=1e-13)


def test_silu_closed_forms():
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert O.silu_grad(np.array([0.0]))[0] == 0.5
    z = np.linspace(-8, 8, 101)
    np.testing.assert_allclose(O.silu(z), torch.nn.functional.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-15)
    h = 1e-6
    np.testing.assert_allclose(O.silu_grad(z), (O.silu(z + h) - O.silu(z - h)) / (2 * h), rtol=1e-8, atol=1e-9)


def test_grouped_swiglu_matches_per_token_layer():
    rng = np.random.default_rng(13)
    T, H, E, k, F = 30, 16, 5, 2, 8
    x = rng.standard_normal((T, H)); w_r = rng.standard_normal((E, H))
    W1, W3, W2 = _experts(rng, E, H, F)
    rt = O.route(x, w_r, k)
    _, off, row = O.permute_plan(rt["topk_idx"], E)
    _, _, yp = O.grouped_swiglu(O.permute_rows(x, row), off, W1, W3, W2, O.EXACT)
    out = O.layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT)
    np.testing.assert_allclose(O.combine(yp, row, rt["topk_gate"]), out["y"], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- aux loss
def test_aux_loss_uniform_balanced_equals_alpha():
    T, E, k = 64, 8, 2
    p = np.full((T, E), 1.0 / E)
    counts = np.full(E, T * k // E)
    assert abs(O.aux_loss(p, counts, k, 1e-2) - 1e-2) < 1e-17


# ---------------------------------------------------------------- backward
def _loss(x, w_r, W1, W3, W2, dO, k, kw, Ws=None):
    out = O.layer_fwd(x, w_r, W1, W3, W2, k, Ws=Ws, prec=O.EXACT, **kw)
    val = float(np.sum(out["y"] * dO))
    if kw.get("aux_coeff"):
        pass
    return val, out


def _margins_ok(x, w_r, k, kw, step):
    rt = O.route(x, w_r, k, kw.get("score", "softmax"), kw.get("expert_bias"), None,
                 kw.get("n_groups", 1), kw.get("topk_groups", 1), kw.get("gate_scale", 1.0))
    z = np.sort(rt["z"], 1)[:, ::-1]
    zz = np.where(np.isfinite(z), z, -1e9)
    return np.min(zz[:, k - 1] - zz[:, k]) > 100 * step


@pytest.mark.parametrize("variant", ["softmax_aux", "sigmoid_groups_shared", "force_balanced_aux"])
def test_backward_against_central_differences(variant):
    rng = np.random.default_rng({"softmax_aux": 14, "sigmoid_groups_shared": 15}.get(variant, 16))
    T, H, E, k, F = 8, 6, 4, 2, 5
    kw = {}
    aux = 0.0
    Ws = None
    if variant == "softmax_aux":
        aux = 1e-1
    elif variant == "force_balanced_aux":
        aux = 1e-1
        kw = dict(force_balanced=True)
    else:
        kw = dict(score="sigmoid", expert_bias=rng.uniform(-.1, .1, E), n_groups=2,
                  topk_groups=1, gate_scale=2.5)
        Ws = [rng.standard_normal((H, 3)) / 2, rng.standard_normal((H, 3)) / 2, rng.standard_normal((3, H)) / 2]
    for _ in range(50):
        x = rng.standard_normal((T, H)); w_r = rng.standard_normal((E, H))
        if _margins_ok(x, w_r, k, kw, 1e-6):
            break
    else:
        pytest.fail("no tie-free draw")
    W1, W3, W2 = _experts(rng, E, H, F)
    dO = rng.standard_normal((T, H))

    def L(x_, w_r_, W1_, W3_, W2_, Ws_=Ws):
        out = O.layer_fwd(x_, w_r_, W1_, W3_, W2_, k, Ws=Ws_, prec=O.EXACT, **kw)
        val = float(np.sum(out["y"] * dO))
        if aux:
            val += O.aux_loss(out["scores"], out["counts"], k, aux)
        return val

    g = O.layer_bwd(x, w_r, W1, W3, W2, dO, k, aux_coeff=aux, Ws=Ws, prec=O.EXACT, **kw)
    h = 1e-6

    def fd(arr, fn):
        out = np.zeros_like(arr)
        for ix in np.ndindex(arr.shape):
            old = arr[ix]
            arr[ix] = old + h; lp = fn()
            arr[ix] = old - h; lm = fn()
            arr[ix] = old
            out[ix] = (lp - lm) / (2 * h)
        return out

    def close(a, b):
        np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-7 * max(1.0, np.abs(b).max()))

    close(g["dx"], fd(x, lambda: L(x, w_r, W1, W3, W2)))
    close(g["dW_r"], fd(w_r, lambda: L(x, w_r, W1, W3, W2)))
    dW1 = np.stack([g["dW1"][e] for e in range(E)])
    dW3 = np.stack([g["dW3"][e] for e in range(E)])
    dW2 = np.stack([g["dW2"][e] for e in range(E)])
    close(dW1, fd(W1, lambda: L(x, w_r, W1, W3, W2)))
    close(dW3, fd(W3, lambda: L(x, w_r, W1, W3, W2)))
    close(dW2, fd(W2, lambda: L(x, w_r, W1, W3, W2)))
    if Ws is not None:
        close(g["dWs1"], fd(Ws[0], lambda: L(x, w_r, W1, W3, W2)))
        close(g["dWs2"], fd(Ws[2], lambda: L(x, w_r, W1, W3, W2)))
    if aux:
        out = O.layer_fwd(x, w_r, W1, W3, W2, k, prec=O.EXACT, **kw)
        assert abs(g["aux_loss"] - O.aux_loss(out["scores"], out["counts"], k, aux)) < 1e-15


def test_backward_sampled_matches_full():
    rng = np.random.default_rng(16)
    T, H, E, k, F = 40, 12, 6, 2, 8
    x = rng.standard_normal((T, H)); w_r = rng.standard_normal((E, H))
    W1, W3, W2 = _experts(rng, E, H, F)
    dO = rng.standard_normal((T, H))
    full = O.layer_bwd(x, w_r, W1, W3, W2, dO, k, aux_coeff=1e-2)
    part = O.layer_bwd(x, w_r, W1, W3, W2, dO, k, aux_coeff=1e-2, experts=[1, 4], tokens=[0, 7, 33])
    np.testing.assert_allclose(part["dx"][[0, 7, 33]], full["dx"][[0, 7, 33]], rtol=1e-13, atol=1e-13)
    for e in (1, 4):
        np.testing.assert_allclose(part["dW1"][e], full["dW1"][e], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(part["dW2"][e], full["dW2"][e], rtol=1e-13, atol=1e-13)


def test_storage_rounding_points():
    # CONTRACT rounds exactly the stored tensors: a is a bf16 value, y_perm too.
    rng = np.random.default_rng(17)
    x = O.bf16_rne(rng.standard_normal((7, 8)))
    W1, W3, W2 = _experts(rng, 1, 8, 4)
    h1, h3, a, out = O.swiglu_expert(x, W1[0], W3[0], W2[0], O.CONTRACT)
    assert np.array_equal(a, O.bf16_rne(a))
    np.testing.assert_allclose(out, a @ W2[0], rtol=1e-15)
