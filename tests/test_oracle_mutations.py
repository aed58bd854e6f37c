"""Planted mistakes in the oracle (CPU): each test replaces one oracle function
with a plausibly wrong version and checks that at least one pin of
test_oracle_pins fails. This shows the pins are sharp enough to catch a
dropped term, a wrong sign, a reversed tie rule, a swapped operand or an
unstable order."""
import numpy as np
import pytest

import oracle as O
import oracle.moe_oracle as M
from tests import test_oracle_pins as P


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(M, name, fn)
    monkeypatch.setattr(O, name, fn)


def _route_unnormalised(x, w_r, k, score="softmax", expert_bias=None, logit_bias=None, n_groups=1,
                        topk_groups=1, gate_scale=1.0):
    out = _orig_route(x, w_r, k, score, expert_bias, logit_bias, n_groups, topk_groups, gate_scale)
    sel = np.take_along_axis(out["scores"], out["topk_idx"], axis=1)
    out["topk_gate"] = gate_scale * sel  # renormalisation dropped
    return out


_orig_route = M.route


def _topk_high_index_wins(z, k):
    idx = np.arange(z.shape[1])
    return np.stack([np.lexsort((-idx, -row))[:k] for row in z])


def _silu_grad_wrong_sign(z):
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 - z * (1.0 - s))


def _permute_plan_reversed_tokens(topk_idx, E):
    idx = np.asarray(topk_idx, np.int64)
    T, k = idx.shape
    counts = np.bincount(idx.ravel(), minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    tok = np.repeat(np.arange(T), k)
    order = np.lexsort((-tok, idx.ravel()))  # tokens in descending order inside an expert
    row = np.empty(T * k, np.int64)
    row[order] = np.arange(T * k)
    return counts, offsets, row.reshape(T, k)


def _aux_without_E(p, counts, k, alpha):
    T, E = p.shape
    return alpha * float(np.sum(np.asarray(counts) / (T * k) * p.mean(axis=0)))


def _group_limit_top1(z, n_groups, topk_groups):
    T, E = z.shape
    if n_groups <= 1 or topk_groups >= n_groups:
        return z.copy()
    gsz = E // n_groups
    gscore = z.reshape(T, n_groups, gsz).max(axis=2)  # best value only, not the two best
    keep = M.topk_select(gscore, topk_groups)
    mask = np.zeros((T, n_groups), bool)
    np.put_along_axis(mask, keep, True, axis=1)
    out = z.copy().reshape(T, n_groups, gsz)
    out[~mask] = -np.inf
    return out.reshape(T, E)


def _swiglu_gate_on_w3(xr, W1e, W3e, W2e, prec=O.CONTRACT):
    h1 = xr @ W3e  # operands swapped: the gate taken from the up projection
    h3 = xr @ W1e
    a = prec.r("a", M.silu(h1) * h3)
    return h1, h3, a, a @ W2e


def _router_bwd_no_inner(logits, topk_idx, topk_gate, dgate, score="softmax", gate_scale=1.0, counts=None,
                         k=None, aux_coeff=0.0, T_total=None):
    T, E = logits.shape
    dL = np.zeros((T, E))
    q = topk_gate / gate_scale
    np.put_along_axis(dL, topk_idx, gate_scale * q * dgate, axis=1)  # the -<q, dg> term dropped
    return dL


def _balanced_by_token(T, E, k):
    t = np.arange(T)[:, None]
    return (t + np.arange(k)[None, :]) % E  # the token's slots start at t, not at t k


MUTATIONS = [
    ("route", _route_unnormalised, [P.test_gates_sum_and_closed_form]),
    ("topk_select", _topk_high_index_wins, [P.test_topk_tie_rule]),
    ("silu_grad", _silu_grad_wrong_sign, [P.test_silu_closed_forms]),
    ("permute_plan", _permute_plan_reversed_tokens, [P.test_permute_invariants_and_brute_force]),
    ("aux_loss", _aux_without_E, [P.test_aux_loss_uniform_balanced_equals_alpha]),
    ("group_limit_mask", _group_limit_top1, [P.test_group_limit_against_enumeration]),
    ("swiglu_expert", _swiglu_gate_on_w3, [P.test_single_expert_is_textbook_swiglu_mlp]),
    ("balanced_assignment", _balanced_by_token, [P.test_force_balanced_assignment]),
    ("router_backward", _router_bwd_no_inner,
     [lambda: P.test_backward_against_central_differences("softmax_aux")]),
]


@pytest.mark.parametrize("name,fn,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, fn, pins):
    _patch(monkeypatch, name, fn)
    caught = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin caught the planted mistake in {name}"
