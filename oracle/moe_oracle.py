"""Plain fp64 definition of the single-GPU MoE layer hot path.

TEST INFRASTRUCTURE: the independent checker of the CUDA library. Only the
tests, the smoke check and the benchmark's CPU-baseline leg use it. Nothing here
is tuned; every step is the textbook definition written out with numpy in
float64, a matmul or a stable sort being the only library primitives.

Sources (all from the report "Scalable Training of Mixture-of-Experts Models
with Megatron Core"; "summary page" = its paper-summary page, "captions page" =
its figures & tables page):

* layer equation y = sum_i g(x)_i * E_i(x): summary page, "Problem Definition";
* Router -> Dispatcher -> Experts -> Combiner: summary page, "Pipeline Flow" and
  "System Modules"; captions page, Fig. 1 (Route, Dispatch, Compute, Combine);
* router = learned linear layer + score function + top-k + load balancing:
  summary page, "System Modules" (Router); captions page, Fig. 2 and Fig. 39;
* experts are feed-forward networks with the SwiGLU activation: summary page,
  "System Modules" (Experts); captions page, Table 4 (activation function
  SwiGLU) and the GLU-variants reference of the report;
* grouped GEMM = several GEMMs of different sizes at once: summary page,
  "Key Terms" (Grouped GEMM);
* shared expert sees every token: captions page, Fig. 40;
* memory-efficient permutation (probabilities applied at combine): captions
  page, Fig. 7 and Table 6.

What the report leaves open is fixed by the readings listed with each function
(sigmoid scores, selection-only expert bias, group-limited selection, gate
scale, the auxiliary-loss formula, tie rules and the storage precision).

Storage precision. The layer stores activations in bf16 and accumulates in
fp32. Wherever the layer stores a tensor in bf16 (the SwiGLU activation ``a``,
the saved pre-activations ``h13``, the expert outputs ``y_perm`` when kept in
bf16, the backward's ``dy_perm``, ``dh13`` and ``dx_perm``, and a bf16 layer
output) this oracle rounds the fp64 value to bf16 (round to nearest even) at the
same point, and computes everything else in fp64. ``EXACT`` turns every such
rounding off (used by the finite-difference pins).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "Precision", "EXACT", "CONTRACT", "bf16_rne", "router_logits", "softmax",
    "sigmoid", "group_limit_mask", "topk_select", "balanced_assignment", "route", "permute_plan",
    "permute_rows", "silu", "silu_grad", "swiglu_expert", "grouped_swiglu",
    "combine", "layer_fwd", "aux_loss", "router_backward", "layer_bwd",
    "expert_backward",
]


# ----------------------------------------------------------------------------
# bf16 storage rounding
# ----------------------------------------------------------------------------
def bf16_rne(a):
    """Round float64 values to the nearest bfloat16 (ties to even), returned as
    float64. bfloat16 keeps 8 significant bits and the float32 exponent range;
    the rounding is done once, directly from the float64 bit pattern (no
    intermediate float32 rounding). Inputs are finite (non-finite values are
    outside the layer's contract)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    u = a.view(np.uint64)
    drop = np.uint64(52 - 7)  # float64 has 52 stored mantissa bits, bf16 has 7
    lsb = (u >> drop) & np.uint64(1)
    half = np.uint64(1) << (drop - np.uint64(1))
    r = (u + (half - np.uint64(1)) + lsb) & ~((np.uint64(1) << drop) - np.uint64(1))
    return r.view(np.float64).reshape(a.shape)


@dataclass(frozen=True)
class Precision:
    """Which stored tensors are rounded to bf16 (True) or kept exact (False)."""
    a: bool = True          # SwiGLU activation fed to the down projection
    h13: bool = True        # saved gate/up pre-activations (backward input)
    y_perm: bool = True     # expert outputs, one row per (token, slot)
    shared: bool = True     # shared-expert output
    y: bool = False         # layer output
    dy_perm: bool = True    # gate-weighted output gradient per row
    dh13: bool = True       # SwiGLU-backward output
    dx_perm: bool = True    # input gradient per row
    dx: bool = False        # layer input gradient

    def r(self, name, v):
        return bf16_rne(v) if getattr(self, name) else v


CONTRACT = Precision()
EXACT = Precision(a=False, h13=False, y_perm=False, shared=False, y=False,
                  dy_perm=False, dh13=False, dx_perm=False, dx=False)


# ----------------------------------------------------------------------------
# Router: linear projection, score function, top-k, gates
# (summary page "System Modules" Router; captions page Fig. 2)
# ----------------------------------------------------------------------------
def router_logits(x, w_r, logit_bias=None):
    """L[t,e] = sum_h x[t,h] * w_r[e,h] (+ logit_bias[e]).

    ``w_r`` is [E,H], the layout of a linear layer mapping H features to E
    outputs. ``logit_bias`` is an optional additive per-expert logit offset (an
    input, used by the benchmark to create a skewed expert popularity)."""
    L = np.asarray(x, np.float64) @ np.asarray(w_r, np.float64).T
    if logit_bias is not None:
        L = L + np.asarray(logit_bias, np.float64)[None, :]
    return L


def softmax(L):
    """p = exp(L - max L) / sum exp(L - max L) over the expert axis."""
    m = L.max(axis=1, keepdims=True)
    e = np.exp(L - m)
    return e / e.sum(axis=1, keepdims=True)


def sigmoid(L):
    """s = 1 / (1 + exp(-L))."""
    return 1.0 / (1.0 + np.exp(-L))


def topk_select(z, k):
    """Indices of the k largest entries of each row of z.

    Reading (the report is silent on ties): a lower expert index wins a tie, and
    the k slots are ordered by descending z, then ascending index. A stable
    sort of -z keeps equal values in ascending index order."""
    order = np.argsort(-z, axis=1, kind="stable")
    return order[:, :k]


def group_limit_mask(z, n_groups, topk_groups):
    """Group-limited selection: split the E experts into ``n_groups`` contiguous
    groups, score each group by the sum of its two largest z values (one value
    if a group holds one expert), keep the ``topk_groups`` best groups (lower
    group index wins a tie) and return z with every expert of a dropped group
    set to -inf. With topk_groups == n_groups it returns z unchanged."""
    T, E = z.shape
    if n_groups <= 1 or topk_groups >= n_groups:
        return z.copy()
    gsz = E // n_groups
    zg = z.reshape(T, n_groups, gsz)
    top2 = -np.sort(-zg, axis=2)[:, :, : min(2, gsz)]
    gscore = top2.sum(axis=2)                        # [T, n_groups]
    keep = topk_select(gscore, topk_groups)          # [T, topk_groups]
    mask = np.zeros((T, n_groups), dtype=bool)
    np.put_along_axis(mask, keep, True, axis=1)
    out = z.copy().reshape(T, n_groups, gsz)
    out[~mask] = -np.inf
    return out.reshape(T, E)


def balanced_assignment(T, E, k):
    """Force-balanced routing (throughput page, Table 11: every configuration
    of the unified benchmark uses force-balanced routing; the page gives no
    rule). Reading: slot i of token t goes to expert (t k + i) mod E, so the
    T k assignments cycle through the experts and every expert receives
    floor(T k / E) or one more; a token's k experts are distinct when k <= E."""
    t = np.arange(T)[:, None]
    i = np.arange(k)[None, :]
    return (t * k + i) % E


def route(x, w_r, k, score="softmax", expert_bias=None, logit_bias=None,
          n_groups=1, topk_groups=1, gate_scale=1.0, force_balanced=False):
    """The router of the MoE layer.

    1. logits L = x w_r^T (+ logit_bias);
    2. scores: softmax over all E experts, or element-wise sigmoid;
    3. selection value z = scores (+ expert_bias, selection only), optionally
       group-limited, then top-k (force_balanced: the fixed assignment of
       ``balanced_assignment`` instead of the top-k);
    4. gates g_i = gate_scale * score[e_i] / sum_j score[e_j] over the k
       selected experts (renormalised; for sigmoid the unbiased score).

    Returns a dict with logits [T,E], scores [T,E], z [T,E] (after the group
    mask), topk_idx [T,k] int64 and topk_gate [T,k]."""
    L = router_logits(x, w_r, logit_bias)
    if score == "softmax":
        s = softmax(L)
    elif score == "sigmoid":
        s = sigmoid(L)
    else:
        raise ValueError(score)
    z = s if expert_bias is None else s + np.asarray(expert_bias, np.float64)[None, :]
    z = group_limit_mask(z, n_groups, topk_groups)
    if force_balanced:
        idx = balanced_assignment(L.shape[0], L.shape[1], k)
    else:
        idx = topk_select(z, k)
    sel = np.take_along_axis(s, idx, axis=1)
    gate = gate_scale * sel / sel.sum(axis=1, keepdims=True)
    return {"logits": L, "scores": s, "z": z, "topk_idx": idx, "topk_gate": gate}


# ----------------------------------------------------------------------------
# Local dispatch: histogram, prefix sum, stable scatter into expert-contiguous
# rows (summary page "Key Terms" Grouped GEMM; captions page Fig. 7, Fig. 20)
# ----------------------------------------------------------------------------
def permute_plan(topk_idx, E):
    """counts[e] = #{(t,i): topk_idx[t,i] == e}; offsets = exclusive prefix sum
    (offsets[E] = T*k); row_id_map[t,i] = the row of (t,i) when all (t,i) pairs
    are sorted by the key (expert, token). Reading: dropless (no capacity), and
    within one expert the rows follow ascending token index."""
    idx = np.asarray(topk_idx, np.int64)
    T, k = idx.shape
    counts = np.bincount(idx.ravel(), minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    tok = np.repeat(np.arange(T), k)
    order = np.lexsort((tok, idx.ravel()))           # primary key e, then t
    row = np.empty(T * k, np.int64)
    row[order] = np.arange(T * k)
    return counts, offsets, row.reshape(T, k)


def permute_rows(x, row_id_map):
    """x_perm[row_id_map[t,i]] = x[t]."""
    T, k = row_id_map.shape
    out = np.empty((T * k, x.shape[1]), dtype=x.dtype)
    for i in range(k):
        out[row_id_map[:, i]] = x
    return out


# ----------------------------------------------------------------------------
# Experts: SwiGLU FFN, E(x) = (SiLU(x W1) * (x W3)) W2
# (captions page Table 4; summary page "System Modules" Experts)
# ----------------------------------------------------------------------------
def silu(z):
    """SiLU(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def silu_grad(z):
    """d/dz SiLU(z) = s(z) * (1 + z * (1 - s(z))), s the logistic function."""
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def swiglu_expert(xr, W1e, W3e, W2e, prec=CONTRACT):
    """One expert on the rows xr [n,H]: h1 = xr W1e, h3 = xr W3e (W1e, W3e
    [H,F]; W1 is the gate), a = SiLU(h1) * h3 stored per ``prec.a``, out = a W2e
    (W2e [F,H]) stored per ``prec.y_perm``. No biases (reading of the SwiGLU
    variant)."""
    h1 = xr @ W1e
    h3 = xr @ W3e
    a = prec.r("a", silu(h1) * h3)
    out = a @ W2e
    return h1, h3, a, out


def _weights_getter(W1, W3, W2):
    if callable(W1):
        return W1
    return lambda e: (np.asarray(W1[e], np.float64), np.asarray(W3[e], np.float64),
                      np.asarray(W2[e], np.float64))


def grouped_swiglu(x_perm, offsets, W1, W3, W2, prec=CONTRACT, experts=None):
    """Grouped GEMM over the experts: rows offsets[e]..offsets[e+1] of x_perm go
    through expert e. W1/W3 are [E,H,F], W2 is [E,F,H] (or pass a callable
    e -> (W1e, W3e, W2e)). Returns (h13 [R,2F] rounded per prec.h13, a [R,F],
    y_perm [R,H] rounded per prec.y_perm), only for ``experts`` if given (other
    rows stay NaN)."""
    get = _weights_getter(W1, W3, W2)
    R, H = x_perm.shape
    W1e0, _, _ = get(0) if (experts is None or len(experts) == 0 or 0 in experts) else get(experts[0])
    F = W1e0.shape[1]
    h13 = np.full((R, 2 * F), np.nan)
    a = np.full((R, F), np.nan)
    y = np.full((R, H), np.nan)
    E = len(offsets) - 1
    for e in (range(E) if experts is None else experts):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        W1e, W3e, W2e = get(e)
        h1, h3, ae, out = swiglu_expert(x_perm[lo:hi], W1e, W3e, W2e, prec)
        h13[lo:hi, :F] = prec.r("h13", h1)
        h13[lo:hi, F:] = prec.r("h13", h3)
        a[lo:hi] = ae
        y[lo:hi] = prec.r("y_perm", out)
    return h13, a, y


# ----------------------------------------------------------------------------
# Combine: y[t] = sum_i g[t,i] * E_{e_i}(x[t]) (+ S(x[t]))
# (summary page "Problem Definition" and "System Modules" Combiner;
#  captions page Fig. 40 for the ungated shared expert)
# ----------------------------------------------------------------------------
def combine(y_perm, row_id_map, topk_gate, shared=None):
    """Weighted gather-sum in slot order i = 0..k-1, in fp64."""
    T, k = row_id_map.shape
    y = np.zeros((T, y_perm.shape[1]))
    if shared is not None:
        y = y + shared
    for i in range(k):
        y = y + topk_gate[:, i:i + 1] * y_perm[row_id_map[:, i]]
    return y


def layer_fwd(x, w_r, W1, W3, W2, k, score="softmax", expert_bias=None,
              logit_bias=None, n_groups=1, topk_groups=1, gate_scale=1.0,
              Ws=None, prec=CONTRACT, tokens=None, force_balanced=False):
    """Forward of the whole layer.

    ``tokens`` (optional) restricts the expert and combine stages to a token
    subset (routing is still computed for every token, since counts and offsets
    depend on all of them); y rows of other tokens are NaN. ``Ws`` is the
    optional shared expert (Ws1 [H,Fs], Ws3 [H,Fs], Ws2 [Fs,H]), added ungated.
    """
    x = np.asarray(x, np.float64)
    T, H = x.shape
    rt = route(x, w_r, k, score, expert_bias, logit_bias, n_groups, topk_groups, gate_scale, force_balanced)
    E = np.asarray(w_r).shape[0]
    counts, offsets, row = permute_plan(rt["topk_idx"], E)
    get = _weights_getter(W1, W3, W2)
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    y = np.full((T, H), np.nan)
    yp = {}  # (t, i) -> expert output row for the requested tokens
    idx = rt["topk_idx"]
    for e in range(E):
        sel_t, sel_i = np.nonzero(idx[tok] == e)
        if len(sel_t) == 0:
            continue
        t_e = tok[sel_t]
        W1e, W3e, W2e = get(e)
        _, _, _, out = swiglu_expert(x[t_e], W1e, W3e, W2e, prec)
        out = prec.r("y_perm", out)
        for j in range(len(t_e)):
            yp[(int(t_e[j]), int(sel_i[j]))] = out[j]
    shared = None
    if Ws is not None:
        Ws1, Ws3, Ws2 = (np.asarray(w, np.float64) for w in Ws)
        _, _, _, shared = swiglu_expert(x[tok], Ws1, Ws3, Ws2, prec)
        shared = prec.r("shared", shared)
    acc = np.zeros((len(tok), H)) if shared is None else shared.copy()
    for i in range(k):
        rows = np.stack([yp[(int(t), i)] for t in tok]) if len(tok) else np.zeros((0, H))
        acc = acc + rt["topk_gate"][tok, i:i + 1] * rows
    y[tok] = prec.r("y", acc)
    return {**rt, "counts": counts, "offsets": offsets, "row_id_map": row,
            "y": y, "y_perm_rows": yp, "shared": shared}


# ----------------------------------------------------------------------------
# Load-balancing auxiliary loss (captions page Fig. 2 "load balancing" and
# Fig. 39). Reading: the Switch/GShard form
#   L_aux = alpha * E * sum_e f_e * P_e,  f_e = c_e / (T k),  P_e = mean_t p[t,e]
# with p the full softmax; f is piecewise constant (no gradient).
# ----------------------------------------------------------------------------
def aux_loss(p, counts, k, alpha):
    T, E = p.shape
    f = np.asarray(counts, np.float64) / (T * k)
    P = p.mean(axis=0)
    return alpha * E * float(np.sum(f * P))


# ----------------------------------------------------------------------------
# Backward: the analytic chain rule of the forward (top-k selection and the
# counts are piecewise constant, so they carry no gradient). The loss is
# <dO, y> + L_aux.
# ----------------------------------------------------------------------------
def router_backward(logits, topk_idx, topk_gate, dgate, score="softmax",
                    gate_scale=1.0, counts=None, k=None, aux_coeff=0.0, T_total=None):
    """dL [T,E] from the gate gradients dgate [T,k] (and the aux loss).

    softmax: g_i = c * q_i with q = softmax over the selected logits (equal to
    the renormalised full softmax), so dL_j = c q_j (dg_j - sum_i q_i dg_i) on
    selected experts and 0 elsewhere.
    sigmoid: g_i = c s_i / S, S = sum over the selected s, so
    ds_j = (c / S)(dg_j - sum_i dg_i s_i / S) and dL_j = ds_j s_j (1 - s_j).
    aux (softmax only): dp[t,e] = alpha E f_e / T, pushed through the full
    softmax: dL += p * (dp - <p, dp>). ``T_total`` is the layer's token count
    when ``logits`` holds only a subset of the tokens (default: all rows)."""
    T, E = logits.shape
    Tt = T if T_total is None else T_total
    dL = np.zeros((T, E))
    if score == "softmax":
        q = topk_gate / gate_scale
        inner = np.sum(q * dgate, axis=1, keepdims=True)
        np.put_along_axis(dL, topk_idx, gate_scale * q * (dgate - inner), axis=1)
        if aux_coeff:
            p = softmax(logits)
            f = np.asarray(counts, np.float64) / (Tt * k)
            dp = np.broadcast_to(aux_coeff * E * f / Tt, (T, E))
            dL = dL + p * (dp - np.sum(p * dp, axis=1, keepdims=True))
    else:
        s_all = sigmoid(logits)
        s = np.take_along_axis(s_all, topk_idx, axis=1)
        S = s.sum(axis=1, keepdims=True)
        ds = (gate_scale / S) * (dgate - np.sum(dgate * s, axis=1, keepdims=True) / S)
        np.put_along_axis(dL, topk_idx, ds * s * (1.0 - s), axis=1)
    return dL


def expert_backward(xr, h1, h3, a, dyr, W1e, W3e, W2e, prec=CONTRACT):
    """Backward of one SwiGLU expert over rows xr with output gradient dyr
    (already gate-weighted and stored per prec.dy_perm). h1, h3 are the saved
    pre-activations (stored per prec.h13), a the stored activation.
    Returns dx rows (stored per prec.dx_perm), dW1e, dW3e, dW2e."""
    da = dyr @ W2e.T
    dW2 = a.T @ dyr
    dh1 = prec.r("dh13", da * h3 * silu_grad(h1))
    dh3 = prec.r("dh13", da * silu(h1))
    dx = prec.r("dx_perm", dh1 @ W1e.T + dh3 @ W3e.T)
    return dx, xr.T @ dh1, xr.T @ dh3, dW2


def layer_bwd(x, w_r, W1, W3, W2, dO, k, score="softmax", expert_bias=None,
              logit_bias=None, n_groups=1, topk_groups=1, gate_scale=1.0,
              aux_coeff=0.0, Ws=None, prec=CONTRACT, experts=None, tokens=None,
              force_balanced=False, recompute=False):
    """Forward and backward of the layer for the loss <dO, y> + L_aux.

    ``recompute`` is the memory-saving variant (captions page, Fig. 7 and
    Table 4 "SwiGLU recompute"): the forward keeps neither a nor y_perm; the
    backward recomputes a = SiLU(h1) h3 from the stored pre-activations (and
    stores it per prec.a) and takes the gate gradient from the dgrad of the
    down projection, dg = <da, a> / g with da = dy W2^T and dy = g dO, which
    equals <dO, y_perm> in exact arithmetic (0 where g = 0, whose dg carries
    no weight in the router backward).

    Returns a dict with the forward results plus dx [T,H], dW_r [E,H],
    dW1/dW3 [E,H,F], dW2 [E,F,H], aux_loss (and dWs1/dWs3/dWs2 with a shared
    expert). ``experts`` restricts dW1/dW3/dW2 to those experts and ``tokens``
    restricts dx to those tokens (dW_r then needs every token and is only
    returned when ``tokens`` is None)."""
    x = np.asarray(x, np.float64)
    dO = np.asarray(dO, np.float64)
    T, H = x.shape
    w_r = np.asarray(w_r, np.float64)
    E = w_r.shape[0]
    rt = route(x, w_r, k, score, expert_bias, logit_bias, n_groups, topk_groups, gate_scale, force_balanced)
    idx, gate = rt["topk_idx"], rt["topk_gate"]
    counts, offsets, row = permute_plan(idx, E)
    get = _weights_getter(W1, W3, W2)
    need_tok = np.zeros(T, bool)
    if tokens is None:
        need_tok[:] = True
    else:
        need_tok[np.asarray(tokens)] = True
    exp_set = set(range(E)) if experts is None else set(int(e) for e in experts)
    dgate = np.full((T, k), np.nan)
    dx = np.zeros((T, H))
    W1e0 = get(int(idx[0, 0]))[0]
    F = W1e0.shape[1]
    dW1 = {e: np.zeros((H, F)) for e in exp_set}
    dW3 = {e: np.zeros((H, F)) for e in exp_set}
    dW2 = {e: np.zeros((F, H)) for e in exp_set}
    for e in range(E):
        tt, ii = np.nonzero(idx == e)                 # rows of expert e, ascending t
        if len(tt) == 0:
            continue
        want = need_tok[tt] if e not in exp_set else np.ones(len(tt), bool)
        if not want.any():
            continue
        tt, ii = tt[want], ii[want]
        W1e, W3e, W2e = get(e)
        h1, h3, a, out = swiglu_expert(x[tt], W1e, W3e, W2e, prec)
        out = prec.r("y_perm", out)
        h1s, h3s = prec.r("h13", h1), prec.r("h13", h3)
        gsel = gate[tt, ii]
        dyr = prec.r("dy_perm", gsel[:, None] * dO[tt])
        if recompute:
            a = prec.r("a", silu(h1s) * h3s)
            dot = np.sum((dyr @ W2e.T) * a, axis=1)
            dgate[tt, ii] = np.where(gsel != 0, dot / np.where(gsel != 0, gsel, 1.0), 0.0)
        else:
            dgate[tt, ii] = np.sum(dO[tt] * out, axis=1)
        dxr, g1, g3, g2 = expert_backward(x[tt], h1s, h3s, a, dyr, W1e, W3e, W2e, prec)
        np.add.at(dx, tt, dxr)
        if e in exp_set:
            dW1[e] += g1
            dW3[e] += g3
            dW2[e] += g2
    res = {**rt, "counts": counts, "offsets": offsets, "row_id_map": row,
           "dgate": dgate, "dW1": dW1, "dW3": dW3, "dW2": dW2}
    if Ws is not None:
        Ws1, Ws3, Ws2 = (np.asarray(w, np.float64) for w in Ws)
        h1, h3, a, _ = swiglu_expert(x, Ws1, Ws3, Ws2, prec)
        dxs, g1, g3, g2 = expert_backward(x, prec.r("h13", h1), prec.r("h13", h3), a,
                                          prec.r("dy_perm", dO), Ws1, Ws3, Ws2, prec)
        dx += dxs
        res.update(dWs1=g1, dWs3=g3, dWs2=g2)
    tok_full = tokens is None
    rows_ok = need_tok
    lg = rt["logits"][rows_ok]
    aux = aux_coeff if score == "softmax" else 0.0
    dL = router_backward(lg, idx[rows_ok], gate[rows_ok], dgate[rows_ok], score,
                         gate_scale, counts, k, aux, T_total=T)
    if aux:
        res["aux_loss"] = aux_loss(softmax(rt["logits"]), counts, k, aux)
    dx[rows_ok] += dL @ w_r
    res["dlogits"] = dL
    res["dx"] = np.where(rows_ok[:, None], prec.r("dx", dx), np.nan)
    if tok_full:
        res["dW_r"] = dL.T @ x
    return res
