"""Comparison helpers for the parity tests."""
import numpy as np
import torch

# Floating-point bar of the layer: relative L2 error <= 5e-3 and max-abs error
# <= 2e-2 against the fp64 oracle, for bf16 inputs with fp32 accumulation.
REL_L2 = 5e-3
MAX_ABS = 2e-2
# Selection margin below which a token's top-k is not compared exactly: the
# k-th and (k+1)-th selection scores differ by less than this.
TIE_MARGIN = 1e-6


def f64(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def wgrad_atol(want):
    """Max-abs bound of an fp32 weight gradient. Weight gradients are sums over
    many rows of products with activations the training step stores in bf16
    (dh13, a, dy_perm). Where such an activation's fp32 value lies within the
    fp32-vs-fp64 accumulation difference of a bf16 rounding boundary, the kernel
    and the oracle round it to different neighbours; each such flip moves the
    gradient by one bf16 ulp of the activation times the other operand. The
    bound is the layer's 2e-2 or one bf16 ulp (2^-7 relative) of the gradient's
    largest magnitude, whichever is larger; the relative L2 bound stays 5e-3."""
    return max(MAX_ABS, 2.0 ** -7 * float(np.abs(np.asarray(want, np.float64)).max()))


def mx_wgrad_atol(want, amax_a, amax_b):
    """Max-abs bound of an MXFP8 weight gradient Q(A)^T Q(B) (both operands
    quantised along the tokens). An operand's E4M3 code is decided from a bf16
    value that fp32 and fp64 accumulation can put on either side of a rounding
    boundary (see wgrad_atol); such a flip moves the code by one E4M3 step, at
    most 2^-3 of the block's largest magnitude, and every entry of the
    gradient's row or column through that element by at most the step times
    the other operand's magnitude. The bound admits two flips on one entry:
    2 * 2^-3 * max|A| * max|B|, and never less than the bf16 bound."""
    return max(wgrad_atol(want), 2.0 ** -2 * float(amax_a) * float(amax_b))


def assert_close_but_flips(name, got, ref, atol, rank=2, rel=REL_L2):
    """assert_close for weight gradients whose low-precision operand codes may
    differ in rare places from the oracle's: a code is decided from a bf16
    value that the kernel (fp32) and the oracle (fp64) can round to
    neighbouring values, and a coarse code (E2M1) then moves by a whole step.
    One flipped code of a routed row r changes that row of dh13 (or dy_perm),
    so the gradient sum_r X[r]^T D[r] moves by one outer product: a rank-one
    error. Relative L2 <= rel over everything; per matrix (the last two axes),
    the error left after removing its `rank` largest singular components must
    be within `atol` (the bf16 bound), i.e. up to `rank` flips are admitted."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    r = rel_l2(got, ref)
    assert r <= rel, f"{name}: rel_l2={r:.3e} (<= {rel})"
    err = (got - ref).reshape((-1,) + got.shape[-2:])
    flips = 0
    m_left = 0.0
    for i in range(err.shape[0]):
        e = err[i]
        if np.abs(e).max(initial=0.0) <= atol:
            continue
        u, sv, vt = np.linalg.svd(e, full_matrices=False)
        left = e - (u[:, :rank] * sv[:rank]) @ vt[:rank]
        m_left = max(m_left, float(np.abs(left).max()))
        flips += 1
        assert m_left <= atol, f"{name}[{i}]: max_abs beyond rank {rank}: {m_left:.3e} (<= {atol})"
    return r, flips


def rel_l2(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def assert_close(name, got, ref, rel=REL_L2, atol=MAX_ABS):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    r = rel_l2(got, ref)
    m = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert r <= rel and m <= atol, f"{name}: rel_l2={r:.3e} (<= {rel}), max_abs={m:.3e} (<= {atol})"
    return r, m


def topk_margin(z, k):
    """Gap between the k-th and (k+1)-th largest selection values per token
    (inf when k == E)."""
    zs = -np.sort(-np.where(np.isfinite(z), z, -1e300), axis=1)
    if zs.shape[1] == k:
        return np.full(zs.shape[0], np.inf)
    return zs[:, k - 1] - zs[:, k]


def compare_topk(got_idx, ref_idx, z, k, margin=TIE_MARGIN):
    """Exact comparison of the selected experts on tokens whose selection margin
    is >= `margin`; the slot order is compared where the selected values are
    themselves separated by >= margin. Returns the number of excluded tokens;
    for them only validity (k distinct experts, each within `margin` of the
    selection threshold) is checked."""
    got_idx = np.asarray(got_idx, np.int64)
    ref_idx = np.asarray(ref_idx, np.int64)
    T = got_idx.shape[0]
    mg = topk_margin(z, k)
    excl = mg < margin
    for t in range(T):
        g, r = got_idx[t], ref_idx[t]
        assert len(set(g.tolist())) == k and g.min() >= 0 and g.max() < z.shape[1], f"token {t}: invalid {g}"
        if excl[t]:
            thr = np.sort(z[t])[::-1][k - 1]
            assert np.all(z[t, g] >= thr - margin), f"token {t}: selected value below threshold"
            continue
        assert set(g.tolist()) == set(r.tolist()), f"token {t}: got {g} want {r} (margin {mg[t]:.2e})"
        zr = z[t, r]
        sep = np.all(np.abs(np.diff(zr)) >= margin) if k > 1 else True
        if sep:
            assert np.array_equal(g, r), f"token {t}: slot order {g} want {r}"
    return int(excl.sum())


# Error of CUDA outputs against the fully unrounded fp64 oracle (oracle.EXACT:
# no bf16 rounding of any stored intermediate). Reported for information next
# to the contract comparison (which rounds where the layer stores bf16); never
# asserted. Collected here, printed in pytest's terminal summary.
EXACT_REPORT = []


def report_exact(name, got, exact):
    """Record rel-L2 and max-abs of `got` against the unrounded oracle value."""
    got, exact = np.asarray(got, np.float64), np.asarray(exact, np.float64)
    ok = np.isfinite(exact)
    if not ok.any():
        return
    r = rel_l2(got[ok], exact[ok])
    m = float(np.max(np.abs(got[ok] - exact[ok])))
    EXACT_REPORT.append((name, r, m))
