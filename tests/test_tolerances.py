"""The comparison helpers themselves (CPU): the low-rank allowance for flipped
low-precision codes admits what one or two flipped codes do to a weight
gradient (rank-one changes x_r^T d_r beyond the bf16 bound) and nothing that a
wrong GEMM does (a dropped term, a transposed block, noise on every entry)."""
import numpy as np
import pytest

from tests._util import assert_close_but_flips, wgrad_atol


def _grad(seed, rows=512, H=256, F=192):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (rows, H))
    d = rng.normal(0, 0.05, (rows, F))
    return x, d, x.T @ d


def _flip(x, rows, F, scale, seed):
    """The change of x^T d when the listed rows of d move (a flipped code of a
    routed row moves that row of d along one direction): sum_r x_r^T v_r."""
    rng = np.random.default_rng(seed)
    out = np.zeros((x.shape[1], F))
    for r in rows:
        v = 0.1 * rng.normal(0, 1, F)
        v[rng.integers(F)] = 1.0  # mostly along one column, as a code step on one element
        out += np.outer(x[r], scale * v / np.abs(v).max())
    return out


def test_one_and_two_flipped_rows_are_admitted():
    x, d, want = _grad(1)
    atol = wgrad_atol(want)
    rows = np.argsort(-np.abs(x).max(axis=1))[:2]  # flips where x is large
    got = want + _flip(x, rows, want.shape[1], 1.5 * atol / np.abs(x[rows]).max(), 5)
    assert np.abs(got - want).max() > atol  # beyond the bf16 bound
    _, flips = assert_close_but_flips("dW", got, want, atol)
    assert flips == 1


def test_three_flips_need_rank_three():
    x, d, want = _grad(2)
    atol = wgrad_atol(want)
    rows = np.argsort(-np.abs(x).max(axis=1))[:3]
    got = want + _flip(x, rows, want.shape[1], 1.5 * atol / np.abs(x[rows]).max(), 6)
    with pytest.raises(AssertionError):
        assert_close_but_flips("dW", got, want, atol, rank=2)
    assert_close_but_flips("dW", got, want, atol, rank=3)


@pytest.mark.parametrize("mistake", ["dropped_rows", "transposed_block", "noise"])
def test_gemm_errors_are_not_admitted(mistake):
    x, d, want = _grad(3)
    atol = wgrad_atol(want)
    if mistake == "dropped_rows":      # a k block of the contraction left out
        got = x[64:].T @ d[64:]
    elif mistake == "transposed_block":  # one 64 x 64 output block written transposed
        got = want.copy()
        got[:64, :64] = want[:64, :64].T
    else:                               # every entry off by a little more than the bf16 bound
        got = want + np.random.default_rng(4).normal(0, 2 * atol, want.shape)
    with pytest.raises(AssertionError):
        assert_close_but_flips("dW", got, want, atol, rank=4)
