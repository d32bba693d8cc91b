"""Blockwise (m, l, u) recurrence and split combine equal the full softmax
on brute-forced tiny inputs (exact in real arithmetic; 1e-12 in fp64)."""
import numpy as np
import pytest

from oracle import recurrence as R


def _cases():
    rng = np.random.default_rng(0)
    for trial in range(200):
        n = int(rng.integers(1, 65))
        d = int(rng.integers(1, 9))
        s = rng.normal(size=n) * rng.choice([0.1, 1.0, 5.0, 40.0])
        if trial % 5 == 0 and n > 2:  # masked (-inf) entries, never the whole row
            k = rng.integers(1, n)
            s[rng.choice(n, size=k, replace=False)] = -np.inf
            s[rng.integers(0, n)] = rng.normal()
        V = rng.normal(size=(n, d))
        k = int(rng.integers(0, n))
        cuts = sorted(rng.choice(np.arange(1, n + 1), size=k, replace=True).tolist())
        yield s, V, cuts


@pytest.mark.parametrize("form", [R.deferred, R.normalised])
def test_blockwise_equals_full(form):
    for s, V, cuts in _cases():
        o_ref, lse_ref = R.full_softmax_row(s, V)
        o, lse = form(s, V, cuts)
        assert np.abs(o - o_ref).max() < 1e-12
        assert abs(lse - lse_ref) < 1e-12 * max(1.0, abs(lse_ref))


def test_split_combine_equals_full():
    rng = np.random.default_rng(1)
    for s, V, cuts in _cases():
        edges = [0] + cuts + [len(s)]
        order = rng.permutation(len(edges) - 1)  # combine order does not matter
        states = [R.partial_state(s[edges[i]:edges[i + 1]], V[edges[i]:edges[i + 1]])
                  for i in order]
        o, lse = R.combine(states)
        o_ref, lse_ref = R.full_softmax_row(s, V)
        assert np.abs(o - o_ref).max() < 1e-12
        assert abs(lse - lse_ref) < 1e-12 * max(1.0, abs(lse_ref))


def test_single_block_is_plain_softmax():
    rng = np.random.default_rng(2)
    s = rng.normal(size=17)
    V = rng.normal(size=(17, 3))
    assert np.abs(R.deferred(s, V, [])[0] - R.full_softmax_row(s, V)[0]).max() < 1e-15
