"""Pins of the heavy-hitter selection oracle (oracle/select.py)."""
import numpy as np
import pytest

from oracle import select


def test_scores_sum_to_rows_times_group():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((5, 6, 8))
    k = rng.standard_normal((40, 2, 8))
    s = select.scores(q, k)
    np.testing.assert_allclose(s.sum(axis=1), [3 * 5, 3 * 5], rtol=1e-12)
    assert (s >= 0).all()


def test_uniform_queries_closed_form():
    # q = 0: every row spreads its mass evenly over keys 0..pos, so
    # score_j = group * sum over observation positions pos >= j of 1 / (pos + 1)
    n, n_obs, g = 30, 7, 2
    q = np.zeros((n_obs, g, 4))
    k = np.random.default_rng(1).standard_normal((n, 1, 4))
    s = select.scores(q, k)[0]
    pos = np.arange(n - n_obs, n)
    want = np.array([g * sum(1.0 / (p + 1) for p in pos if p >= j) for j in range(n)])
    np.testing.assert_allclose(s, want, rtol=1e-12)


def test_dominant_key_collects_its_rows():
    # one key aligned with every query and 50 units longer: it takes almost all
    # the mass of every row that sees it
    n, n_obs, d = 20, 6, 4
    q = np.zeros((n_obs, 1, d)); q[:, 0, 0] = 1.0
    k = np.zeros((n, 1, d)); k[:, 0, 1] = 1.0
    k[9, 0, 0] = 100.0
    s = select.scores(q, k)[0]
    assert s[9] == pytest.approx(n_obs, rel=1e-9)


def test_rule_ties_window_and_edges():
    sc = [0.5, 0.9, 0.5, 0.9, 0.1, 0.7]
    assert select.select(sc, 6, 2, 0) == [1, 3]
    assert select.select(sc, 6, 3, 0) == [1, 3, 5]
    assert select.select(sc, 6, 4, 0) == [0, 1, 3, 5]         # tie 0.5: lower index first
    assert select.select(sc, 6, 2, 2) == [1, 3, 4, 5]         # candidates 0..3, window 4, 5
    assert select.select(sc, 6, 10, 1) == [0, 1, 2, 3, 4, 5]  # everything
    assert select.select(sc, 6, 0, 0) == []
    assert select.select(sc, 6, 3, 9) == [0, 1, 2, 3, 4, 5]   # window longer than n
