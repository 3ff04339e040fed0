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


def _brute_top_p(score_row, n, p, max_keys, recent):
    """Every prefix length tried in turn, masses summed with math.fsum
    (correctly rounded) over exact binary values: the first length whose
    mass reaches p * total."""
    import math
    ncand = max(n - recent, 0)
    order = sorted(range(ncand), key=lambda j: (-float(score_row[j]), j))
    total = math.fsum(float(score_row[j]) for j in range(ncand))
    for m in range(ncand + 1):
        if math.fsum(float(score_row[j]) for j in order[:m]) >= float(p) * total:
            return min(m, max_keys)
    return min(ncand, max_keys)


def test_top_p_closed_forms():
    ones = np.ones(10, np.float32)
    # uniform scores: ceil(p * n) keys, the lowest indices (ties)
    assert select.top_p_count(ones, 10, 0.35, 100, 0)[0] == 4
    assert select.select_top_p(ones, 10, 0.35, 100, 0) == [0, 1, 2, 3]
    assert select.top_p_count(ones, 10, 0.5, 100, 0)[0] == 5
    # p = 1 keeps every key with positive score and no zero-score key
    s = np.array([1, 0, 2, 0, 3], np.float32)
    assert select.select_top_p(s, 5, 1.0, 100, 0) == [0, 2, 4]
    # geometric scores 2^-j: p = 3/4 of the total (2 - 2^-9) needs 3 keys
    g = (2.0 ** -np.arange(10)).astype(np.float32)
    assert select.top_p_count(g, 10, 0.75, 100, 0)[0] == 2   # 1 + 1/2 = 1.5 >= 0.75 * 1.998
    assert select.top_p_count(g, 10, 0.76, 100, 0)[0] == 3
    # the page budget caps the count; the recent window is kept whole
    assert select.top_p_count(ones, 10, 0.9, 3, 0)[0] == 3
    assert select.select_top_p(ones, 12, 0.5, 100, 2) == [0, 1, 2, 3, 4, 10, 11]
    # nothing to keep: no candidates, or no mass
    assert select.top_p_count(ones, 4, 0.5, 100, 4)[0] == 0
    assert select.top_p_count(np.zeros(6, np.float32), 6, 0.5, 100, 0)[0] == 0


def test_top_p_equals_top_k_of_its_count_and_brute_force():
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(1, 300))
        recent = int(rng.integers(0, 20))
        s = rng.exponential(size=n).astype(np.float32)
        if trial % 3 == 0:
            s[rng.integers(0, n, n // 3)] = s[0]            # ties
        p = np.float32(rng.uniform(0.05, 1.0))
        cap = int(rng.integers(1, 400))
        m, ok = select.top_p_count(s, n, p, cap, recent)
        assert _brute_top_p(s, n, p, cap, recent) in ok
        assert select.select_top_p(s, n, p, cap, recent) == select.select(s, n, m, recent)
        # the kept mass reaches the target and one key fewer does not (uncapped)
        m_free, _ = select.top_p_count(s, n, p, 10 ** 9, recent)
        order = sorted(range(max(n - recent, 0)), key=lambda j: (-float(s[j]), j))
        tot = sum(float(s[j]) for j in order)
        assert sum(float(s[j]) for j in order[:m_free]) >= float(p) * tot * (1 - 1e-12)
        if m_free > 0:
            assert sum(float(s[j]) for j in order[:m_free - 1]) < float(p) * tot * (1 + 1e-12)
