"""Heavy-hitter retrieval selection -- the plain definition.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The runtime article (section 2) gives retrieval heads "the top-p important
tokens" and (section 5) measures an H2O heavy-hitter decode scenario; H2O
keeps the keys with the largest accumulated attention.  Reading taken here
(the pages fix no more): for KV head h the score of key j is the causal
softmax probability of j, scale 1/sqrt(d), summed over h's query heads and
over the observation rows (the last n_obs prompt rows); the selection is the
topk highest scores among keys below n - recent (ties: lower index first),
united with the recent window, ascending.

The "top-p" form read from the same sentence: among those candidates, in
the order (score descending, index ascending), keep the shortest prefix
whose summed score reaches p times the candidates' total score, at most
max_keys of them (a page budget), then the recent window.  Sums here are
exact (rational arithmetic on the given float values, p included: pass the
float the kernel receives, e.g. a float32 p as np.float32).
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Set, Tuple

import numpy as np


def scores(q_obs: np.ndarray, k: np.ndarray) -> np.ndarray:
    """q_obs [n_obs, Hq, d], k [n, Hkv, d] (any float type) -> [Hkv, n] float64."""
    q = np.asarray(q_obs, dtype=np.float64)
    kk = np.asarray(k, dtype=np.float64)
    n_obs, hq, d = q.shape
    n, hkv, _ = kk.shape
    g = hq // hkv
    out = np.zeros((hkv, n))
    for h in range(hkv):
        for qh in range(h * g, (h + 1) * g):
            for oi in range(n_obs):
                pos = n - n_obs + oi
                logits = kk[: pos + 1, h] @ q[oi, qh] / np.sqrt(d)
                p = np.exp(logits - logits.max())
                out[h, : pos + 1] += p / p.sum()
    return out


def select(score_row, n: int, topk: int, recent: int) -> List[int]:
    """The selection rule on one head's scores (any float type, compared as
    given): topk largest among j < n - recent, ties to the lower j, then the
    recent window; ascending."""
    ncand = max(n - recent, 0)
    kk = min(topk, ncand)
    order = sorted(range(ncand), key=lambda j: (-float(score_row[j]), j))[:kk]
    return sorted(order) + list(range(ncand, ncand + min(recent, n)))


def top_p_count(score_row, n: int, p: float, max_keys: int, recent: int,
                rel: float = 1e-9) -> Tuple[int, Set[int]]:
    """How many candidates the top-p rule keeps for one head, with exact
    sums: the smallest m such that the m highest-ranked candidates (score
    descending, index ascending, j < n - recent) hold at least p times the
    candidates' total score, capped at max_keys (0 when p * total is 0).
    Also returns every count a float64 evaluation of the same comparison may
    give: m - 1 (or m + 1) when the exact prefix mass at m - 1 (or m) lies
    within rel * total of the boundary."""
    ncand = max(n - recent, 0)
    vals = [Fraction(float(score_row[j])) for j in range(ncand)]
    total = sum(vals, Fraction(0))
    target = Fraction(float(p)) * total
    if ncand == 0 or target <= 0:
        return 0, {0}
    order = sorted(range(ncand), key=lambda j: (-float(score_row[j]), j))
    prefix = [Fraction(0)]
    for j in order:
        prefix.append(prefix[-1] + vals[j])
    m = next(i for i in range(ncand + 1) if prefix[i] >= target)
    ok = {m}
    slack = Fraction(rel) * total
    if m > 1 and target - prefix[m - 1] <= slack:
        ok.add(m - 1)
    if m < ncand and prefix[m] - target <= slack:
        ok.add(m + 1)
    return min(m, max_keys), {min(x, max_keys) for x in ok}


def select_top_p(score_row, n: int, p: float, max_keys: int, recent: int) -> List[int]:
    """The top-p selection of one head: the top_p_count highest-ranked
    candidates, then the recent window; ascending."""
    m, _ = top_p_count(score_row, n, p, max_keys, recent)
    return select(score_row, n, m, recent)
