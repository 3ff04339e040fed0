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
"""
from __future__ import annotations

from typing import List

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
