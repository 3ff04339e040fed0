"""Work accounting for the head-aware attention path.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

  * visible pairs of a prefill: sum over query heads and query rows of
    |V(i)| -- the pairs the mask-free kernel must touch (runtime article
    section 4: every (query head, KV head) pair attends over exactly its own
    visible tokens); FLOP = 4 d per pair (QK^T and PV, 2 d each).
  * visible KV bytes of a decode step: sum over units of |V(t)| * 2 * d *
    bytes_per_element (K and V rows), the per-head form of the KV-cache
    tutorial's size formula 2 x L x H_kv x D_head x T x bytes (section 3.2).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import visible

GLOBAL, LOCAL, RETRIEVAL = 0, 1, 2


def vis_count(kind: int, sink: int, window: int, idx: Optional[Sequence[int]],
              i: int) -> int:
    """|V(i)| by materialising V(i)."""
    return int(visible(kind, sink, window, idx, i).size)


def vis_count_closed(kind: int, sink: int, window: int,
                     idx: Optional[Sequence[int]], i: np.ndarray) -> np.ndarray:
    """|V(i)| in closed form, vectorised over positions i (int64 array)."""
    i = np.asarray(i, dtype=np.int64)
    if kind == GLOBAL:
        return i + 1
    if kind == LOCAL:
        return np.minimum(i + 1, sink + window)
    if kind == RETRIEVAL:
        arr = np.asarray([] if idx is None else list(idx), dtype=np.int64)
        return np.searchsorted(arr, i, side="right").astype(np.int64)
    raise ValueError("unknown head class")


def prefill_pairs(policies, hq: int, n0: int, c: int) -> int:
    """Visible (query, key) pairs of a prefill of rows n0 .. n0+c-1 for one
    sequence and layer; policies: per KV head (kind, sink, window, idx)."""
    hkv = len(policies)
    group = hq // hkv
    rows = np.arange(n0, n0 + c, dtype=np.int64)
    total = 0
    for (kind, sink, window, idx) in policies:
        total += group * int(vis_count_closed(kind, sink, window, idx, rows).sum())
    return total


def decode_kv_bytes(policies, t: int, d: int, elem_bytes: int = 2) -> int:
    """Visible K+V bytes one decode query at position t reads, per layer."""
    total = 0
    for (kind, sink, window, idx) in policies:
        total += int(vis_count_closed(kind, sink, window, idx, np.array([t]))[0])
    return total * 2 * d * elem_bytes


def dense_kv_bytes(layers: int, hkv: int, d: int, tokens: int, elem_bytes: int) -> int:
    """2 x L x H_kv x D_head x T x bytes (KV-cache tutorial section 3.2)."""
    return 2 * layers * hkv * d * tokens * elem_bytes
