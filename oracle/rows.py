"""Row-sampled form of the attention oracle, for sequences too long for the
C oracle's scalar loops (the 131,072-token prefill, checked on sampled rows).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU baseline may use it; the product never does.

It computes the same definition as ``segpaged_oracle.c`` (RedKnot
SegPagedAttention runtime article, section 4: the fused kernel equals dense
attention under a head-wise mask; section 2 for the head classes): for every
query head h of KV head h // (Hq / Hkv) (KV-cache tutorial section 5.3,
0-indexed) and every requested row at absolute position i,

    O_i = sum_{j in V(i)} softmax_j(q_i . k_j / sqrt(d)) v_j,
    LSE_i = log sum_{j in V(i)} exp(q_i . k_j / sqrt(d)),

with V(i) the class's visibility set, written here as the position ranges
it is made of:
    GLOBAL          [0, i]
    LOCAL(s, W)     [0, min(s, i+1)) and [max(min(s, i+1), i-W+1), i]
                    (sink tokens, then the W most recent, query included,
                    with no position counted twice)
    RETRIEVAL(I)    the listed positions j <= i
An empty V(i) gives O_i = 0 and LSE_i = -inf.

Arithmetic, per (row, KV head): gather the visible keys and values, scores of
the head's query group by one matrix product, the maximum, exp(score - max),
their sum, the weighted sum of values by one matrix product, one division
(torch on the CPU, float64 by default).  No blocking across rows and no
online rescaling: the same two passes as the C oracle, with library matrix
products as steps.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np
import torch

GLOBAL, LOCAL, RETRIEVAL = 0, 1, 2


def visible_ranges(kind: int, sink: int, window: int, i: int) -> List[Tuple[int, int]]:
    """V(i) of a GLOBAL or LOCAL head as half-open position ranges, ascending
    and disjoint (runtime article section 2)."""
    if i < 0:
        return []
    if kind == GLOBAL:
        return [(0, i + 1)]
    if kind == LOCAL:
        a = min(sink, i + 1)
        b = max(a, i - window + 1)
        return [r for r in ((0, a), (b, i + 1)) if r[1] > r[0]]
    raise ValueError("visible_ranges: GLOBAL or LOCAL only")


def attend_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, row_pos: Sequence[int],
                policies, dtype: torch.dtype = torch.float64):
    """O [rows, Hq, d], LSE [rows, Hq] for queries q [rows, Hq, d] at absolute
    positions row_pos, over keys / values k, v [n_keys, Hkv, d] of positions
    0 .. n_keys-1.  policies: per KV head (kind, sink, window, idx|None)."""
    n_rows, hq, d = q.shape
    n_keys, hkv, d2 = k.shape
    assert d2 == d and v.shape == k.shape and hq % hkv == 0 and len(policies) == hkv
    rows = [int(i) for i in row_pos]
    assert len(rows) == n_rows
    if rows and max(rows) >= n_keys:
        raise ValueError("attend_rows: a row's position lies past the given keys")
    g = hq // hkv
    scale = 1.0 / math.sqrt(d)
    qt = torch.from_numpy(np.ascontiguousarray(q)).to(dtype)
    o = torch.zeros(n_rows, hq, d, dtype=dtype)
    lse = torch.full((n_rows, hq), -math.inf, dtype=dtype)
    for h, (kind, sink, window, idx) in enumerate(policies):
        kh = torch.from_numpy(np.ascontiguousarray(k[:, h])).to(dtype)
        vh = torch.from_numpy(np.ascontiguousarray(v[:, h])).to(dtype)
        ind = None
        if kind == RETRIEVAL:
            ind = torch.as_tensor(np.asarray([] if idx is None else list(idx), dtype=np.int64))
        elif kind not in (GLOBAL, LOCAL):
            raise ValueError("attend_rows: unknown head class")
        heads = slice(h * g, (h + 1) * g)
        for r, i in enumerate(rows):
            if kind == RETRIEVAL:
                sel = ind[ind <= i]
                if sel.numel() == 0:
                    continue
                kk, vv = kh.index_select(0, sel), vh.index_select(0, sel)
            else:
                rg = visible_ranges(kind, sink, window, i)
                if not rg:
                    continue
                if len(rg) == 1:
                    kk, vv = kh[rg[0][0]:rg[0][1]], vh[rg[0][0]:rg[0][1]]
                else:
                    kk = torch.cat([kh[a:b] for a, b in rg])
                    vv = torch.cat([vh[a:b] for a, b in rg])
            s = (qt[r, heads] @ kk.T) * scale                # [g, |V(i)|]
            m = s.max(dim=1, keepdim=True).values
            p = torch.exp(s - m)
            den = p.sum(dim=1, keepdim=True)
            o[r, heads] = (p @ vv) / den
            lse[r, heads] = (m + torch.log(den))[:, 0]
    return o.numpy(), lse.numpy()
