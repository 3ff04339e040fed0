"""Canonical page-table model of the head-aware paged KV cache.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Plain Python, written
token by token so that it can be checked by eye.

Storage per (sequence, layer, KV head) -- a *unit* -- follows the RedKnot
SegPagedAttention runtime article, section 3 ("paged storage"): a three-level
page table (layer, head, segment) -> pages in one physical pool, where a
global head holds pages for its whole context, a local head holds only its
sink pages plus pages for the recent window (so its page count does not grow
with the context), and (summary paragraph) a retrieval head holds pages for
its selected tokens only.  The runtime article leaves the slot layout open;
the readings taken here are:

  * GLOBAL: token t lives in page t // P, slot t % P.
  * LOCAL(s, W): token t < s lives in sink page t // P, slot t % P; a token
    t >= s lives in a ring of R = ceil(W / P) + 1 pages after the
    ceil(s / P) sink pages, at ring slot (t - s) mod (R * P); a newer token
    overwrites the older one in its slot.
  * RETRIEVAL(I): token t is stored only if t is in I, at slot rank(t in I),
    i.e. page rank // P, slot rank % P.
  * Pages are taken from the pool when first needed: a unit holding n tokens
    owns exactly pages_needed(n) pages.

Physical page ids come from one deterministic stack allocator: the free stack
starts as [N-1, ..., 1, 0] (top = 0); one call that needs d_k new pages for
its units k = 0, 1, ... (in call order: sequences in the order given, then KV
heads) gives unit k the entries top-o_k, top-o_k-1, ... where o_k is the
exclusive prefix sum of d; releasing a sequence pushes its pages back in
(layer, KV head, page) order.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

GLOBAL, LOCAL, RETRIEVAL = 0, 1, 2


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def ring_pages(window: int, page: int) -> int:
    """R = ceil(W / P) + 1 ring pages of a LOCAL head."""
    return cdiv(window, page) + 1


def pages_needed(kind: int, sink: int, window: int, idx: Optional[Sequence[int]],
                 n: int, page: int) -> int:
    """Pages a unit owns after its first n tokens were written."""
    if kind == GLOBAL:
        return cdiv(n, page)
    if kind == LOCAL:
        sink_part = cdiv(min(n, sink), page)
        ring_part = min(ring_pages(window, page), cdiv(max(0, n - sink), page))
        return sink_part + ring_part
    if kind == RETRIEVAL:
        return cdiv(sum(1 for t in idx if t < n), page)
    raise ValueError("unknown head class")


def slot_of(kind: int, sink: int, window: int, idx: Optional[Sequence[int]],
            t: int, page: int) -> Optional[Tuple[int, int]]:
    """(page index within the unit, slot) where token t is written, or None."""
    if kind == GLOBAL:
        return t // page, t % page
    if kind == LOCAL:
        if t < sink:
            return t // page, t % page
        ring = ring_pages(window, page) * page
        q = (t - sink) % ring
        return cdiv(sink, page) + q // page, q % page
    if kind == RETRIEVAL:
        for rank, x in enumerate(idx):
            if x == t:
                return rank // page, rank % page
        return None
    raise ValueError("unknown head class")


def stored_positions(kind: int, sink: int, window: int,
                     idx: Optional[Sequence[int]], n: int, page: int) -> List[List[int]]:
    """Position held by every slot of every page after writing tokens 0..n-1
    in order (-1 = empty slot)."""
    npg = pages_needed(kind, sink, window, idx, n, page)
    table = [[-1] * page for _ in range(npg)]
    for t in range(n):
        ps = slot_of(kind, sink, window, idx, t, page)
        if ps is None:
            continue
        p, s = ps
        table[p][s] = t
    return table


class OutOfPages(Exception):
    pass


class PoolModel:
    """The deterministic free-stack allocator described in the module doc."""

    def __init__(self, num_pages: int):
        self.stack = list(range(num_pages - 1, -1, -1))  # stack[-1] is the top

    @property
    def free(self) -> int:
        return len(self.stack)

    def alloc(self, demands: Sequence[int]) -> List[List[int]]:
        total = sum(demands)
        if total > len(self.stack):
            raise OutOfPages
        top = len(self.stack) - 1
        out, off = [], 0
        for d in demands:
            out.append([self.stack[top - (off + j)] for j in range(d)])
            off += d
        del self.stack[len(self.stack) - total:]
        return out

    def release(self, pages_in_order: Sequence[int]) -> None:
        self.stack.extend(pages_in_order)


class CacheModel:
    """Per-unit state: policy, token count and page list, plus the pool."""

    def __init__(self, layers: int, hkv: int, page: int, num_pages: int):
        self.layers, self.hkv, self.page = layers, hkv, page
        self.pool = PoolModel(num_pages)
        self.policy: Dict[int, list] = {}
        self.n: Dict[Tuple[int, int], int] = {}
        self.pages: Dict[Tuple[int, int, int], List[int]] = {}

    def set_policy(self, seq: int, pol) -> None:
        """pol[layer][kvh] = (kind, sink, window, idx)."""
        assert all(self.n.get((seq, l), 0) == 0 for l in range(self.layers))
        self.policy[seq] = [[tuple(p) for p in row] for row in pol]
        for l in range(self.layers):
            self.n[(seq, l)] = 0
            for h in range(self.hkv):
                self.pages[(seq, l, h)] = []

    def append(self, layer: int, seqs: Sequence[int], counts: Sequence[int]) -> None:
        """Write counts[k] new tokens of seqs[k] (positions n .. n+c-1)."""
        demands, keys = [], []
        for seq, c in zip(seqs, counts):
            n = self.n[(seq, layer)]
            for h in range(self.hkv):
                kind, sink, window, idx = self.policy[seq][layer][h]
                d = (pages_needed(kind, sink, window, idx, n + c, self.page)
                     - pages_needed(kind, sink, window, idx, n, self.page))
                demands.append(d)
                keys.append((seq, layer, h))
        got = self.pool.alloc(demands)
        for key, new in zip(keys, got):
            self.pages[key].extend(new)
        for seq, c in zip(seqs, counts):
            self.n[(seq, layer)] += c

    def build(self, seq: int, layer: int, n: int) -> None:
        assert self.n[(seq, layer)] == 0
        self.append(layer, [seq], [n])

    def release(self, seq: int) -> None:
        order = []
        for l in range(self.layers):
            for h in range(self.hkv):
                order.extend(self.pages[(seq, l, h)])
                self.pages[(seq, l, h)] = []
            self.n[(seq, l)] = 0
        self.pool.release(order)

    def table(self, seq: int, layer: int, h: int):
        """(page ids, stored positions per page) of one unit."""
        kind, sink, window, idx = self.policy[seq][layer][h]
        n = self.n[(seq, layer)]
        pos = stored_positions(kind, sink, window, idx, n, self.page)
        ids = list(self.pages[(seq, layer, h)])
        assert len(ids) == len(pos)
        return ids, pos
