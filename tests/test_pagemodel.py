"""Pins for the oracle's page-table model (no GPU)."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import pagemodel as pm

G, L, R = 0, 1, 2
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_block_table_17_tokens():
    with open(os.path.join(GOLDEN, "block_table_17_tokens.json")) as f:
        gd = json.load(f)
    P, n = gd["page_size"], gd["tokens"]
    assert pm.pages_needed(G, 0, 0, None, n, P) == gd["expect_pages"]
    table = pm.stored_positions(G, 0, 0, None, n, P)
    assert [p[0] for p in table] == gd["expect_page_first_token"]
    assert [sum(x >= 0 for x in p) for p in table] == gd["expect_page_filled_slots"]


@pytest.mark.parametrize("n", [1, 15, 16, 17, 255, 256, 257, 4096])
def test_global_pages_closed_form(n):
    P = 16
    assert pm.pages_needed(G, 0, 0, None, n, P) == -(-n // P)
    tab = pm.stored_positions(G, 0, 0, None, n, P)
    flat = [x for p in tab for x in p if x >= 0]
    assert flat == list(range(n))


def test_local_page_count_independent_of_context():
    """A local head's storage does not grow with the context (runtime article
    section 3): sink pages + R ring pages once the ring is full."""
    for (s, w, P) in [(4, 32, 16), (4, 1024, 64), (4, 2048, 64), (4, 8192, 64), (0, 5, 4),
                      (5, 3, 4), (17, 64, 16)]:
        Rg = -(-w // P) + 1
        full = -(-s // P) + Rg
        counts = {pm.pages_needed(L, s, w, None, n, P) for n in (256, 1024, 4096, 65536)
                  if n >= s + (Rg - 1) * P + 1}
        assert counts == {full}
        # grows monotonically up to that count
        prev = 0
        for n in range(0, s + Rg * P + 3 * P):
            c = pm.pages_needed(L, s, w, None, n, P)
            assert prev <= c <= full
            prev = c


def test_pages_workload_totals():
    """Page totals of the pages-shaped workloads."""
    # tiny: P 16, G 16 pages at n=256, 17 after 4 decodes; LOCAL(4, 32) 1 + 3
    assert pm.pages_needed(G, 0, 0, None, 256, 16) == 16
    assert pm.pages_needed(G, 0, 0, None, 260, 16) == 17
    assert pm.pages_needed(L, 4, 32, None, 260, 16) == 4
    # Mistral-shaped: 1 G (128) + 7 LOCAL(4, 1024) (1 + 17) = 254
    assert 128 + 7 * pm.pages_needed(L, 4, 1024, None, 8192, 64) == 254
    # Llama-3-8B-shaped decode: 32 seqs x (32 G x 513 + 224 L x 34) at n = 32768 + 64
    n = 32768 + 64
    assert 32 * (32 * pm.pages_needed(G, 0, 0, None, n, 64)
                 + 224 * pm.pages_needed(L, 4, 2048, None, n, 64)) == 769_024
    # Llama-3.3-70B-shaped: 77 G x 2048 + 435 L(4, 8192) x 130
    assert (77 * pm.pages_needed(G, 0, 0, None, 131072, 64)
            + 435 * pm.pages_needed(L, 4, 8192, None, 131072, 64)) == 214_246


def _brute_local_store(s, w, n, P):
    """What a LOCAL head must keep: every token t < s, plus the newest
    min(n - s, R*P) tokens t >= s; returns {position}."""
    Rg = -(-w // P) + 1
    keep = {t for t in range(min(n, s))}
    keep |= {t for t in range(max(s, n - Rg * P), n)}
    return keep


@pytest.mark.parametrize("s,w,P", [(4, 32, 16), (0, 1, 4), (5, 3, 4), (4, 16, 16), (9, 40, 8)])
def test_local_storage_holds_exactly_the_ring(s, w, P):
    for n in range(0, s + 5 * w + 40):
        tab = pm.stored_positions(L, s, w, None, n, P)
        flat = [x for p in tab for x in p if x >= 0]
        assert sorted(flat) == sorted(_brute_local_store(s, w, n, P))
        assert len(set(flat)) == len(flat)
        # storage suffices: every token a later query (i >= n-1) can see is kept
        for i in range(max(0, n - 1), n + 3):
            need = {j for j in oracle.visible(L, s, w, None, i) if j < n}
            assert need <= set(flat)


def test_retrieval_storage():
    rng = np.random.default_rng(1)
    for P in (4, 16):
        idx = sorted(rng.choice(500, 77, replace=False).tolist())
        for n in (0, 1, 100, 321, 500):
            tab = pm.stored_positions(R, 0, 0, idx, n, P)
            flat = [x for p in tab for x in p if x >= 0]
            assert flat == [t for t in idx if t < n]
            assert len(tab) == -(-len(flat) // P)


def test_allocator_is_injective_and_deterministic():
    model = pm.CacheModel(layers=2, hkv=3, page=4, num_pages=200)
    pol = [[(G, 0, 0, None), (L, 2, 5, None), (R, 0, 0, [1, 3, 8, 20, 21])]] * 2
    model.set_policy(0, pol)
    model.set_policy(1, pol)
    model.append(0, [1, 0], [9, 30])
    model.append(1, [0], [30])
    model.append(0, [0, 1], [3, 1])
    ids = []
    for seq in (0, 1):
        for layer in (0, 1):
            for h in range(3):
                pages, pos = model.table(seq, layer, h)
                ids.extend(pages)
    assert len(ids) == len(set(ids))
    assert 200 - model.pool.free == len(ids)
    # first call: seq 1 then seq 0, KV heads in order, pages popped 0, 1, 2, ...
    assert model.table(1, 0, 0)[0][:3] == [0, 1, 2]
    # releasing and re-allocating the same demand hands back the same ids
    released = sum((model.table(1, 0, h)[0] for h in range(3)), [])
    assert len(released) == 7           # G 3 + LOCAL(2, 5) 1 + 2 + RETRIEVAL 1
    model.release(1)
    model.set_policy(1, pol)
    model.append(0, [1], [10])          # the same demand: 3 + 3 + 1 pages
    after = sum((model.table(1, 0, h)[0] for h in range(3)), [])
    # the stack hands the released pages back, last pushed first
    assert after == released[::-1]


def test_allocator_out_of_pages():
    model = pm.CacheModel(layers=1, hkv=1, page=4, num_pages=3)
    model.set_policy(0, [[(G, 0, 0, None)]])
    model.append(0, [0], [12])
    with pytest.raises(pm.OutOfPages):
        model.append(0, [0], [1])
    assert model.n[(0, 0)] == 12
