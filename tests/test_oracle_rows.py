"""Pins for the row-sampled oracle (oracle/rows.py), no GPU.

It must agree with things other than itself:
  * its visibility ranges, position by position, with the C oracle's
    materialised V(i) (itself pinned by brute force from the class
    descriptions in test_oracle.py);
  * its attention with the C oracle (pinned separately) and with dense
    attention under an explicit head-wise mask (the runtime article's
    section 4 equivalence), on mixed GLOBAL / LOCAL / RETRIEVAL heads, GQA
    groups 1-4, empty rows and rows at the sequence's ends;
  * closed forms: constant values give that constant, q = 0 gives the mean
    of the visible values, LOCAL(0, 1) gives v_i, GLOBAL row 0 gives v_0,
    LSE of q = 0 is log |V(i)|.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import rows as orows
from test_oracle import dense_masked

G, L, R = 0, 1, 2


@pytest.mark.parametrize("kind", [G, L])
def test_ranges_equal_the_materialised_sets(kind):
    for s in (0, 1, 3, 4, 7, 64):
        for w in (1, 2, 5, 16, 100):
            for i in list(range(0, 40)) + [63, 64, 65, 127, 128, 500]:
                got = [p for a, b in orows.visible_ranges(kind, s, w, i) for p in range(a, b)]
                want = oracle.visible(kind, s, w, None, i).tolist()
                assert got == want, (kind, s, w, i)
            if kind == G:
                break


def _case(seed, n, rows, hq, hkv, d):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((len(rows), hq, d))
    k = rng.standard_normal((n, hkv, d)) * 0.7
    v = rng.standard_normal((n, hkv, d))
    pols = []
    for h in range(hkv):
        kind = (h + seed) % 3
        if kind == G:
            pols.append((G, 0, 0, None))
        elif kind == L:
            pols.append((L, int(rng.integers(0, 6)), int(rng.integers(1, n)), None))
        else:
            idx = np.sort(rng.choice(n, size=int(rng.integers(1, n // 3)), replace=False))
            idx[0] = max(idx[0], 3)                      # rows 0..2 see nothing
            pols.append((R, 0, 0, sorted(set(int(x) for x in idx))))
    return q, k, v, pols


@pytest.mark.parametrize("seed,n,hq,hkv,d", [(0, 97, 4, 2, 64), (1, 256, 6, 3, 32),
                                             (2, 300, 8, 2, 128), (3, 130, 3, 3, 16),
                                             (4, 200, 12, 3, 64)])
def test_agrees_with_the_c_oracle_and_dense_mask(seed, n, hq, hkv, d):
    rows = np.unique(np.concatenate([[0, 1, 2, n - 1], np.random.default_rng(seed).integers(0, n, 20)]))
    q, k, v, pols = _case(seed, n, rows, hq, hkv, d)
    o, lse = orows.attend_rows(q, k, v, rows, pols)
    oc, lc = oracle.attend(q, k, v, rows, pols, "f64")
    od, ld = dense_masked(q, k, v, rows, pols)
    for ref, lref in ((oc, lc), (od, ld)):
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-11)
        assert np.array_equal(np.isfinite(lse), np.isfinite(lref))
        fin = np.isfinite(lref)
        np.testing.assert_allclose(lse[fin], lref[fin], rtol=0, atol=1e-11)
    # the retrieval rows before the first index see nothing
    assert (lse[:, [h for h in range(hq) if pols[h // (hq // hkv)][0] == R]][:1] == -np.inf).all()


def test_closed_forms():
    n, d, hkv, hq = 120, 32, 3, 6
    pols = [(G, 0, 0, None), (L, 2, 9, None), (R, 0, 0, [5, 17, 40, 41, 99])]
    rows = np.arange(n)
    rng = np.random.default_rng(9)
    k = rng.standard_normal((n, hkv, d))
    # constant values -> that constant wherever something is visible
    v = np.full((n, hkv, d), 0.375)
    o, lse = orows.attend_rows(rng.standard_normal((n, hq, d)), k, v, rows, pols)
    fin = np.isfinite(lse)
    assert np.all(np.abs(o[fin] - 0.375) <= 1e-14)
    # q = 0 -> mean of the visible values, LSE = log |V(i)|
    v = rng.standard_normal((n, hkv, d))
    o, lse = orows.attend_rows(np.zeros((n, hq, d)), k, v, rows, pols)
    for i in (0, 1, 8, 9, 10, 60, 119):
        for h, p in enumerate(pols):
            vis = oracle.visible(p[0], p[1], p[2], p[3], i)
            for hh in (2 * h, 2 * h + 1):
                if len(vis) == 0:
                    assert lse[i, hh] == -np.inf and not o[i, hh].any()
                    continue
                np.testing.assert_allclose(o[i, hh], v[vis, h].mean(0), atol=1e-13)
                assert abs(lse[i, hh] - math.log(len(vis))) <= 1e-13
    # LOCAL(0, 1) sees only its own position; GLOBAL row 0 sees only key 0
    o, _ = orows.attend_rows(rng.standard_normal((n, 2, d)), k[:, :2], v[:, :2], rows,
                             [(L, 0, 1, None), (G, 0, 0, None)])
    np.testing.assert_array_equal(o[:, 0], v[:, 0])
    np.testing.assert_array_equal(o[0, 1], v[0, 1])


def test_rejects_rows_past_the_keys_and_unknown_classes():
    q = np.zeros((1, 2, 8))
    k = np.zeros((4, 1, 8))
    with pytest.raises(ValueError):
        orows.attend_rows(q, k, k, [4], [(G, 0, 0, None)])
    with pytest.raises(ValueError):
        orows.attend_rows(q, k, k, [1], [(7, 0, 0, None)])
