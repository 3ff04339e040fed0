"""The oracle pins catch planted mistakes (no GPU).

Each variant of the C oracle is built with one deliberate error (a dropped
scale, an off-by-one window or sink, a wrong retrieval bound, interleaved GQA
grouping, a shifted index, a dropped normaliser term, LSE in the wrong base);
the dense+mask equivalence, the brute-force check or a golden fixture must
reject every one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from test_oracle import dense_masked, _brute_visible, _brute_attend

G, L, R = 0, 1, 2
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pins_pass(mut):
    rng = np.random.default_rng(0)
    n, hq, hkv, d = 96, 4, 2, 8
    q = rng.standard_normal((n, hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = rng.standard_normal((n, hkv, d))
    ok = True
    for pols in ([(G, 0, 0, None), (L, 3, 10, None)],
                 [(R, 0, 0, sorted(rng.choice(n, 20, replace=False).tolist())), (L, 0, 1, None)]):
        o, lse = oracle.attend(q, k, v, np.arange(n), pols, "f64", _mutation=mut)
        od, ld = dense_masked(q, k, v, np.arange(n), pols)
        fin = np.isfinite(ld)
        ok &= bool(np.abs(o - od).max() < 1e-10)
        ok &= bool(np.array_equal(np.isfinite(lse), fin))
        ok &= bool(np.abs(lse[fin] - ld[fin]).max() < 1e-10)
    # visibility lists against brute-force sets
    for (kind, s, w, idx) in [(L, 4, 7, None), (R, 0, 0, [2, 5, 9])]:
        for i in range(20):
            got = oracle.visible(kind, s, w, idx, i, _mutation=mut).tolist()
            ok &= got == sorted(_brute_visible(kind, s, w, idx, i))
    with open(os.path.join(GOLDEN, "two_key_softmax.json")) as f:
        gd = json.load(f)
    o, lse = oracle.attend(np.array(gd["q"]).reshape(1, 1, 4), np.array(gd["k"]).reshape(2, 1, 4),
                           np.array(gd["v"]).reshape(2, 1, 4), [1], [(G, 0, 0, None)], "f64",
                           _mutation=mut)
    ok &= bool(np.abs(o[0, 0] - gd["expect_o"]).max() < 1e-12)
    ok &= abs(lse[0, 0] - gd["expect_lse"]) < 1e-12
    return ok


def test_unmutated_oracle_passes_the_pins():
    assert _pins_pass(0)


@pytest.mark.parametrize("mut", range(1, 9))
def test_planted_mistake_is_caught(mut):
    assert not _pins_pass(mut)
