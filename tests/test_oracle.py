"""Pins for the CPU attention oracle (no GPU).

Each test ties the oracle to something other than itself:
  * the runtime article's equivalence claim (section 4): identical to dense
    attention under an explicit head-wise mask -> a NumPy fp64 dense+mask
    formulation with vectorised masks and np.repeat GQA;
  * brute force on tiny inputs: visibility from Python sets built from the
    class descriptions, attention with math.exp in pure Python;
  * closed forms: |V(i)|, a hand-derived two-key softmax, special inputs;
  * worked examples printed on the pages (tests/golden/);
  * invariants of the method.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
G, L, R = 0, 1, 2


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def dense_masked(q, k, v, row_pos, policies):
    """Dense fp64 attention with an explicit [Hq, rows, keys] boolean mask."""
    q = q.astype(np.float64)
    k = k.astype(np.float64)
    v = v.astype(np.float64)
    rows, hq, d = q.shape
    n, hkv, _ = k.shape
    grp = hq // hkv
    kk = np.repeat(k, grp, axis=1)
    vv = np.repeat(v, grp, axis=1)
    i = np.asarray(row_pos)[:, None]
    j = np.arange(n)[None, :]
    masks = []
    for (kind, s, w, idx) in policies:
        if kind == G:
            m = j <= i
        elif kind == L:
            m = (j <= i) & ((j < s) | (j > i - w))
        else:
            m = (j <= i) & np.isin(j, np.asarray(idx if idx is not None else [], dtype=np.int64))
        masks.append(m)
    mask = np.repeat(np.stack(masks), grp, axis=0)           # [hq, rows, n]
    S = np.einsum("rhd,nhd->hrn", q, kk) / math.sqrt(d)
    S = np.where(mask, S, -np.inf)
    mx = S.max(-1, keepdims=True)
    empty = ~np.isfinite(mx)
    mx = np.where(empty, 0.0, mx)
    P = np.exp(S - mx)
    den = P.sum(-1, keepdims=True)
    out = np.einsum("hrn,nhd->rhd", P / np.where(den == 0, 1, den), vv)
    lse = np.where(empty[..., 0], -np.inf, (mx + np.log(np.where(den == 0, 1, den)))[..., 0])
    return out, lse.T


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _mixed_policies(hkv, L_, seed):
    rng = np.random.default_rng(seed)
    pols = []
    for h in range(hkv):
        kind = h % 3
        if kind == G:
            pols.append((G, 0, 0, None))
        elif kind == L:
            pols.append((L, int(rng.integers(0, 6)), int(rng.integers(1, L_)), None))
        else:
            idx = np.sort(rng.choice(L_, size=max(1, L_ // 5), replace=False)).astype(np.int32)
            pols.append((R, 0, 0, idx.tolist()))
    return pols


# ---------------------------------------------------------------- golden pins

def test_golden_two_key_softmax():
    gd = _golden("two_key_softmax.json")
    d = gd["d"]
    q = np.array(gd["q"], dtype=np.float64).reshape(1, 1, d)
    k = np.array(gd["k"], dtype=np.float64).reshape(2, 1, d)
    v = np.array(gd["v"], dtype=np.float64).reshape(2, 1, d)
    for prec, tol in (("f64", 1e-12), ("f32", 2e-6)):
        o, lse = oracle.attend(q, k, v, [1], [(G, 0, 0, None)], prec)
        np.testing.assert_allclose(o[0, 0], gd["expect_o"], atol=tol)
        assert abs(lse[0, 0] - gd["expect_lse"]) < tol


def test_golden_gqa_grouping():
    """Query head h uses KV head (1-indexed) ceil(h / (H/G)) (tutorial 5.3)."""
    gd = _golden("gqa_h8_g2.json")
    hq, hkv, d, n = gd["num_q_heads"], gd["num_kv_heads"], 16, 9
    q = _rand((1, hq, d), 1)
    k = _rand((n, hkv, d), 2)
    v = _rand((n, hkv, d), 3)
    pols = [(G, 0, 0, None)] * hkv
    o, _ = oracle.attend(q, k, v, [n - 1], pols, "f64")
    for h in range(hq):
        grp = gd["expect_group_1_indexed"][h] - 1
        o1, _ = oracle.attend(q[:, h:h + 1], k[:, grp:grp + 1], v[:, grp:grp + 1],
                              [n - 1], [(G, 0, 0, None)], "f64")
        np.testing.assert_allclose(o[0, h], o1[0, 0], atol=1e-14)
        other = 1 - grp
        o2, _ = oracle.attend(q[:, h:h + 1], k[:, other:other + 1], v[:, other:other + 1],
                              [n - 1], [(G, 0, 0, None)], "f64")
        assert np.abs(o[0, h] - o2[0, 0]).max() > 1e-3


def test_golden_kv_bytes():
    gd = _golden("kv_bytes_example.json")
    b = accounting.dense_kv_bytes(gd["layers"], gd["kv_heads"], gd["head_dim"],
                                  gd["tokens"], gd["bytes_per_element"])
    assert b == gd["expect_bytes_exact"]
    assert abs(b / 1e9 - gd["expect_bytes_approx_gb"]) < 0.05
    # all-GLOBAL heads at the last position see every token: visible == dense
    pols = [(G, 0, 0, None)] * gd["kv_heads"]
    per_layer = accounting.decode_kv_bytes(pols, gd["tokens"] - 1, gd["head_dim"],
                                           gd["bytes_per_element"])
    assert per_layer * gd["layers"] == b


# ------------------------------------------------------- dense+mask equivalence

@pytest.mark.parametrize("prec,atol", [("f64", 1e-11), ("f32", 2e-5)])
def test_equivalence_tiny_config(prec, atol):
    """Tiny case: Hq 4 / Hkv 2, d 64, L 256, KV0 GLOBAL, KV1 LOCAL(4, 32)."""
    Lq = 256
    q = _rand((Lq, 4, 64), 10)
    k = _rand((Lq, 2, 64), 11)
    v = _rand((Lq, 2, 64), 12)
    pols = [(G, 0, 0, None), (L, 4, 32, None)]
    o, lse = oracle.attend(q, k, v, np.arange(Lq), pols, prec)
    od, ld = dense_masked(q, k, v, np.arange(Lq), pols)
    np.testing.assert_allclose(o, od, atol=atol)
    np.testing.assert_allclose(lse, ld, atol=atol * 10)
    cos = (o * od).sum() / np.sqrt((o * o).sum() * (od * od).sum())
    assert cos >= 0.999999


def test_equivalence_mistral_shaped_reduced():
    """Hq 32 / Hkv 8, d 128, L 1024 (reduced), K x 0.5, 1 GLOBAL + 7 LOCAL(4, 256)
    plus a mixed-class variant with RETRIEVAL heads."""
    Lq, hq, hkv, d = 1024, 32, 8, 128
    q = _rand((Lq, hq, d), 20)
    k = _rand((Lq, hkv, d), 21, 0.5)
    v = _rand((Lq, hkv, d), 22)
    rows = np.arange(0, Lq, 3)
    for pols in ([(G, 0, 0, None)] + [(L, 4, 256, None)] * 7,
                 _mixed_policies(hkv, Lq, 5)):
        o, lse = oracle.attend(q[rows], k, v, rows, pols, "f64")
        od, ld = dense_masked(q[rows], k, v, rows, pols)
        assert np.abs(o - od).max() <= 1e-10
        fin = np.isfinite(ld)
        np.testing.assert_allclose(lse[fin], ld[fin], atol=1e-10)
        assert np.array_equal(np.isfinite(lse), fin)
        o32, _ = oracle.attend(q[rows], k, v, rows, pols, "f32")
        assert np.abs(o32 - od).max() <= 1e-5


# ------------------------------------------------------------- brute force

def _brute_visible(kind, s, w, idx, i):
    if kind == G:
        return set(range(i + 1))
    if kind == L:
        sinks = {j for j in range(i + 1) if j < s}
        recent = {i - back for back in range(w) if i - back >= 0}
        return sinks | recent
    return {t for t in idx if t <= i}


def _brute_attend(q, k, v, i, vis):
    d = len(q)
    if not vis:
        return [0.0] * d, -math.inf
    js = sorted(vis)
    sc = [sum(q[c] * k[j][c] for c in range(d)) / math.sqrt(d) for j in js]
    mx = max(sc)
    w = [math.exp(x - mx) for x in sc]
    den = sum(w)
    o = [sum(w[t] * v[js[t]][c] for t in range(len(js))) / den for c in range(d)]
    return o, mx + math.log(den)


@pytest.mark.parametrize("s", [0, 1, 4, 5])
@pytest.mark.parametrize("w", [1, 3, 16, 64])
def test_brute_force_local(s, w):
    Lq, d = 48, 8
    q = _rand((Lq, 1, d), 100 + s)
    k = _rand((Lq, 1, d), 200 + w)
    v = _rand((Lq, 1, d), 300)
    o, lse = oracle.attend(q, k, v, np.arange(Lq), [(L, s, w, None)], "f64")
    for i in range(Lq):
        vis = _brute_visible(L, s, w, None, i)
        assert len(vis) == min(i + 1, s + w)
        assert list(oracle.visible(L, s, w, None, i)) == sorted(vis)
        ob, lb = _brute_attend(q[i, 0], k[:, 0], v[:, 0], i, vis)
        np.testing.assert_allclose(o[i, 0], ob, atol=1e-12)
        assert abs(lse[i, 0] - lb) < 1e-12


@pytest.mark.parametrize("seed", range(4))
def test_brute_force_global_and_retrieval(seed):
    rng = np.random.default_rng(seed)
    Lq, d = 64, 4
    idx = sorted(rng.choice(Lq, size=int(rng.integers(1, 20)), replace=False).tolist())
    q = _rand((Lq, 2, d), seed + 1)
    k = _rand((Lq, 2, d), seed + 2)
    v = _rand((Lq, 2, d), seed + 3)
    pols = [(G, 0, 0, None), (R, 0, 0, idx)]
    o, lse = oracle.attend(q, k, v, np.arange(Lq), pols, "f64")
    for i in range(Lq):
        for h, (kind, s, w, ind) in enumerate(pols):
            vis = _brute_visible(kind, s, w, ind, i)
            ob, lb = _brute_attend(q[i, h], k[:, h], v[:, h], i, vis)
            np.testing.assert_allclose(o[i, h], ob, atol=1e-12)
            if vis:
                assert abs(lse[i, h] - lb) < 1e-12
            else:
                assert lse[i, h] == -np.inf and not o[i, h].any()


# ----------------------------------------------------------- closed forms

def test_visible_count_closed_forms():
    rng = np.random.default_rng(7)
    idx = np.sort(rng.choice(300, 40, replace=False)).tolist()
    rows = np.arange(300)
    for (kind, s, w, ind) in [(G, 0, 0, None), (L, 4, 32, None), (L, 0, 1, None),
                              (L, 7, 100, None), (R, 0, 0, idx)]:
        closed = accounting.vis_count_closed(kind, s, w, ind, rows)
        brute = [accounting.vis_count(kind, s, w, ind, int(i)) for i in rows]
        assert closed.tolist() == brute
        if kind == G:
            assert closed.tolist() == (rows + 1).tolist()
        if kind == L:
            assert closed.tolist() == np.minimum(rows + 1, s + w).tolist()


def test_visible_pairs_match_pages_workload_totals():
    """Mistral-shaped prefill (L 8192, 1 GLOBAL + 7 LOCAL(4, 1024), Hq 32):
    355,252,056 visible pairs = 0.1819 TFLOP at 4 d FLOP per pair."""
    pols = [(G, 0, 0, None)] + [(L, 4, 1024, None)] * 7
    pairs = accounting.prefill_pairs(pols, 32, 0, 8192)
    assert pairs == 4 * (8192 * 8193 // 2) + 7 * 4 * (
        sum(i + 1 for i in range(1028)) + (8192 - 1028) * 1028)
    assert pairs == 355_252_056


def test_special_inputs():
    Lq, d = 40, 16
    rng = np.random.default_rng(3)
    k = _rand((Lq, 3, d), 4)
    pols = [(G, 0, 0, None), (L, 2, 5, None), (R, 0, 0, [1, 5, 9, 30])]
    # constant value rows -> O = c wherever V(i) is non-empty
    c = rng.standard_normal(d)
    v = np.broadcast_to(c, (Lq, 3, d)).copy()
    q = _rand((Lq, 3, d), 5)
    o, lse = oracle.attend(q, k, v, np.arange(Lq), pols, "f64")
    for h in range(3):
        for i in range(Lq):
            if len(_brute_visible(*pols[h], i)):
                np.testing.assert_allclose(o[i, h], c, atol=1e-12)
    # q = 0 -> uniform weights -> mean of the visible values
    v = _rand((Lq, 3, d), 6)
    o, lse = oracle.attend(np.zeros((Lq, 3, d)), k, v, np.arange(Lq), pols, "f64")
    for h in range(3):
        for i in range(Lq):
            vis = sorted(_brute_visible(*pols[h], i))
            if vis:
                np.testing.assert_allclose(o[i, h], v[vis, h].mean(0), atol=1e-12)
                assert abs(lse[i, h] - math.log(len(vis))) < 1e-12
    # LOCAL with sink 0 and window 1 sees only itself: O_i = v_i
    q = _rand((Lq, 1, d), 8)
    o, _ = oracle.attend(q, k[:, :1], v[:, :1], np.arange(Lq), [(L, 0, 1, None)], "f64")
    np.testing.assert_allclose(o[:, 0], v[:, 0], atol=1e-14)


def test_empty_visibility_gives_zero_and_neg_inf():
    d = 8
    q = _rand((3, 1, d), 1)
    k = _rand((12, 1, d), 2)
    v = _rand((12, 1, d), 3)
    o, lse = oracle.attend(q, k, v, [0, 4, 11], [(R, 0, 0, [5, 9])], "f64")
    assert not o[0].any() and not o[1].any()
    assert lse[0, 0] == -np.inf and lse[1, 0] == -np.inf
    assert np.isfinite(lse[2, 0])


# -------------------------------------------------------------- invariants

def test_invariants():
    Lq, d = 200, 32
    q = _rand((Lq, 4, d), 40)
    k = _rand((Lq, 2, d), 41)
    v = _rand((Lq, 2, d), 42)
    rows = np.arange(Lq)
    og, lg = oracle.attend(q, k, v, rows, [(G, 0, 0, None)] * 2, "f64")
    # LOCAL with s + W >= L is GLOBAL
    ol, ll = oracle.attend(q, k, v, rows, [(L, 3, Lq - 3, None)] * 2, "f64")
    np.testing.assert_allclose(ol, og, atol=1e-13)
    # RETRIEVAL of every index is GLOBAL
    orr, lr = oracle.attend(q, k, v, rows, [(R, 0, 0, list(range(Lq)))] * 2, "f64")
    np.testing.assert_allclose(orr, og, atol=1e-13)
    # query heads of one group with equal Q give identical O
    q2 = q.copy()
    q2[:, 1] = q2[:, 0]
    o2, _ = oracle.attend(q2, k, v, rows, [(L, 4, 20, None)] * 2, "f64")
    assert np.array_equal(o2[:, 0], o2[:, 1])
    # a decode query at position t equals prefill row t
    pols = [(G, 0, 0, None), (L, 4, 20, None)]
    op, _ = oracle.attend(q, k, v, rows, pols, "f64")
    for t in (0, 19, 24, 150, Lq - 1):
        od, _ = oracle.attend(q[t:t + 1], k[:t + 1], v[:t + 1], [t], pols, "f64")
        np.testing.assert_allclose(od[0], op[t], atol=1e-14)
    # keys beyond the query position never matter (causality)
    k3 = k.copy()
    k3[150:] = 1e3
    o3, _ = oracle.attend(q[:150], k3, v, rows[:150], pols, "f64")
    np.testing.assert_allclose(o3, op[:150], atol=1e-14)


def test_fp32_agrees_with_fp64():
    Lq, d = 300, 128
    q = _rand((Lq, 8, d), 50)
    k = _rand((Lq, 2, d), 51, 0.5)
    v = _rand((Lq, 2, d), 52)
    pols = [(G, 0, 0, None), (L, 4, 64, None)]
    o64, l64 = oracle.attend(q, k, v, np.arange(Lq), pols, "f64")
    o32, l32 = oracle.attend(q, k, v, np.arange(Lq), pols, "f32")
    assert np.abs(o64 - o32).max() < 1e-5
    assert np.abs(l64 - l32).max() < 1e-4


def test_bad_inputs_rejected():
    q = _rand((1, 1, 4), 1)
    k = _rand((3, 1, 4), 2)
    with pytest.raises(ValueError):
        oracle.attend(q, k, k, [5], [(G, 0, 0, None)], "f64")   # position beyond keys
    with pytest.raises(ValueError):
        oracle.attend(q, k, k, [1], [(7, 0, 0, None)], "f64")   # unknown class
