"""The library's tile planner and storage rules, run on the CPU, against the
oracle (no GPU).

`plan_host_check.cpp` compiles the product's own rule headers
(`csrc/sp_rules.h`, `csrc/sp_plan.h`, the code the kernels run) for the
host.  For seeded random head policies, page sizes, history lengths and row
ranges this test checks, bit for bit:
  * prefill: the keys each query row attends over, collected from the tile
    plan with the kernels' own mask test, equal the oracle's V(i) (runtime
    article section 2), each position once; tiles marked "full" (no mask on
    the GPU) are visible to every row; paged tiles stay inside the unit's
    pages (section 3: per-head page lists);
  * decode: the slot ranges one query reads hold exactly V(t);
  * storage: the position held by every slot of a unit equals the oracle's
    page model of the same write rule, both from the closed-form slot rule
    and after the scatter kernels' per-write rule applied chunk by chunk.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle import pagemodel

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "head_aware_paged_gb300", "csrc")
G, L, R = 0, 1, 2


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_host_check")
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", CSRC, os.path.join(HERE, "plan_host_check.cpp"),
                    "-o", exe], check=True, capture_output=True)
    return exe


def _run(exe, cases):
    lines = [str(len(cases))]
    for c in cases:
        mode, kind, sink, window, P, n, i_lo, i_hi, idx = c[:9]
        extra = list(c[9]) if len(c) > 9 else []
        lines.append(" ".join(str(x) for x in [mode, kind, sink, window, P, n, i_lo, i_hi, len(idx)]
                              + list(idx) + extra))
    out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True).stdout
    res, cur = [], None
    for ln in out.splitlines():
        f = ln.split()
        if f[0] == "C":
            cur = {"R": {}, "L": {}, "D": None, "S": None, "P": [], "ERR": []}
            res.append(cur)
        elif f[0] == "ERR":
            cur["ERR"].append(ln)
        elif f[0] == "R":
            cur["R"][int(f[1])] = tuple(int(x) for x in f[2:])
        elif f[0] == "L":
            cur["L"][int(f[1])] = [int(x) for x in f[2:]]
        elif f[0] == "D":
            cur["D"] = tuple(int(x) for x in f[1:])
        elif f[0] == "S":
            cur["S"] = int(f[1])
            cur.setdefault("tables", []).append([])
        elif f[0] == "P":
            cur["P"].append([int(x) for x in f[1:]])
            cur["tables"][-1].append([int(x) for x in f[1:]])
    assert len(res) == len(cases)
    return res


def _policy(rng, limit):
    kind = int(rng.integers(0, 3))
    sink = int(rng.choice([0, 1, 4, 5, 17, 70]))
    window = int(rng.choice([1, 3, 16, 64, 100, 257, 1024]))
    idx = []
    if kind == R:
        m = int(rng.integers(0, 120))
        idx = sorted(set(int(x) for x in rng.integers(0, max(limit, 1), size=m)))
    return kind, sink, window, idx


def _stats(pos):
    p = np.asarray(pos, dtype=np.int64)
    return (int(p.size), int(p.sum()), int((p * p).sum()))


def _visible(kind, sink, window, idx, i):
    return oracle.visible(kind, sink, window, idx if kind == R else None, i)


def test_prefill_plans_cover_exactly_the_visible_sets(harness):
    rng = np.random.default_rng(11)
    cases = []
    for _ in range(160):
        P = int(rng.choice([16, 32, 64, 128]))
        n_b = int(rng.choice([0, 0, 1, 5, 63, 64, 65, 200, 777, 1200]))
        rb = int(rng.integers(0, 3))
        rows = int(rng.choice([1, 2, 17, 64, 127, 128]))
        i_lo = n_b + 128 * rb
        kind, sink, window, idx = _policy(rng, i_lo + rows + 40)
        cases.append((0, kind, sink, window, P, n_b, i_lo, i_lo + rows - 1, idx))
    # fixed edge cases: sink longer than the history, a window of one, an
    # empty retrieval list, a list entirely after the rows
    cases += [(0, L, 70, 1, 16, 40, 40, 167, []), (0, L, 0, 1, 64, 300, 300, 427, []),
              (0, R, 0, 0, 32, 100, 100, 227, []), (0, R, 0, 0, 32, 100, 100, 227, [500, 600]),
              (0, L, 4, 1024, 64, 0, 0, 127, []), (0, G, 0, 0, 128, 129, 257, 384, [])]
    res = _run(harness, cases)
    checked = 0
    for c, r in zip(cases, res):
        _, kind, sink, window, P, n_b, i_lo, i_hi, idx = c
        assert not r["ERR"], (c[:8], r["ERR"][:3])
        for i in range(i_lo, i_hi + 1):
            want = _visible(kind, sink, window, idx, i)
            assert r["R"][i] == _stats(want), (c[:8], i)
            if i in r["L"]:
                assert r["L"][i] == want.tolist(), (c[:8], i)
                checked += 1
    assert checked >= len(cases)


def test_decode_ranges_hold_exactly_the_visible_set(harness):
    rng = np.random.default_rng(12)
    cases = []
    for _ in range(300):
        P = int(rng.choice([16, 32, 64, 128]))
        t = int(rng.choice([0, 1, 3, 15, 16, 63, 64, 65, 300, 1000, 2047, 2048, 2049, 4000]))
        kind, sink, window, idx = _policy(rng, t + 30)
        cases.append((1, kind, sink, window, P, t + 1, t, t, idx))
    res = _run(harness, cases)
    for c, r in zip(cases, res):
        _, kind, sink, window, P, n, t, _, idx = c
        assert not r["ERR"], (c[:8], r["ERR"][:3])
        want = _visible(kind, sink, window, idx, t)
        assert r["D"] == _stats(want), c[:8]
        assert r["L"][t] == want.tolist(), c[:8]


def test_slot_tables_match_the_page_model(harness):
    rng = np.random.default_rng(13)
    cases = []
    for _ in range(200):
        P = int(rng.choice([16, 32, 64, 128]))
        n = int(rng.choice([0, 1, 4, 5, 16, 64, 65, 129, 500, 1023, 1024, 1025, 3000]))
        kind, sink, window, idx = _policy(rng, n + 30)
        cases.append((2, kind, sink, window, P, n, 0, 0, idx))
    res = _run(harness, cases)
    for c, r in zip(cases, res):
        _, kind, sink, window, P, n, _, _, idx = c
        want = pagemodel.stored_positions(kind, sink, window, idx if kind == R else None, n, P)
        assert r["S"] == len(want), c[:6]
        assert r["P"] == want, c[:6]


def test_chunked_writes_leave_the_page_model_state(harness):
    """The scatter kernels' write rule (kept tokens per write, the slot of
    each) applied chunk by chunk leaves after every chunk exactly the slot
    contents of the oracle's token-by-token page model."""
    rng = np.random.default_rng(14)
    cases = []
    for _ in range(150):
        P = int(rng.choice([16, 32, 64, 128]))
        m = int(rng.integers(1, 6))
        chunks = [int(x) for x in rng.choice([1, 2, 15, 16, 17, 64, 100, 333, 1000], size=m)]
        kind, sink, window, idx = _policy(rng, sum(chunks) + 30)
        cases.append((3, kind, sink, window, P, sum(chunks), m, 0, idx, chunks))
    res = _run(harness, cases)
    for c, r in zip(cases, res):
        _, kind, sink, window, P, _, m, _, idx, chunks = c
        assert not r["ERR"], (c[:8], r["ERR"][:3])
        assert len(r["tables"]) == m
        n = 0
        for ch, got in zip(chunks, r["tables"]):
            n += ch
            want = pagemodel.stored_positions(kind, sink, window, idx if kind == R else None, n, P)
            assert got == want, (c[:8], n)
