"""The seeded input generators (no GPU): the recipe the design notes state
for each workload -- class counts, retrieval lists, ragged lengths, tensor
shapes and scales -- and determinism, since the oracle and the CUDA path
must see the same numbers."""
import math

import numpy as np
import pytest
import torch

import workloads as W


@pytest.mark.parametrize("name,units,n_g,n_r", [
    ("mistral7b_prefill_8k", 8, 1, 0),
    ("llama3_8b_decode_32k", 256, 32, 0),        # 12.5 %
    ("llama33_70b_prefill_128k", 512, 77, 0),    # 15 %
    ("ragged_mixed", 256, 38, 38),               # 15 % / 15 %
])
def test_class_counts(name, units, n_g, n_r):
    wl = W.WORKLOADS[name]
    kinds = W.class_assignment(wl)
    assert kinds.shape == (wl.layers, wl.hkv) and kinds.size == units
    assert int((kinds == W.GLOBAL).sum()) == n_g
    assert int((kinds == W.RETRIEVAL).sum()) == n_r
    assert int((kinds == W.LOCAL).sum()) == units - n_g - n_r
    assert np.array_equal(kinds, W.class_assignment(wl))          # same seed, same draw
    assert not np.array_equal(kinds, W.class_assignment(wl, seed=1)) or n_g == units


def test_tiny_classes_are_fixed():
    kinds = W.class_assignment(W.WORKLOADS["tiny"])
    assert kinds.tolist() == [[W.GLOBAL, W.LOCAL]]
    pols = W.policies(W.WORKLOADS["tiny"])
    assert (pols[0][1].sink, pols[0][1].window) == (4, 32)


def test_local_policies_carry_the_workload_window():
    for name, (s, w) in {"mistral7b_prefill_8k": (4, 1024), "llama3_8b_decode_32k": (4, 2048),
                         "llama33_70b_prefill_128k": (4, 8192), "ragged_mixed": (4, 4096)}.items():
        for row in W.policies(W.WORKLOADS[name], length=5000):
            for p in row:
                if p.kind == W.LOCAL:
                    assert (p.sink, p.window) == (s, w)


def test_retrieval_lists():
    for L in (100, 2048, 2049, 65536):
        idx = W.retrieval_indices(L, 2048, seed=7)
        assert idx.dtype == np.int32
        assert len(idx) == min(L, 2048)
        assert np.all(np.diff(idx) > 0) and idx[0] >= 0 and idx[-1] < L
        assert np.array_equal(idx, W.retrieval_indices(L, 2048, seed=7))
    # the lists are the top-k of the seeded scores: every kept index scores at
    # least as high as every dropped one
    L, k = 5000, 300
    idx = W.retrieval_indices(L, k, seed=3)
    rng = np.random.default_rng(W._seed(3, L, 31))
    score = rng.random(L, dtype=np.float32)
    kept = np.zeros(L, bool)
    kept[idx] = True
    assert score[kept].min() >= score[~kept].max()


def test_ragged_lengths_are_log_uniform_in_range():
    wl = W.WORKLOADS["ragged_mixed"]
    lens = W.ragged_lengths(wl)
    assert len(lens) == wl.seqs and lens == W.ragged_lengths(wl)
    assert all(2048 <= n < 65536 for n in lens)
    # many draws: log-lengths spread evenly over [ln 2048, ln 65536)
    draws = [n for s in range(200) for n in W.ragged_lengths(wl, seed=s)]
    u = (np.log(draws) - math.log(2048)) / (math.log(65536) - math.log(2048))
    hist, _ = np.histogram(u, bins=4, range=(0, 1))
    assert hist.min() > 0.8 * len(draws) / 4


def test_tensors_are_seeded_and_scaled():
    wl = W.WORKLOADS["mistral7b_prefill_8k"]
    q, k, v = W.qkv(wl, 512, 0, 0)
    assert q.shape == (512, 32, 128) and k.shape == (512, 8, 128) and v.shape == (512, 8, 128)
    assert q.dtype == torch.bfloat16
    q2, k2, v2 = W.qkv(wl, 512, 0, 0)
    assert torch.equal(q, q2) and torch.equal(k, k2) and torch.equal(v, v2)
    q3, _, _ = W.qkv(wl, 512, 1, 0)
    assert not torch.equal(q, q3)
    # N(0, 1) for q and v, K scaled by 0.5 (the Mistral-shaped recipe)
    assert abs(q.float().std().item() - 1.0) < 0.02
    assert abs(v.float().std().item() - 1.0) < 0.02
    assert abs(k.float().std().item() - 0.5) < 0.01
    assert abs(q.float().mean().item()) < 0.01
