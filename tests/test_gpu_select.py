"""GPU: heavy-hitter retrieval selection (sp_select_heavy_hitters) against
the selection oracle (oracle/select.py).

The scores are floating point, so parity is split: the GPU's scores must
match the oracle's fp64 scores within a tolerance, and the GPU's index set
must be exactly what the oracle's selection rule picks from the GPU's own
fp32 scores (the integer decision taken on the same values)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import select
from _gpu_common import compare, f64, gpu_ready, pol_tuple, to_c_policies

pytestmark = pytest.mark.gpu


def _run(q, k, topk, recent):
    from head_aware_paged_gb300 import sp_select_heavy_hitters
    idx, counts, sc = sp_select_heavy_hitters(q, k, topk, recent, want_scores=True)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), counts.cpu().numpy(), sc.cpu().numpy()


def _check(q, k, topk, recent, rtol=2e-3):
    n = k.shape[0]
    idx, counts, sc = _run(q, k, topk, recent)
    ref = select.scores(f64(q), f64(k))
    np.testing.assert_allclose(sc, ref, rtol=rtol, atol=1e-6 * ref.max())
    for h in range(k.shape[1]):
        want = select.select(sc[h], n, topk, recent)          # the rule on the GPU's own scores
        got = idx[h, : counts[h]].tolist()
        assert got == want, (h, got[:10], want[:10])
        assert (idx[h, counts[h]:] == -1).all()
    return idx, counts, sc


@pytest.mark.parametrize("d,n,n_obs,hq,hkv", [(64, 1000, 37, 8, 2), (128, 777, 64, 6, 3),
                                              (128, 64, 1, 2, 1), (64, 200, 200, 4, 4)])
def test_scores_and_selection(d, n, n_obs, hq, hkv):
    gpu_ready()
    q = W.normal((n_obs, hq, d), 1, device="cuda")
    k = W.normal((n, hkv, d), 2, scale=0.5, device="cuda")
    _check(q, k, 50, 16)


def test_edges_and_ties():
    gpu_ready()
    d, n = 64, 300
    q = W.normal((20, 4, d), 3, device="cuda")
    k = W.normal((n, 2, d), 4, device="cuda")
    # duplicated keys score identically: the lower positions must win the ties
    k[100:140] = k[60].clone()
    k[200:210] = k[60].clone()
    for topk, recent in [(5, 0), (0, 10), (290, 10), (400, 0), (10, 400), (1, 1)]:
        _check(q, k, topk, recent)


def test_selected_indices_drive_a_retrieval_head():
    # select on a prompt, set RETRIEVAL(I) from the selection, attend: the
    # result matches the oracle over the same index list
    gpu_ready()
    from head_aware_paged_gb300 import Config, Policy, SegPagedCache
    d, n, hq, hkv = 128, 700, 4, 2
    q = W.normal((n, hq, d), 5, device="cuda")
    k = W.normal((n, hkv, d), 6, device="cuda")
    v = W.normal((n, hkv, d), 7, device="cuda")
    idx, counts, _ = _check(q[-32:].contiguous(), k, 96, 32)
    pols = [[Policy(2, idx=idx[h, : counts[h]].tolist()) for h in range(hkv)]]
    cache = SegPagedCache(Config(num_layers=1, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                 page_size=16, max_seqs=1, max_seq_len=n + 16, num_pages=64,
                                 max_idx_per_seq=1024, max_tokens=n + 16, max_batch=1))
    cache.set_policy(0, pols)
    cache.build(0, 0, k, v)
    qd = W.normal((1, hq, d), 8, device="cuda")
    kd = W.normal((1, hkv, d), 9, device="cuda")
    vd = W.normal((1, hkv, d), 10, device="cuda")
    cache.append_kv(0, [0], [0, 1], kd, vd)
    out, lse = cache.decode(0, [0], qd)
    pt = [(2, 0, 0, idx[h, : counts[h]].tolist()) for h in range(hkv)]
    kk = np.concatenate([f64(k), f64(kd)], axis=0)
    vv = np.concatenate([f64(v), f64(vd)], axis=0)
    ref, lref = oracle.attend(f64(qd), kk, vv, np.array([n]), pt, "f64")
    compare(out, ref, lse, lref, "decode over selected indices")
    assert cache.status() == 0


def _check_top_p(q, k, top_p, max_keys, recent, rtol=2e-3):
    """GPU top-p selection: scores against the oracle's float64 scores; each
    head's count is the exact rule's count on the GPU's own fp32 scores (or
    its float64-boundary neighbour), and the kept keys are exactly the
    highest-ranked ones of that count."""
    from head_aware_paged_gb300 import sp_select_heavy_hitters_top_p
    n = k.shape[0]
    idx, counts, sc = sp_select_heavy_hitters_top_p(q, k, top_p, max_keys, recent, want_scores=True)
    torch.cuda.synchronize()
    idx, counts, sc = idx.cpu().numpy(), counts.cpu().numpy(), sc.cpu().numpy()
    ref = select.scores(f64(q), f64(k))
    np.testing.assert_allclose(sc, ref, rtol=rtol, atol=1e-6 * ref.max())
    nrec = min(recent, n)
    for h in range(k.shape[1]):
        m, ok = select.top_p_count(sc[h], n, np.float32(top_p), max_keys, recent)
        got_m = int(counts[h]) - nrec
        assert got_m in ok, (h, got_m, m, ok)
        assert idx[h, :counts[h]].tolist() == select.select(sc[h], n, got_m, recent)
        assert (idx[h, counts[h]:] == -1).all()
    return counts


@pytest.mark.parametrize("d,n,n_obs,hq,hkv", [(64, 1000, 37, 8, 2), (128, 777, 64, 6, 3),
                                              (128, 4096, 64, 32, 8), (64, 200, 200, 4, 4)])
def test_top_p_selection(d, n, n_obs, hq, hkv):
    gpu_ready()
    q = W.normal((n_obs, hq, d), 11, device="cuda")
    k = W.normal((n, hkv, d), 12, scale=0.5, device="cuda")
    for top_p, max_keys, recent in [(0.9, n, 16), (0.5, 64, 0), (0.25, n, 0), (1.0, n, 8),
                                    (0.999, 50, 3)]:
        _check_top_p(q, k, top_p, max_keys, recent)


def test_top_p_ties_and_arguments():
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError, sp_select_heavy_hitters_top_p
    d, n = 64, 300
    q = W.normal((20, 4, d), 3, device="cuda")
    k = W.normal((n, 2, d), 4, device="cuda")
    k[100:140] = k[60].clone()                  # equal scores: lower positions first
    for top_p, max_keys, recent in [(0.3, 400, 0), (0.7, 10, 5), (0.05, 1, 0), (0.6, 0, 20)]:
        _check_top_p(q, k, top_p, max_keys, recent)
    for bad in (0.0, -0.5, 1.5, float("nan")):
        with pytest.raises(SegPagedError):
            sp_select_heavy_hitters_top_p(q, k, bad, 10, 0)
