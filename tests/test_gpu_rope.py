"""GPU: RoPE realignment of stored keys (sp_rope_realign) against the
closed-form oracle (oracle/rope.py), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import rope
from _gpu_common import compare, f64, gpu_ready, pol_tuple, to_c_policies

pytestmark = pytest.mark.gpu

G, L, R = W.GLOBAL, W.LOCAL, W.RETRIEVAL
ULP = 2.0 ** -8          # one bf16 ulp, relative


def _cache(d, P, max_len, pages, seqs=2):
    from head_aware_paged_gb300 import Config, SegPagedCache
    return SegPagedCache(Config(num_layers=2, num_q_heads=6, num_kv_heads=3, head_dim=d,
                                page_size=P, max_seqs=seqs, max_seq_len=max_len,
                                num_pages=pages, max_idx_per_seq=4096, max_tokens=max_len,
                                max_batch=seqs))


def _stored_rows(cache, seq, layer, h):
    """(position, page id, slot) of every stored row of a unit, from the
    device table."""
    ids, pos = cache.export_table(seq, layer, h)
    out = []
    for pg, slots in zip(ids, pos):
        for s, p in enumerate(slots):
            if p >= 0:
                out.append((p, pg, s))
    return out


def _pair_norm(x):
    """sqrt(x[i]^2 + x[i + d/2]^2) spread back over both elements of a pair."""
    h = x.shape[-1] // 2
    n = np.sqrt(x[..., :h] ** 2 + x[..., h:] ** 2)
    return np.concatenate([n, n], axis=-1)


def _within_ulp(got, ref, what):
    """One bf16 ulp of the element, plus fp32 rounding slack relative to the
    rotated pair (an element much smaller than its partner carries the fp32
    error of the pair)."""
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    bound = ULP * np.abs(ref) + 2.0 ** -18 * _pair_norm(ref) + 2.0 ** -40
    bad = err > bound
    assert not bad.any(), "%s: %d elements beyond one bf16 ulp, worst %.3g at ref %.3g" % (
        what, bad.sum(), err.max(), ref.flat[np.argmax(err)])


@pytest.mark.parametrize("d,P", [(64, 16), (128, 64)])
def test_realign_rotates_exactly_the_requested_rows(d, P):
    gpu_ready()
    n = 600
    cache = _cache(d, P, n + 64, 400)
    pols = [[W.HeadPolicy(G), W.HeadPolicy(L, 5, 70),
             W.HeadPolicy(R, idx=np.array(sorted({3, 40, 41, 99, 250, 251, 252, 400, 599}), np.int32))]] * 2
    cache.set_policy(0, to_c_policies(pols))
    cache.set_policy(1, to_c_policies(pols))
    ks, vs = {}, {}
    for s in range(2):
        for l in range(2):
            ks[s, l] = W.normal((n, 3, d), W.tensor_seed(11, "k", s, l), device="cuda")
            vs[s, l] = W.normal((n, 3, d), W.tensor_seed(11, "v", s, l), device="cuda")
            cache.build(s, l, ks[s, l], vs[s, l])
    torch.cuda.synchronize()
    k_before = cache.k_pool().clone()
    v_before = cache.v_pool().clone()
    lo, hi, delta = 30, 560, 123457
    cache.rope_realign(1, [0], delta, kv_head=-1, pos_lo=lo, pos_hi=hi, rope_theta=10000.0)
    torch.cuda.synchronize()
    assert cache.status() == 0
    k_after = cache.k_pool()
    assert torch.equal(cache.v_pool(), v_before), "V must not change"
    touched = torch.zeros(k_after.shape[:2], dtype=torch.bool, device="cuda")
    for h in range(3):
        rows = _stored_rows(cache, 0, 1, h)
        assert rows
        sel = [(p, pg, s) for p, pg, s in rows if lo <= p < hi]
        assert sel
        pgs = torch.tensor([pg for _, pg, _ in sel], device="cuda")
        sls = torch.tensor([s for _, _, s in sel], device="cuda")
        before = f64(k_before[pgs, sls])
        ref = rope.realign(before, delta)
        _within_ulp(f64(k_after[pgs, sls]), ref, "head %d" % h)
        # the rows held the original keys at their positions
        pos = torch.tensor([p for p, _, _ in sel], device="cuda")
        assert torch.equal(k_before[pgs, sls], ks[0, 1][pos, h])
        touched[pgs, sls] = True
    # everything else in the K pool (other sequence, other layer, rows outside
    # [lo, hi), empty slots) is bit-identical
    assert torch.equal(k_after[~touched], k_before[~touched])


def test_single_head_round_trip_and_attention():
    gpu_ready()
    d, P, n = 128, 16, 300
    cache = _cache(d, P, n + 64, 200, seqs=1)
    pols = [[W.HeadPolicy(G), W.HeadPolicy(L, 4, 40), W.HeadPolicy(G)]] * 2
    cache.set_policy(0, to_c_policies(pols))
    k = W.normal((n, 3, d), 21, device="cuda")
    v = W.normal((n, 3, d), 22, device="cuda")
    cache.build(0, 0, k, v)
    torch.cuda.synchronize()
    k0 = cache.k_pool().clone()
    # one head only, then back: within two bf16 roundings of the start
    cache.rope_realign(0, [0], 777, kv_head=2)
    torch.cuda.synchronize()
    ids2, _ = cache.export_table(0, 0, 2)
    others = torch.ones(k0.shape[0], dtype=torch.bool, device="cuda")
    others[torch.tensor(ids2, device="cuda")] = False
    assert torch.equal(cache.k_pool()[others], k0[others]), "other heads must not change"
    cache.rope_realign(0, [0], -777, kv_head=2)
    torch.cuda.synchronize()
    rows = [pg for pg in ids2]
    back, start = f64(cache.k_pool()[rows]), f64(k0[rows])
    # two bf16 roundings of a norm-preserving rotation: within two ulps of the pair norm
    assert np.all(np.abs(back - start) <= 2 * ULP * _pair_norm(start) + 2.0 ** -40)
    # attention after moving every key of head 0 by delta equals the oracle
    # over keys rotated by the oracle (prefill of one new row at position n)
    delta = 4321
    cache2 = _cache(d, P, n + 64, 200, seqs=1)
    cache2.set_policy(0, to_c_policies(pols))
    cache2.build(0, 0, k, v)
    cache2.rope_realign(0, [0], delta)
    q = W.normal((1, 6, d), 23, device="cuda")
    kn = W.normal((1, 3, d), 24, device="cuda")
    vn = W.normal((1, 3, d), 25, device="cuda")
    out, lse = cache2.prefill(0, [0], [0, 1], q, kn, vn)
    k_rot = rope.realign(f64(k), delta)
    # the kernel reads the bf16-rounded rotated keys
    k_rot_bf16 = torch.tensor(k_rot, dtype=torch.float64).to(torch.bfloat16).to(torch.float64).numpy()
    kk = np.concatenate([k_rot_bf16, f64(kn)], axis=0)
    vv = np.concatenate([f64(v), f64(vn)], axis=0)
    ref, lref = oracle.attend(f64(q), kk, vv, np.array([n]), [pol_tuple(p) for p in pols[0]], "f64")
    compare(out, ref, lse, lref, "attention over realigned keys")
    assert cache2.status() == 0


def test_bad_arguments_rejected():
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError
    cache = _cache(64, 16, 128, 64, seqs=1)
    cache.set_policy(0, to_c_policies([[W.HeadPolicy(G)] * 3] * 2))
    for kw in ({"kv_head": 3}, {"kv_head": -2}, {"pos_lo": 5, "pos_hi": 4}, {"rope_theta": 0.0},
               {"rope_theta": -1.0}):
        with pytest.raises(SegPagedError):
            cache.rope_realign(0, [0], 5, **kw)
    with pytest.raises(SegPagedError):
        cache.rope_realign(0, [0], 1 << 41)
    with pytest.raises(SegPagedError):
        cache.rope_realign(0, [0, 0], 5)
    cache.rope_realign(0, [0], 0)          # no-op
    assert cache.status() == 0
