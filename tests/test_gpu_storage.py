"""GPU: page-pool allocator, page tables and KV scatter/trim, bit-exact against
the oracle's page model (through the C ABI)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import pagemodel as pm
from oracle import accounting
from _gpu_common import gpu_ready, pol_tuple, to_c_policies

pytestmark = pytest.mark.gpu

G, L, R = W.GLOBAL, W.LOCAL, W.RETRIEVAL


def _mk(layers, hq, hkv, d, P, max_seqs, max_len, num_pages, max_batch=8, max_idx=4096):
    from head_aware_paged_gb300 import Config, SegPagedCache
    cfg = Config(num_layers=layers, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=P,
                 max_seqs=max_seqs, max_seq_len=max_len, num_pages=num_pages,
                 max_idx_per_seq=max_idx, max_tokens=max_len, max_batch=max_batch)
    return SegPagedCache(cfg)


def _check_tables(cache, model, seq, layer, hkv, kpool, vpool, dense_k, dense_v):
    """Page ids and slot positions bit-exact; stored rows equal the dense rows."""
    for h in range(hkv):
        ids, pos = cache.export_table(seq, layer, h)
        mids, mpos = model.table(seq, layer, h)
        assert ids == mids, (seq, layer, h)
        assert pos == mpos, (seq, layer, h)
        for pid, slots in zip(ids, pos):
            s = np.array(slots)
            live = np.nonzero(s >= 0)[0]
            if live.size == 0:
                continue
            got_k = kpool[pid, live]
            got_v = vpool[pid, live]
            src = torch.as_tensor(s[live], device=dense_k.device)
            assert torch.equal(got_k, dense_k[src, h]), (seq, layer, h, pid)
            assert torch.equal(got_v, dense_v[src, h]), (seq, layer, h, pid)


def test_tiny_build_tables_bit_exact():
    gpu_ready()
    wl = W.WORKLOADS["tiny"]
    cache = _mk(1, wl.hq, wl.hkv, wl.d, wl.page, 2, 512, 64)
    pols = W.policies(wl)
    cache.set_policy(0, to_c_policies(pols))
    _, k, v = W.qkv(wl, 256, 0, 0, device="cuda")
    cache.build(0, 0, k, v)
    model = pm.CacheModel(1, wl.hkv, wl.page, 64)
    model.set_policy(0, [[pol_tuple(p) for p in row] for row in pols])
    model.build(0, 0, 256)
    torch.cuda.synchronize()
    assert cache.status() == 0
    _check_tables(cache, model, 0, 0, wl.hkv, cache.k_pool(), cache.v_pool(), k, v)
    # GLOBAL 16 pages, LOCAL(4, 32) 1 + 3 pages
    assert len(cache.export_table(0, 0, 0)[0]) == 16
    assert len(cache.export_table(0, 0, 1)[0]) == 4
    assert cache.free_pages() == 64 - 20


def _mixed_policies(layers, hkv, P, max_len, rng):
    pols = []
    for l in range(layers):
        row = []
        for h in range(hkv):
            kind = (l * hkv + h) % 3
            if kind == G:
                row.append(W.HeadPolicy(G))
            elif kind == L:
                row.append(W.HeadPolicy(L, int(rng.integers(0, 70)), int(rng.integers(1, 300))))
            else:
                idx = np.sort(rng.choice(max_len, int(rng.integers(0, 200)), replace=False))
                row.append(W.HeadPolicy(R, idx=idx.astype(np.int32)))
        pols.append(row)
    return pols


@pytest.mark.parametrize("P,d", [(16, 64), (64, 128), (32, 128), (128, 64)])
def test_ragged_appends_match_model(P, d):
    """Several sequences, mixed classes, ragged chunk sizes, release and reuse."""
    gpu_ready()
    rng = np.random.default_rng(P + d)
    layers, hq, hkv, max_len, npages = 2, 9, 3, 1200, 2000
    cache = _mk(layers, hq, hkv, d, P, 4, max_len, npages)
    model = pm.CacheModel(layers, hkv, P, npages)
    dense = {}
    for seq in range(3):
        pols = _mixed_policies(layers, hkv, P, max_len, rng)
        cache.set_policy(seq, to_c_policies(pols))
        model.set_policy(seq, [[pol_tuple(p) for p in row] for row in pols])
        for l in range(layers):
            dense[(seq, l)] = (W.normal((max_len, hkv, d), 1000 + seq * 10 + l, device="cuda"),
                               W.normal((max_len, hkv, d), 2000 + seq * 10 + l, device="cuda"))
    held = {(s, l): 0 for s in range(3) for l in range(layers)}
    for step in range(6):
        for l in range(layers):
            seqs = [s for s in range(3) if rng.random() < 0.8]
            if not seqs:
                continue
            counts = [int(rng.choice([1, 7, 63, 64, 65, 130, 257])) for _ in seqs]
            counts = [min(c, max_len - held[(s, l)]) for s, c in zip(seqs, counts)]
            cu = np.concatenate([[0], np.cumsum(counts)]).astype(int)
            kk = torch.cat([dense[(s, l)][0][held[(s, l)]:held[(s, l)] + c] for s, c in zip(seqs, counts)])
            vv = torch.cat([dense[(s, l)][1][held[(s, l)]:held[(s, l)] + c] for s, c in zip(seqs, counts)])
            cache.append_kv(l, seqs, cu.tolist(), kk.contiguous(), vv.contiguous())
            model.append(l, seqs, counts)
            for s, c in zip(seqs, counts):
                held[(s, l)] += c
        torch.cuda.synchronize()
        assert cache.status() == 0
        assert cache.free_pages() == model.pool.free
        for s in range(3):
            for l in range(layers):
                assert cache.seq_len(s, l) == held[(s, l)]
                _check_tables(cache, model, s, l, hkv, cache.k_pool(), cache.v_pool(),
                              dense[(s, l)][0], dense[(s, l)][1])
        if step == 3:
            cache.release(1)
            model.release(1)
            for l in range(layers):
                held[(1, l)] = 0
            assert cache.free_pages() == model.pool.free


def test_out_of_pages_leaves_state_unchanged():
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError
    cache = _mk(1, 4, 1, 64, 16, 2, 4096, 12)
    cache.set_policy(0, [[(G, 0, 0, None)]])
    k = W.normal((200, 1, 64), 5, device="cuda")
    cache.append_kv(0, [0], [0, 150], k[:150].contiguous(), k[:150].contiguous())
    free = cache.free_pages()
    with pytest.raises(SegPagedError) as ei:
        cache.append_kv(0, [0], [0, 50], k[150:].contiguous(), k[150:].contiguous())
    assert ei.value.status == 2
    assert cache.free_pages() == free and cache.seq_len(0, 0) == 150
    # a LOCAL head's pages stop growing: its 2 ring pages fit where GLOBAL did not
    cache.set_policy(1, [[(L, 0, 8, None)]])
    for _ in range(5):
        cache.append_kv(0, [1], [0, 150], k[:150].contiguous(), k[:150].contiguous())
    assert cache.seq_len(1, 0) == 750
    assert cache.status() == 0


def test_bad_arguments_rejected_before_launch():
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError
    cache = _mk(1, 4, 2, 64, 16, 2, 256, 64)
    with pytest.raises(SegPagedError):          # no policy yet
        cache.append_kv(0, [0], [0, 1], torch.zeros(1, 2, 64, dtype=torch.bfloat16, device="cuda"),
                        torch.zeros(1, 2, 64, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(SegPagedError):          # descending retrieval list
        cache.set_policy(0, [[(R, 0, 0, [5, 3]), (G, 0, 0, None)]])
    with pytest.raises(SegPagedError):          # window 0
        cache.set_policy(0, [[(L, 4, 0, None), (G, 0, 0, None)]])
    with pytest.raises(SegPagedError):          # unknown class
        cache.set_policy(0, [[(9, 0, 0, None), (G, 0, 0, None)]])
    cache.set_policy(0, [[(G, 0, 0, None), (L, 2, 8, None)]])
    z = torch.zeros(4, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(SegPagedError):          # duplicate sequence in one call
        cache.append_kv(0, [0, 0], [0, 2, 4], z, z)
    with pytest.raises(SegPagedError):          # sequence id out of range
        cache.append_kv(0, [5], [0, 4], z, z)
    with pytest.raises(SegPagedError):          # decode before any token
        cache.decode(0, [0], torch.zeros(1, 4, 64, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(SegPagedError):          # past max_seq_len
        big = torch.zeros(300, 2, 64, dtype=torch.bfloat16, device="cuda")
        cache.append_kv(0, [0], [0, 300], big, big)
    assert cache.free_pages() == 64 and cache.status() == 0


def test_visible_counts_bit_exact():
    """Decode-view and prefill-view |V(i)| from the device equal the oracle's."""
    gpu_ready()
    rng = np.random.default_rng(3)
    P, d, hkv = 16, 64, 3
    cache = _mk(1, 6, hkv, d, P, 2, 2048, 600)
    idx = np.sort(rng.choice(1500, 300, replace=False)).astype(np.int32)
    pols = [[W.HeadPolicy(G), W.HeadPolicy(L, 5, 37), W.HeadPolicy(R, idx=idx)]]
    cache.set_policy(0, to_c_policies(pols))
    kv = W.normal((1500, hkv, d), 9, device="cuda")
    held = 0
    for c in (1, 40, 333, 126):
        cache.append_kv(0, [0], [0, c], kv[held:held + c].contiguous(), kv[held:held + c].contiguous())
        held += c
        for h, p in enumerate(pols[0]):
            pt = pol_tuple(p)
            positions = [held - 1] + list(range(held, held + 300, 7))
            got = cache.visible_count(0, 0, h, positions)
            want = [accounting.vis_count(*pt, i) for i in positions]
            assert got == want, (c, h)
    assert cache.status() == 0
