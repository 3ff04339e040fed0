"""GPU: split-KV decode against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _gpu_common import compare, f64, gpu_ready, ncores, pol_tuple, to_c_policies

pytestmark = pytest.mark.gpu

G, L, R = W.GLOBAL, W.LOCAL, W.RETRIEVAL


def _mk(layers, hq, hkv, d, P, max_seqs, max_len, num_pages, max_batch=8, max_idx=8192):
    from head_aware_paged_gb300 import Config, SegPagedCache
    cfg = Config(num_layers=layers, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=P,
                 max_seqs=max_seqs, max_seq_len=max_len, num_pages=num_pages,
                 max_idx_per_seq=max_idx, max_tokens=max_len, max_batch=max_batch)
    return SegPagedCache(cfg)


def test_tiny_decode_steps():
    """Tiny case: build 256 tokens, then 4 steps of append-one + decode."""
    gpu_ready()
    wl = W.WORKLOADS["tiny"]
    cache = _mk(1, wl.hq, wl.hkv, wl.d, wl.page, 1, 512, 64)
    pols = W.policies(wl)
    cache.set_policy(0, to_c_policies(pols))
    _, k, v = W.qkv(wl, 256 + wl.decode_steps, 0, 0, device="cuda")
    cache.build(0, 0, k[:256], v[:256])
    pt = [pol_tuple(p) for p in pols[0]]
    for step in range(wl.decode_steps):
        t = 256 + step
        cache.append_kv(0, [0], [0, 1], k[t:t + 1].contiguous(), v[t:t + 1].contiguous())
        q = W.normal((1, wl.hq, wl.d), 77 + step, device="cuda")
        out, lse = cache.decode(0, [0], q)
        ref, lref = oracle.attend(f64(q), f64(k[:t + 1]), f64(v[:t + 1]), [t], pt, "f64")
        compare(out, ref, lse, lref, "tiny decode step %d" % step)
    assert cache.status() == 0


@pytest.mark.parametrize("P,d,hq,hkv", [(64, 128, 32, 8), (16, 64, 8, 2), (128, 128, 16, 2),
                                        (32, 128, 24, 8), (64, 64, 16, 16)])
def test_decode_mixed_classes_ragged_batch(P, d, hq, hkv):
    gpu_ready()
    rng = np.random.default_rng(P * 7 + d + hq)
    B, max_len = 5, 3000
    lens = [int(x) for x in rng.integers(1, max_len, size=B)]
    lens[0] = 1
    cache = _mk(1, hq, hkv, d, P, B, max_len, B * hkv * (max_len // P + 2), max_batch=B)
    kvs, pols = [], []
    for b in range(B):
        row = []
        for h in range(hkv):
            kind = int(rng.integers(0, 3))
            if kind == G:
                row.append(W.HeadPolicy(G))
            elif kind == L:
                row.append(W.HeadPolicy(L, int(rng.integers(0, 9)), int(rng.integers(1, 700))))
            else:
                idx = np.sort(rng.choice(max_len, int(rng.integers(0, 400)), replace=False))
                row.append(W.HeadPolicy(R, idx=idx.astype(np.int32)))
        pols.append([row])
        cache.set_policy(b, to_c_policies([row]))
        k = W.normal((lens[b], hkv, d), 10 * b + 1, 0.5, device="cuda")
        v = W.normal((lens[b], hkv, d), 10 * b + 2, device="cuda")
        kvs.append((k, v))
        cache.build(b, 0, k, v)
    q = W.normal((B, hq, d), 99, device="cuda")
    out, lse = cache.decode(0, list(range(B)), q)
    for b in range(B):
        pt = [pol_tuple(p) for p in pols[b][0]]
        t = lens[b] - 1
        ref, lref = oracle.attend(f64(q[b:b + 1]), f64(kvs[b][0]), f64(kvs[b][1]), [t], pt, "f64",
                                  threads=ncores())
        compare(out[b:b + 1], ref, lse[b:b + 1], lref, "seq %d" % b)
    assert cache.status() == 0


def test_decode_repeat_is_stable():
    """Split partials and tickets reset between calls: two identical calls agree."""
    gpu_ready()
    cache = _mk(1, 32, 8, 128, 64, 4, 20000, 4 * 8 * 320, max_batch=4)
    for b in range(4):
        cache.set_policy(b, [[(G, 0, 0, None)] * 8])
        k = W.normal((19000 - 3000 * b, 8, 128), b + 5, device="cuda")
        cache.build(b, 0, k, k)
    q = W.normal((4, 32, 128), 3, device="cuda")
    o1, l1 = cache.decode(0, [0, 1, 2, 3], q)
    o1b, l1b = cache.decode(0, [0, 1, 2, 3], q)
    # same call, same split partition, fixed merge order: bitwise identical
    assert torch.equal(o1, o1b) and torch.equal(l1, l1b)
    # another sequence order splits the pages differently: equal within rounding
    o2, l2 = cache.decode(0, [3, 1, 2, 0], q[[3, 1, 2, 0]].contiguous())
    assert (o1[[3, 1, 2, 0]].float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1[[3, 1, 2, 0]] - l2).abs().max().item() <= 1e-4
    assert cache.status() == 0


def test_decode_llama3_8b_shape_64_steps_all_layers():
    """Llama-3-8B-shaped decode batch as the benchmark runs it: 32 layers x
    32 sequences of 32,768 cached tokens (12.5 % GLOBAL units, LOCAL(4,
    2048)), 64 decode steps of one token per sequence in every layer, so
    GLOBAL units cross a page boundary (position 32,768) and LOCAL rings
    turn over a page.  The oracle checks sequences 0 and 31 in every layer
    at steps 0 and 63."""
    gpu_ready()
    wl = W.WORKLOADS["llama3_8b_decode_32k"]
    layers, B, n, steps = wl.layers, wl.seqs, wl.seq_len, wl.decode_steps
    pols = W.policies(wl)
    pages = B * sum(pm_pages(p, n + steps, wl.page) for row in pols for p in row) + 64
    cache = _mk(layers, wl.hq, wl.hkv, wl.d, wl.page, B, n + steps + 8, pages, max_batch=B)
    watched = (0, B - 1)
    full = {}                       # (b, l) -> whole K / V token streams of watched sequences
    new_k = [[None] * B for _ in range(layers)]
    new_v = [[None] * B for _ in range(layers)]
    for b in range(B):
        cache.set_policy(b, to_c_policies(pols))
    for l in range(layers):
        for b in range(B):
            k = W.normal((n + steps, wl.hkv, wl.d), W.tensor_seed(3, "k", b, l), device="cuda")
            v = W.normal((n + steps, wl.hkv, wl.d), W.tensor_seed(3, "v", b, l), device="cuda")
            cache.build(b, l, k[:n], v[:n])
            new_k[l][b], new_v[l][b] = k[n:].clone(), v[n:].clone()
            if b in watched:
                full[(b, l)] = (k, v)
            del k, v
    torch.cuda.synchronize()
    assert cache.status() == 0
    seqs = list(range(B))
    cu = list(range(B + 1))
    kept = {}
    for step in range(steps):
        for l in range(layers):
            kd = torch.stack([new_k[l][b][step] for b in seqs]).contiguous()
            vd = torch.stack([new_v[l][b][step] for b in seqs]).contiguous()
            cache.append_kv(l, seqs, cu, kd, vd)
            q = W.normal((B, wl.hq, wl.d), W.tensor_seed(3, "q", l, step), device="cuda")
            out, lse = cache.decode(l, seqs, q)
            if step in (0, steps - 1):
                kept[(l, step)] = (q[list(watched)].clone(), out[list(watched)].clone(),
                                   lse[list(watched)].clone())
    torch.cuda.synchronize()
    assert cache.status() == 0
    for l in range(layers):
        pt = [pol_tuple(p) for p in pols[l]]
        for j, b in enumerate(watched):
            k, v = full[(b, l)]
            k64, v64 = f64(k), f64(v)
            for step in (0, steps - 1):
                q, out, lse = kept[(l, step)]
                t = n + step
                ref, lref = oracle.attend(f64(q[j:j + 1]), k64[:t + 1], v64[:t + 1], [t], pt, "f64",
                                          threads=ncores())
                compare(out[j:j + 1], ref, lse[j:j + 1], lref,
                        "layer %d seq %d step %d" % (l, b, step))


def pm_pages(p, n, P):
    from oracle import pagemodel
    return pagemodel.pages_needed(p.kind, p.sink, p.window,
                                  None if p.idx is None else p.idx.tolist(), n, P)
