"""GPU: the ragged mixed-policy serving batch at full size.

8 sequences with lengths log-uniform in [2048, 65536], Hq 32 / Hkv 8, d 128,
page 64; per (layer, KV head) 15 % GLOBAL, 70 % LOCAL(4, 4096), 15 %
RETRIEVAL (top-2048 indices from seeded scores).  Schedule (the reading of
the unstated interleaving): every step prefills one 4096-token chunk of the
lowest-index sequence still prefilling, then decodes one token for every
sequence whose prefill is done; after all prefills, 16 more decode steps.
All 32 layers are run, each with its own policy rows; at every step the
oracle checks sampled prefill rows and decode rows of two layers, taken in
turn, so every layer is checked at several steps.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _gpu_common import compare, f64, gpu_ready, ncores, pol_tuple, to_c_policies

pytestmark = pytest.mark.gpu


def test_ragged_mixed_serving_batch():
    gpu_ready()
    from head_aware_paged_gb300 import Config, SegPagedCache
    wl = W.WORKLOADS["ragged_mixed"]
    layers = wl.layers
    lens = W.seq_lengths(wl)
    B, chunk, extra = wl.seqs, wl.chunk, wl.decode_steps
    n_dec_max = sum(-(-L // chunk) for L in lens) + extra + 4
    max_len = max(lens) + n_dec_max
    pols = [W.policies(wl, seq=b, length=lens[b])[:layers] for b in range(B)]
    pages = 0
    for b in range(B):
        for row in pols[b]:
            for p in row:
                pages += (max_len + wl.page - 1) // wl.page + 2 if p.kind != W.LOCAL else \
                    (p.sink + wl.page - 1) // wl.page + p.window // wl.page + 2
    cache = SegPagedCache(Config(num_layers=layers, num_q_heads=wl.hq, num_kv_heads=wl.hkv,
                                 head_dim=wl.d, page_size=wl.page, max_seqs=B,
                                 max_seq_len=max_len, num_pages=pages + 64,
                                 max_idx_per_seq=layers * wl.hkv * wl.retrieval_topk,
                                 max_tokens=chunk + B, max_batch=B))
    for b in range(B):
        cache.set_policy(b, to_c_policies(pols[b]))
    # the whole token stream of every (sequence, layer): prompt then decode tokens
    total = [lens[b] + n_dec_max for b in range(B)]
    K = {(b, l): W.normal((total[b], wl.hkv, wl.d), W.tensor_seed(7, "k", b, l), 1.0, "cuda")
         for b in range(B) for l in range(layers)}
    V = {(b, l): W.normal((total[b], wl.hkv, wl.d), W.tensor_seed(7, "v", b, l), 1.0, "cuda")
         for b in range(B) for l in range(layers)}
    Q = {(b, l): W.normal((total[b], wl.hq, wl.d), W.tensor_seed(7, "q", b, l), 1.0, "cuda")
         for b in range(B) for l in range(layers)}
    held = [0] * B
    rng = np.random.default_rng(3)
    checked = 0

    from oracle import rows as orows

    def check_rows(b, l, rows, got, lse):
        nonlocal checked
        e = int(rows.max()) + 1
        pt = [pol_tuple(p) for p in pols[b][l]]
        k32 = K[(b, l)][:e].float().cpu().numpy()
        v32 = V[(b, l)][:e].float().cpu().numpy()
        q32 = Q[(b, l)][torch.as_tensor(rows, device="cuda")].float().cpu().numpy()
        ref, lref = orows.attend_rows(q32, k32, v32, rows, pt)
        compare(got, ref, lse, lref, "seq %d layer %d rows %s" % (b, l, rows[:3]))
        checked += 1

    torch.set_num_threads(ncores())
    seen = set()
    step = 0
    while any(held[b] < lens[b] for b in range(B)) or extra > 0:
        watch = {(2 * step) % layers, (2 * step + 1) % layers}   # layers checked this step
        pre = [b for b in range(B) if held[b] < lens[b]]
        dec = [b for b in range(B) if held[b] >= lens[b]]
        if pre:
            b = pre[0]
            c = min(chunk, lens[b] - held[b])
            n0 = held[b]
            for l in range(layers):
                qc = Q[(b, l)][n0:n0 + c].contiguous()
                kc = K[(b, l)][n0:n0 + c].contiguous()
                vc = V[(b, l)][n0:n0 + c].contiguous()
                out, lse = cache.prefill(l, [b], [0, c], qc, kc, vc)
                if l in watch:
                    sel = np.unique(np.concatenate([[0, c - 1], rng.integers(0, c, 4)]))
                    ts = torch.as_tensor(sel, device="cuda")
                    check_rows(b, l, n0 + sel, out[ts], lse[ts])
                    seen.add(l)
                cache.append_kv(l, [b], [0, c], kc, vc)
            held[b] += c
        if dec:
            for l in range(layers):
                kd = torch.stack([K[(b, l)][held[b]] for b in dec]).contiguous()
                vd = torch.stack([V[(b, l)][held[b]] for b in dec]).contiguous()
                qd = torch.stack([Q[(b, l)][held[b]] for b in dec]).contiguous()
                cache.append_kv(l, dec, list(range(len(dec) + 1)), kd, vd)
                out, lse = cache.decode(l, dec, qd)
                if l in watch:
                    for n, b in enumerate(dec[:3]):
                        check_rows(b, l, np.array([held[b]]), out[n:n + 1], lse[n:n + 1])
            for b in dec:
                held[b] += 1
        if not pre:
            extra -= 1
        step += 1
    assert cache.status() == 0
    assert checked > 40
    assert seen == set(range(layers))
