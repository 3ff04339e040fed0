"""GPU: tcgen05 prefill against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _gpu_common import compare, f64, gpu_ready, ncores, pol_tuple, to_c_policies

pytestmark = pytest.mark.gpu

G, L, R = W.GLOBAL, W.LOCAL, W.RETRIEVAL


def _mk(layers, hq, hkv, d, P, max_seqs, max_len, num_pages, max_batch=8, max_idx=8192,
        max_tokens=None):
    from head_aware_paged_gb300 import Config, SegPagedCache
    cfg = Config(num_layers=layers, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=P,
                 max_seqs=max_seqs, max_seq_len=max_len, num_pages=num_pages,
                 max_idx_per_seq=max_idx, max_tokens=max_tokens or max_len, max_batch=max_batch)
    return SegPagedCache(cfg)


def test_tiny_prefill_then_decode():
    """Tiny case end to end: 256-row causal prefill, append, 4 decode steps."""
    gpu_ready()
    wl = W.WORKLOADS["tiny"]
    cache = _mk(1, wl.hq, wl.hkv, wl.d, wl.page, 1, 512, 64)
    pols = W.policies(wl)
    pt = [pol_tuple(p) for p in pols[0]]
    cache.set_policy(0, to_c_policies(pols))
    q, k, v = W.qkv(wl, 256 + 4, 0, 0, device="cuda")
    out, lse = cache.prefill(0, [0], [0, 256], q[:256].contiguous(), k[:256].contiguous(),
                             v[:256].contiguous())
    ref, lref = oracle.attend(f64(q[:256]), f64(k[:256]), f64(v[:256]), np.arange(256), pt, "f64")
    compare(out, ref, lse, lref, "tiny prefill")
    cache.append_kv(0, [0], [0, 256], k[:256].contiguous(), v[:256].contiguous())
    for step in range(4):
        t = 256 + step
        cache.append_kv(0, [0], [0, 1], k[t:t + 1].contiguous(), v[t:t + 1].contiguous())
        o, l_ = cache.decode(0, [0], q[t:t + 1].contiguous())
        r, lr = oracle.attend(f64(q[t:t + 1]), f64(k[:t + 1]), f64(v[:t + 1]), [t], pt, "f64")
        compare(o, r, l_, lr, "tiny decode %d" % step)
    assert cache.status() == 0


def test_mistral7b_shape_one_shot():
    """Mistral-7B-shaped layer: Hq 32 / Hkv 8, d 128, L 8192, P 64, 1 GLOBAL +
    7 LOCAL(4, 1024); oracle on every 5th row plus the first and last 128."""
    gpu_ready()
    wl = W.WORKLOADS["mistral7b_prefill_8k"]
    Lq = wl.seq_len
    cache = _mk(1, wl.hq, wl.hkv, wl.d, wl.page, 1, Lq, 400)
    pols = W.policies(wl)
    cache.set_policy(0, to_c_policies(pols))
    q, k, v = W.qkv(wl, Lq, 0, 0, device="cuda")
    out, lse = cache.prefill(0, [0], [0, Lq], q, k, v)
    rows = np.unique(np.concatenate([np.arange(0, Lq, 5), np.arange(128), np.arange(Lq - 128, Lq)]))
    pt = [pol_tuple(p) for p in pols[0]]
    ref, lref = oracle.attend(f64(q[rows]), f64(k), f64(v), rows, pt, "f64", threads=ncores())
    compare(out[rows], ref, lse[rows], lref, "mistral one-shot")
    assert cache.status() == 0


def _rand_policies(hkv, max_len, rng, sink_hi=9, win_hi=700, idx_hi=500):
    row = []
    for h in range(hkv):
        kind = h % 3 if hkv >= 3 else int(rng.integers(0, 3))
        if kind == G:
            row.append(W.HeadPolicy(G))
        elif kind == L:
            row.append(W.HeadPolicy(L, int(rng.integers(0, sink_hi)), int(rng.integers(1, win_hi))))
        else:
            idx = np.sort(rng.choice(max_len, int(rng.integers(0, idx_hi)), replace=False))
            row.append(W.HeadPolicy(R, idx=idx.astype(np.int32)))
    return row


@pytest.mark.parametrize("P,d,hq,hkv", [(64, 128, 16, 4), (16, 64, 8, 4), (128, 128, 12, 3),
                                        (32, 64, 6, 3),
                                        # odd GQA groups (one query tile per item) and the
                                        # remaining (head_dim, page size) kernel instances
                                        (16, 128, 6, 2), (32, 128, 8, 8), (64, 64, 4, 2),
                                        (128, 64, 9, 3)])
def test_chunked_ragged_prefill_with_history(P, d, hq, hkv):
    """Several sequences prefilled in ragged chunks (history from pages, the
    rest from the chunk), mixed classes incl. RETRIEVAL, then decode; every
    chunk's output against the oracle; chunked equals one-shot."""
    gpu_ready()
    rng = np.random.default_rng(P + 3 * d + hq)
    B, max_len = 3, 1700
    lens = [1700, 901, 333]
    cache = _mk(1, hq, hkv, d, P, B, max_len + 16, B * hkv * (max_len // P + 3), max_batch=B)
    oneshot = _mk(1, hq, hkv, d, P, B, max_len, B * hkv * (max_len // P + 3), max_batch=B,
                  max_tokens=B * max_len)
    pols, data = [], []
    for b in range(B):
        row = _rand_policies(hkv, max_len, rng)
        pols.append(row)
        cache.set_policy(b, to_c_policies([row]))
        oneshot.set_policy(b, to_c_policies([row]))
        data.append((W.normal((lens[b], hq, d), 100 + b, device="cuda"),
                     W.normal((lens[b], hkv, d), 200 + b, 0.5, device="cuda"),
                     W.normal((lens[b], hkv, d), 300 + b, device="cuda")))
    outs = [torch.zeros(lens[b], hq, d, dtype=torch.bfloat16, device="cuda") for b in range(B)]
    held = [0] * B
    chunk_sizes = [1, 77, 128, 129, 300, 511, 64, 2000]
    step = 0
    while any(held[b] < lens[b] for b in range(B)):
        seqs = [b for b in range(B) if held[b] < lens[b]]
        counts = [min(chunk_sizes[(step + b) % len(chunk_sizes)], lens[b] - held[b]) for b in seqs]
        cu = [0] + list(np.cumsum(counts))
        qc = torch.cat([data[b][0][held[b]:held[b] + c] for b, c in zip(seqs, counts)]).contiguous()
        kc = torch.cat([data[b][1][held[b]:held[b] + c] for b, c in zip(seqs, counts)]).contiguous()
        vc = torch.cat([data[b][2][held[b]:held[b] + c] for b, c in zip(seqs, counts)]).contiguous()
        o, lse = cache.prefill(0, seqs, cu, qc, kc, vc)
        for n, (b, c) in enumerate(zip(seqs, counts)):
            rows = np.arange(held[b], held[b] + c)
            pt = [pol_tuple(p) for p in pols[b]]
            e = held[b] + c
            ref, lref = oracle.attend(f64(data[b][0][held[b]:e]), f64(data[b][1][:e]),
                                      f64(data[b][2][:e]), rows, pt, "f64", threads=ncores())
            compare(o[cu[n]:cu[n + 1]], ref, lse[cu[n]:cu[n + 1]], lref,
                    "step %d seq %d rows %d..%d" % (step, b, held[b], e))
            outs[b][held[b]:e] = o[cu[n]:cu[n + 1]]
        cache.append_kv(0, seqs, cu, kc, vc)
        for b, c in zip(seqs, counts):
            held[b] += c
        step += 1
    # chunking invariance against a one-shot prefill of the whole sequences
    cu = [0] + list(np.cumsum(lens))
    o1, _ = oneshot.prefill(0, list(range(B)), cu, torch.cat([x[0] for x in data]).contiguous(),
                            torch.cat([x[1] for x in data]).contiguous(),
                            torch.cat([x[2] for x in data]).contiguous())
    for b in range(B):
        diff = (o1[cu[b]:cu[b + 1]].float() - outs[b].float()).abs().max().item()
        assert diff <= 2e-2, (b, diff)
    # decode after the chunked prefill
    for b in range(B):
        kn = W.normal((1, hkv, d), 400 + b, device="cuda")
        cache.append_kv(0, [b], [0, 1], kn, kn)
    qd = W.normal((B, hq, d), 500, device="cuda")
    od, ld = cache.decode(0, list(range(B)), qd)
    for b in range(B):
        kn = W.normal((1, hkv, d), 400 + b, device="cuda")
        kk = torch.cat([data[b][1], kn])
        vv = torch.cat([data[b][2], kn])
        pt = [pol_tuple(p) for p in pols[b]]
        ref, lref = oracle.attend(f64(qd[b:b + 1]), f64(kk), f64(vv), [lens[b]], pt, "f64")
        compare(od[b:b + 1], ref, ld[b:b + 1], lref, "decode after chunks, seq %d" % b)
    assert cache.status() == 0 and oneshot.status() == 0


@pytest.mark.parametrize("P,d,hq,hkv", [(64, 128, 8, 4), (16, 64, 6, 3)])
def test_long_history_short_chunks_split_items(P, d, hq, hkv):
    """A few query rows over a long history: every work item is far longer
    than a CTA's share of the call, so the planner splits each along its key
    tiles into pieces (up to eight, of at least six tiles) whose partial
    results the merge kernel combines.  GLOBAL, LOCAL (a ring tile can hold
    nothing a row sees, so a piece may leave a row empty) and RETRIEVAL heads;
    chunks of 1, 128 and 200 rows; every row against the oracle."""
    gpu_ready()
    rng = np.random.default_rng(5 + d)
    n_hist, max_len = 9000, 9400
    pols = []
    for h in range(hkv):
        kind = h % 3
        if kind == G:
            pols.append(W.HeadPolicy(G))
        elif kind == L:
            pols.append(W.HeadPolicy(L, 4, 3000))
        else:
            idx = np.sort(rng.choice(np.arange(40, max_len), 1500, replace=False)).astype(np.int32)
            pols.append(W.HeadPolicy(R, idx=idx))
    cache = _mk(1, hq, hkv, d, P, 1, max_len + 16, hkv * (max_len // P + 4), max_batch=1,
                max_tokens=max_len)
    cache.set_policy(0, to_c_policies([pols]))
    q = W.normal((max_len, hq, d), 31, device="cuda")
    k = W.normal((max_len, hkv, d), 32, 0.5, device="cuda")
    v = W.normal((max_len, hkv, d), 33, device="cuda")
    cache.build(0, 0, k[:n_hist].contiguous(), v[:n_hist].contiguous())
    pt = [pol_tuple(p) for p in pols]
    held = n_hist
    for c in (1, 128, 200):
        sl = slice(held, held + c)
        o, lse = cache.prefill(0, [0], [0, c], q[sl].contiguous(), k[sl].contiguous(),
                               v[sl].contiguous())
        ref, lref = oracle.attend(f64(q[sl]), f64(k[:held + c]), f64(v[:held + c]),
                                  np.arange(held, held + c), pt, "f64", threads=ncores())
        compare(o, ref, lse, lref, "split items, chunk of %d at %d" % (c, held))
        cache.append_kv(0, [0], [0, c], k[sl].contiguous(), v[sl].contiguous())
        held += c
    assert cache.status() == 0


def test_edge_cases():
    """One-row chunks, rows with no visible key (RETRIEVAL before its first
    index: O = 0, LSE = -inf), sink larger than a tile, window 1, odd group."""
    gpu_ready()
    d, P = 64, 16
    cache = _mk(1, 3, 3, d, P, 2, 600, 600, max_batch=2)
    pols = [W.HeadPolicy(R, idx=np.array([50, 51, 300], np.int32)),
            W.HeadPolicy(L, 150, 1), W.HeadPolicy(L, 0, 1)]
    cache.set_policy(0, to_c_policies([pols]))
    n = 400
    q = W.normal((n, 3, d), 1, device="cuda")
    k = W.normal((n, 3, d), 2, device="cuda")
    v = W.normal((n, 3, d), 3, device="cuda")
    pt = [pol_tuple(p) for p in pols]
    held = 0
    for c in (1, 1, 60, 1, 200, 137):
        o, lse = cache.prefill(0, [0], [0, c], q[held:held + c].contiguous(),
                               k[held:held + c].contiguous(), v[held:held + c].contiguous())
        ref, lref = oracle.attend(f64(q[held:held + c]), f64(k[:held + c]), f64(v[:held + c]),
                                  np.arange(held, held + c), pt, "f64")
        compare(o, ref, lse, lref, "edge chunk at %d" % held)
        cache.append_kv(0, [0], [0, c], k[held:held + c].contiguous(), v[held:held + c].contiguous())
        held += c
    assert cache.status() == 0


def test_prefill_rejects_out_not_32_byte_aligned():
    """out is written with 32-byte vector stores: a 16-byte offset is refused
    before anything is launched, and the aligned call still works."""
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError
    d, P = 64, 16
    cache = _mk(1, 2, 1, d, P, 1, 128, 64)
    cache.set_policy(0, to_c_policies([[W.HeadPolicy(G)]]))
    n = 32
    q = W.normal((n, 2, d), 4, device="cuda")
    k = W.normal((n, 1, d), 5, device="cuda")
    v = W.normal((n, 1, d), 6, device="cuda")
    buf = torch.empty(n * 2 * d + 16, dtype=torch.bfloat16, device="cuda")
    assert buf.data_ptr() % 32 == 0
    bad = buf[8:8 + n * 2 * d].view(n, 2, d)          # 16 bytes past a 32-byte boundary
    with pytest.raises(SegPagedError, match="32-byte"):
        cache.prefill(0, [0], [0, n], q, k, v, bad)
    o, lse = cache.prefill(0, [0], [0, n], q, k, v)
    ref, lref = oracle.attend(f64(q), f64(k), f64(v), np.arange(n), [pol_tuple(W.HeadPolicy(G))], "f64")
    compare(o, ref, lse, lref, "aligned out after a refused call")
    assert cache.status() == 0


def _unit_pages(p, n, P):
    from oracle import pagemodel
    return pagemodel.pages_needed(p.kind, p.sink, p.window,
                                  None if p.idx is None else [int(x) for x in p.idx], n, P)


def test_llama33_70b_shape_all_layers_sampled():
    """Llama-3.3-70B-shaped long prefill as the benchmark runs it: all 64
    layers, each with its own policy row (77 of the 512 (layer, KV head)
    units GLOBAL by seed, the rest LOCAL(4, 8192)) and its own Q/K/V,
    Hq 64 / Hkv 8, d 128, one sequence of 131,072 tokens prefilled as one
    chunk per layer and then written to the cache.  256 sampled query rows
    of every query head of every layer (the first and last rows and the
    window edges among them) are checked against the row-sampled oracle."""
    gpu_ready()
    from oracle import rows as orows
    wl = W.WORKLOADS["llama33_70b_prefill_128k"]
    Lq, n_rows = wl.seq_len, 256
    pols = W.policies(wl)
    pages = sum(_unit_pages(p, Lq, wl.page) for row in pols for p in row) + 64
    cache = _mk(wl.layers, wl.hq, wl.hkv, wl.d, wl.page, 1, Lq + 64, pages, max_batch=1,
                max_idx=1, max_tokens=Lq)
    cache.set_policy(0, to_c_policies(pols))
    out = torch.empty(Lq, wl.hq, wl.d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(Lq, wl.hq, dtype=torch.float32, device="cuda")
    rng = np.random.default_rng(11)
    fixed = np.array([0, 1, 127, 128, 8191, 8192, 8195, Lq - 129, Lq - 1])
    torch.set_num_threads(ncores())
    for l in range(wl.layers):
        q, k, v = W.qkv(wl, Lq, 0, l, device="cuda")
        cache.prefill(l, [0], [0, Lq], q, k, v, out, lse)
        cache.append_kv(l, [0], [0, Lq], k, v)
        rest = np.setdiff1d(np.arange(Lq), fixed)
        rows = np.sort(np.concatenate([fixed, rng.choice(rest, n_rows - len(fixed), replace=False)]))
        ts = torch.as_tensor(rows, device="cuda")
        pt = [pol_tuple(p) for p in pols[l]]
        ref, lref = orows.attend_rows(q[ts].float().cpu().numpy(), k.float().cpu().numpy(),
                                      v.float().cpu().numpy(), rows, pt)
        compare(out[ts], ref, lse[ts], lref, "llama-70B-shaped layer %d" % l)
        del q, k, v
    assert cache.status() == 0
    cache.release(0)
    assert cache.status() == 0


def test_work_list_in_parameters_or_uploaded_gives_identical_rows():
    """A call whose work list fits the kernel parameters (one 8192-row
    sequence, Hq 32 / Hkv 8: 1024 items) and a call that uploads it (the same
    sequence batched with a second one: 2048 items) compute every item the
    same way, whichever CTA runs it: the first sequence's rows are bitwise
    equal, and sampled rows of both match the oracle."""
    gpu_ready()
    wl = W.WORKLOADS["mistral7b_prefill_8k"]
    Lq = wl.seq_len
    pols = W.policies(wl)
    cache = _mk(1, wl.hq, wl.hkv, wl.d, wl.page, 2, Lq, 800, max_tokens=2 * Lq)
    cache.set_policy(0, to_c_policies(pols))
    cache.set_policy(1, to_c_policies(pols))
    q, k, v = W.qkv(wl, 2 * Lq, 0, 0, device="cuda")
    alone, lse_a = cache.prefill(0, [0], [0, Lq], q[:Lq].contiguous(), k[:Lq].contiguous(),
                                 v[:Lq].contiguous())
    both, lse_b = cache.prefill(0, [0, 1], [0, Lq, 2 * Lq], q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(alone, both[:Lq]) and torch.equal(lse_a, lse_b[:Lq])
    pt = [pol_tuple(p) for p in pols[0]]
    rows = np.array([0, 1, 127, 128, 1000, 4095, 4096, Lq - 1])
    for b in range(2):
        kb, vb = f64(k[b * Lq:(b + 1) * Lq]), f64(v[b * Lq:(b + 1) * Lq])
        ref, lref = oracle.attend(f64(q[b * Lq + rows]), kb, vb, rows, pt, "f64", threads=ncores())
        compare(both[b * Lq + rows], ref, lse_b[b * Lq + rows], lref, "batched sequence %d" % b)
    assert cache.status() == 0
