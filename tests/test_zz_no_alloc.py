"""GPU: the allocation-free decode entry point.

sp_attention_decode_static_scratch serves callers that cannot allocate device
memory when they decode (a plain C host with no device allocator, or a
serving loop that must not call cudaMalloc mid-step): its split scratch is a
fixed device array inside the library.  Its output must match the regular
sp_attention_decode on the same cache, on two calls in a row (the array keeps
the previous call's contents, so the second call checks that what must start
at zero is cleared), and calls beyond the array's limit must be refused
before any launch.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu_common import ATOL, gpu_ready, to_c_policies

pytestmark = pytest.mark.gpu

G, L, R = W.GLOBAL, W.LOCAL, W.RETRIEVAL


def _cache(hq, hkv, d, P, B, max_len, pages, max_batch):
    from head_aware_paged_gb300 import Config, SegPagedCache
    return SegPagedCache(Config(num_layers=1, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                page_size=P, max_seqs=B, max_seq_len=max_len, num_pages=pages,
                                max_idx_per_seq=4096, max_tokens=max_len, max_batch=max_batch))


def test_static_scratch_decode_matches_regular_decode_twice():
    gpu_ready()
    from head_aware_paged_gb300 import sp_attention_decode_static_scratch
    rng = np.random.default_rng(21)
    B, hq, hkv, d, P, n_max = 6, 32, 8, 128, 64, 9000
    cache = _cache(hq, hkv, d, P, B, n_max + 8, B * hkv * (n_max // P + 3), B)
    for b in range(B):
        row = []
        for h in range(hkv):
            kind = (b + h) % 3
            if kind == G:
                row.append(W.HeadPolicy(G))
            elif kind == L:
                row.append(W.HeadPolicy(L, 4, int(rng.integers(16, 2048))))
            else:
                idx = np.sort(rng.choice(n_max, 700, replace=False)).astype(np.int32)
                row.append(W.HeadPolicy(R, idx=idx))
        cache.set_policy(b, to_c_policies([row]))
        n = int(rng.integers(2000, n_max))
        k = W.normal((n, hkv, d), 40 + b, device="cuda")
        v = W.normal((n, hkv, d), 60 + b, device="cuda")
        cache.build(b, 0, k, v)
    seqs = list(range(B))
    q = W.normal((B, hq, d), 5, device="cuda")
    ref, lref = cache.decode(0, seqs, q)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
        sp_attention_decode_static_scratch(cache.handle, 0, seqs, q, out, lse)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all(), call
        assert (out.float() - ref.float()).abs().max().item() <= ATOL, call
        assert (lse - lref).abs().max().item() <= 2e-3, call
    assert cache.status() == 0


def test_static_scratch_refuses_calls_beyond_its_limit():
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError, sp_attention_decode_static_scratch
    # 64 sequences x 8 KV heads, 16 query heads per KV head, d 128: the split
    # scratch would exceed the 4 MiB array
    B, hq, hkv, d, P = 64, 128, 8, 128, 16
    cache = _cache(hq, hkv, d, P, B, 64, B * hkv * 2, B)
    pol = [[W.HeadPolicy(G)] * hkv]
    k = W.normal((1, hkv, d), 1, device="cuda")
    for b in range(B):
        cache.set_policy(b, to_c_policies(pol))
        cache.build(b, 0, k, k)
    q = W.normal((B, hq, d), 2, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(SegPagedError) as ei:
        sp_attention_decode_static_scratch(cache.handle, 0, list(range(B)), q, out)
    assert ei.value.status == 3 and "scratch" in str(ei.value)
    # the regular entry point handles the same call
    ref, _ = cache.decode(0, list(range(B)), q)
    assert torch.isfinite(ref.float()).all()
    assert cache.status() == 0
