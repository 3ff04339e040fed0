"""GPU: the allocation-free decode entry point.

sp_attention_decode_static_scratch serves callers that cannot allocate device
memory when they decode (a plain C host with no device allocator, or a
serving loop that must not call cudaMalloc mid-step): its split scratch is a
fixed device array inside the library.  It runs the same decode launch as
sp_attention_decode with only the scratch's address changed, so on the same
cache its output and LSE must be bitwise equal to the regular entry point's,
and both must match the CPU oracle, on two calls in a row (the array keeps
the previous call's contents between calls); bf16 and FP8 pages.  Calls
beyond the array's limit must be refused before any launch.  This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import fp8
from _gpu_common import compare, f64, gpu_ready, ncores, pol_tuple, to_c_policies

pytestmark = pytest.mark.gpu

G, L, R = W.GLOBAL, W.LOCAL, W.RETRIEVAL


def _cache(hq, hkv, d, P, B, max_len, pages, max_batch, kv_dtype=0):
    from head_aware_paged_gb300 import Config, SegPagedCache
    return SegPagedCache(Config(num_layers=1, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                page_size=P, max_seqs=B, max_seq_len=max_len, num_pages=pages,
                                max_idx_per_seq=4096, max_tokens=max_len, max_batch=max_batch,
                                kv_dtype=kv_dtype))


def _dq(x, s):
    """The oracle's dequantised rows of x [n, hkv, d] under scales [hkv, d]."""
    xs = f64(x)
    out = np.empty_like(xs)
    for h in range(xs.shape[1]):
        out[:, h] = fp8.dequantize(fp8.quantize(xs[:, h], s[h]), s[h])
    return out


@pytest.mark.parametrize("kv_dtype", [0, 1], ids=["bf16", "fp8"])
def test_static_scratch_decode_matches_regular_decode_and_oracle_twice(kv_dtype):
    gpu_ready()
    from head_aware_paged_gb300 import sp_attention_decode_static_scratch
    rng = np.random.default_rng(21 + kv_dtype)
    B, hq, hkv, d, P, n_max = 6, 32, 8, 128, 64, 9000
    cache = _cache(hq, hkv, d, P, B, n_max + 8, B * hkv * (n_max // P + 3), B, kv_dtype)
    data, pols, lens = [], [], []
    for b in range(B):
        n = int(rng.integers(2000, n_max))
        data.append((W.normal((n, hkv, d), 40 + b, device="cuda"),
                     W.normal((n, hkv, d), 60 + b, device="cuda")))
        lens.append(n)
    if kv_dtype:
        # one scale per (KV head, channel): absmax over all rows / 448
        ks = np.clip(torch.cat([k for k, _ in data]).float().abs().amax(0).cpu().numpy() / 448.0,
                     2.0 ** -14, 128.0).astype(np.float32)
        vs = np.clip(torch.cat([v for _, v in data]).float().abs().amax(0).cpu().numpy() / 448.0,
                     2.0 ** -14, 128.0).astype(np.float32)
        cache.set_kv_scales(0, ks, vs)
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
        pols.append(row)
        cache.set_policy(b, to_c_policies([row]))
        cache.build(b, 0, *data[b])
    seqs = list(range(B))
    q = W.normal((B, hq, d), 5, device="cuda")
    ref, lref = cache.decode(0, seqs, q)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
        sp_attention_decode_static_scratch(cache.handle, 0, seqs, q, out, lse)
        torch.cuda.synchronize()
        # the same launch with another scratch address: bit for bit the same
        assert torch.equal(out, ref), call
        assert torch.equal(lse, lref), call
        for b in range(B):
            k, v = data[b]
            kk, vv = (_dq(k, ks), _dq(v, vs)) if kv_dtype else (f64(k), f64(v))
            o_ref, l_ref = oracle.attend(f64(q[b:b + 1]), kk, vv, [lens[b] - 1],
                                         [pol_tuple(p) for p in pols[b]], "f64", threads=ncores())
            compare(out[b:b + 1], o_ref, lse[b:b + 1], l_ref,
                    "static-scratch decode, call %d, seq %d" % (call, b))
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
    # argument errors are the regular entry point's, also before any launch
    with pytest.raises(SegPagedError, match="listed twice"):
        sp_attention_decode_static_scratch(cache.handle, 0, [0, 0], q[:2].contiguous(), out[:2])
    # the regular entry point handles the over-limit call
    ref, _ = cache.decode(0, list(range(B)), q)
    assert torch.isfinite(ref.float()).all()
    assert cache.status() == 0
