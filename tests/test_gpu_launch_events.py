"""GPU: the launch-event hook (sp_set_launch_events) times a call's kernels
and leaves the results unchanged."""
import pytest
import torch

import workloads as W
from _gpu_common import gpu_ready, to_c_policies

pytestmark = pytest.mark.gpu


def _cache_with_history(n):
    from head_aware_paged_gb300 import Config, SegPagedCache
    wl = W.WORKLOADS["tiny"]
    cfg = Config(num_layers=1, num_q_heads=wl.hq, num_kv_heads=wl.hkv, head_dim=wl.d,
                 page_size=wl.page, max_seqs=1, max_seq_len=2 * n + 64,
                 num_pages=wl.hkv * (2 * n // wl.page + 8), max_idx_per_seq=2 * n,
                 max_tokens=2 * n, max_batch=1)
    cache = SegPagedCache(cfg)
    cache.set_policy(0, to_c_policies(W.policies(wl)))
    q, k, v = W.qkv(wl, n, 0, 0, device="cuda")
    return wl, cache, q, k, v


def _timing_events():
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for e in evs:
        e.record()          # creates the CUDA event behind the torch object
    torch.cuda.synchronize()
    return evs


def test_prefill_and_decode_kernel_intervals():
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError
    wl, cache, q, k, v = _cache_with_history(1024)
    ref_out, ref_lse = cache.prefill(0, [0], [0, 1024], q, k, v)
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()

    s, e = _timing_events()
    outer = _timing_events()
    cache.set_launch_events(s, e)
    outer[0].record()
    out, lse = cache.prefill(0, [0], [0, 1024], q, k, v)
    outer[1].record()
    torch.cuda.synchronize()
    inner_ms, outer_ms = s.elapsed_time(e), outer[0].elapsed_time(outer[1])
    assert 0.0 < inner_ms <= outer_ms + 1e-3
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)

    # disarmed after one call: a second call leaves the pair where it was
    cache.prefill(0, [0], [0, 1024], q, k, v)
    torch.cuda.synchronize()
    assert s.elapsed_time(e) == inner_ms

    # decode: the same hook times the decode kernel
    cache.append_kv(0, [0], [0, 1024], k, v)
    q1 = W.normal((1, wl.hq, wl.d), 5, device="cuda")
    ref1, _ = cache.decode(0, [0], q1)
    ref1 = ref1.clone()
    cache.set_launch_events(s, e)
    out1, _ = cache.decode(0, [0], q1)
    torch.cuda.synchronize()
    assert s.elapsed_time(e) > 0.0
    assert torch.equal(out1, ref1)

    # both or neither
    with pytest.raises(SegPagedError):
        cache.set_launch_events(s, None)
    cache.set_launch_events()              # disarm
    with pytest.raises(ValueError):
        cache.set_launch_events(torch.cuda.Event(enable_timing=True), e)
    assert cache.status() == 0
