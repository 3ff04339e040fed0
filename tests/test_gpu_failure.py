"""GPU: the bounded waits that every kernel of the library uses, exercised
without a fault or a hang (sp_selftest_bounded_wait): a wait that nothing
completes gives up after its cycle limit, the status word reports
SP_ERR_TIMEOUT, and the context keeps computing correct attention."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _gpu_common import compare, f64, gpu_ready, pol_tuple, to_c_policies

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_recovers():
    gpu_ready()
    from head_aware_paged_gb300 import Config, SegPagedCache, SegPagedError, sp_selftest_bounded_wait
    d, P, n = 64, 16, 300
    cache = SegPagedCache(Config(num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=d, page_size=P,
                                 max_seqs=1, max_seq_len=n + 16, num_pages=64, max_tokens=n + 16,
                                 max_batch=1))
    pols = [W.HeadPolicy(W.GLOBAL), W.HeadPolicy(W.LOCAL, 4, 40)]
    cache.set_policy(0, to_c_policies([pols]))
    # a wait that is completed: no flag
    sp_selftest_bounded_wait(cache.handle, 2_000_000, 1)
    assert cache.status() == 0
    # a wait that nothing completes: gives up after ~1 ms of cycles
    t0 = time.time()
    sp_selftest_bounded_wait(cache.handle, 2_000_000, 0)
    with pytest.raises(SegPagedError, match="SP_ERR_TIMEOUT"):
        cache.status()
    assert time.time() - t0 < 10
    assert cache.status() == 0                 # the read cleared the flag
    # two warps that must leave together, one of whose waits never completes
    # (the FP8 converter pair's pattern): both leave, the kernel returns
    t0 = time.time()
    sp_selftest_bounded_wait(cache.handle, 2_000_000, 2)
    with pytest.raises(SegPagedError, match="SP_ERR_TIMEOUT"):
        cache.status()
    assert time.time() - t0 < 10
    assert cache.status() == 0
    # the same context still computes attention correctly
    k = W.normal((n, 2, d), 1, device="cuda")
    v = W.normal((n, 2, d), 2, device="cuda")
    cache.build(0, 0, k[: n - 1].contiguous(), v[: n - 1].contiguous())
    cache.append_kv(0, [0], [0, 1], k[n - 1:].contiguous(), v[n - 1:].contiguous())
    q = W.normal((1, 4, d), 3, device="cuda")
    out, lse = cache.decode(0, [0], q)
    ref, lref = oracle.attend(f64(q), f64(k), f64(v), [n - 1], [pol_tuple(p) for p in pols], "f64")
    compare(out, ref, lse, lref, "decode after a timed-out wait")
    assert cache.status() == 0
    # arguments outside the documented range are refused before any launch
    for limit, mode in ((10, 0), (2_000_000, 3), (2_000_000, -1), (3_000_000_000, 0)):
        with pytest.raises(SegPagedError):
            sp_selftest_bounded_wait(cache.handle, limit, mode)
    assert cache.status() == 0
