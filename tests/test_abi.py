"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from head_aware_paged_gb300 import build
    build.build()
    from head_aware_paged_gb300 import _lib
    return _lib.load()


def _declared():
    with open(os.path.join(ROOT, "include", "segpaged.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"\b(sp_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    from head_aware_paged_gb300._lib import EXPORTS
    declared = _declared()
    assert sorted(EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def _cfg(**kw):
    from head_aware_paged_gb300 import Config
    base = dict(num_layers=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64,
                max_seqs=4, max_seq_len=4096, num_pages=512, max_idx_per_seq=256,
                max_tokens=4096, max_batch=4)
    base.update(kw)
    return Config(**base)


def test_required_bytes(lib):
    from head_aware_paged_gb300 import sp_required_bytes
    pool, meta, ws = sp_required_bytes(_cfg())
    assert pool == 2 * 512 * 64 * 128 * 2
    assert meta > 0 and ws > 0
    pool2, _, _ = sp_required_bytes(_cfg(num_pages=1024))
    assert pool2 == 2 * pool


@pytest.mark.parametrize("bad", [dict(head_dim=96), dict(page_size=48), dict(num_q_heads=7),
                                 dict(num_q_heads=64, num_kv_heads=2), dict(num_layers=0),
                                 dict(max_batch=1000), dict(num_pages=0)])
def test_bad_config_rejected(lib, bad):
    from head_aware_paged_gb300 import SegPagedError, sp_required_bytes
    with pytest.raises(SegPagedError) as ei:
        sp_required_bytes(_cfg(**bad))
    assert ei.value.status in (1, 3)


def test_create_rejects_null_and_misaligned_buffers(lib):
    from head_aware_paged_gb300._lib import SpConfig
    cfg = _cfg().to_c()
    h = ctypes.c_void_p()
    rc = lib.sp_cache_create(ctypes.byref(cfg), None, None, None, ctypes.byref(h))
    assert rc == 1 and b"null" in lib.sp_last_error()
    rc = lib.sp_cache_create(ctypes.byref(cfg), ctypes.c_void_p(4096 + 16), ctypes.c_void_p(8192),
                             ctypes.c_void_p(16384), ctypes.byref(h))
    assert rc == 1 and b"aligned" in lib.sp_last_error()
    assert not h.value


def test_null_handle_calls_fail_cleanly(lib):
    from head_aware_paged_gb300._lib import i32_array
    assert lib.sp_cache_destroy(None) == 1
    assert lib.sp_release_seq(None, 0, None) == 1
    assert lib.sp_attention_decode(None, 0, i32_array([0]), 1, None, None, None, None) == 1
    n = ctypes.c_int32()
    assert lib.sp_free_pages(None, ctypes.byref(n)) == 1
