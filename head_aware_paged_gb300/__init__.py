"""head_aware_paged_gb300 -- head-aware paged KV cache and mask-free attention
for one GB300 GPU.

Thin Python binding over libsegpaged.so (include/segpaged.h).  The functions
below carry the C-ABI names and only marshal arguments: torch tensors are
passed as device pointers together with torch's current CUDA stream; torch
supplies device memory and streams, the library's kernels do all the work.

    cache = SegPagedCache(cfg)                        # allocates pool/meta/ws
    cache.set_policy(seq, policies)                   # [layers][kv_heads]
    out, lse = cache.prefill(layer, [seq], [0, T], q, k, v)
    cache.append_kv(layer, [seq], [0, T], k, v)
    cache.append_kv(layer, [seq], [0, 1], k1, v1)
    out, lse = cache.decode(layer, [seq], q1)
"""
from __future__ import annotations

import ctypes
from ctypes import byref, c_int32, c_int64, c_size_t, c_void_p
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from ._lib import (EXPORTS, GLOBAL, KV_BF16, KV_FP8, LOCAL, RETRIEVAL, SegPagedError, SpConfig, SpHeadPolicy,
                   check, i32_array, i64_array, load)

__all__ = ["Config", "Policy", "SegPagedCache", "SegPagedError", "GLOBAL", "LOCAL",
           "RETRIEVAL", "KV_BF16", "KV_FP8", "load", "EXPORTS"] + list(EXPORTS)


@dataclass
class Config:
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    max_seqs: int
    max_seq_len: int
    num_pages: int
    max_idx_per_seq: int = 0
    max_tokens: int = 8192
    max_batch: int = 1
    kv_dtype: int = 0          # KV_BF16, or KV_FP8 (e4m3 pages with per-channel scales)

    def to_c(self) -> SpConfig:
        return SpConfig(self.num_layers, self.num_q_heads, self.num_kv_heads, self.head_dim,
                        self.page_size, self.max_seqs, self.max_seq_len, self.num_pages,
                        self.max_idx_per_seq, self.max_tokens, self.max_batch, self.kv_dtype)


@dataclass
class Policy:
    kind: int
    sink: int = 0
    window: int = 0
    idx: Optional[Sequence[int]] = None


def _stream(stream=None) -> c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: Optional[torch.Tensor]) -> c_void_p:
    return c_void_p(0 if t is None else t.data_ptr())


# ---------------------------------------------------------------- C-ABI names

def sp_required_bytes(cfg: Config):
    lib = load()
    a, b, c = c_size_t(), c_size_t(), c_size_t()
    check(lib.sp_required_bytes(byref(cfg.to_c()), byref(a), byref(b), byref(c)))
    return a.value, b.value, c.value


def sp_cache_create(cfg: Config, pool: torch.Tensor, meta: torch.Tensor, ws: torch.Tensor):
    lib = load()
    h = c_void_p()
    check(lib.sp_cache_create(byref(cfg.to_c()), _ptr(pool), _ptr(meta), _ptr(ws), byref(h)))
    return h


def sp_cache_destroy(handle) -> None:
    check(load().sp_cache_destroy(handle))


def _policy_array(policies: Sequence[Policy]):
    arr = (SpHeadPolicy * len(policies))()
    keep = []
    for n, p in enumerate(policies):
        idx = list(p.idx) if p.idx is not None else []
        buf = i32_array(idx)
        keep.append(buf)
        arr[n] = SpHeadPolicy(p.kind, p.sink, p.window, len(idx),
                              ctypes.cast(buf, ctypes.POINTER(c_int32)))
    return arr, keep


def sp_set_policy(handle, seq: int, policies: Sequence[Policy], stream=None) -> None:
    arr, keep = _policy_array(policies)
    check(load().sp_set_policy(handle, seq, arr, _stream(stream)))
    del keep


def sp_build_cache(handle, seq: int, layer: int, k: torch.Tensor, v: torch.Tensor,
                   n_tokens: int, row_stride: int, stream=None) -> None:
    check(load().sp_build_cache(handle, seq, layer, _ptr(k), _ptr(v), n_tokens, row_stride,
                                _stream(stream)))


def sp_append_kv(handle, layer: int, seq_ids: Sequence[int], cu_new: Sequence[int],
                 k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
    check(load().sp_append_kv(handle, layer, i32_array(seq_ids), len(seq_ids),
                              i32_array(cu_new), _ptr(k), _ptr(v), _stream(stream)))


def sp_attention_prefill(handle, layer: int, seq_ids: Sequence[int], cu_q: Sequence[int],
                         q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                         lse: Optional[torch.Tensor] = None, stream=None) -> None:
    check(load().sp_attention_prefill(handle, layer, i32_array(seq_ids), len(seq_ids),
                                      i32_array(cu_q), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                      _ptr(lse), _stream(stream)))


def sp_attention_decode(handle, layer: int, seq_ids: Sequence[int], q: torch.Tensor,
                        out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    check(load().sp_attention_decode(handle, layer, i32_array(seq_ids), len(seq_ids), _ptr(q),
                                     _ptr(out), _ptr(lse), _stream(stream)))


def sp_attention_decode_static_scratch(handle, layer: int, seq_ids: Sequence[int],
                                       q: torch.Tensor, out: torch.Tensor,
                                       lse: Optional[torch.Tensor] = None, stream=None) -> None:
    """Decode whose split scratch is the library's built-in device array, for
    callers that cannot allocate device memory when they decode (see the C
    header for the 4 MiB limit and the sharing rules)."""
    check(load().sp_attention_decode_static_scratch(handle, layer, i32_array(seq_ids),
                                                    len(seq_ids), _ptr(q), _ptr(out), _ptr(lse),
                                                    _stream(stream)))


def sp_rope_realign(handle, layer: int, seq_ids: Sequence[int], kv_head: int, pos_lo: int,
                    pos_hi: int, delta: int, rope_theta: float = 10000.0, stream=None) -> None:
    check(load().sp_rope_realign(handle, layer, i32_array(seq_ids), len(seq_ids), kv_head,
                                 pos_lo, pos_hi, delta, float(rope_theta), _stream(stream)))


def sp_pack_seq(handle, seq: int, dst: Optional[torch.Tensor], stream=None) -> int:
    """Pack `seq` into dst (a 256-byte aligned device buffer); with dst None
    only return the packed size in bytes."""
    n = c_size_t()
    nbytes = 0 if dst is None else dst.numel() * dst.element_size()
    check(load().sp_pack_seq(handle, seq, _ptr(dst), nbytes, byref(n), _stream(stream)))
    return n.value


def sp_unpack_seq(handle, seq: int, src: torch.Tensor, stream=None) -> None:
    check(load().sp_unpack_seq(handle, seq, _ptr(src), src.numel() * src.element_size(),
                               _stream(stream)))


def sp_select_heavy_hitters(q_obs: torch.Tensor, k: torch.Tensor, topk: int, recent: int = 0,
                            want_scores: bool = False, stream=None):
    """Heavy-hitter retrieval selection on dense q_obs [n_obs, Hq, d] and k
    [n, Hkv, d] (bf16, on the device).  Returns (idx [Hkv, topk + recent]
    int32 padded with -1, counts [Hkv] int32, scores [Hkv, n] fp32 or None)."""
    n_obs, hq, d = q_obs.shape
    n, hkv, _ = k.shape
    nbytes = c_size_t()
    check(load().sp_select_workspace_bytes(n_obs, n, hq, hkv, byref(nbytes)))
    ws = torch.empty(nbytes.value + 256, dtype=torch.uint8, device=k.device)
    off = (-ws.data_ptr()) % 256
    idx = torch.empty(hkv, topk + recent, dtype=torch.int32, device=k.device)
    counts = torch.empty(hkv, dtype=torch.int32, device=k.device)
    scores = torch.empty(hkv, n, dtype=torch.float32, device=k.device) if want_scores else None
    check(load().sp_select_heavy_hitters(
        _ptr(q_obs), n_obs, _ptr(k), n, hq, hkv, d, topk, recent,
        ctypes.cast(idx.data_ptr(), ctypes.POINTER(c_int32)),
        ctypes.cast(counts.data_ptr(), ctypes.POINTER(c_int32)),
        _ptr(scores), c_void_p(ws.data_ptr() + off), nbytes.value, _stream(stream)))
    return idx, counts, scores


def sp_select_heavy_hitters_top_p(q_obs: torch.Tensor, k: torch.Tensor, top_p: float,
                                  max_keys: int, recent: int = 0, want_scores: bool = False,
                                  stream=None):
    """The top-p form of the selection: per KV head the shortest prefix of
    the ranked candidates whose summed score reaches top_p of their total, at
    most max_keys, then the recent window.  Returns (idx [Hkv, max_keys +
    recent] int32 padded with -1, counts [Hkv] int32, scores or None)."""
    n_obs, hq, d = q_obs.shape
    n, hkv, _ = k.shape
    nbytes = c_size_t()
    check(load().sp_select_workspace_bytes(n_obs, n, hq, hkv, byref(nbytes)))
    ws = torch.empty(nbytes.value + 256, dtype=torch.uint8, device=k.device)
    off = (-ws.data_ptr()) % 256
    idx = torch.empty(hkv, max_keys + recent, dtype=torch.int32, device=k.device)
    counts = torch.empty(hkv, dtype=torch.int32, device=k.device)
    scores = torch.empty(hkv, n, dtype=torch.float32, device=k.device) if want_scores else None
    check(load().sp_select_heavy_hitters_top_p(
        _ptr(q_obs), n_obs, _ptr(k), n, hq, hkv, d, float(top_p), max_keys, recent,
        ctypes.cast(idx.data_ptr(), ctypes.POINTER(c_int32)),
        ctypes.cast(counts.data_ptr(), ctypes.POINTER(c_int32)),
        _ptr(scores), c_void_p(ws.data_ptr() + off), nbytes.value, _stream(stream)))
    return idx, counts, scores


def sp_set_kv_scales(handle, layer: int, k_scale, v_scale, stream=None) -> None:
    """Per-channel FP8 scales of one layer: host float arrays [Hkv][d]."""
    ks = np.ascontiguousarray(np.asarray(k_scale, dtype=np.float32).reshape(-1))
    vs = np.ascontiguousarray(np.asarray(v_scale, dtype=np.float32).reshape(-1))
    fp = ctypes.POINTER(ctypes.c_float)
    check(load().sp_set_kv_scales(handle, layer, ks.ctypes.data_as(fp), vs.ctypes.data_as(fp),
                                  _stream(stream)))


def sp_release_seq(handle, seq: int, stream=None) -> None:
    check(load().sp_release_seq(handle, seq, _stream(stream)))


def sp_export_table(handle, seq: int, layer: int, kv_head: int, cap: int, page_size: int,
                    stream=None):
    np_ = c_int32()
    ids = (c_int32 * max(cap, 1))()
    pos = (c_int32 * max(cap * page_size, 1))()
    check(load().sp_export_table(handle, seq, layer, kv_head, byref(np_), ids, pos, cap,
                                 _stream(stream)))
    n = np_.value
    return list(ids[:n]), [list(pos[j * page_size:(j + 1) * page_size]) for j in range(n)]


def sp_visible_count(handle, seq: int, layer: int, kv_head: int, positions: Sequence[int],
                     stream=None) -> List[int]:
    out = (c_int32 * max(1, len(positions)))()
    check(load().sp_visible_count(handle, seq, layer, kv_head, i64_array(positions),
                                  len(positions), out, _stream(stream)))
    return list(out[:len(positions)])


def sp_seq_len(handle, seq: int, layer: int) -> int:
    n = c_int32()
    check(load().sp_seq_len(handle, seq, layer, byref(n)))
    return n.value


def sp_free_pages(handle) -> int:
    n = c_int32()
    check(load().sp_free_pages(handle, byref(n)))
    return n.value


def sp_count_prefill_pairs(handle, seq: int, layer: int, n0: int, c: int) -> int:
    r = c_int64()
    check(load().sp_count_prefill_pairs(handle, seq, layer, n0, c, byref(r)))
    return r.value


def sp_count_decode_bytes(handle, layer: int, seq_ids: Sequence[int], t: Sequence[int]) -> int:
    r = c_int64()
    check(load().sp_count_decode_bytes(handle, layer, i32_array(seq_ids), len(seq_ids),
                                       i64_array(t), byref(r)))
    return r.value


def sp_get_status(handle, stream=None) -> int:
    w = c_int32()
    check(load().sp_get_status(handle, _stream(stream), byref(w)))
    return w.value


def sp_selftest_bounded_wait(handle, limit_cycles: int, mode: int, stream=None) -> None:
    """Launch the bounded-wait self-test (mode 0: the wait gives up and the
    next status read reports SP_ERR_TIMEOUT; mode 1: the wait completes;
    mode 2: two warps, one wait completes and one gives up, both leave
    together and the status reports SP_ERR_TIMEOUT)."""
    check(load().sp_selftest_bounded_wait(handle, limit_cycles, mode, _stream(stream)))


def sp_set_launch_events(handle, start=None, end=None) -> None:
    """Arm two torch.cuda.Event objects for the next attention call on the
    cache: it records `start` right before its first kernel and `end` right
    after its last (see the C header); no events disarm.  Each event must
    have been recorded once already, so that its CUDA event exists."""
    def raw(e):
        if e is None:
            return c_void_p(0)
        h = int(e.cuda_event)
        if h == 0:
            raise ValueError("record the event once before arming it")
        return c_void_p(h)
    check(load().sp_set_launch_events(handle, raw(start), raw(end)))


def sp_last_error() -> str:
    return load().sp_last_error().decode(errors="replace")


# ------------------------------------------------------------ convenience class

class SegPagedCache:
    """Owns the three device buffers (torch tensors) and the library handle."""

    def __init__(self, cfg: Config, device: str = "cuda"):
        self.cfg = cfg
        self.device = device
        pool_b, meta_b, ws_b = sp_required_bytes(cfg)
        # 1024-byte alignment: torch's caching allocator returns 512-byte
        # aligned blocks, so over-allocate and offset.
        self._pool_raw, self.pool = self._aligned(pool_b, device)
        self._meta_raw, self.meta = self._aligned(meta_b, device)
        self._ws_raw, self.ws = self._aligned(ws_b, device)
        self.handle = sp_cache_create(cfg, self.pool, self.meta, self.ws)

    @staticmethod
    def _aligned(nbytes: int, device: str):
        raw = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device)
        off = (-raw.data_ptr()) % 1024
        return raw, raw[off:off + nbytes]

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            sp_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # views of the page pool: [num_pages, page_size, head_dim] bf16 each
    def k_pool(self) -> torch.Tensor:
        """K pages [num_pages][page_size][head_dim]: bf16, or uint8 e4m3 codes."""
        c = self.cfg
        half = c.num_pages * c.page_size * c.head_dim
        dt = torch.uint8 if c.kv_dtype == KV_FP8 else torch.bfloat16
        return self.pool.view(dt)[:half].view(c.num_pages, c.page_size, c.head_dim)

    def v_pool(self) -> torch.Tensor:
        c = self.cfg
        half = c.num_pages * c.page_size * c.head_dim
        dt = torch.uint8 if c.kv_dtype == KV_FP8 else torch.bfloat16
        return self.pool.view(dt)[half:2 * half].view(c.num_pages, c.page_size, c.head_dim)

    def set_policy(self, seq: int, policies, stream=None) -> None:
        flat = []
        for row in policies:
            for p in row:
                flat.append(p if isinstance(p, Policy) else Policy(*p))
        sp_set_policy(self.handle, seq, flat, stream)

    def build(self, seq: int, layer: int, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
        assert k.dtype == torch.bfloat16 and k.is_cuda and k.stride(-1) == 1
        n = k.shape[0]
        sp_build_cache(self.handle, seq, layer, k, v, n, k.stride(0), stream)

    def append_kv(self, layer: int, seq_ids, cu_new, k, v, stream=None) -> None:
        assert k.is_contiguous() and v.is_contiguous()
        sp_append_kv(self.handle, layer, seq_ids, cu_new, k, v, stream)

    def prefill(self, layer: int, seq_ids, cu_q, q, k, v, out=None, lse=None, want_lse=True,
                stream=None):
        assert q.is_contiguous() and k.is_contiguous() and v.is_contiguous()
        if out is None:
            out = torch.empty_like(q)
        if lse is None and want_lse:
            lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
        sp_attention_prefill(self.handle, layer, seq_ids, cu_q, q, k, v, out, lse, stream)
        return out, lse

    def decode(self, layer: int, seq_ids, q, out=None, lse=None, want_lse=True, stream=None):
        assert q.is_contiguous()
        if out is None:
            out = torch.empty_like(q)
        if lse is None and want_lse:
            lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
        sp_attention_decode(self.handle, layer, seq_ids, q, out, lse, stream)
        return out, lse

    def rope_realign(self, layer: int, seq_ids, delta: int, kv_head: int = -1, pos_lo: int = 0,
                     pos_hi: int = 1 << 62, rope_theta: float = 10000.0, stream=None) -> None:
        """Rotate the stored K rows at positions [pos_lo, pos_hi) by `delta`
        positions of rotary embedding (see sp_rope_realign in the C header)."""
        sp_rope_realign(self.handle, layer, seq_ids, kv_head, pos_lo, pos_hi, delta, rope_theta,
                        stream)

    def pack(self, seq: int, stream=None) -> torch.Tensor:
        """The packed transfer form of `seq` (header + trimmed rows) in a new
        uint8 device tensor."""
        n = sp_pack_seq(self.handle, seq, None)
        _, buf = self._aligned(n, self.device)     # the view keeps its storage alive
        sp_pack_seq(self.handle, seq, buf, stream)
        return buf

    def unpack(self, seq: int, buf: torch.Tensor, stream=None) -> None:
        """Restore a packed sequence into the empty slot `seq`."""
        sp_unpack_seq(self.handle, seq, buf, stream)

    def set_kv_scales(self, layer: int, k_scale, v_scale, stream=None) -> None:
        sp_set_kv_scales(self.handle, layer, k_scale, v_scale, stream)

    def release(self, seq: int, stream=None) -> None:
        sp_release_seq(self.handle, seq, stream)

    def export_table(self, seq: int, layer: int, kv_head: int):
        cap = (self.cfg.max_seq_len + self.cfg.page_size - 1) // self.cfg.page_size + 1
        return sp_export_table(self.handle, seq, layer, kv_head, cap, self.cfg.page_size)

    def visible_count(self, seq: int, layer: int, kv_head: int, positions) -> List[int]:
        return sp_visible_count(self.handle, seq, layer, kv_head, positions)

    def seq_len(self, seq: int, layer: int) -> int:
        return sp_seq_len(self.handle, seq, layer)

    def free_pages(self) -> int:
        return sp_free_pages(self.handle)

    def count_prefill_pairs(self, seq: int, layer: int, n0: int, c: int) -> int:
        return sp_count_prefill_pairs(self.handle, seq, layer, n0, c)

    def count_decode_bytes(self, layer: int, seq_ids, t) -> int:
        return sp_count_decode_bytes(self.handle, layer, seq_ids, t)

    def status(self, stream=None) -> int:
        return sp_get_status(self.handle, stream)

    def set_launch_events(self, start=None, end=None) -> None:
        """Time the next attention call's kernels with two recorded-once
        torch.cuda.Event objects (sp_set_launch_events)."""
        sp_set_launch_events(self.handle, start, end)
