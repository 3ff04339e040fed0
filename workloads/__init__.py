"""Seeded synthetic workloads shaped like the SegPagedAttention pages' experiments.

This module only draws numbers: shapes, per-(layer, KV head) head classes,
retrieval index lists, sequence lengths and Q/K/V tensors.  It holds none of
the method's arithmetic (no visibility rule, no page rule, no attention), so
both the CPU oracle and the CUDA path can take their inputs from it.

Shapes follow the pages' workloads:
  * head classes per (layer, KV head): GLOBAL / LOCAL(sink, window) /
    RETRIEVAL(indices) -- RedKnot SegPagedAttention runtime article,
    section 2 ("four head-class policies"), with ~12-15 % global heads
    (RedKnot news summary, "Head-Class Sparsification" paragraph);
  * sink 4, windows 1024 / 2048 / 4096 / 8192 and page size 64 -- runtime
    article sections 2 and 6;
  * GQA shapes of Mistral-7B, Llama-3-8B and Llama-3.3-70B.

The pages measured on LongBench-style QA sets with trained models; those are
not available here, so N(0, 1) tensors of the same shapes stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

GLOBAL, LOCAL, RETRIEVAL = 0, 1, 2
KIND_NAMES = {GLOBAL: "GLOBAL", LOCAL: "LOCAL", RETRIEVAL: "RETRIEVAL"}


@dataclass(frozen=True)
class HeadPolicy:
    """One (sequence, layer, KV head) head class as drawn by the harness."""
    kind: int
    sink: int = 0
    window: int = 0
    idx: Optional[np.ndarray] = None  # int32, strictly ascending (RETRIEVAL)

    def as_tuple(self):
        return (self.kind, self.sink, self.window,
                None if self.idx is None else self.idx.tolist())


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    hq: int
    hkv: int
    d: int
    page: int
    seqs: int
    seq_len: Optional[int]          # None -> ragged, see ragged_lengths()
    local_sink: int
    local_window: int
    n_global: int                   # GLOBAL units per sequence (of layers*hkv)
    n_retrieval: int = 0
    retrieval_topk: int = 0
    k_scale: float = 1.0
    fp32_inputs: bool = False
    decode_steps: int = 0
    chunk: Optional[int] = None
    len_range: Optional[tuple] = None
    extra: Dict = field(default_factory=dict)

    @property
    def units(self) -> int:
        return self.layers * self.hkv


# The five workloads.  The global/retrieval counts are round(fraction * units):
# 1 of 8, 32 of 256 (12.5 %), 77 of 512 (15 %), and 38 / 38 of 256 (15 % each).
WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", layers=1, hq=4, hkv=2, d=64, page=16, seqs=1,
                     seq_len=256, local_sink=4, local_window=32, n_global=1,
                     fp32_inputs=True, decode_steps=4),
    "mistral7b_prefill_8k": Workload(
        "mistral7b_prefill_8k", layers=1, hq=32, hkv=8, d=128, page=64, seqs=1,
        seq_len=8192, local_sink=4, local_window=1024, n_global=1, k_scale=0.5),
    "llama3_8b_decode_32k": Workload(
        "llama3_8b_decode_32k", layers=32, hq=32, hkv=8, d=128, page=64, seqs=32,
        seq_len=32768, local_sink=4, local_window=2048, n_global=32,
        decode_steps=64),
    "llama33_70b_prefill_128k": Workload(
        "llama33_70b_prefill_128k", layers=64, hq=64, hkv=8, d=128, page=64,
        seqs=1, seq_len=131072, local_sink=4, local_window=8192, n_global=77),
    "ragged_mixed": Workload(
        "ragged_mixed", layers=32, hq=32, hkv=8, d=128, page=64, seqs=8,
        seq_len=None, local_sink=4, local_window=4096, n_global=38,
        n_retrieval=38, retrieval_topk=2048, chunk=4096, decode_steps=16,
        len_range=(2048, 65536)),
}


def _seed(*parts: int) -> int:
    """Fold integer tags into one 63-bit seed (splitmix64 finaliser)."""
    x = 0x9E3779B97F4A7C15
    for p in parts:
        x = (x ^ (int(p) & 0xFFFFFFFFFFFFFFFF)) * 0xBF58476D1CE4E5B9 & 0xFFFFFFFFFFFFFFFF
        x ^= x >> 31
    return x & 0x7FFFFFFFFFFFFFFF


def class_assignment(wl: Workload, seed: int = 0) -> np.ndarray:
    """Head class per (layer, KV head): int array [layers, hkv].

    The GLOBAL (and RETRIEVAL) units are the first n_global (then next
    n_retrieval) entries of a seeded permutation of all units; the rest are
    LOCAL.  The tiny workload fixes KV head 0 GLOBAL and KV head 1 LOCAL.
    """
    if wl.name == "tiny":
        return np.array([[GLOBAL, LOCAL]], dtype=np.int32)
    rng = np.random.default_rng(_seed(seed, 17))
    perm = rng.permutation(wl.units)
    kinds = np.full(wl.units, LOCAL, dtype=np.int32)
    kinds[perm[:wl.n_global]] = GLOBAL
    kinds[perm[wl.n_global:wl.n_global + wl.n_retrieval]] = RETRIEVAL
    return kinds.reshape(wl.layers, wl.hkv)


def retrieval_indices(length: int, topk: int, seed: int) -> np.ndarray:
    """Top-k token indices by seeded uniform scores, ascending int32.

    Ties are broken by lower index first; if length <= topk every index is
    kept.  This stands in for an attention-score based selection.
    """
    if length <= topk:
        return np.arange(length, dtype=np.int32)
    rng = np.random.default_rng(_seed(seed, length, 31))
    score = rng.random(length, dtype=np.float32)
    order = np.lexsort((np.arange(length), -score))  # score desc, index asc
    return np.sort(order[:topk]).astype(np.int32)


def policies(wl: Workload, seq: int = 0, length: Optional[int] = None,
             seed: int = 0) -> List[List[HeadPolicy]]:
    """Per-(layer, KV head) policy list for one sequence."""
    kinds = class_assignment(wl, seed)
    L = wl.seq_len if length is None else length
    out = []
    for layer in range(wl.layers):
        row = []
        for h in range(wl.hkv):
            k = int(kinds[layer, h])
            if k == GLOBAL:
                row.append(HeadPolicy(GLOBAL))
            elif k == LOCAL:
                row.append(HeadPolicy(LOCAL, wl.local_sink, wl.local_window))
            else:
                idx = retrieval_indices(L, wl.retrieval_topk,
                                        _seed(seed, seq, layer, h))
                row.append(HeadPolicy(RETRIEVAL, idx=idx))
        out.append(row)
    return out


def ragged_lengths(wl: Workload, seed: int = 0) -> List[int]:
    """Sequence lengths log-uniform in wl.len_range (floor of exp(U))."""
    lo, hi = wl.len_range
    rng = np.random.default_rng(_seed(seed, 53))
    u = rng.uniform(math.log(lo), math.log(hi), size=wl.seqs)
    return [int(math.floor(math.exp(x))) for x in u]


def seq_lengths(wl: Workload, seed: int = 0) -> List[int]:
    if wl.seq_len is None:
        return ragged_lengths(wl, seed)
    return [wl.seq_len] * wl.seqs


def normal(shape: Sequence[int], seed: int, scale: float = 1.0,
           device: str = "cpu", dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """Seeded N(0, scale^2) tensor drawn in fp32 and rounded to `dtype`."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(dtype)


def tensor_seed(seed: int, tag: str, *parts: int) -> int:
    """Seed for one tensor: tag is 'q', 'k', 'v' plus (seq, layer, step...)."""
    return _seed(seed, sum(ord(c) << (8 * i) for i, c in enumerate(tag)), *parts)


def qkv(wl: Workload, n_tokens: int, seq: int, layer: int, seed: int = 0,
        device: str = "cpu", step: int = 0, dtype: torch.dtype = torch.bfloat16):
    """Q [n, hq, d], K [n, hkv, d], V [n, hkv, d] for one (sequence, layer, step)."""
    q = normal((n_tokens, wl.hq, wl.d), tensor_seed(seed, "q", seq, layer, step),
               1.0, device, dtype)
    k = normal((n_tokens, wl.hkv, wl.d), tensor_seed(seed, "k", seq, layer, step),
               wl.k_scale, device, dtype)
    v = normal((n_tokens, wl.hkv, wl.d), tensor_seed(seed, "v", seq, layer, step),
               1.0, device, dtype)
    return q, k, v
