"""Shared helpers for the GPU parity tests: build caches through the C ABI,
run the CPU oracle on the same bf16 inputs, compare."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from workloads import GLOBAL, LOCAL, RETRIEVAL, HeadPolicy

# Parity bar for bf16 outputs against the oracle: max |err| <= 2e-2 over all
# compared elements and cosine >= 0.9999 per (sequence, query head).
ATOL = 2e-2
COS_MIN = 0.9999
LSE_ATOL = 2e-3


def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_aware_paged_gb300 import build
    build.build()


def ncores() -> int:
    return os.cpu_count() or 4


def pol_tuple(p: HeadPolicy):
    return (p.kind, p.sink, p.window, None if p.idx is None else [int(x) for x in p.idx])


def to_c_policies(pols):
    from head_aware_paged_gb300 import Policy
    return [[Policy(p.kind, p.sink, p.window, None if p.idx is None else [int(x) for x in p.idx])
             for p in row] for row in pols]


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(out_gpu: torch.Tensor, ref: np.ndarray, lse_gpu=None, lse_ref=None,
            what: str = ""):
    """out_gpu [rows, hq, d] bf16; ref [rows, hq, d] float64."""
    got = f64(out_gpu)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what + ": non-finite output"
    assert err.max() <= ATOL, "%s: max abs err %.3g" % (what, err.max())
    for h in range(ref.shape[1]):
        a, b = got[:, h].ravel(), ref[:, h].ravel()
        na, nb = np.linalg.norm(a), np.linalg.norm(b)
        if nb == 0 and na == 0:
            continue
        cos = float(a @ b / (na * nb))
        assert cos >= COS_MIN, "%s: head %d cosine %.6f" % (what, h, cos)
    if lse_gpu is not None and lse_ref is not None:
        lg = lse_gpu.detach().cpu().numpy().astype(np.float64)
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lg), fin), what + ": LSE finiteness differs"
        if fin.any():
            assert np.abs(lg[fin] - lse_ref[fin]).max() <= LSE_ATOL, what + ": LSE error"
    return float(err.max())
