"""CPU oracle for head-aware (SegPaged) attention and its paged storage.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may import this package; the
product (``head_aware_paged_gb300``) never does, and shares no code with it.

Contents
  * ``attend`` -- plain two-pass softmax attention over materialised
    visibility sets, in C (``segpaged_oracle.c``), fp32 and fp64 builds.
  * ``visible`` -- V(i) for one head (same C file).
  * ``pagemodel`` -- canonical page table and deterministic allocator model.
  * ``accounting`` -- visible-pair FLOPs and visible-KV bytes.

Every function cites the passage of the SegPagedAttention pages it follows.
Parity pins: see tests/test_oracle.py and tests/test_pagemodel.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SRC = os.path.join(_HERE, "segpaged_oracle.c")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()

GLOBAL, LOCAL, RETRIEVAL = 0, 1, 2


def build(force: bool = False, mutation: int = 0) -> str:
    """Compile the C oracle (fp32 and fp64 objects) into one shared library.

    mutation != 0 builds a variant with one planted mistake (see the C file);
    only the mutation test asks for one."""
    os.makedirs(_BUILD, exist_ok=True)
    lib = _LIB if mutation == 0 else os.path.join(_BUILD, "liboracle_mut%d.so" % mutation)
    if (not force and os.path.exists(lib)
            and os.path.getmtime(lib) >= os.path.getmtime(_SRC)):
        return lib
    flags = ["-O2", "-fPIC", "-fopenmp", "-std=c11", "-ffp-contract=off",
             "-DORACLE_MUTATION=%d" % mutation]
    tag = "" if mutation == 0 else "_mut%d" % mutation
    o32 = os.path.join(_BUILD, "oracle_f32%s.o" % tag)
    o64 = os.path.join(_BUILD, "oracle_f64%s.o" % tag)
    subprocess.check_call(["gcc", *flags, "-c", _SRC, "-o", o32])
    subprocess.check_call(["gcc", *flags, "-DORACLE_DOUBLE", "-c", _SRC, "-o", o64])
    tmp = lib + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-shared", "-fopenmp", o32, o64, "-o", tmp, "-lm"])
    os.replace(tmp, lib)
    return lib


_libs = {}


def _load(mutation: int = 0):
    with _lock:
        if mutation not in _libs:
            lib = ctypes.CDLL(build(mutation=mutation))
            P = ctypes.c_void_p
            for sfx in ("f32", "f64"):
                f = getattr(lib, "oracle_attend_" + sfx)
                f.restype = ctypes.c_int
                f.argtypes = [ctypes.c_int64, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              P, P, P, P, P, P, ctypes.c_int64, P, P, P, P, ctypes.c_int]
                g = getattr(lib, "oracle_visible_" + sfx)
                g.restype = ctypes.c_int64
                g.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, P,
                              ctypes.c_int64, ctypes.c_int64, P]
            _libs[mutation] = lib
    return _libs[mutation]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _policy_arrays(policies):
    """policies: sequence over KV heads of (kind, sink, window, idx|None)."""
    kinds, sinks, wins, offs, idx = [], [], [], [0], []
    for p in policies:
        kind, sink, window, ind = p
        kinds.append(kind)
        sinks.append(sink)
        wins.append(window)
        ind = [] if ind is None else list(ind)
        idx.extend(ind)
        offs.append(len(idx))
    return (np.asarray(kinds, np.int32), np.asarray(sinks, np.int32),
            np.asarray(wins, np.int32), np.asarray(offs, np.int64),
            np.asarray(idx if idx else [0], np.int32))


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, row_pos: Sequence[int],
           policies, precision: str = "f64", threads: int = 0, _mutation: int = 0):
    """O, LSE for queries q [n_rows, Hq, d] at absolute positions row_pos.

    k, v: [n_keys, Hkv, d] hold keys/values of positions 0 .. n_keys-1 of the
    same sequence.  policies: per KV head (kind, sink, window, idx).
    Follows the runtime article section 4 equivalence (dense attention under a
    head-wise mask) through the C oracle.
    """
    lib = _load(_mutation)
    dt = np.float64 if precision == "f64" else np.float32
    q = np.ascontiguousarray(q, dtype=dt)
    k = np.ascontiguousarray(k, dtype=dt)
    v = np.ascontiguousarray(v, dtype=dt)
    n_rows, hq, d = q.shape
    n_keys, hkv, d2 = k.shape
    assert d2 == d and v.shape == k.shape and hq % hkv == 0
    assert len(policies) == hkv
    rp = np.ascontiguousarray(np.asarray(row_pos, dtype=np.int64))
    assert rp.shape == (n_rows,)
    kinds, sinks, wins, offs, idx = _policy_arrays(policies)
    o = np.zeros((n_rows, hq, d), dtype=dt)
    lse = np.zeros((n_rows, hq), dtype=dt)
    fn = getattr(lib, "oracle_attend_" + precision)
    rc = fn(n_rows, _ptr(rp), hq, hkv, d, _ptr(kinds), _ptr(sinks), _ptr(wins),
            _ptr(offs), _ptr(idx), _ptr(q), n_keys, _ptr(k), _ptr(v), _ptr(o),
            _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError("oracle: visible position outside the given keys or bad class")
    return o, lse


def visible(kind: int, sink: int, window: int, idx: Optional[Sequence[int]],
            i: int, _mutation: int = 0) -> np.ndarray:
    """V(i) of one head as an ascending int64 array (runtime article section 2)."""
    lib = _load(_mutation)
    ind = np.asarray([] if idx is None else list(idx), dtype=np.int32)
    if ind.size == 0:
        ind_buf = np.zeros(1, np.int32)
    else:
        ind_buf = np.ascontiguousarray(ind)
    out = np.zeros(max(i + 1, 1), dtype=np.int64)
    n = lib.oracle_visible_f64(kind, sink, window, _ptr(ind_buf), ind.size, i, _ptr(out))
    if n < 0:
        raise ValueError("unknown head class")
    return out[:n].copy()
