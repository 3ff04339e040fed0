"""ctypes binding of libsegpaged.so: the C-ABI entry points under their own
names, with argument marshalling only (every step of the path runs in the
library's CUDA kernels).  No fallback: if the library is missing, loading
raises."""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_int32, c_int64, c_size_t, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsegpaged.so")

SP_OK = 0
STATUS_NAMES = {0: "SP_OK", 1: "SP_ERR_INVALID_ARG", 2: "SP_ERR_OUT_OF_PAGES",
                3: "SP_ERR_UNSUPPORTED", 4: "SP_ERR_CUDA", 5: "SP_ERR_DEVICE_STATUS",
                6: "SP_ERR_TIMEOUT"}
GLOBAL, LOCAL, RETRIEVAL = 0, 1, 2
KV_BF16, KV_FP8 = 0, 1

# Every symbol include/segpaged.h declares.
EXPORTS = ("sp_required_bytes", "sp_cache_create", "sp_cache_destroy", "sp_set_policy",
           "sp_build_cache", "sp_append_kv", "sp_attention_prefill", "sp_attention_decode",
           "sp_attention_decode_static_scratch", "sp_rope_realign", "sp_pack_seq",
           "sp_unpack_seq", "sp_select_workspace_bytes", "sp_select_heavy_hitters",
           "sp_select_heavy_hitters_top_p", "sp_set_kv_scales",
           "sp_release_seq", "sp_export_table", "sp_visible_count", "sp_seq_len",
           "sp_free_pages", "sp_count_prefill_pairs", "sp_count_decode_bytes",
           "sp_get_status", "sp_selftest_bounded_wait", "sp_set_launch_events",
           "sp_last_error")


class SegPagedError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, str(status)), message))


class SpConfig(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in (
        "num_layers", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "max_seqs",
        "max_seq_len", "num_pages", "max_idx_per_seq", "max_tokens", "max_batch", "kv_dtype")]


class SpHeadPolicy(ctypes.Structure):
    _fields_ = [("kind", c_int32), ("sink", c_int32), ("window", c_int32),
                ("n_idx", c_int32), ("idx", POINTER(c_int32))]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (built by __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libsegpaged.so not built at %s; run head_aware_paged_gb300/build.py"
                           % path)
    lib = ctypes.CDLL(path)
    P = c_void_p
    I32P, I64P = POINTER(c_int32), POINTER(c_int64)
    sig = {
        "sp_required_bytes": [POINTER(SpConfig), POINTER(c_size_t), POINTER(c_size_t), POINTER(c_size_t)],
        "sp_cache_create": [POINTER(SpConfig), P, P, P, POINTER(P)],
        "sp_cache_destroy": [P],
        "sp_set_policy": [P, c_int32, POINTER(SpHeadPolicy), P],
        "sp_build_cache": [P, c_int32, c_int32, P, P, c_int64, c_int64, P],
        "sp_append_kv": [P, c_int32, I32P, c_int32, I32P, P, P, P],
        "sp_attention_prefill": [P, c_int32, I32P, c_int32, I32P, P, P, P, P, P, P],
        "sp_attention_decode": [P, c_int32, I32P, c_int32, P, P, P, P],
        "sp_attention_decode_static_scratch": [P, c_int32, I32P, c_int32, P, P, P, P],
        "sp_rope_realign": [P, c_int32, I32P, c_int32, c_int32, c_int64, c_int64, c_int64,
                            c_double, P],
        "sp_pack_seq": [P, c_int32, P, c_size_t, POINTER(c_size_t), P],
        "sp_unpack_seq": [P, c_int32, P, c_size_t, P],
        "sp_select_workspace_bytes": [c_int32, c_int32, c_int32, c_int32, POINTER(c_size_t)],
        "sp_select_heavy_hitters": [P, c_int32, P, c_int32, c_int32, c_int32, c_int32, c_int32,
                                    c_int32, I32P, I32P, P, P, c_size_t, P],
        "sp_select_heavy_hitters_top_p": [P, c_int32, P, c_int32, c_int32, c_int32, c_int32,
                                          ctypes.c_float, c_int32, c_int32, I32P, I32P, P, P,
                                          c_size_t, P],
        "sp_set_kv_scales": [P, c_int32, POINTER(ctypes.c_float), POINTER(ctypes.c_float), P],
        "sp_release_seq": [P, c_int32, P],
        "sp_export_table": [P, c_int32, c_int32, c_int32, I32P, I32P, I32P, c_int32, P],
        "sp_visible_count": [P, c_int32, c_int32, c_int32, I64P, c_int32, I32P, P],
        "sp_seq_len": [P, c_int32, c_int32, I32P],
        "sp_free_pages": [P, I32P],
        "sp_count_prefill_pairs": [P, c_int32, c_int32, c_int64, c_int64, I64P],
        "sp_count_decode_bytes": [P, c_int32, I32P, c_int32, I64P, I64P],
        "sp_get_status": [P, P, I32P],
        "sp_selftest_bounded_wait": [P, c_int64, c_int32, P],
        "sp_set_launch_events": [P, P, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = c_int32
    lib.sp_last_error.argtypes = []
    lib.sp_last_error.restype = c_char_p
    _lib = lib
    return lib


def check(status: int) -> None:
    if status != SP_OK:
        msg = load().sp_last_error().decode(errors="replace")
        raise SegPagedError(status, msg)


def i32_array(values):
    values = [int(x) for x in values]
    return (c_int32 * max(1, len(values)))(*values)


def i64_array(values):
    values = [int(x) for x in values]
    return (c_int64 * max(1, len(values)))(*values)
