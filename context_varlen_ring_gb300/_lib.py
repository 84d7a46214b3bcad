"""Loads libra.so (built in-tree) and declares its C ABI for ctypes.

There is no fallback: if the library is missing or fails to load, every
call raises.  Build it with `python -m context_varlen_ring_gb300.build`
or `__graft_entry__.build()`.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libra.so")

RA_OK = 0
RA_ERR_INVALID_ARG = 1
RA_ERR_UNSUPPORTED = 2
RA_ERR_CUDA = 3
RA_ERR_WORKSPACE = 4
RA_ERR_TIMEOUT = 5
RA_ERR_DEVICE_BOUNDS = 6

RA_ZZ_GLOBAL = 0
RA_ZZ_PER_DOC = 1
RA_BWD_FWD_RESERVE = 1
RA_BF16 = 0
RA_FP32 = 1
RA_SCHED_FUSED = 0
RA_SCHED_STEPWISE = 1
RA_SCHED_ALLGATHER = 2

# every symbol include/ra.h declares
EXPORTS = (
    "ra_zigzag_plan", "ra_zigzag_permute", "ra_zigzag_unpermute",
    "ra_partial_workspace_bytes", "ra_varlen_attn_partial", "ra_lse_merge",
    "ra_ring_workspace_bytes", "ra_ring_attn_fwd", "ra_ring_attn_bwd",
    "ra_ring_rank_pairs", "ra_get_device_status", "ra_selftest_wait_timeout",
    "ra_status_string", "ra_last_error", "ra_version", "ra_profile_enable", "ra_profile_read",
    "ra_varlen_attn_partial_noalloc", "ra_ring_plan_stats", "ra_partial_table_bytes",
    "ra_ring_workspace_bytes_masked", "ra_ring_attn_fwd_masked", "ra_ring_attn_bwd_masked",
    "ra_ring_plan_stats_masked", "ra_varlen_attn_partial_dev",
)

_lib = None


class RaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where} failed: status {status} ({detail})")
        self.status = status


def _declare(L):
    P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    sig = {
        "ra_zigzag_plan": (i32, [P, i32, i32, i32, P, P, P]),
        "ra_zigzag_permute": (i32, [P, P, P, i64, i64, P]),
        "ra_zigzag_unpermute": (i32, [P, P, P, i64, i64, P]),
        "ra_partial_workspace_bytes": (sz, [i64, i64, i32, i32, i32, i32, i32]),
        "ra_partial_table_bytes": (sz, [i64, i64, i32, i32, i32, i32, P, P, i32, P, P, i32, i32]),
        "ra_varlen_attn_partial": (i32, [P, P, P, i32, i64, i64, i32, i32, i32, P, P, i32, P, P, i32, i32, f32,
                                         P, P, P, sz, P]),
        "ra_varlen_attn_partial_dev": (i32, [P, P, P, i32, i64, i64, i32, i32, i32, P, P, i32, P, P, i32, i32, f32,
                                             P, P, P, sz, P]),
        "ra_varlen_attn_partial_noalloc": (i32, [P, P, P, i32, i64, i64, i32, i32, i32, P, P, i32, P, P, i32,
                                                 i32, f32, P, P, P]),
        "ra_lse_merge": (i32, [i32, P, P, i64, i32, i32, P, i32, P, P]),
        "ra_ring_workspace_bytes": (sz, [i64, i32, i32, i32, i32, P, i32, i32, i32, i32, i32]),
        "ra_ring_attn_fwd": (i32, [P, P, P, i32, i64, i32, i32, i32, P, i32, i32, i32, i32, i32, f32, i32,
                                   P, P, P, sz, P]),
        "ra_ring_attn_bwd": (i32, [P, P, P, i32, i64, i32, i32, i32, P, i32, i32, i32, i32, i32, f32, i32,
                                   P, P, P, P, P, P, i32, i32, P, sz, P]),
        "ra_ring_workspace_bytes_masked": (sz, [i64, i32, i32, i32, i32, P, i32, i32, i32, P, P, i32, i32]),
        "ra_ring_attn_fwd_masked": (i32, [P, P, P, i32, i64, i32, i32, i32, P, i32, i32, i32, P, P, f32, i32,
                                          P, P, P, sz, P]),
        "ra_ring_attn_bwd_masked": (i32, [P, P, P, i32, i64, i32, i32, i32, P, i32, i32, i32, P, P, f32, i32,
                                          P, P, P, P, P, P, i32, i32, P, sz, P]),
        "ra_ring_rank_pairs": (i32, [P, i32, i32, i32, i32, i32, P]),
        "ra_ring_plan_stats": (i32, [P, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, P]),
        "ra_ring_plan_stats_masked": (i32, [P, i32, i32, i32, i32, i32, P, P, i32, i32, i32, P]),
        "ra_get_device_status": (i32, [P]),
        "ra_selftest_wait_timeout": (i32, [i64, P]),
        "ra_status_string": (ctypes.c_char_p, [i32]),
        "ra_last_error": (ctypes.c_char_p, []),
        "ra_version": (ctypes.c_char_p, []),
        "ra_profile_enable": (i32, [i32]),
        "ra_profile_read": (i32, [i32, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def lib():
    """The loaded library; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        _declare(L)
        _lib = L
    return _lib


def check(status: int, where: str):
    if status != RA_OK:
        detail = lib().ra_last_error().decode(errors="replace")
        raise RaError(status, where, detail)
