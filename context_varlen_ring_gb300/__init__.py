"""Packed causal varlen ring attention with zigzag CP balancing on GB300.

A thin PyTorch binding over the C ABI in include/ra.h (libra.so): it checks
shapes, allocates outputs and the workspace with PyTorch, and passes raw
pointers and the current CUDA stream.  Every step of the data path runs in
the library's CUDA kernels; there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

from ._lib import (RA_BF16, RA_BWD_FWD_RESERVE, RA_FP32, RA_SCHED_ALLGATHER, RA_SCHED_FUSED, RA_SCHED_STEPWISE,
                   RA_ZZ_GLOBAL, RA_ZZ_PER_DOC, RaError, check, lib)

__all__ = [
    "zigzag_plan", "zigzag_permute", "zigzag_unpermute", "varlen_attn_partial", "varlen_attn_partial_dev",
    "lse_merge",
    "ring_attn_fwd", "ring_attn_bwd", "ring_rank_pairs", "ring_plan_stats", "device_status", "selftest_wait_timeout",
    "RA_ZZ_GLOBAL", "RA_ZZ_PER_DOC", "RA_SCHED_FUSED", "RA_SCHED_STEPWISE", "RA_SCHED_ALLGATHER", "RaError",
]

_SCHED = {"fused": RA_SCHED_FUSED, "stepwise": RA_SCHED_STEPWISE, "allgather": RA_SCHED_ALLGATHER}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return RA_BF16
    if t.dtype == torch.float32:
        return RA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _host_i32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def zigzag_plan(cu_seqlens, cp: int, mode: int = RA_ZZ_GLOBAL):
    """Host zigzag plan: (perm [T], off [cp+1], cu_local [cp, B+1]) int32 numpy."""
    cu = _host_i32(cu_seqlens)
    B = len(cu) - 1
    T = int(cu[-1]) if B >= 1 else 0
    perm = np.zeros(max(T, 1), dtype=np.int32)
    off = np.zeros(cp + 1, dtype=np.int32)
    cl = np.zeros((cp, B + 1), dtype=np.int32)
    check(lib().ra_zigzag_plan(_np_ptr(cu), B, cp, mode, _np_ptr(perm), _np_ptr(off), _np_ptr(cl)),
          "ra_zigzag_plan")
    return perm[:T], off, cl


def ring_rank_pairs(cu_seqlens, cp: int, mode: int = RA_ZZ_GLOBAL, causal: bool = True,
                    window: int = -1) -> np.ndarray:
    cu = _host_i32(cu_seqlens)
    counts = np.zeros(cp, dtype=np.int64)
    check(lib().ra_ring_rank_pairs(_np_ptr(cu), len(cu) - 1, cp, mode, int(causal), int(window), _np_ptr(counts)),
          "ra_ring_rank_pairs")
    return counts


PLAN_STATS = ("q_tiles", "kv_tiles", "fwd_items", "dkdv_items", "dq_items", "fwd_visited", "fwd_full",
              "two_run_q_rows", "two_run_kv_rows", "fwd_capacity", "fwd_allowed", "full_disallowed",
              "dkdv_allowed", "dq_allowed", "dkdv_visited", "dq_visited",
              "fwd_makespan", "dkdv_makespan", "dq_makespan", "fwd_steps")


def ring_plan_stats(cu_seqlens, cp: int, mode: int = RA_ZZ_GLOBAL, G: int = 4, Hkv: int = 8, causal: bool = True,
                    window: int = -1, sched: str = "fused", exact: bool = False, n_sm: int = 152, key_lo=None,
                    key_hi=None) -> dict:
    """Host-only counts of what the tensor-core passes visit (tiles, work
    items, visited tile pairs, rows copied into rank order; with exact=True
    also the allowed pairs inside the visited tile pairs of each pass) and a
    scheduling model of each pass over n_sm SMs (makespans in tile visits)."""
    cu = _host_i32(cu_seqlens)
    out = np.zeros(len(PLAN_STATS), dtype=np.int64)
    if key_lo is not None or key_hi is not None:
        lo, hi = _host_i32(key_lo), _host_i32(key_hi)
        check(lib().ra_ring_plan_stats_masked(_np_ptr(cu), len(cu) - 1, cp, mode, G, Hkv, _np_ptr(lo), _np_ptr(hi),
                                              _SCHED[sched], int(exact), int(n_sm), _np_ptr(out)),
              "ra_ring_plan_stats_masked")
        return dict(zip(PLAN_STATS, (int(x) for x in out)))
    check(lib().ra_ring_plan_stats(_np_ptr(cu), len(cu) - 1, cp, mode, G, Hkv, int(causal), int(window),
                                   _SCHED[sched], int(exact), int(n_sm), _np_ptr(out)), "ra_ring_plan_stats")
    return dict(zip(PLAN_STATS, (int(x) for x in out)))


def _perm_dev(perm, device):
    if isinstance(perm, torch.Tensor):
        return perm.to(device=device, dtype=torch.int32).contiguous()
    return torch.from_numpy(_host_i32(perm)).to(device)


def zigzag_permute(x: torch.Tensor, perm) -> torch.Tensor:
    """y[i] = x[perm[i]] along dim 0 (bit-exact)."""
    _check_cuda(x)
    p = _perm_dev(perm, x.device)
    y = torch.empty_like(x)
    T = x.shape[0]
    rb = x[0].numel() * x.element_size() if T else 1
    check(lib().ra_zigzag_permute(_ptr(x), _ptr(y), _ptr(p), T, rb, _stream(x.device)), "ra_zigzag_permute")
    return y


def zigzag_unpermute(y: torch.Tensor, perm) -> torch.Tensor:
    """x[perm[i]] = y[i] along dim 0 (bit-exact)."""
    _check_cuda(y)
    p = _perm_dev(perm, y.device)
    x = torch.empty_like(y)
    T = y.shape[0]
    rb = y[0].numel() * y.element_size() if T else 1
    check(lib().ra_zigzag_unpermute(_ptr(y), _ptr(x), _ptr(p), T, rb, _stream(y.device)), "ra_zigzag_unpermute")
    return x


def varlen_attn_partial(q, k, v, cu_seqlens_q, cu_seqlens_k, q_pos=None, k_pos=None, causal: bool = True,
                        scale: float | None = None, out=None, lse=None, window: int = -1):
    """One ring step: (out fp32 [Tq,Hq,d], lse fp32 [Hq,Tq]) of q against k/v
    over pairs in the same segment with k_pos <= q_pos (when causal) and
    k_pos >= q_pos - window (when window >= 0)."""
    _check_cuda(q, k, v)
    Tq, Hq, d = q.shape
    Tk, Hkv, _ = k.shape
    dt = _dtype_code(q)
    cuq, cuk = _host_i32(cu_seqlens_q), _host_i32(cu_seqlens_k)
    nseg = len(cuq) - 1
    qp = _host_i32(q_pos) if q_pos is not None else None
    kp = _host_i32(k_pos) if k_pos is not None else None
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty((Tq, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    L = lib()
    ws_bytes = L.ra_partial_workspace_bytes(Tq, Tk, nseg, Hq, Hkv, d, dt)
    ws = torch.empty(max(int(ws_bytes), 1), dtype=torch.uint8, device=q.device)
    check(L.ra_varlen_attn_partial(_ptr(q), _ptr(k), _ptr(v), dt, Tq, Tk, Hq, Hkv, d, _np_ptr(cuq), _np_ptr(cuk),
                                   nseg, _np_ptr(qp) if qp is not None else None,
                                   _np_ptr(kp) if kp is not None else None, int(causal), int(window), scale, _ptr(out),
                                   _ptr(lse), _ptr(ws), ws.numel(), _stream(q.device)),
          "ra_varlen_attn_partial")
    return out, lse


def varlen_attn_partial_dev(q, k, v, cu_seqlens_q, cu_seqlens_k, q_pos=None, k_pos=None, causal: bool = True,
                            scale: float | None = None, out=None, lse=None, window: int = -1, workspace=None):
    """varlen_attn_partial with the segment boundaries and positions as int32
    tensors on q's device (no host round trip; capturable).  Tensor-core
    path only (bf16, d = 128, Hq / Hkv a power of two <= 16)."""
    _check_cuda(q, k, v, cu_seqlens_q, cu_seqlens_k)
    for t in (q_pos, k_pos):
        if t is not None:
            _check_cuda(t)
    for t in (cu_seqlens_q, cu_seqlens_k, q_pos, k_pos):
        if t is not None and t.dtype != torch.int32:
            raise TypeError("segment boundaries and positions must be int32")
    Tq, Hq, d = q.shape
    Tk, Hkv, _ = k.shape
    nseg = cu_seqlens_q.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty((Tq, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    L = lib()
    ws_bytes = int(L.ra_partial_workspace_bytes(Tq, Tk, nseg, Hq, Hkv, d, _dtype_code(q)))
    ws = workspace if workspace is not None else torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    check(L.ra_varlen_attn_partial_dev(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), Tq, Tk, Hq, Hkv, d,
                                       _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), nseg, _ptr(q_pos), _ptr(k_pos),
                                       int(causal), int(window), scale, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                       _stream(q.device)), "ra_varlen_attn_partial_dev")
    return out, lse


def lse_merge(outs, lses, out_dtype=torch.float32):
    """Merge partials (fp32 [Tq,Hq,d], fp32 [Hq,Tq]) -> (out, lse)."""
    _check_cuda(*outs, *lses)
    Tq, Hq, d = outs[0].shape
    n = len(outs)
    op = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    lp = (ctypes.c_void_p * n)(*[l.data_ptr() for l in lses])
    out = torch.empty((Tq, Hq, d), dtype=out_dtype, device=outs[0].device)
    lse = torch.empty((Hq, Tq), dtype=torch.float32, device=outs[0].device)
    check(lib().ra_lse_merge(n, op, lp, Tq, Hq, d, _ptr(out), _dtype_code(out), _ptr(lse),
                             _stream(out.device)), "ra_lse_merge")
    return out, lse


class _Workspace:
    """A per-device byte buffer reused across calls (grown on demand)."""

    def __init__(self):
        self.buf = {}

    def get(self, device, nbytes: int) -> torch.Tensor:
        key = (device.type, device.index)
        b = self.buf.get(key)
        if b is None or b.numel() < nbytes:
            b = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
            self.buf[key] = b
        return b


_WS = _Workspace()


def ring_workspace_bytes(T, Hq, Hkv, d, dtype, cu_seqlens, cp, mode, sched="fused", bwd=False, key_lo=None,
                         key_hi=None) -> int:
    cu = _host_i32(cu_seqlens)
    if key_lo is not None or key_hi is not None:
        lo, hi = _host_i32(key_lo), _host_i32(key_hi)
        return int(lib().ra_ring_workspace_bytes_masked(T, Hq, Hkv, d, dtype, _np_ptr(cu), len(cu) - 1, cp, mode,
                                                        _np_ptr(lo), _np_ptr(hi), _SCHED[sched], int(bwd)))
    return int(lib().ra_ring_workspace_bytes(T, Hq, Hkv, d, dtype, _np_ptr(cu), len(cu) - 1, cp, mode,
                                             _SCHED[sched], int(bwd)))


def ring_attn_fwd(q, k, v, cu_seqlens, cp: int, mode: int = RA_ZZ_GLOBAL, causal: bool = True,
                  scale: float | None = None, sched: str = "fused", out=None, lse=None, workspace=None,
                  window: int = -1, key_lo=None, key_hi=None):
    """Simulated zigzag ring attention forward; returns (out [T,Hq,d] in q's
    dtype, lse fp32 [Hq,T]) in the original token order.  window >= 0: a key
    is visible only up to `window` positions behind its query.  sched:
    "fused" (ring steps in one launch), "stepwise" (a launch per ring step,
    then the LSE merge) or "allgather" (each rank's queries over the gathered
    K/V of all ranks).  key_lo / key_hi (int32 [T], host or device, both
    non-decreasing inside each document): an interval mask instead of
    causal and window -- query i sees key j of its document iff
    key_lo[i] <= j <= key_hi[i]."""
    _check_cuda(q, k, v)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    dt = _dtype_code(q)
    cu = _host_i32(cu_seqlens)
    B = len(cu) - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    L = lib()
    if key_lo is not None or key_hi is not None:
        lo, hi = _host_i32(key_lo), _host_i32(key_hi)
        need = L.ra_ring_workspace_bytes_masked(T, Hq, Hkv, d, dt, _np_ptr(cu), B, cp, mode, _np_ptr(lo), _np_ptr(hi),
                                                _SCHED[sched], 0)
        ws = workspace if workspace is not None else _WS.get(q.device, int(need))
        check(L.ra_ring_attn_fwd_masked(_ptr(q), _ptr(k), _ptr(v), dt, T, Hq, Hkv, d, _np_ptr(cu), B, cp, mode,
                                        _np_ptr(lo), _np_ptr(hi), scale, _SCHED[sched], _ptr(out), _ptr(lse), _ptr(ws),
                                        ws.numel(), _stream(q.device)), "ra_ring_attn_fwd_masked")
        return out, lse
    need = L.ra_ring_workspace_bytes(T, Hq, Hkv, d, dt, _np_ptr(cu), B, cp, mode, _SCHED[sched], 0)
    ws = workspace if workspace is not None else _WS.get(q.device, int(need))
    check(L.ra_ring_attn_fwd(_ptr(q), _ptr(k), _ptr(v), dt, T, Hq, Hkv, d, _np_ptr(cu), B, cp, mode, int(causal),
                             int(window), scale, _SCHED[sched], _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(q.device)),
          "ra_ring_attn_fwd")
    return out, lse


def ring_attn_bwd(q, k, v, out, lse, dout, cu_seqlens, cp: int, mode: int = RA_ZZ_GLOBAL, causal: bool = True,
                  scale: float | None = None, sched: str = "fused", grad_dtype=None, dq=None, dk=None, dv=None,
                  workspace=None, reuse_fwd_workspace: bool = False, window: int = -1, key_lo=None, key_hi=None):
    """Gradients (dq, dk, dv) in the original token order (window, or
    key_lo / key_hi, as in ring_attn_fwd; pass the forward's).

    reuse_fwd_workspace: `workspace` is the one the preceding ring_attn_fwd
    used with these same q, k, v and arguments, untouched since; its
    rank-ordered Q, K, V and tile tables are reused (RA_BWD_FWD_RESERVE).
    """
    _check_cuda(q, k, v, out, lse, dout)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    dt = _dtype_code(q)
    gd = grad_dtype or q.dtype
    cu = _host_i32(cu_seqlens)
    B = len(cu) - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty((T, Hq, d), dtype=gd, device=q.device) if dq is None else dq
    dk = torch.empty((T, Hkv, d), dtype=gd, device=q.device) if dk is None else dk
    dv = torch.empty((T, Hkv, d), dtype=gd, device=q.device) if dv is None else dv
    L = lib()
    if key_lo is not None or key_hi is not None:
        lo, hi = _host_i32(key_lo), _host_i32(key_hi)
        need = L.ra_ring_workspace_bytes_masked(T, Hq, Hkv, d, dt, _np_ptr(cu), B, cp, mode, _np_ptr(lo), _np_ptr(hi),
                                                _SCHED[sched], 1)
        ws = workspace if workspace is not None else _WS.get(q.device, int(need))
        check(L.ra_ring_attn_bwd_masked(_ptr(q), _ptr(k), _ptr(v), dt, T, Hq, Hkv, d, _np_ptr(cu), B, cp, mode,
                                        _np_ptr(lo), _np_ptr(hi), scale, _SCHED[sched], _ptr(out), _ptr(lse),
                                        _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _dtype_code(dq),
                                        RA_BWD_FWD_RESERVE if reuse_fwd_workspace else 0, _ptr(ws), ws.numel(),
                                        _stream(q.device)), "ra_ring_attn_bwd_masked")
        return dq, dk, dv
    need = L.ra_ring_workspace_bytes(T, Hq, Hkv, d, dt, _np_ptr(cu), B, cp, mode, _SCHED[sched], 1)
    ws = workspace if workspace is not None else _WS.get(q.device, int(need))
    check(L.ra_ring_attn_bwd(_ptr(q), _ptr(k), _ptr(v), dt, T, Hq, Hkv, d, _np_ptr(cu), B, cp, mode, int(causal),
                             int(window), scale, _SCHED[sched], _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                             _dtype_code(dq), RA_BWD_FWD_RESERVE if reuse_fwd_workspace else 0, _ptr(ws), ws.numel(),
                             _stream(q.device)),
          "ra_ring_attn_bwd")
    return dq, dk, dv


def device_status(stream=None) -> int:
    """Reads and clears the device status word (0 = ok)."""
    s = ctypes.c_void_p(stream) if stream is not None else _stream(torch.device("cuda"))
    return int(lib().ra_get_device_status(s))


def selftest_wait_timeout(budget_us: int = 1000):
    check(lib().ra_selftest_wait_timeout(int(budget_us), _stream(torch.device("cuda"))),
          "ra_selftest_wait_timeout")
