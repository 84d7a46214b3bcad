"""fp64 CPU oracle for packed causal varlen ring attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline / reference legs import this package; the product
path (the CUDA library and its Python binding) never does.

The arithmetic lives in `ra_oracle.c` (plain C, fp64, OpenMP); this module
marshals numpy/torch arrays into it.  bf16 inputs are converted to float64
exactly, so the oracle sees the same values as the GPU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ra_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ra_oracle.c with gcc into oracle/liboracle.so (in-tree)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.orc_set_threads.argtypes = [i32]
        L.orc_set_threads.restype = i32
        L.orc_partial_fwd.argtypes = [P, P, P, i64, i64, i32, i32, i32, P, P, P, P, i32, i64, dbl, P, P, P, i64, P, P]
        L.orc_partial_fwd.restype = i32
        L.orc_lse_merge.argtypes = [i32, P, P, i64, i32, i32, P, P]
        L.orc_lse_merge.restype = i32
        L.orc_attn_bwd.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, P, P, i32, i64, dbl, P, P, P, i64, P, i64, P, P,
                                   P]
        L.orc_attn_bwd.restype = i32
        L.orc_zigzag_owner.argtypes = [P, i32, i32, i32, P]
        L.orc_zigzag_owner.restype = i32
        L.orc_zigzag_plan.argtypes = [P, i32, i32, i32, P, P, P]
        L.orc_zigzag_plan.restype = i32
        L.orc_rank_pairs.argtypes = [P, i32, i32, i32, i32, i64, P]
        L.orc_rank_pairs.restype = i32
        _lib = L
    return _lib


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (0 = leave as is); returns the count in use."""
    return int(lib().orc_set_threads(int(n)))


def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _i64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def doc_ids(cu) -> np.ndarray:
    """Per-token document index from cumulative lengths."""
    cu = np.asarray(cu, dtype=np.int64)
    ids = np.empty(int(cu[-1]), dtype=np.int32)
    for b in range(len(cu) - 1):
        ids[cu[b]:cu[b + 1]] = b
    return ids


def _bounds(b, n):
    if b is None:
        return None, None
    a = _i64(b)
    assert a.shape == (n,)
    return a, _p(a)


def partial_fwd(q, k, v, seg_q, seg_k, q_pos, k_pos, causal: bool, scale: float, rows=None, window: int = -1,
                q_lo=None, q_hi=None):
    """Attention of queries against keys over the allowed pairs
    {(i,j): seg_k[j]==seg_q[i] and (not causal or k_pos[j] <= q_pos[i])
    and (window < 0 or k_pos[j] >= q_pos[i] - window)
    and (q_lo is None or k_pos[j] >= q_lo[i]) and (q_hi is None or k_pos[j] <= q_hi[i])}.

    q [Tq,Hq,d], k/v [Tk,Hkv,d]; q_lo / q_hi [Tq] (per query, indexed like
    q).  Returns (out [R,Hq,d], lse [R,Hq]) in fp64, R = len(rows) or Tq.
    Empty rows give out = 0 and lse = -inf."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, Hq, d = q.shape
    Tk, Hkv, _ = k.shape
    sq, sk = _i32(seg_q), _i32(seg_k)
    pq, pk = _i64(q_pos), _i64(k_pos)
    assert sq.shape == (Tq,) and pq.shape == (Tq,) and sk.shape == (Tk,) and pk.shape == (Tk,)
    if rows is None:
        R, rp, rr = Tq, None, None
    else:
        rr = _i64(rows)
        R, rp = len(rr), _p(rr)
    lo_a, lo_p = _bounds(q_lo, Tq)
    hi_a, hi_p = _bounds(q_hi, Tq)
    out = np.zeros((R, Hq, d), dtype=np.float64)
    lse = np.zeros((R, Hq), dtype=np.float64)
    rc = lib().orc_partial_fwd(_p(q), _p(k), _p(v), Tq, Tk, Hq, Hkv, d, _p(sq), _p(sk), _p(pq), _p(pk),
                               int(bool(causal)), int(window), float(scale), lo_p, hi_p, rp, R, _p(out), _p(lse))
    if rc:
        raise ValueError(f"orc_partial_fwd failed ({rc})")
    return out, lse


def attn_fwd(q, k, v, cu, causal: bool, scale: float, rows=None, window: int = -1, q_lo=None, q_hi=None):
    """Full packed (block-diagonal, optionally causal, optionally
    sliding-window, optionally interval-masked by per-token key bounds
    q_lo / q_hi on packed positions) attention."""
    T = int(np.asarray(cu)[-1])
    seg = doc_ids(cu)
    pos = np.arange(T, dtype=np.int64)
    return partial_fwd(q, k, v, seg, seg, pos, pos, causal, scale, rows, window, q_lo, q_hi)


def lse_merge(outs, lses):
    """Merge n partials (out [R,H,d], lse [R,H]) of the same queries."""
    outs = [_f64(o) for o in outs]
    lses = [_f64(l) for l in lses]
    R, H, d = outs[0].shape
    n = len(outs)
    op = (ctypes.c_void_p * n)(*[o.ctypes.data for o in outs])
    lp = (ctypes.c_void_p * n)(*[l.ctypes.data for l in lses])
    out = np.zeros((R, H, d), dtype=np.float64)
    lse = np.zeros((R, H), dtype=np.float64)
    rc = lib().orc_lse_merge(n, op, lp, R, H, d, _p(out), _p(lse))
    if rc:
        raise ValueError("orc_lse_merge failed")
    return out, lse


def attn_bwd(q, k, v, o, lse, dout, cu, causal: bool, scale: float, dq_rows=None, dk_rows=None, window: int = -1,
             q_lo=None, q_hi=None):
    """Gradients (dq, dk, dv) in fp64 given the oracle's own forward (o, lse)
    over the allowed set of attn_fwd with the same arguments.

    o/lse/dout are [T,Hq,d]/[T,Hq]/[T,Hq,d]; rows that no requested output
    depends on may hold zeros."""
    q, k, v, o, lse, dout = map(_f64, (q, k, v, o, lse, dout))
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    seg = doc_ids(cu)
    pos = np.arange(T, dtype=np.int64)
    if dq_rows is None:
        nq, qp, qa = T, None, None
    else:
        qa = _i64(dq_rows)
        nq, qp = len(qa), _p(qa)
    if dk_rows is None:
        nk, kp, ka = T, None, None
    else:
        ka = _i64(dk_rows)
        nk, kp = len(ka), _p(ka)
    lo_a, lo_p = _bounds(q_lo, T)
    hi_a, hi_p = _bounds(q_hi, T)
    dq = np.zeros((nq, Hq, d))
    dk = np.zeros((nk, Hkv, d))
    dv = np.zeros((nk, Hkv, d))
    rc = lib().orc_attn_bwd(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(dout), T, Hq, Hkv, d,
                            _p(seg), _p(pos), int(bool(causal)), int(window), float(scale), lo_p, hi_p, qp, nq,
                            kp, nk, _p(dq), _p(dk), _p(dv))
    if rc:
        raise ValueError("orc_attn_bwd failed")
    return dq, dk, dv


def zigzag_owner(cu, cp: int, mode: int) -> np.ndarray:
    cu = _i32(cu)
    T = int(cu[-1])
    owner = np.zeros(T, dtype=np.int32)
    rc = lib().orc_zigzag_owner(_p(cu), len(cu) - 1, cp, mode, _p(owner))
    if rc:
        raise ValueError(f"orc_zigzag_owner failed ({rc})")
    return owner


def zigzag_plan(cu, cp: int, mode: int):
    """(perm [T], off [cp+1], cu_local [cp, B+1]) as int32."""
    cu = _i32(cu)
    B = len(cu) - 1
    T = int(cu[-1])
    perm = np.zeros(T, dtype=np.int32)
    off = np.zeros(cp + 1, dtype=np.int32)
    cl = np.zeros((cp, B + 1), dtype=np.int32)
    rc = lib().orc_zigzag_plan(_p(cu), B, cp, mode, _p(perm), _p(off), _p(cl))
    if rc:
        raise ValueError(f"orc_zigzag_plan failed ({rc})")
    return perm, off, cl


def rank_pairs(cu, cp: int, mode: int, causal: bool = True, window: int = -1) -> np.ndarray:
    cu = _i32(cu)
    counts = np.zeros(cp, dtype=np.int64)
    rc = lib().orc_rank_pairs(_p(cu), len(cu) - 1, cp, mode, int(bool(causal)), int(window), _p(counts))
    if rc:
        raise ValueError("orc_rank_pairs failed")
    return counts


def ring_fwd(q, k, v, cu, cp: int, mode: int, causal: bool, scale: float, window: int = -1):
    """The ring schedule written out step by step in fp64: zigzag-permute,
    for every rank r and step t take the partial of rank r's queries against
    rank s=(r-t) mod cp's keys, merge the cp partials, undo the permutation.
    Returns (out [T,Hq,d], lse [T,Hq]) in the original token order."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, d = q.shape
    perm, off, _ = zigzag_plan(cu, cp, mode)
    seg = doc_ids(cu)
    out = np.zeros((T, Hq, d))
    lse = np.zeros((T, Hq))
    for r in range(cp):
        qi = perm[off[r]:off[r + 1]]
        parts_o, parts_l = [], []
        for t in range(cp):
            s = (r - t) % cp
            ki = perm[off[s]:off[s + 1]]
            o_p, l_p = partial_fwd(q[qi], k[ki], v[ki], seg[qi], seg[ki], qi, ki, causal, scale, window=window)
            parts_o.append(o_p)
            parts_l.append(l_p)
        o_r, l_r = lse_merge(parts_o, parts_l)
        out[qi] = o_r
        lse[qi] = l_r
    return out, lse
