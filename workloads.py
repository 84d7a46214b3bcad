"""Seeded synthetic workloads for packed causal varlen ring attention.

This module only *generates inputs*: document lengths, cumulative sequence
lengths and N(0,1) Q/K/V/dO tensors.  It holds none of the attention,
zigzag or merge arithmetic, so both the CUDA path and the CPU oracle can
draw their inputs from it without sharing any of the method.

The five workloads follow the packing scenarios discussed on the pages:
packed variable-length documents (EasyDeL issue #129, "Attention Mask for
Packed Sequences"), long single sequences split over context-parallel ranks
with zigzag balancing (ring-attention-pytorch issue #20, `extract_local`;
maxtext PR #1133, review comment on load-balanced reordering) and GQA
(ring-attention-pytorch issue #20, the Llama 3 remark).  No public dataset
is named by the pages; document lengths are drawn log-uniformly instead.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

ZZ_GLOBAL = 0
ZZ_PER_DOC = 1


@dataclass(frozen=True)
class Workload:
    name: str
    doc_lens: tuple
    hq: int
    hkv: int
    d: int
    dtype: torch.dtype
    cp: int
    zz_mode: int
    causal: bool = True
    bwd: bool = False
    note: str = field(default="", compare=False)

    @property
    def T(self) -> int:
        return int(sum(self.doc_lens))

    @property
    def B(self) -> int:
        return len(self.doc_lens)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def cu_seqlens(self) -> np.ndarray:
        return cu_seqlens(self.doc_lens)


def cu_seqlens(doc_lens) -> np.ndarray:
    """int32 cumulative lengths [0, L0, L0+L1, ...] (B+1 entries)."""
    cu = np.zeros(len(doc_lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(doc_lens, dtype=np.int64))
    assert cu[-1] < 2**31
    return cu.astype(np.int32)


def loguniform_doc_lens(total: int, lo: int = 128, hi: int = 8192, seed: int = 0) -> list:
    """Draw floor(exp(U(ln lo, ln hi))) lengths from numpy's default_rng(seed)
    until they cover `total` tokens; the last document is truncated."""
    rng = np.random.default_rng(seed)
    lens, s = [], 0
    while s < total:
        x = int(math.floor(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
        x = min(x, total - s)
        lens.append(x)
        s += x
    return lens


def _c2_lens():
    return tuple(loguniform_doc_lens(32768, 128, 8192, 0))


# The five synthetic configurations (named C0..C4).
C0 = Workload("C0 tiny packed fp32: docs {37,64,27}=128 tok, 2/2 heads, d64, global zigzag CP=2, fwd",
              (37, 64, 27), 2, 2, 64, torch.float32, 2, ZZ_GLOBAL)
C1 = Workload("C1 single seq 8192, GQA 32/8, d128, bf16, zigzag CP=4, fwd",
              (8192,), 32, 8, 128, torch.bfloat16, 4, ZZ_GLOBAL)
C2 = Workload("C2 packed varlen 32768 tok (log-uniform [128,8192] docs, seed 0), GQA 32/8, d128, bf16, per-doc zigzag CP=8, fwd",
              _c2_lens(), 32, 8, 128, torch.bfloat16, 8, ZZ_PER_DOC)
C3 = Workload("C3 long single seq 131072, GQA 64/8, d128, bf16, zigzag CP=16, fwd",
              (131072,), 64, 8, 128, torch.bfloat16, 16, ZZ_GLOBAL)
C4 = Workload("C4 fwd+bwd of the packed 32768-token workload, GQA 32/8, d128, bf16, per-doc zigzag CP=8",
              _c2_lens(), 32, 8, 128, torch.bfloat16, 8, ZZ_PER_DOC, bwd=True)

ALL = {"C0": C0, "C1": C1, "C2": C2, "C3": C3, "C4": C4}

SEED_Q, SEED_K, SEED_V, SEED_DO = 1, 2, 3, 4


def randn(shape, seed: int, dtype: torch.dtype) -> torch.Tensor:
    """N(0,1) drawn in fp32 on the CPU from torch.Generator(seed), then cast."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)


def make_qkv(T: int, hq: int, hkv: int, d: int, dtype: torch.dtype, seed_offset: int = 0):
    """Q [T,hq,d], K/V [T,hkv,d] on the CPU (THD layout, d contiguous)."""
    q = randn((T, hq, d), SEED_Q + seed_offset, dtype)
    k = randn((T, hkv, d), SEED_K + seed_offset, dtype)
    v = randn((T, hkv, d), SEED_V + seed_offset, dtype)
    return q, k, v


def make_dout(T: int, hq: int, d: int, dtype: torch.dtype, seed_offset: int = 0):
    return randn((T, hq, d), SEED_DO + seed_offset, dtype)


def random_doc_lens(rng: np.random.Generator, total_max: int, lmin: int = 1, lmax: int = 300) -> list:
    """Small random packings for edge-case tests (lengths in [lmin, lmax])."""
    lens, s = [], 0
    while True:
        x = int(rng.integers(lmin, lmax + 1))
        if s + x > total_max:
            break
        lens.append(x)
        s += x
    if not lens:
        lens = [max(1, min(lmax, total_max))]
    return lens


def sample_rows(T: int, n: int, seed: int, must_include=()) -> np.ndarray:
    """Sorted unique query rows: `must_include` plus seeded random rows."""
    rng = np.random.default_rng(seed)
    rows = set(int(x) for x in must_include if 0 <= int(x) < T)
    while len(rows) < min(n, T):
        rows.add(int(rng.integers(0, T)))
    return np.array(sorted(rows), dtype=np.int64)


def interval_bounds(cu, kind: str, param: int = 0, seed: int = 0):
    """Per-token key intervals of a packed batch, on packed positions: query
    i sees key j of its own document iff lo[i] <= j <= hi[i].  Both arrays
    are non-decreasing inside every document.  Kinds:
      causal         lo = document start, hi = i
      window         lo = max(start, i - param), hi = i  (param = window)
      chunked        lo = start of i's block of `param` tokens, hi = i
      prefix         bidirectional over the first `param` tokens of each
                     document, causal after: lo = start,
                     hi = max(i, start + param - 1) (capped at the end)
      bidirectional  lo = start, hi = end - 1
      random         seeded non-decreasing lo and hi inside each document,
                     with some rows empty (lo > hi)
    Returns (lo, hi) as int32 arrays [T]."""
    cu = np.asarray(cu, dtype=np.int64)
    T = int(cu[-1])
    lo = np.zeros(T, dtype=np.int64)
    hi = np.zeros(T, dtype=np.int64)
    rng = np.random.default_rng(seed)
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        if e <= s:
            continue
        i = np.arange(s, e, dtype=np.int64)
        if kind == "causal":
            lo[s:e], hi[s:e] = s, i
        elif kind == "window":
            lo[s:e], hi[s:e] = np.maximum(s, i - param), i
        elif kind == "chunked":
            lo[s:e], hi[s:e] = s + (i - s) // param * param, i
        elif kind == "prefix":
            lo[s:e], hi[s:e] = s, np.minimum(np.maximum(i, s + param - 1), e - 1)
        elif kind == "bidirectional":
            lo[s:e], hi[s:e] = s, e - 1
        elif kind == "random":
            L = e - s
            a = np.sort(rng.integers(s, e, L))
            c = np.sort(rng.integers(s - 2, e + 2, L))
            lo[s:e], hi[s:e] = a, np.clip(c, s - 1, e - 1)
        else:
            raise ValueError(kind)
    return lo.astype(np.int32), hi.astype(np.int32)


def interval_pairs(cu, lo, hi) -> int:
    """Allowed (query, key) pairs of an interval mask (keys of the query's
    own document inside [lo, hi])."""
    cu = np.asarray(cu, dtype=np.int64)
    T = int(cu[-1])
    start = np.repeat(cu[:-1], np.diff(cu))
    end = np.repeat(cu[1:], np.diff(cu)) - 1
    a = np.maximum(np.asarray(lo, np.int64), start)
    b = np.minimum(np.asarray(hi, np.int64), end)
    return int(np.maximum(b - a + 1, 0).sum()) if T else 0
