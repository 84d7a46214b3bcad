"""C-ABI checks that need no GPU: the library loads and exports every
symbol include/ra.h declares; the host planner matches the oracle bit for
bit; argument checks return their status without launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def ra():
    from context_varlen_ring_gb300 import build as b
    b.build()
    import context_varlen_ring_gb300 as m
    m.lib()
    return m


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "ra.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(ra):
    from context_varlen_ring_gb300 import _lib
    names = _declared_symbols()
    assert len(names) >= 15
    L = ra.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.EXPORTS)
    assert b"sm_103a" in L.ra_version()


@pytest.mark.parametrize("mode", [0, 1])
def test_host_planner_matches_oracle(ra, orc, mode):
    rng = np.random.default_rng(11)
    cases = [W.C0.cu_seqlens(), W.C2.cu_seqlens(), np.array([0, 130]), np.array([0, 3, 4, 6])]
    for _ in range(25):
        cases.append(W.cu_seqlens(W.random_doc_lens(rng, 900, 1, 300)))
    for cu in cases:
        for cp in (1, 2, 3, 4, 8, 16):
            p1, o1, c1 = ra.zigzag_plan(cu, cp, mode)
            p2, o2, c2 = orc.zigzag_plan(cu, cp, mode)
            assert np.array_equal(p1, p2) and np.array_equal(o1, o2) and np.array_equal(c1, c2)


def test_rank_pairs_match_oracle(ra, orc):
    rng = np.random.default_rng(12)
    for _ in range(10):
        cu = W.cu_seqlens(W.random_doc_lens(rng, 2000, 1, 600))
        for cp in (1, 2, 4, 8):
            for mode in (0, 1):
                for causal in (True, False):
                    assert np.array_equal(ra.ring_rank_pairs(cu, cp, mode, causal),
                                          orc.rank_pairs(cu, cp, mode, causal))


def test_c3_rank_pairs_closed_form(ra):
    counts = ra.ring_rank_pairs(W.C3.cu_seqlens(), 16, W.ZZ_GLOBAL)
    assert np.all(counts == 536_875_008) and counts.sum() == 8_590_000_128


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def test_invalid_arguments_return_status(ra):
    from context_varlen_ring_gb300 import _lib
    L = ra.lib()
    perm = np.zeros(8, np.int32)
    off = np.zeros(3, np.int32)
    cl = np.zeros(6, np.int32)
    bad_cus = [np.array([1, 8], np.int32), np.array([0, 5, 3], np.int32)]
    for cu in bad_cus:
        assert L.ra_zigzag_plan(_p(cu), len(cu) - 1, 2, 0, _p(perm), _p(off), _p(cl)) == _lib.RA_ERR_INVALID_ARG
        assert L.ra_last_error()
    cu = np.array([0, 8], np.int32)
    assert L.ra_zigzag_plan(_p(cu), 1, 0, 0, _p(perm), _p(off), _p(cl)) == _lib.RA_ERR_INVALID_ARG
    assert L.ra_zigzag_plan(_p(cu), 1, 2, 7, _p(perm), _p(off), _p(cl)) == _lib.RA_ERR_INVALID_ARG
    fake = ctypes.c_void_p(256)  # never dereferenced: checks fail before any launch
    ws = ctypes.c_void_p(4096)
    args = dict(dt=_lib.RA_BF16, T=8, hq=4, hkv=2, d=128)

    def fwd(cu, T=8, hq=4, hkv=2, d=128, cp=2, mode=0, sched=0, dt=_lib.RA_BF16, q=fake):
        return L.ra_ring_attn_fwd(q, fake, fake, dt, T, hq, hkv, d, _p(cu), len(cu) - 1, cp, mode, 1, -1, 0.1, sched,
                                  fake, fake, ws, 1 << 40, None)
    assert fwd(np.array([0, 7], np.int32)) == _lib.RA_ERR_INVALID_ARG          # cu[B] != T
    assert fwd(np.array([0, 8], np.int32), hq=3) == _lib.RA_ERR_INVALID_ARG    # Hq % Hkv
    assert fwd(np.array([0, 8], np.int32), cp=0) == _lib.RA_ERR_INVALID_ARG
    assert fwd(np.array([0, 8], np.int32), mode=5) == _lib.RA_ERR_INVALID_ARG
    assert fwd(np.array([0, 8], np.int32), sched=9) == _lib.RA_ERR_INVALID_ARG
    assert fwd(np.array([0, 8], np.int32), d=100) == _lib.RA_ERR_UNSUPPORTED
    assert fwd(np.array([0, 8], np.int32), dt=7) == _lib.RA_ERR_INVALID_ARG
    assert fwd(np.array([0, 8], np.int32), q=ctypes.c_void_p(258)) == _lib.RA_ERR_UNSUPPORTED  # misaligned
    # too-small workspace is caught before launching
    cu = np.array([0, 8], np.int32)
    rc = L.ra_ring_attn_fwd(fake, fake, fake, _lib.RA_BF16, 8, 4, 2, 128, _p(cu), 1, 2, 0, 1, -1, 0.1, 0, fake, fake,
                            ws, 16, None)
    assert rc == _lib.RA_ERR_WORKSPACE
    # the all-gather schedule is accepted by both ring calls (the check that
    # stops them here is the workspace size, after the plan is built)
    rc = L.ra_ring_attn_fwd(fake, fake, fake, _lib.RA_BF16, 8, 4, 2, 128, _p(cu), 1, 2, 0, 1, -1, 0.1,
                            _lib.RA_SCHED_ALLGATHER, fake, fake, ws, 16, None)
    assert rc == _lib.RA_ERR_WORKSPACE
    rc = L.ra_ring_attn_bwd(fake, fake, fake, _lib.RA_BF16, 8, 4, 2, 128, _p(cu), 1, 2, 0, 1, -1, 0.1,
                            _lib.RA_SCHED_ALLGATHER, fake, fake, fake, fake, fake, fake, _lib.RA_BF16, 0, ws, 16, None)
    assert rc == _lib.RA_ERR_WORKSPACE
    # merge argument checks
    assert L.ra_lse_merge(0, None, None, 4, 2, 128, fake, 0, fake, None) == _lib.RA_ERR_INVALID_ARG
    assert L.ra_lse_merge(65, None, None, 4, 2, 128, fake, 0, fake, None) == _lib.RA_ERR_INVALID_ARG
    assert L.ra_selftest_wait_timeout(0, None) == _lib.RA_ERR_INVALID_ARG
    assert L.ra_status_string(_lib.RA_ERR_TIMEOUT) == b"device wait timed out"


def test_workspace_sizes(ra):
    cu = W.C2.cu_seqlens()
    f = ra.ring_workspace_bytes(32768, 32, 8, 128, 0, cu, 8, W.ZZ_PER_DOC, "fused")
    s = ra.ring_workspace_bytes(32768, 32, 8, 128, 0, cu, 8, W.ZZ_PER_DOC, "stepwise")
    b = ra.ring_workspace_bytes(32768, 32, 8, 128, 0, cu, 8, W.ZZ_PER_DOC, "fused", bwd=True)
    qkv = 32768 * (32 + 16) * 128 * 2
    assert qkv < f < qkv + (64 << 20)
    assert s > f + 8 * 32768 * 32 * 128 * 4
    assert b > f
    # the all-gather schedule keeps the fused layout; its key side is tiled
    # per document (fewer KV tiles and key-side items than the ring shards)
    a = ra.ring_workspace_bytes(32768, 32, 8, 128, 0, cu, 8, W.ZZ_PER_DOC, "allgather")
    ab = ra.ring_workspace_bytes(32768, 32, 8, 128, 0, cu, 8, W.ZZ_PER_DOC, "allgather", bwd=True)
    assert qkv < a <= f and ab <= b and f - a < (1 << 20)
    import ctypes
    from context_varlen_ring_gb300 import _lib
    c = np.ascontiguousarray(cu, dtype=np.int32)
    assert _lib.lib().ra_ring_workspace_bytes(32768, 32, 8, 128, 0, c.ctypes.data_as(ctypes.c_void_p), len(c) - 1,
                                              8, W.ZZ_PER_DOC, 3, 0) == 0  # unknown schedule


def test_ring_rank_pairs_window_matches_oracle(orc):
    """The library's per-rank pair counts under a sliding window equal the
    oracle's (host logic, no GPU)."""
    import context_varlen_ring_gb300 as ra
    rng = np.random.default_rng(21)
    for _ in range(4):
        cu = W.cu_seqlens(W.random_doc_lens(rng, 5000, 1, 900))
        for cp in (1, 3, 8):
            for mode in (0, 1):
                for causal in (True, False):
                    for window in (0, 13, 256, 10**6):
                        assert np.array_equal(ra.ring_rank_pairs(cu, cp, mode, causal, window),
                                              orc.rank_pairs(cu, cp, mode, causal, window))


@pytest.mark.parametrize("G", [1, 4, 16])
def test_partial_workspace_bound_covers_tables(ra, G):
    """ra_partial_workspace_bytes bounds the tables a partial call uploads for
    every position pattern, including positions that break each tile into
    the most runs (a stride of 2 leaves two rows per tile, so the tile and
    item counts are the largest a segment can have)."""
    L = ra.lib()
    hkv = 8
    hq = hkv * G
    rng = np.random.default_rng(21)
    cases = []
    for Tq, Tk, nseg in ((4096, 128, 1), (4096, 4096, 3), (777, 1500, 5), (1, 1, 1), (300, 0, 2)):
        cuq = np.sort(np.concatenate([[0, Tq], rng.integers(0, Tq + 1, nseg - 1)])).astype(np.int32)
        cuk = np.sort(np.concatenate([[0, Tk], rng.integers(0, Tk + 1, nseg - 1)])).astype(np.int32)
        for name in ("contiguous", "stride2", "random"):
            if name == "contiguous":
                qp, kp = np.arange(Tq, dtype=np.int32), np.arange(Tk, dtype=np.int32)
            elif name == "stride2":
                qp, kp = 2 * np.arange(Tq, dtype=np.int32), 2 * np.arange(Tk, dtype=np.int32)
            else:
                qp = rng.integers(0, 10 * Tq + 1, Tq).astype(np.int32)
                kp = rng.integers(0, 10 * Tk + 1, max(Tk, 0)).astype(np.int32)
            cases.append((Tq, Tk, nseg, cuq, cuk, qp, kp))
    for Tq, Tk, nseg, cuq, cuk, qp, kp in cases:
        bound = L.ra_partial_workspace_bytes(Tq, Tk, nseg, hq, hkv, 128, 0)
        for causal in (0, 1):
            exact = L.ra_partial_table_bytes(Tq, Tk, hq, hkv, 128, 0, _p(cuq), _p(cuk), nseg, _p(qp),
                                             _p(kp) if Tk else None, causal, -1)
            assert 0 < exact <= bound, (Tq, Tk, nseg, causal, exact, bound)
    # the case of the finding: 4096 queries at a stride of 2 against 128 keys
    cu_q, cu_k = np.array([0, 4096], np.int32), np.array([0, 128], np.int32)
    qp, kp = 2 * np.arange(4096, dtype=np.int32), np.arange(128, dtype=np.int32)
    exact = L.ra_partial_table_bytes(4096, 128, 32, 8, 128, 0, _p(cu_q), _p(cu_k), 1, _p(qp), _p(kp), 1, -1)
    assert exact <= L.ra_partial_workspace_bytes(4096, 128, 1, 32, 8, 128, 0)
