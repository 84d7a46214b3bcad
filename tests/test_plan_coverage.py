"""Host-only pins of the tile planner (no GPU): walking every work item of
the three tensor-core passes over its ring steps, with the kernels' own
step-to-rank rule and tile classifier, must meet every allowed (query, key)
pair exactly once, and a tile pair classified "full" (run without a mask)
must hold no masked pair.  The allowed-pair totals come from the oracle's
own per-rank count (a separate restatement of the zigzag split and the
mask), so a dropped ring step, a wrong step range of a work item, a
misclassified tile or a tile that straddles a document fails here."""
import numpy as np
import pytest

import workloads as W


@pytest.fixture(scope="module")
def ra():
    import context_varlen_ring_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("sched", ["fused", "allgather"])
@pytest.mark.parametrize("causal", [True, False])
def test_every_allowed_pair_once(ra, orc, sched, causal):
    rng = np.random.default_rng(40 + causal + 2 * (sched == "allgather"))
    n = 0
    for trial in range(6):
        cu = W.cu_seqlens(W.random_doc_lens(rng, int(rng.integers(60, 1500)), 1, 500))
        for cp in (1, 2, 3, 8, 16):
            for mode in (0, 1):
                G = int(rng.choice([1, 2, 4, 8, 16]))
                window = int(rng.choice([-1, -1, 0, 5, 130]))
                ref = int(orc.rank_pairs(cu, cp, mode, causal, window=window).sum())
                st = ra.ring_plan_stats(cu, cp, mode, G, 2, causal, window, sched, exact=True)
                case = (sched, causal, list(np.diff(cu)), cp, mode, G, window)
                assert st["fwd_allowed"] == ref, case
                assert st["dkdv_allowed"] == ref, case
                assert st["dq_allowed"] == ref, case
                assert st["full_disallowed"] == 0, case
                assert st["fwd_visited"] == st["dq_visited"] == st["dkdv_visited"], case
                assert st["fwd_capacity"] == st["fwd_visited"] * (128 // G) * 128
                assert st["dq_items"] == 2 * st["q_tiles"]  # one per query tile and KV head (Hkv = 2)
                if sched == "allgather":
                    assert st["two_run_kv_rows"] == 0, case
                n += 1
    assert n == 60


def test_packed_workload_tiling(ra, orc):
    """The 32768-token packing (GQA 32/8, CP 8, per-document zigzag): both
    schedules cover the 67 823 768 allowed pairs in every pass; per-document
    key tiles leave less of the tensor work masked or padded than the
    ring's per-rank shards (265 against 328 key tiles)."""
    wl = W.C2
    cu = wl.cu_seqlens()
    ref = int(orc.rank_pairs(cu, wl.cp, wl.zz_mode, True).sum())
    assert ref == 67823768
    ring = ra.ring_plan_stats(cu, wl.cp, wl.zz_mode, 4, 8, True, -1, "fused", exact=True)
    ag = ra.ring_plan_stats(cu, wl.cp, wl.zz_mode, 4, 8, True, -1, "allgather", exact=True)
    for st in (ring, ag):
        assert st["fwd_allowed"] == st["dkdv_allowed"] == st["dq_allowed"] == ref
        assert st["full_disallowed"] == 0
        assert st["q_tiles"] == 1080 and st["two_run_q_rows"] == 3174
    assert ring["kv_tiles"] == 328 and ag["kv_tiles"] == 265
    assert ring["two_run_kv_rows"] == 10938 and ag["two_run_kv_rows"] == 0
    # forward items pair a document's query tiles across ranks by visit
    # count: the KV steps they walk match a separate restatement of the
    # tiling and the pairing (10 700 per KV head, the lower bound of half the
    # 21 264 visits being 10 632; pairing within each rank's share walks 11 236,
    # consecutive tiles of a share 11 768)
    lens, qtok = np.diff(cu), 128 // (wl.hq // wl.hkv)
    assert ring["fwd_steps"] == _ring_fwd_steps(lens, wl.cp, qtok) == 10700
    assert _ring_fwd_steps(lens, wl.cp, qtok, cross_rank=False) == 11236
    assert _ring_fwd_steps(lens, wl.cp, qtok, pair_sorted=False, cross_rank=False) == 11768
    for st in (ring, ag):
        assert 2 * st["fwd_steps"] >= st["fwd_visited"]
    assert ag["fwd_capacity"] < ring["fwd_capacity"]
    assert ref / ag["fwd_capacity"] > 0.9 > ref / ring["fwd_capacity"] > 0.75


def test_one_run_tiling_has_the_most_kv_tiles(ra):
    """The workspace size query counts the KV tiles of the tiling that cuts
    every rank's share at its chunk boundary (one position run per tile).
    Whatever a mask or window makes the planner choose per share, its plan
    has no more KV tiles than that (per-document zigzag, restated here)."""
    rng = np.random.default_rng(23)
    for trial in range(12):
        lens = W.random_doc_lens(rng, int(rng.integers(300, 6000)), 1, 2500)
        cu = W.cu_seqlens(lens)
        for cp in (2, 4, 8):
            one_run = 0
            for L in (int(x) for x in lens):
                bnd = [c * L // (2 * cp) for c in range(2 * cp + 1)]
                for r in range(cp):
                    sh = list(range(bnd[r], bnd[r + 1])) + list(range(bnd[2 * cp - 1 - r], bnd[2 * cp - r]))
                    one_run += len(_runs_tiles(sh, 128, 1))
            cases = [dict(window=w) for w in (-1, 0, 64, 1024)]
            for kind, par in (("chunked", 200), ("random", 0), ("window", 100)):
                lo, hi = W.interval_bounds(cu, kind, par, seed=trial)
                cases.append(dict(key_lo=lo, key_hi=hi))
            for kw in cases:
                st = ra.ring_plan_stats(cu, cp, 1, 4, 2, True, sched="fused", **kw)
                assert st["kv_tiles"] <= one_run, (trial, cp, kw.keys())


def _runs_tiles(pos, rows, max_runs=2):
    """Greedy tiles of at most `rows` positions and at most `max_runs` runs
    of consecutive positions (the planner's rule), as arrays of positions."""
    out, i, n = [], 0, len(pos)
    while i < n:
        s = i
        i += 1
        while i < n and i - s < rows and pos[i] == pos[i - 1] + 1:
            i += 1
        if max_runs > 1 and i < n and i - s < rows:
            i += 1
            while i < n and i - s < rows and pos[i] == pos[i - 1] + 1:
                i += 1
        out.append(np.asarray(pos[s:i]))
    return out


def _ring_fwd_steps(lens, cp, q_tokens, pair_sorted=True, window=-1, kv_runs=2, visits=False, cross_rank=True):
    # kv_runs: 1 or 2 runs per KV tile, or 0: per rank shard, the tiling the
    # forward visits less
    """KV tiles walked by the causal ring forward's items of one KV head:
    per document and rank, the rank's two zigzag chunks (floor(c*L/2cp)
    bounds) cut into query tiles of q_tokens and KV tiles of 128 (of at
    most kv_runs position runs); a query tile needs every KV tile of its
    document (all ranks) starting at or before its last position (and, with
    a window w, ending at or after its first position - w); tiles of a
    document (across ranks; cross_rank=False: of each rank's share) paired
    by need, largest first (or consecutively); an item walks the union of
    its pair's needs.  visits=True: the query tiles' needs summed instead."""
    steps = 0
    for L in (int(x) for x in lens):
        n = 2 * cp
        bnd = [c * L // n for c in range(n + 1)]
        shards = [list(range(bnd[r], bnd[r + 1])) + list(range(bnd[n - 1 - r], bnd[n - r])) for r in range(cp)]
        qall = [t for sh in shards for t in _runs_tiles(sh, q_tokens)]
        qmax, qmin = np.array([t.max() for t in qall]), np.array([t.min() for t in qall])

        def seg_visits(kt):  # tile pairs of this shard's KV tiles with every query tile of the document
            return sum(int(((k.min() <= qmax) & ((k.max() >= qmin - window) if window >= 0 else True)).sum())
                       for k in kt)

        kt = []
        for sh in shards:  # kv_runs 0: each shard's tiling with fewer visits (two runs on a tie)
            one, two = _runs_tiles(sh, 128, 1), _runs_tiles(sh, 128, 2)
            pick = {1: one, 2: two}.get(kv_runs) or (one if seg_visits(one) < seg_visits(two) else two)
            kt += pick
        kmin = np.array([t.min() for t in kt])
        kmax = np.array([t.max() for t in kt])
        # pairing groups: the whole document across ranks, or each rank's share
        groups = [qall] if cross_rank else [_runs_tiles(sh, q_tokens) for sh in shards]
        for qt in groups:
            need = [(kmin <= t.max()) & ((kmax >= t.min() - window) if window >= 0 else True) for t in qt]
            if visits:
                steps += int(sum(x.sum() for x in need))
                continue
            idx = list(range(len(qt)))
            if pair_sorted:
                idx.sort(key=lambda i: (int(need[i].sum()), int(qt[i].max())), reverse=True)
            for j in range(0, len(idx), 2):
                u = need[idx[j]] | (need[idx[j + 1]] if j + 1 < len(idx) else False)
                steps += int(u.sum())
    return steps


@pytest.mark.parametrize("window", [-1, 1024, 256, 64])
def test_ring_kv_tiling_takes_fewer_visits(ra, window):
    """The ring planner keeps, per rank's share of a document, whichever KV
    tiling (tiles of at most two position runs, or of one) the forward
    visits less: its visits and steps match the restatement, and they are at
    most those of either tiling throughout (the causal mask keeps two runs
    everywhere; a window takes one run in most shares)."""
    wl = W.C2
    cu = wl.cu_seqlens()
    lens, qtok = np.diff(cu), 128 // (wl.hq // wl.hkv)
    v = {r: _ring_fwd_steps(lens, wl.cp, qtok, window=window, kv_runs=r, visits=True) for r in (0, 1, 2)}
    st = ra.ring_plan_stats(cu, wl.cp, wl.zz_mode, wl.hq // wl.hkv, wl.hkv, True, window, "fused")
    assert st["fwd_visited"] == v[0] <= min(v[1], v[2])
    assert st["fwd_steps"] == _ring_fwd_steps(lens, wl.cp, qtok, window=window, kv_runs=0)
    if window < 0:
        assert v[0] == v[2] and st["two_run_kv_rows"] == 10938
    else:
        assert v[0] < v[1] < v[2]


def test_scheduling_model_bounds(ra):
    """The scheduling model: on one SM every pass takes its whole work (all
    KV heads' visits); on many it takes at least the even share and at most
    the whole."""
    rng = np.random.default_rng(5)
    for _ in range(4):
        cu = W.cu_seqlens(W.random_doc_lens(rng, int(rng.integers(500, 3000)), 1, 900))
        for sched in ("fused", "allgather"):
            one = ra.ring_plan_stats(cu, 4, 1, 4, 2, True, -1, sched, n_sm=1)
            assert one["fwd_makespan"] == 2 * one["fwd_visited"]
            assert one["dkdv_makespan"] == 2 * one["dkdv_visited"]
            assert one["dq_makespan"] == 2 * one["dq_visited"]
            many = ra.ring_plan_stats(cu, 4, 1, 4, 2, True, -1, sched, n_sm=7)
            for k, tot in (("fwd_makespan", 2 * many["fwd_visited"]), ("dkdv_makespan", 2 * many["dkdv_visited"]),
                           ("dq_makespan", 2 * many["dq_visited"])):
                assert -(-tot // 7) <= many[k] <= tot


def test_plan_stats_argument_checks(ra):
    import ctypes
    from context_varlen_ring_gb300 import _lib
    L = _lib.lib()
    cu = np.array([0, 100], np.int32)
    out = np.zeros(20, np.int64)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 4, 2, 1, -1, 7, 0, 152, p(out)) == _lib.RA_ERR_INVALID_ARG  # schedule
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 3, 2, 1, -1, 0, 0, 152, p(out)) == _lib.RA_ERR_INVALID_ARG  # G
    assert L.ra_ring_plan_stats(p(cu), 1, 0, 0, 4, 2, 1, -1, 0, 0, 152, p(out)) == _lib.RA_ERR_INVALID_ARG  # cp
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 4, 2, 1, -1, 0, 0, 152, None) == _lib.RA_ERR_INVALID_ARG
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 4, 2, 1, -1, 0, 0, 0, p(out)) == _lib.RA_ERR_INVALID_ARG  # n_sm
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 4, 2, 1, -1, 0, 0, 152, p(out)) == 0
    assert out[10] == -1 and out[0] > 0


MASKS = [("causal", 0), ("window", 40), ("chunked", 64), ("prefix", 100), ("bidirectional", 0), ("random", 0)]


@pytest.mark.parametrize("sched", ["fused", "allgather"])
def test_interval_masks_cover_every_allowed_pair_once(ra, sched):
    """Interval masks (per-token key bounds): every pass's visited tile
    pairs hold each allowed pair exactly once and no "full" pair holds a
    masked one.  The totals are the brute-force interval counts
    (workloads.interval_pairs, pinned against dense masks in
    test_oracle_bounds.py)."""
    rng = np.random.default_rng(70 + (sched == "allgather"))
    n = 0
    for trial in range(4):
        cu = W.cu_seqlens(W.random_doc_lens(rng, int(rng.integers(60, 1500)), 1, 500))
        for kind, par in MASKS:
            lo, hi = W.interval_bounds(cu, kind, par, seed=trial)
            ref = W.interval_pairs(cu, lo, hi)
            for cp, mode in ((1, 0), (3, 1), (8, int(rng.integers(0, 2)))):
                G = int(rng.choice([1, 2, 4, 8, 16]))
                st = ra.ring_plan_stats(cu, cp, mode, G, 2, sched=sched, exact=True, key_lo=lo, key_hi=hi)
                case = (sched, kind, list(np.diff(cu)), cp, mode, G)
                assert st["fwd_allowed"] == st["dkdv_allowed"] == st["dq_allowed"] == ref, case
                assert st["full_disallowed"] == 0, case
                assert st["fwd_visited"] == st["dq_visited"] == st["dkdv_visited"], case
                n += 1
    assert n == 4 * len(MASKS) * 3


def test_causal_intervals_plan_like_the_causal_mask(ra):
    """Bounds that spell out the causal mask (document start to the query)
    give the block map of the causal plan: the same visited, full and
    capacity counts on the packed workload."""
    wl = W.C2
    cu = wl.cu_seqlens()
    lo, hi = W.interval_bounds(cu, "causal")
    for sched in ("fused", "allgather"):
        a = ra.ring_plan_stats(cu, wl.cp, wl.zz_mode, 4, 8, True, -1, sched)
        b = ra.ring_plan_stats(cu, wl.cp, wl.zz_mode, 4, 8, sched=sched, key_lo=lo, key_hi=hi)
        for key in ("fwd_visited", "fwd_full", "fwd_capacity", "dkdv_visited", "dq_visited", "fwd_items"):
            assert a[key] == b[key], (sched, key)


def test_interval_mask_argument_checks(ra):
    """Host-side refusals, before any device work: bounds that decrease
    inside a document, fp32 (no tensor-core path), the stepwise schedule."""
    import ctypes
    L = ra.lib()
    cu = W.cu_seqlens((50, 30))
    T = 80
    lo, hi = W.interval_bounds(cu, "causal")
    bad = hi.copy()
    bad[10] = bad[9] - 1
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    assert L.ra_ring_workspace_bytes_masked(T, 8, 2, 128, 0, P(cu), 2, 2, 1, P(lo), P(hi), 0, 0) > 0
    assert L.ra_ring_workspace_bytes_masked(T, 8, 2, 128, 0, P(cu), 2, 2, 1, P(lo), P(bad), 0, 0) == 0
    fake = ctypes.c_void_p(256)
    args = lambda dt, l, h, sched: (fake, fake, fake, dt, T, 8, 2, 128, P(cu), 2, 2, 1, P(l), P(h), 0.1, sched,
                                    fake, fake, fake, 1 << 30, None)
    assert L.ra_ring_attn_fwd_masked(*args(0, lo, bad, 0)) == 1  # RA_ERR_INVALID_ARG
    assert b"non-decreasing" in L.ra_last_error()
    assert L.ra_ring_attn_fwd_masked(*args(1, lo, hi, 0)) == 2   # fp32: RA_ERR_UNSUPPORTED
    assert L.ra_ring_attn_fwd_masked(*args(0, lo, hi, 1)) == 2   # stepwise: RA_ERR_UNSUPPORTED
