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
        for cp in (1, 2, 3, 8):
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
    assert n == 48


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
    assert ag["fwd_capacity"] < ring["fwd_capacity"]
    assert ref / ag["fwd_capacity"] > 0.9 > ref / ring["fwd_capacity"] > 0.75


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
    out = np.zeros(19, np.int64)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 4, 2, 1, -1, 7, 0, 152, p(out)) == _lib.RA_ERR_INVALID_ARG  # schedule
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 3, 2, 1, -1, 0, 0, 152, p(out)) == _lib.RA_ERR_INVALID_ARG  # G
    assert L.ra_ring_plan_stats(p(cu), 1, 0, 0, 4, 2, 1, -1, 0, 0, 152, p(out)) == _lib.RA_ERR_INVALID_ARG  # cp
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 4, 2, 1, -1, 0, 0, 152, None) == _lib.RA_ERR_INVALID_ARG
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 4, 2, 1, -1, 0, 0, 0, p(out)) == _lib.RA_ERR_INVALID_ARG  # n_sm
    assert L.ra_ring_plan_stats(p(cu), 1, 2, 0, 4, 2, 1, -1, 0, 0, 152, p(out)) == 0
    assert out[10] == -1 and out[0] > 0
