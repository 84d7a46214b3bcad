"""Pins for the oracle's zigzag plan and per-rank pair counts (CPU only).

The zigzag rule (ring-attention-pytorch #20, `extract_local`; maxtext
PR #1133, review comment on load-balanced reordering): cut the stream into
2*CP chunks, rank r keeps chunks r and 2*CP-1-r.  The pages use
torch.chunk, which is only well defined here when 2*CP divides the length;
the restatement below uses it exactly there.  Longer checks: a hand-derived
worked example (tests/golden/c0_zigzag.txt) and the closed-form per-rank
causal work of a single sequence.
"""
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden", "c0_zigzag.txt")


def _read_golden():
    vals = {}
    for line in open(GOLD):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        vals[key] = rest
    return vals


def _ranges(tokens):
    out = []
    for t in tokens:
        a, b = t.split(":")
        out.extend(range(int(a), int(b)))
    return out


def test_c0_worked_example(orc):
    g = _read_golden()
    cu = np.array([int(x) for x in g["cu"]])
    cp = int(g["cp"][0])
    perm, off, cl = orc.zigzag_plan(cu, cp, W.ZZ_GLOBAL)
    assert list(off) == [int(x) for x in g["off"]]
    assert list(cl[0]) == [int(x) for x in g["cu_local0"]]
    assert list(cl[1]) == [int(x) for x in g["cu_local1"]]
    assert list(perm[off[0]:off[1]]) == _ranges(g["perm_rank0"])
    assert list(perm[off[1]:off[2]]) == _ranges(g["perm_rank1"])
    assert list(orc.rank_pairs(cu, cp, W.ZZ_GLOBAL)) == [int(x) for x in g["pairs"]]


def _chunk_restatement(L, cp, r):
    """Rank r's token indices per the pages' recipe, using torch.chunk on an
    index vector (valid when 2*cp divides L)."""
    pieces = torch.arange(L).chunk(2 * cp)
    assert len(pieces) == 2 * cp
    mine = [pieces[r], pieces[2 * cp - 1 - r]]
    return torch.cat(mine).tolist()


@pytest.mark.parametrize("L,cp", [(8, 1), (16, 2), (96, 3), (128, 4), (1024, 8), (64, 16)])
def test_matches_chunk_restatement_when_divisible(orc, L, cp):
    perm, off, cl = orc.zigzag_plan(np.array([0, L]), cp, W.ZZ_GLOBAL)
    for r in range(cp):
        assert list(perm[off[r]:off[r + 1]]) == _chunk_restatement(L, cp, r)
    # per-document mode of a single document is the same split
    perm2, off2, _ = orc.zigzag_plan(np.array([0, L]), cp, W.ZZ_PER_DOC)
    assert np.array_equal(perm, perm2) and np.array_equal(off, off2)


def test_per_doc_mode_applies_rule_to_each_doc(orc):
    docs = (32, 64, 16)
    cu = W.cu_seqlens(docs)
    cp = 4
    perm, off, cl = orc.zigzag_plan(cu, cp, W.ZZ_PER_DOC)
    for r in range(cp):
        expect = []
        for b, L in enumerate(docs):
            expect += [int(cu[b]) + x for x in _chunk_restatement(L, cp, r)]
        assert list(perm[off[r]:off[r + 1]]) == expect
        assert list(np.diff(cl[r])) == [2 * L // (2 * cp) for L in docs]


@pytest.mark.parametrize("mode", [0, 1])
def test_plan_is_a_bijection_and_sorted_per_rank(orc, mode):
    rng = np.random.default_rng(5)
    for _ in range(20):
        docs = W.random_doc_lens(rng, 700, 1, 200)
        cu = W.cu_seqlens(docs)
        T = int(cu[-1])
        for cp in (1, 2, 3, 5, 8):
            perm, off, cl = orc.zigzag_plan(cu, cp, mode)
            assert sorted(perm.tolist()) == list(range(T))
            assert off[0] == 0 and off[-1] == T
            inv = np.empty(T, dtype=np.int64)
            inv[perm] = np.arange(T)
            x = np.arange(T) * 7 + 3
            assert np.array_equal(x[perm][inv], x)          # unpermute(permute(x)) == x
            for r in range(cp):
                mine = perm[off[r]:off[r + 1]]
                assert np.all(np.diff(mine) > 0)            # local order = global order
                assert cl[r, 0] == 0 and cl[r, -1] == off[r + 1] - off[r]
                docs_of = orc.doc_ids(cu)[mine]
                assert np.array_equal(np.diff(cl[r]), np.bincount(docs_of, minlength=len(docs)))


def test_balanced_split_when_not_divisible(orc):
    """Length 130 over 2*CP = 16 chunks: chunk c is [floor(c*130/16), floor((c+1)*130/16));
    sizes differ by at most one and rank r still holds chunks r and 15-r."""
    L, cp = 130, 8
    owner = orc.zigzag_owner(np.array([0, L]), cp, W.ZZ_GLOBAL)
    bounds = [(c * L) // 16 for c in range(17)]
    for c in range(16):
        rank = c if c < cp else 15 - c
        assert np.all(owner[bounds[c]:bounds[c + 1]] == rank)
    sizes = np.diff(bounds)
    assert sizes.max() - sizes.min() <= 1


def test_short_docs_leave_ranks_empty(orc):
    cu = W.cu_seqlens((3, 1, 2))
    perm, off, cl = orc.zigzag_plan(cu, 4, W.ZZ_PER_DOC)
    assert sorted(perm.tolist()) == list(range(6))
    counts = np.diff(off)
    assert counts.sum() == 6 and (counts == 0).any()


@pytest.mark.parametrize("cp,c", [(1, 5), (2, 3), (4, 1024), (3, 17)])
def test_closed_form_rank_work_single_sequence(orc, cp, c):
    """Single causal sequence of T = 2*cp*c tokens: every rank gets
    2*cp*c^2 + c allowed pairs (sum T(T+1)/2)."""
    T = 2 * cp * c
    counts = orc.rank_pairs(np.array([0, T]), cp, W.ZZ_GLOBAL)
    assert np.all(counts == 2 * cp * c * c + c)
    assert counts.sum() == T * (T + 1) // 2


def test_c1_rank_work(orc):
    counts = orc.rank_pairs(W.C1.cu_seqlens(), W.C1.cp, W.C1.zz_mode)
    assert np.all(counts == 8_389_632) and counts.sum() == 33_558_528


def test_c2_total_pairs_and_balance(orc):
    cu = W.C2.cu_seqlens()
    counts = orc.rank_pairs(cu, W.C2.cp, W.C2.zz_mode)
    lens = np.diff(cu).astype(np.int64)
    assert counts.sum() == int((lens * (lens + 1) // 2).sum()) == 67_823_768
    assert counts.max() / counts.mean() - 1 < 0.005
