"""Pins for the fp64 oracle's attention, merge and gradient (CPU only).

Each test checks the oracle against something other than itself: PyTorch's
own scaled_dot_product_attention / logsumexp / autograd in float64 (library
routines), closed forms of degenerate inputs, finite differences, and the
merge invariant (any partition of the keys merges back to full attention).
"""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


def _sdpa_packed(q, k, v, cu, causal, scale):
    """torch SDPA over the packed batch with a dense boolean mask; returns
    (out [T,Hq,d], lse [T,Hq]) with lse from torch.logsumexp of the masked
    score matrix.  GQA by repeat_interleave (kv head g serves q heads gG..gG+G-1)."""
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    kk = k.repeat_interleave(G, dim=1)
    vv = v.repeat_interleave(G, dim=1)
    doc = torch.zeros(T, dtype=torch.long)
    for b in range(len(cu) - 1):
        doc[cu[b]:cu[b + 1]] = b
    mask = doc[:, None] == doc[None, :]
    if causal:
        mask &= torch.ones(T, T, dtype=torch.bool).tril()
    qh, kh, vh = (x.permute(1, 0, 2) for x in (q, kk, vv))
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask, scale=scale)
    scores = torch.einsum("htc,hsc->hts", qh, kh) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
    return out.permute(1, 0, 2), lse.T


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("docs,hq,hkv,d", [((50,), 2, 2, 16), ((37, 64, 27), 4, 2, 32),
                                            ((5, 1, 40, 13, 2), 8, 2, 8), ((3, 90), 6, 1, 24)])
def test_fwd_matches_torch_sdpa(orc, docs, hq, hkv, d, causal):
    cu = W.cu_seqlens(docs)
    T = int(cu[-1])
    q, k, v = _rand((T, hq, d), 1), _rand((T, hkv, d), 2), _rand((T, hkv, d), 3)
    scale = 1.0 / math.sqrt(d)
    out, lse = orc.attn_fwd(q, k, v, cu, causal, scale)
    ref_o, ref_l = _sdpa_packed(q, k, v, cu, causal, scale)
    np.testing.assert_allclose(out, ref_o.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l.numpy(), rtol=0, atol=1e-12)


def test_fwd_rows_subset_equals_full(orc):
    cu = W.cu_seqlens((20, 33, 11))
    T = int(cu[-1])
    q, k, v = _rand((T, 4, 16), 4), _rand((T, 2, 16), 5), _rand((T, 2, 16), 6)
    full_o, full_l = orc.attn_fwd(q, k, v, cu, True, 0.25)
    rows = np.array([0, 5, 19, 20, 52, 63])
    o, l = orc.attn_fwd(q, k, v, cu, True, 0.25, rows=rows)
    np.testing.assert_array_equal(o, full_o[rows])
    np.testing.assert_array_equal(l, full_l[rows])


def test_single_token_doc_closed_form(orc):
    """A document of one token attends only to itself: o = v, lse = s_ii."""
    cu = W.cu_seqlens((7, 1, 9))
    T = int(cu[-1])
    q, k, v = _rand((T, 2, 8), 7), _rand((T, 1, 8), 8), _rand((T, 1, 8), 9)
    out, lse = orc.attn_fwd(q, k, v, cu, True, 0.5)
    i = 7
    for h in range(2):
        np.testing.assert_allclose(out[i, h], v[i, 0].numpy(), atol=1e-15)
        np.testing.assert_allclose(lse[i, h], 0.5 * float(q[i, h] @ k[i, 0]), atol=1e-14)


def test_identical_keys_uniform_weights(orc):
    """All keys equal: every allowed key gets weight 1/|A(i)|, so o is the
    mean of the allowed values and lse = s + log|A(i)|."""
    cu = W.cu_seqlens((12, 5))
    T = int(cu[-1])
    q, v = _rand((T, 2, 8), 10), _rand((T, 2, 8), 11)
    k = _rand((1, 2, 8), 12).expand(T, 2, 8).contiguous()
    out, lse = orc.attn_fwd(q, k, v, cu, True, 0.3)
    for i in range(T):
        b = 0 if i < 12 else 1
        lo = int(cu[b])
        for h in range(2):
            mean = v[lo:i + 1, h].mean(0).numpy()
            np.testing.assert_allclose(out[i, h], mean, atol=1e-13)
            s = 0.3 * float(q[i, h] @ k[0, h])
            np.testing.assert_allclose(lse[i, h], s + math.log(i - lo + 1), atol=1e-13)


def test_empty_rows_give_zero_and_neg_inf(orc):
    Tq, Tk = 6, 5
    q, k, v = _rand((Tq, 2, 4), 13), _rand((Tk, 1, 4), 14), _rand((Tk, 1, 4), 15)
    seg_q = np.array([0, 0, 1, 1, 2, 2])
    seg_k = np.array([0, 0, 0, 1, 1])
    q_pos = np.array([10, 3, 50, 51, 60, 61])
    k_pos = np.array([4, 5, 6, 52, 53])
    out, lse = orc.partial_fwd(q, k, v, seg_q, seg_k, q_pos, k_pos, True, 1.0)
    for i in (1, 2, 3, 4, 5):   # row 1 sees only keys <= 3 (none); seg 1 rows see pos <= 51 (none); seg 2 has no keys
        assert np.all(lse[i] == -np.inf)
        assert np.all(out[i] == 0.0)
    assert np.all(np.isfinite(lse[0]))


def test_merge_of_any_key_partition_equals_full(orc):
    """LSE-merging partials over a partition of the keys (random, including
    empty parts) reproduces full attention (fp64, 1e-12)."""
    rng = np.random.default_rng(0)
    for trial in range(6):
        docs = W.random_doc_lens(rng, 160, 1, 60)
        cu = W.cu_seqlens(docs)
        T = int(cu[-1])
        hq, hkv, d = [(2, 2, 8), (4, 1, 16), (6, 3, 8)][trial % 3]
        q, k, v = _rand((T, hq, d), 20 + trial), _rand((T, hkv, d), 30 + trial), _rand((T, hkv, d), 40 + trial)
        full_o, full_l = orc.attn_fwd(q, k, v, cu, True, 0.3)
        nparts = int(rng.integers(1, 6))
        label = rng.integers(0, nparts + 1, size=T)   # part nparts may stay empty
        seg = orc.doc_ids(cu)
        pos = np.arange(T)
        outs, lses = [], []
        for p in range(nparts + 1):
            idx = np.nonzero(label == p)[0]
            o_p, l_p = orc.partial_fwd(q, k[idx], v[idx], seg, seg[idx], pos, idx, True, 0.3)
            outs.append(o_p)
            lses.append(l_p)
        mo, ml = orc.lse_merge(outs, lses)
        np.testing.assert_allclose(mo, full_o, atol=1e-12, rtol=0)
        np.testing.assert_allclose(ml, full_l, atol=1e-12, rtol=0)


def test_merge_all_empty_and_single_part(orc):
    o1 = np.random.default_rng(1).standard_normal((3, 2, 4))
    l1 = np.array([[0.5, -np.inf], [1.0, 2.0], [-np.inf, -np.inf]])
    o1[0, 1] = 0.0
    o1[2] = 0.0
    mo, ml = orc.lse_merge([o1], [l1])
    np.testing.assert_array_equal(ml, l1)
    np.testing.assert_allclose(mo, o1, atol=1e-15)
    empty_o = np.zeros_like(o1)
    empty_l = np.full_like(l1, -np.inf)
    mo, ml = orc.lse_merge([empty_o, empty_o], [empty_l, empty_l])
    assert np.all(ml == -np.inf) and np.all(mo == 0.0)


@pytest.mark.parametrize("mode", [0, 1])
def test_oracle_ring_schedule_equals_full_attention(orc, mode):
    """The ring written out step by step (zigzag, partial per step, merge,
    un-permute) equals full packed attention for any CP."""
    docs = (37, 64, 27) if mode == 0 else (9, 40, 3, 31)
    cu = W.cu_seqlens(docs)
    T = int(cu[-1])
    q, k, v = _rand((T, 4, 16), 50), _rand((T, 2, 16), 51), _rand((T, 2, 16), 52)
    full_o, full_l = orc.attn_fwd(q, k, v, cu, True, 0.25)
    for cp in (1, 2, 3, 4):
        ro, rl = orc.ring_fwd(q, k, v, cu, cp, mode, True, 0.25)
        np.testing.assert_allclose(ro, full_o, atol=1e-12, rtol=0)
        np.testing.assert_allclose(rl, full_l, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [True, False])
def test_bwd_matches_torch_autograd(orc, causal):
    docs = (11, 1, 23, 6)
    cu = W.cu_seqlens(docs)
    T = int(cu[-1])
    hq, hkv, d = 4, 2, 8
    scale = 1.0 / math.sqrt(d)
    q, k, v = _rand((T, hq, d), 60), _rand((T, hkv, d), 61), _rand((T, hkv, d), 62)
    do = _rand((T, hq, d), 63)
    o, l = orc.attn_fwd(q, k, v, cu, causal, scale)
    dq, dk, dv = orc.attn_bwd(q, k, v, o, l, do, cu, causal, scale)
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    ref_o, _ = _sdpa_packed(qq, kk, vv, cu, causal, scale)
    ref_o.backward(do)
    np.testing.assert_allclose(dq, qq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vv.grad.numpy(), atol=1e-12)


def test_bwd_finite_differences(orc):
    """Central differences of L = sum(dO * O) in fp64."""
    cu = W.cu_seqlens((5, 7))
    T = int(cu[-1])
    q, k, v = _rand((T, 2, 4), 70), _rand((T, 1, 4), 71), _rand((T, 1, 4), 72)
    do = _rand((T, 2, 4), 73)
    o, l = orc.attn_fwd(q, k, v, cu, True, 0.7)
    dq, dk, dv = orc.attn_bwd(q, k, v, o, l, do, cu, True, 0.7)

    def loss(q_, k_, v_):
        oo, _ = orc.attn_fwd(q_, k_, v_, cu, True, 0.7)
        return float((oo * do.numpy()).sum())

    eps = 1e-6
    rng = np.random.default_rng(3)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)
            xp, xm = x.clone(), x.clone()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (loss(**{a + "_": b for a, b in args_p.items()}) -
                  loss(**{a + "_": b for a, b in args_m.items()})) / (2 * eps)
            assert abs(fd - g[idx]) < 1e-7, (name, idx, fd, g[idx])


def test_bwd_row_subsets_equal_full(orc):
    cu = W.cu_seqlens((13, 20))
    T = int(cu[-1])
    q, k, v = _rand((T, 4, 8), 80), _rand((T, 2, 8), 81), _rand((T, 2, 8), 82)
    do = _rand((T, 4, 8), 83)
    o, l = orc.attn_fwd(q, k, v, cu, True, 0.35)
    dq, dk, dv = orc.attn_bwd(q, k, v, o, l, do, cu, True, 0.35)
    rq, rk = np.array([0, 12, 13, 32]), np.array([1, 30, 13])
    sq, sk, sv = orc.attn_bwd(q, k, v, o, l, do, cu, True, 0.35, dq_rows=rq, dk_rows=rk)
    np.testing.assert_array_equal(sq, dq[rq])
    np.testing.assert_array_equal(sk, dk[rk])
    np.testing.assert_array_equal(sv, dv[rk])


def test_bwd_sum_invariants(orc):
    """sum_j dV_j (per kv head) = sum over its q heads of sum_i dO_i, because
    every row of P sums to 1; and sum_j dK_j = 0 because sum_j dS_ij = 0."""
    cu = W.cu_seqlens((17, 4, 30))
    T = int(cu[-1])
    q, k, v = _rand((T, 4, 8), 90), _rand((T, 2, 8), 91), _rand((T, 2, 8), 92)
    do = _rand((T, 4, 8), 93)
    o, l = orc.attn_fwd(q, k, v, cu, True, 0.35)
    _, dk, dv = orc.attn_bwd(q, k, v, o, l, do, cu, True, 0.35)
    for g in range(2):
        np.testing.assert_allclose(dv[:, g].sum(0), do[:, 2 * g:2 * g + 2].sum((0, 1)).numpy(), atol=1e-12)
        np.testing.assert_allclose(dk[:, g].sum(0), 0.0, atol=1e-12)
