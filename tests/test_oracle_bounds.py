"""Pins for the oracle's interval masks (CPU only).

Flex-style dynamic masks ("[Train] Support custom attention with context
parallel", FlagScale PR #910, description) written as per-token key
intervals: query i sees key j of its own document iff lo[i] <= j <= hi[i].
Each test checks the oracle against something other than itself: PyTorch's
scaled_dot_product_attention / logsumexp / autograd in float64 with a dense
mask built from the intervals, closed forms (a query that sees only itself;
identical keys), brute-force pair counts, and the LSE merge of a key
partition.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W

KINDS = [("causal", 0), ("window", 5), ("chunked", 8), ("prefix", 10), ("bidirectional", 0), ("random", 0)]


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


def _dense_mask(cu, lo, hi):
    T = int(cu[-1])
    doc = torch.zeros(T, dtype=torch.long)
    for b in range(len(cu) - 1):
        doc[cu[b]:cu[b + 1]] = b
    j = torch.arange(T)
    lo_t, hi_t = torch.from_numpy(np.asarray(lo, np.int64)), torch.from_numpy(np.asarray(hi, np.int64))
    return (doc[:, None] == doc[None, :]) & (j[None, :] >= lo_t[:, None]) & (j[None, :] <= hi_t[:, None])


def _sdpa(q, k, v, mask, scale):
    G = q.shape[1] // k.shape[1]
    kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    qh, kh, vh = (x.permute(1, 0, 2) for x in (q, kk, vv))
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask, scale=scale)
    scores = torch.einsum("htc,hsc->hts", qh, kh) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
    return out.permute(1, 0, 2), lse.T


def test_bounds_are_monotone_and_pairs_count(orc):
    cu = W.cu_seqlens((37, 64, 5, 27, 1))
    for kind, par in KINDS:
        lo, hi = W.interval_bounds(cu, kind, par, seed=3)
        for b in range(len(cu) - 1):
            s, e = cu[b], cu[b + 1]
            assert np.all(np.diff(lo[s:e]) >= 0) and np.all(np.diff(hi[s:e]) >= 0), kind
        assert W.interval_pairs(cu, lo, hi) == int(_dense_mask(cu, lo, hi).sum()), kind
    lo, hi = W.interval_bounds(cu, "causal")
    L = np.diff(cu)
    assert W.interval_pairs(cu, lo, hi) == int((L * (L + 1) // 2).sum())


@pytest.mark.parametrize("kind,par", KINDS)
def test_bounds_fwd_matches_torch_sdpa(orc, kind, par):
    cu = W.cu_seqlens((37, 64, 5, 27, 1))
    T = int(cu[-1])
    lo, hi = W.interval_bounds(cu, kind, par, seed=4)
    q, k, v = _rand((T, 4, 16), 110), _rand((T, 2, 16), 111), _rand((T, 2, 16), 112)
    o, l = orc.attn_fwd(q, k, v, cu, False, 0.3, q_lo=lo, q_hi=hi)
    mask = _dense_mask(cu, lo, hi)
    nonempty = mask.any(1).numpy()
    ro, rl = _sdpa(q, k, v, mask, 0.3)
    np.testing.assert_allclose(o[nonempty], ro.numpy()[nonempty], atol=1e-12, rtol=0)
    np.testing.assert_allclose(l[nonempty], rl.numpy()[nonempty], atol=1e-12, rtol=0)
    # rows that see no key: output 0, lse -inf
    assert np.all(o[~nonempty] == 0) and np.all(np.isneginf(l[~nonempty]))
    if kind == "random":
        assert (~nonempty).any()


@pytest.mark.parametrize("kind,par", [k for k in KINDS if k[0] != "random"])
def test_bounds_bwd_matches_torch_autograd(orc, kind, par):
    cu = W.cu_seqlens((11, 1, 23, 6))
    T = int(cu[-1])
    lo, hi = W.interval_bounds(cu, kind, par)
    hq, hkv, d = 4, 2, 8
    scale = 1.0 / math.sqrt(d)
    q, k, v = _rand((T, hq, d), 120), _rand((T, hkv, d), 121), _rand((T, hkv, d), 122)
    do = _rand((T, hq, d), 123)
    o, l = orc.attn_fwd(q, k, v, cu, False, scale, q_lo=lo, q_hi=hi)
    dq, dk, dv = orc.attn_bwd(q, k, v, o, l, do, cu, False, scale, q_lo=lo, q_hi=hi)
    mask = _dense_mask(cu, lo, hi)
    assert mask.any(1).all()
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    ref_o, _ = _sdpa(qq, kk, vv, mask, scale)
    ref_o.backward(do)
    np.testing.assert_allclose(dq, qq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vv.grad.numpy(), atol=1e-12)


def test_bounds_self_only_closed_form(orc):
    """lo = hi = i: every query sees only its own key, so O = V of its KV
    head, lse = scale * q.k, dQ = dK = 0 and dV = the sum of its group's dO."""
    cu = W.cu_seqlens((9, 1, 14))
    T = int(cu[-1])
    lo = hi = np.arange(T, dtype=np.int32)
    q, k, v = _rand((T, 4, 8), 130), _rand((T, 2, 8), 131), _rand((T, 2, 8), 132)
    do = _rand((T, 4, 8), 133)
    o, l = orc.attn_fwd(q, k, v, cu, False, 0.5, q_lo=lo, q_hi=hi)
    vv = v.numpy().repeat(2, axis=1)
    np.testing.assert_array_equal(o, vv)
    ref_l = 0.5 * np.einsum("thc,thc->th", q.numpy(), k.numpy().repeat(2, axis=1))
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-14)
    dq, dk, dv = orc.attn_bwd(q, k, v, o, l, do, cu, False, 0.5, q_lo=lo, q_hi=hi)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    np.testing.assert_allclose(dv, do.numpy().reshape(T, 2, 2, 8).sum(2), atol=1e-14)


def test_bounds_identical_keys_give_mean_of_values(orc):
    """With every key equal, the weights over a query's allowed keys are
    uniform: O is the mean of those V rows and lse = s + log(count)."""
    cu = W.cu_seqlens((20, 13))
    T = int(cu[-1])
    lo, hi = W.interval_bounds(cu, "chunked", 6)
    q, v = _rand((T, 2, 4), 140), _rand((T, 1, 4), 141)
    k = _rand((1, 1, 4), 142).repeat(T, 1, 1)
    o, l = orc.attn_fwd(q, k, v, cu, False, 0.7, q_lo=lo, q_hi=hi)
    for i in range(T):
        cnt = hi[i] - lo[i] + 1
        ref = v.numpy()[lo[i]:hi[i] + 1, 0].mean(0)
        s = 0.7 * (q.numpy()[i] @ k.numpy()[0, 0])
        np.testing.assert_allclose(o[i], np.stack([ref, ref]), atol=1e-13)
        np.testing.assert_allclose(l[i], s + math.log(cnt), atol=1e-13)


def test_bounds_key_partition_merges_to_full(orc):
    """LSE-merging the partials of a random key partition under the same
    interval mask gives the full result."""
    cu = W.cu_seqlens((30, 17, 25))
    T = int(cu[-1])
    lo, hi = W.interval_bounds(cu, "random", seed=7)
    q, k, v = _rand((T, 4, 8), 150), _rand((T, 2, 8), 151), _rand((T, 2, 8), 152)
    seg = orc.doc_ids(cu)
    pos = np.arange(T)
    full_o, full_l = orc.attn_fwd(q, k, v, cu, False, 0.4, q_lo=lo, q_hi=hi)
    part = np.random.default_rng(8).integers(0, 3, T)
    outs, lses = [], []
    for p in range(3):
        ki = np.nonzero(part == p)[0]
        o_p, l_p = orc.partial_fwd(q, k[ki], v[ki], seg, seg[ki], pos, ki, False, 0.4, q_lo=lo, q_hi=hi)
        outs.append(o_p)
        lses.append(l_p)
    mo, ml = orc.lse_merge(outs, lses)
    fin = np.isfinite(full_l)
    np.testing.assert_allclose(mo, full_o, atol=1e-12)
    np.testing.assert_allclose(ml[fin], full_l[fin], atol=1e-12)
    assert np.all(np.isneginf(ml[~fin]))
