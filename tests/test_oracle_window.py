"""Pins for the oracle's sliding-window mask (CPU only).

The window is the window_size argument that the cuDNN flash-attention call
takes ("Add Context Parallelism support to cudnn Flash Attention #1133",
maxtext, diff of cudnn_flash_attention), read as: key j is visible to query
i only if pos[j] >= pos[i] - window (on top of the document and causal
masks).  Each test checks the oracle against something other than itself:
PyTorch's scaled_dot_product_attention / logsumexp / autograd in float64
with a dense mask, closed forms, and the same rows computed without a window
on an explicitly truncated key set.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


def _sdpa_window(q, k, v, cu, causal, scale, window):
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    doc = torch.zeros(T, dtype=torch.long)
    for b in range(len(cu) - 1):
        doc[cu[b]:cu[b + 1]] = b
    i = torch.arange(T)
    mask = (doc[:, None] == doc[None, :]) & (i[None, :] >= i[:, None] - window)
    if causal:
        mask &= i[None, :] <= i[:, None]
    qh, kh, vh = (x.permute(1, 0, 2) for x in (q, kk, vv))
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask, scale=scale)
    scores = torch.einsum("htc,hsc->hts", qh, kh) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
    return out.permute(1, 0, 2), lse.T


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window", [0, 3, 17])
def test_window_fwd_matches_torch_sdpa(orc, causal, window):
    cu = W.cu_seqlens((37, 64, 5, 27))
    T = int(cu[-1])
    q, k, v = _rand((T, 4, 16), 80), _rand((T, 2, 16), 81), _rand((T, 2, 16), 82)
    o, l = orc.attn_fwd(q, k, v, cu, causal, 0.3, window=window)
    ro, rl = _sdpa_window(q, k, v, cu, causal, 0.3, window)
    np.testing.assert_allclose(o, ro.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(l, rl.numpy(), atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [True, False])
def test_window_bwd_matches_torch_autograd(orc, causal):
    cu = W.cu_seqlens((11, 1, 23, 6))
    T = int(cu[-1])
    hq, hkv, d, w = 4, 2, 8, 4
    scale = 1.0 / math.sqrt(d)
    q, k, v = _rand((T, hq, d), 90), _rand((T, hkv, d), 91), _rand((T, hkv, d), 92)
    do = _rand((T, hq, d), 93)
    o, l = orc.attn_fwd(q, k, v, cu, causal, scale, window=w)
    dq, dk, dv = orc.attn_bwd(q, k, v, o, l, do, cu, causal, scale, window=w)
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    ref_o, _ = _sdpa_window(qq, kk, vv, cu, causal, scale, w)
    ref_o.backward(do)
    np.testing.assert_allclose(dq, qq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vv.grad.numpy(), atol=1e-12)


def test_window_zero_closed_form(orc):
    """Causal window 0: every query sees only its own key, so O = V of its
    KV head exactly, lse = scale * q.k, and dQ = dK = 0, dV = sum of the
    group's dO (the softmax over one element is exactly 1)."""
    cu = W.cu_seqlens((9, 1, 14))
    T = int(cu[-1])
    q, k, v = _rand((T, 4, 8), 100), _rand((T, 2, 8), 101), _rand((T, 2, 8), 102)
    do = _rand((T, 4, 8), 103)
    o, l = orc.attn_fwd(q, k, v, cu, True, 0.5, window=0)
    vv = v.repeat_interleave(2, dim=1).numpy()
    assert np.array_equal(o, vv)
    qk = np.einsum("thc,thc->th", q.numpy(), k.repeat_interleave(2, dim=1).numpy()) * 0.5
    np.testing.assert_allclose(l, qk, atol=1e-13, rtol=0)
    dq, dk, dv = orc.attn_bwd(q, k, v, o, l, do, cu, True, 0.5, window=0)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0
    np.testing.assert_allclose(dv, do.numpy().reshape(T, 2, 2, 8).sum(2), atol=1e-13, rtol=0)


def test_window_covering_documents_is_no_window(orc):
    """A window at least as long as the longest document masks nothing:
    bit-identical to the unwindowed result, forward and backward."""
    docs = (30, 7, 45)
    cu = W.cu_seqlens(docs)
    T = int(cu[-1])
    q, k, v = _rand((T, 2, 8), 110), _rand((T, 1, 8), 111), _rand((T, 1, 8), 112)
    do = _rand((T, 2, 8), 113)
    for causal in (True, False):
        o0, l0 = orc.attn_fwd(q, k, v, cu, causal, 0.4)
        o1, l1 = orc.attn_fwd(q, k, v, cu, causal, 0.4, window=max(docs) - 1)
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
        g0 = orc.attn_bwd(q, k, v, o0, l0, do, cu, causal, 0.4)
        g1 = orc.attn_bwd(q, k, v, o1, l1, do, cu, causal, 0.4, window=max(docs) - 1)
        for a, b in zip(g0, g1):
            assert np.array_equal(a, b)


def test_window_rows_equal_truncated_key_sets(orc):
    """Row i under window w equals the unwindowed causal row over the keys
    [i - w, i] alone (same keys in the same order: bit-identical)."""
    T, w = 50, 6
    cu = W.cu_seqlens((T,))
    q, k, v = _rand((T, 2, 8), 120), _rand((T, 2, 8), 121), _rand((T, 2, 8), 122)
    o, l = orc.attn_fwd(q, k, v, cu, True, 0.6, window=w)
    for i in (0, 3, 6, 7, 31, 49):
        lo = max(0, i - w)
        keys = np.arange(lo, i + 1)
        ro, rl = orc.partial_fwd(q[i:i + 1], k[keys], v[keys], np.zeros(1, np.int32), np.zeros(len(keys), np.int32),
                                 np.array([i]), keys, True, 0.6)
        assert np.array_equal(ro[0], o[i]) and np.array_equal(rl[0], l[i])


@pytest.mark.parametrize("mode", [0, 1])
def test_window_rank_pairs_closed_form(orc, mode):
    """Summed over ranks, the pair counts equal sum_i min(i - start + 1, w + 1)
    over each document (causal) and sum_i (min(i + w, end - 1) - start + 1)
    clipped at the window's start (non-causal: keys after i are unbounded)."""
    docs = (100, 3, 250, 17)
    cu = W.cu_seqlens(docs)
    w = 20
    causal_ref = sum(min(i + 1, w + 1) for L in docs for i in range(L))
    full_ref = sum(L - max(0, i - w) for L in docs for i in range(L))
    assert int(orc.rank_pairs(cu, 4, mode, True, window=w).sum()) == causal_ref
    assert int(orc.rank_pairs(cu, 4, mode, False, window=w).sum()) == full_ref
    assert int(orc.rank_pairs(cu, 4, mode, True, window=10**6).sum()) == sum(L * (L + 1) // 2 for L in docs)
