"""GPU parity of the sliding-window mask (a key visible only up to `window`
positions behind its query: the window_size argument of the cuDNN
flash-attention call in "Add Context Parallelism support to cudnn Flash
Attention #1133", maxtext) and of non-causal ring attention, against the
fp64 oracle.  Tolerances as elsewhere: bf16 -> max-abs 2e-2 on outputs and
gradients (relative to max(1, max|ref|)), 1e-3 on LSE; fp32 -> 1e-5."""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available()
    from context_varlen_ring_gb300 import build as b
    b.build()
    import context_varlen_ring_gb300 as m
    m.lib()
    torch.cuda.set_device(0)
    return m


def _status(ra):
    torch.cuda.synchronize()
    assert ra.device_status() == 0


def _err(got, ref):
    """Plain max-abs error (outputs)."""
    return float(np.abs(np.asarray(got, dtype=np.float64) - ref).max())


def _gerr(got, ref):
    """Gradient error: max-abs over max(1, max|ref|).  A gradient of a KV
    head sums the products of its G query heads, formed from bf16 operands
    (P, dS) that carry a relative rounding of 2^-9 each, so its error grows
    with its magnitude, which grows with G and the document length."""
    return _err(got, ref) / max(1.0, float(np.abs(ref).max()))


def _lse_err(got_hq_t, ref_t_hq):
    g = got_hq_t.T
    fin = np.isfinite(ref_t_hq)
    assert np.array_equal(np.isfinite(g), fin)
    return float(np.abs(g[fin] - ref_t_hq[fin]).max()) if fin.any() else 0.0


@pytest.mark.parametrize("sched", ["fused", "stepwise"])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_window_ring_fwd_bwd_bf16(ra, orc, sched, mode, G, causal):
    """Windows shorter than a tile, spanning a few tiles, and longer than
    most documents, over random packings and CP sizes."""
    rng = np.random.default_rng(500 + 10 * G + mode + 2 * causal)
    for trial, window in enumerate((0, 37, 200, 900)):
        docs = W.random_doc_lens(rng, 1500, 1, 700)
        cu = W.cu_seqlens(docs)
        T = int(cu[-1])
        cp = (2, 3, 4, 8)[trial]
        hkv = 2
        q, k, v = W.make_qkv(T, hkv * G, hkv, 128, torch.bfloat16, seed_offset=trial)
        do = W.make_dout(T, hkv * G, 128, torch.bfloat16, seed_offset=trial)
        qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
        out, lse = ra.ring_attn_fwd(qd, kd, vd, cu, cp, mode, causal, None, sched, window=window)
        dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, out, lse, dod, cu, cp, mode, causal, None, sched,
                                      grad_dtype=torch.float32, window=window)
        _status(ra)
        scale = 1 / math.sqrt(128)
        ro, rl = orc.attn_fwd(q, k, v, cu, causal, scale, window=window)
        assert _err(out.float().cpu().numpy(), ro) <= 2e-2, (window, docs)
        assert _lse_err(lse.cpu().numpy(), rl) <= 1e-3, window
        rdq, rdk, rdv = orc.attn_bwd(q, k, v, ro, rl, do, cu, causal, scale, window=window)
        for g, r in ((dq, rdq), (dk, rdk), (dv, rdv)):
            assert _gerr(g.cpu().numpy(), r) <= 2e-2, (window, docs, _err(g.cpu().numpy(), r), float(np.abs(r).max()))


@pytest.mark.parametrize("sched", ["fused", "stepwise"])
def test_window_ring_fp32(ra, orc, sched):
    """fp32 (SIMT path), 1e-5."""
    cu = W.cu_seqlens((37, 64, 27))
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, 2, 2, 64, torch.float32)
    do = W.make_dout(T, 2, 64, torch.float32)
    for window in (0, 5, 30):
        out, lse = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), cu, 2, 0, True, 0.125, sched, window=window)
        g = ra.ring_attn_bwd(q.cuda(), k.cuda(), v.cuda(), out, lse, do.cuda(), cu, 2, 0, True, 0.125, sched,
                             window=window)
        _status(ra)
        ro, rl = orc.attn_fwd(q, k, v, cu, True, 0.125, window=window)
        assert np.abs(out.cpu().numpy() - ro).max() <= 1e-5
        assert _lse_err(lse.cpu().numpy(), rl) <= 1e-5
        rg = orc.attn_bwd(q, k, v, ro, rl, do, cu, True, 0.125, window=window)
        for a, b in zip(g, rg):
            assert _err(a.cpu().numpy(), b) <= 1e-5


def test_window_partial(ra, orc):
    """One ring step's partial with a window (tensor cores: bf16, d 128)."""
    rng = np.random.default_rng(9)
    lq, lk = [300, 0, 250], [280, 120, 0]
    cuq, cuk = W.cu_seqlens(lq), W.cu_seqlens(lk)
    Tq, Tk = int(cuq[-1]), int(cuk[-1])
    qpos = np.concatenate([np.sort(rng.choice(2000, L, replace=False)) for L in lq]).astype(np.int32)
    kpos = np.concatenate([np.sort(rng.choice(2000, L, replace=False)) for L in lk if L]).astype(np.int32)
    q = W.randn((Tq, 8, 128), 31, torch.bfloat16)
    k = W.randn((Tk, 2, 128), 32, torch.bfloat16)
    v = W.randn((Tk, 2, 128), 33, torch.bfloat16)
    for window in (0, 50, 400):
        out, lse = ra.varlen_attn_partial(q.cuda(), k.cuda(), v.cuda(), cuq, cuk, qpos, kpos, True, 0.09,
                                          window=window)
        _status(ra)
        ro, rl = orc.partial_fwd(q, k, v, orc.doc_ids(cuq), orc.doc_ids(cuk), qpos, kpos, True, 0.09,
                                 window=window)
        assert np.abs(out.cpu().numpy() - ro).max() <= 2e-2
        assert _lse_err(lse.cpu().numpy(), rl) <= 1e-3


def test_window_c2_sampled(ra, orc):
    """The packed 32768-token workload with a 1024-token window: sampled
    output rows and gradient rows against the oracle."""
    wl = W.C2
    cu = wl.cu_seqlens()
    T, window = wl.T, 1024
    q, k, v = W.make_qkv(T, wl.hq, wl.hkv, wl.d, wl.dtype)
    do = W.make_dout(T, wl.hq, wl.d, wl.dtype)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    out, lse = ra.ring_attn_fwd(qd, kd, vd, cu, wl.cp, wl.zz_mode, True, wl.scale, window=window)
    dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, out, lse, dod, cu, wl.cp, wl.zz_mode, True, wl.scale,
                                  grad_dtype=torch.float32, window=window)
    _status(ra)
    rows = W.sample_rows(T, 48, 11, list(cu[:-1]) + list(np.maximum(cu[1:] - 1, 0)))
    seg = orc.doc_ids(cu)
    ro, rl = orc.partial_fwd(q[torch.from_numpy(rows)], k, v, seg[rows], seg, rows, np.arange(T), True, wl.scale,
                             window=window)
    idx = torch.from_numpy(rows).cuda()
    assert np.abs(out[idx].float().cpu().numpy() - ro).max() <= 2e-2
    assert np.abs(lse[:, idx].cpu().numpy().T - rl).max() <= 1e-3
    # gradients of whole documents (the oracle needs each document's full
    # forward): the 1809- and 3768-token ones, both longer than the window
    docs = np.array([0, 4])
    assert all(int(cu[b + 1] - cu[b]) > window for b in docs)
    sel = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in docs])
    sub_cu = W.cu_seqlens([int(cu[b + 1] - cu[b]) for b in docs])
    qs, ks, vs, dos = (x[torch.from_numpy(sel)] for x in (q, k, v, do))
    so, sl = orc.attn_fwd(qs, ks, vs, sub_cu, True, wl.scale, window=window)
    rdq, rdk, rdv = orc.attn_bwd(qs, ks, vs, so, sl, dos, sub_cu, True, wl.scale, window=window)
    sidx = torch.from_numpy(sel).cuda()
    for g, r in ((dq, rdq), (dk, rdk), (dv, rdv)):
        assert _gerr(g[sidx].cpu().numpy(), r) <= 2e-2, (_err(g[sidx].cpu().numpy(), r), float(np.abs(r).max()))


def test_noncausal_ring_plan(ra, orc):
    """Non-causal ring attention through the fused tensor-core passes: every
    ring step holds visited tiles (the plan is built for the call's mask)."""
    cu = W.cu_seqlens((500, 77, 900))
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, 8, 2, 128, torch.bfloat16)
    do = W.make_dout(T, 8, 128, torch.bfloat16)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    out, lse = ra.ring_attn_fwd(qd, kd, vd, cu, 4, 1, False, None)
    g = ra.ring_attn_bwd(qd, kd, vd, out, lse, dod, cu, 4, 1, False, None, grad_dtype=torch.float32)
    _status(ra)
    scale = 1 / math.sqrt(128)
    ro, rl = orc.attn_fwd(q, k, v, cu, False, scale)
    assert _err(out.float().cpu().numpy(), ro) <= 2e-2
    assert _lse_err(lse.cpu().numpy(), rl) <= 1e-3
    rg = orc.attn_bwd(q, k, v, ro, rl, do, cu, False, scale)
    for a, b in zip(g, rg):
        assert _err(a.cpu().numpy(), b) <= 2e-2
