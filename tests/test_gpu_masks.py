"""GPU parity of the ring under interval masks (per-token key bounds: the
dynamic attention masks of "[Train] Support custom attention with context
parallel", FlagScale PR #910) against the fp64 oracle with the same bounds.
Tolerances: outputs plain max-abs 2e-2, LSE 1e-3 (-inf rows exactly),
gradients 2e-2 * max(1, max|ref|) (the gradient rule of test_gpu_bwd.py)."""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

MASKS = [("window", 40), ("chunked", 64), ("prefix", 100), ("bidirectional", 0), ("random", 0)]


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available()
    from context_varlen_ring_gb300 import build as b
    b.build()
    import context_varlen_ring_gb300 as m
    m.lib()
    torch.cuda.set_device(0)
    return m


def _err(got, ref):
    return float(np.abs(np.asarray(got, dtype=np.float64) - ref).max())


def _gerr(got, ref):
    return _err(got, ref) / max(1.0, float(np.abs(ref).max()))


def _lse_check(got_hq_t, ref_t_hq, tol):
    g = got_hq_t.T
    fin = np.isfinite(ref_t_hq)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.all(g[~fin] == -np.inf)
    if fin.any():
        assert np.abs(g[fin] - ref_t_hq[fin]).max() <= tol


@pytest.mark.parametrize("sched", ["fused", "allgather"])
@pytest.mark.parametrize("kind,par", MASKS)
def test_masked_ring_fwd_bwd(ra, orc, sched, kind, par):
    rng = np.random.default_rng(600 + MASKS.index((kind, par)) + 10 * (sched == "allgather"))
    for trial in range(2):
        docs = W.random_doc_lens(rng, 1300, 1, 600)
        cu = W.cu_seqlens(docs)
        T = int(cu[-1])
        cp = [2, 5, 8][(trial + len(docs)) % 3]
        mode = trial % 2
        G = [1, 4, 8][(trial + MASKS.index((kind, par))) % 3]
        hkv = 2
        lo, hi = W.interval_bounds(cu, kind, par, seed=trial)
        q, k, v = W.make_qkv(T, hkv * G, hkv, 128, torch.bfloat16, seed_offset=trial)
        do = W.make_dout(T, hkv * G, 128, torch.bfloat16, seed_offset=trial)
        qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
        nb = max(ra.ring_workspace_bytes(T, hkv * G, hkv, 128, 0, cu, cp, mode, sched, bwd=b, key_lo=lo, key_hi=hi)
                 for b in (False, True))
        ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN bytes: every read row must be written
        out, lse = ra.ring_attn_fwd(qd, kd, vd, cu, cp, mode, scale=None, sched=sched, workspace=ws, key_lo=lo,
                                    key_hi=hi)
        dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, out, lse, dod, cu, cp, mode, scale=None, sched=sched,
                                      grad_dtype=torch.float32, workspace=ws, reuse_fwd_workspace=True, key_lo=lo,
                                      key_hi=hi)
        torch.cuda.synchronize()
        assert ra.device_status() == 0
        scale = 1 / math.sqrt(128)
        ro, rl = orc.attn_fwd(q, k, v, cu, False, scale, q_lo=lo, q_hi=hi)
        case = (kind, docs, cp, mode, G)
        assert _err(out.float().cpu().numpy(), ro) <= 2e-2, case
        _lse_check(lse.cpu().numpy(), rl, 1e-3)
        rdq, rdk, rdv = orc.attn_bwd(q, k, v, ro, rl, do, cu, False, scale, q_lo=lo, q_hi=hi)
        for name, g, r in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
            a = g.cpu().numpy()
            assert np.isfinite(a).all(), (name, case)
            assert _gerr(a, r) <= 2e-2, (name, case, _err(a, r), float(np.abs(r).max()))


def test_causal_intervals_equal_causal_path(ra):
    """Bounds spelling out the causal mask run the interval-mask kernels on
    the causal plan's block map with the same per-row limits, so outputs,
    LSE and gradients are bit-identical to the causal call."""
    cu = W.cu_seqlens((700, 33, 1200, 129, 300))
    T = int(cu[-1])
    lo, hi = W.interval_bounds(cu, "causal")
    q, k, v = (x.cuda() for x in W.make_qkv(T, 16, 4, 128, torch.bfloat16))
    do = W.make_dout(T, 16, 128, torch.bfloat16).cuda()
    res = []
    for bounds in (False, True):
        kw = dict(key_lo=lo, key_hi=hi) if bounds else {}
        out, lse = ra.ring_attn_fwd(q, k, v, cu, 4, 1, True, None, "fused", **kw)
        g = ra.ring_attn_bwd(q, k, v, out, lse, do, cu, 4, 1, True, None, "fused", grad_dtype=torch.float32, **kw)
        torch.cuda.synchronize()
        res.append([x.clone() for x in (out, lse) + tuple(g)])
    assert ra.device_status() == 0
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_packed_workload_prefix_mask(ra, orc):
    """The packed 32768-token workload (GQA 32/8, CP 8, per-document
    zigzag) under a prefix-LM mask (the first 512 tokens of each document
    bidirectional, causal after): sampled output rows against the oracle,
    and the whole gradients of a short and a long document for two KV
    heads."""
    wl = W.C4
    cu = wl.cu_seqlens()
    T = wl.T
    lo, hi = W.interval_bounds(cu, "prefix", 512)
    q, k, v = W.make_qkv(T, wl.hq, wl.hkv, wl.d, wl.dtype)
    do = W.make_dout(T, wl.hq, wl.d, wl.dtype)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    out, lse = ra.ring_attn_fwd(qd, kd, vd, cu, wl.cp, wl.zz_mode, scale=wl.scale, key_lo=lo, key_hi=hi)
    dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, out, lse, dod, cu, wl.cp, wl.zz_mode, scale=wl.scale,
                                  grad_dtype=torch.float32, key_lo=lo, key_hi=hi)
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    rows = W.sample_rows(T, 64, 21, list(cu[:-1]) + list(np.maximum(cu[1:] - 1, 0)))
    seg = orc.doc_ids(cu)
    ro, rl = orc.partial_fwd(q[torch.from_numpy(rows)], k, v, seg[rows], seg, rows, np.arange(T), False, wl.scale,
                             q_lo=lo[rows], q_hi=hi[rows])
    idx = torch.from_numpy(rows).cuda()
    assert _err(out[idx].float().cpu().numpy(), ro) <= 2e-2
    assert np.abs(lse[:, idx].cpu().numpy().T - rl).max() <= 1e-3
    G = wl.hq // wl.hkv
    dq, dk, dv = (x.cpu().numpy() for x in (dq, dk, dv))
    for bdoc in (1, 9):  # 393 and 6253 tokens
        a, e = int(cu[bdoc]), int(cu[bdoc + 1])
        sub = np.array([0, e - a])
        for g in (0, 5):
            hs = slice(g * G, (g + 1) * G)
            qs, ks, vs, ds = (x.contiguous() for x in (q[a:e, hs], k[a:e, g:g + 1], v[a:e, g:g + 1], do[a:e, hs]))
            sl, sh = lo[a:e] - a, hi[a:e] - a
            o_r, l_r = orc.attn_fwd(qs, ks, vs, sub, False, wl.scale, q_lo=sl, q_hi=sh)
            rdq, rdk, rdv = orc.attn_bwd(qs, ks, vs, o_r, l_r, ds, sub, False, wl.scale, q_lo=sl, q_hi=sh)
            for name, got, r in (("dq", dq[a:e, hs], rdq), ("dk", dk[a:e, g:g + 1], rdk), ("dv", dv[a:e, g:g + 1], rdv)):
                assert _gerr(got, r) <= 2e-2, (name, bdoc, g, _err(got, r), float(np.abs(r).max()))
