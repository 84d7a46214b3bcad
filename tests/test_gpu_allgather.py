"""GPU parity of the all-gather schedule (each simulated rank's zigzag
queries against the gathered K/V of every rank, read in original order; the
Llama 3 scheme discussed in "Zigzag attention support?",
ring-attention-pytorch issue #20) against the fp64 oracle.  Tolerances as
elsewhere: bf16 -> max-abs 2e-2 on outputs and gradients (relative to
max(1, max|ref|)), 1e-3 on LSE; fp32 -> 1e-5."""
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


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window", [-1, 150])
def test_allgather_fwd_bwd_bf16(ra, orc, mode, G, causal, window):
    """Random packings and CP sizes; the workspace starts NaN-filled (the
    schedule copies no K/V rows, and Q/dO only for two-run query tiles)."""
    rng = np.random.default_rng(900 + 10 * G + mode + 2 * causal + 4 * (window > 0))
    for trial, cp in enumerate((2, 5, 8)):
        docs = W.random_doc_lens(rng, 1300, 1, 600)
        cu = W.cu_seqlens(docs)
        T = int(cu[-1])
        hkv = 2
        q, k, v = W.make_qkv(T, hkv * G, hkv, 128, torch.bfloat16, seed_offset=trial)
        do = W.make_dout(T, hkv * G, 128, torch.bfloat16, seed_offset=trial)
        qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
        nb = max(ra.ring_workspace_bytes(T, hkv * G, hkv, 128, 0, cu, cp, mode, "allgather", bwd=b)
                 for b in (False, True))
        ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda")
        out, lse = ra.ring_attn_fwd(qd, kd, vd, cu, cp, mode, causal, None, "allgather", workspace=ws,
                                    window=window)
        dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, out, lse, dod, cu, cp, mode, causal, None, "allgather",
                                      grad_dtype=torch.float32, workspace=ws, reuse_fwd_workspace=True,
                                      window=window)
        torch.cuda.synchronize()
        assert ra.device_status() == 0
        scale = 1 / math.sqrt(128)
        ro, rl = orc.attn_fwd(q, k, v, cu, causal, scale, window=window)
        assert _err(out.float().cpu().numpy(), ro) <= 2e-2, (docs, cp)
        assert _lse_err(lse.cpu().numpy(), rl) <= 1e-3, (docs, cp)
        rdq, rdk, rdv = orc.attn_bwd(q, k, v, ro, rl, do, cu, causal, scale, window=window)
        for g, r in ((dq, rdq), (dk, rdk), (dv, rdv)):
            a = g.cpu().numpy()
            assert np.isfinite(a).all()
            assert _gerr(a, r) <= 2e-2, (docs, cp, _err(a, r), float(np.abs(r).max()))


def test_allgather_fp32_runs_fused(ra, orc):
    """fp32 has no tensor-core kernels: the schedule runs as the fused ring
    (the same attention), 1e-5 against the oracle."""
    cu = W.cu_seqlens((37, 64, 27))
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, 2, 2, 64, torch.float32)
    do = W.make_dout(T, 2, 64, torch.float32)
    out, lse = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), cu, 2, 0, True, 0.125, "allgather")
    g = ra.ring_attn_bwd(q.cuda(), k.cuda(), v.cuda(), out, lse, do.cuda(), cu, 2, 0, True, 0.125, "allgather")
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    ro, rl = orc.attn_fwd(q, k, v, cu, True, 0.125)
    assert np.abs(out.cpu().numpy() - ro).max() <= 1e-5
    assert _lse_err(lse.cpu().numpy(), rl) <= 1e-5
    rg = orc.attn_bwd(q, k, v, ro, rl, do, cu, True, 0.125)
    for a, b in zip(g, rg):
        assert _err(a.cpu().numpy(), b) <= 1e-5


def test_allgather_c2_sampled_and_ring_agreement(ra, orc):
    """The packed 32768-token workload: sampled output rows against the
    oracle, and the whole output, LSE and gradients against the ring
    schedule's (two tilings of the same attention)."""
    wl = W.C2
    cu = wl.cu_seqlens()
    T = wl.T
    q, k, v = W.make_qkv(T, wl.hq, wl.hkv, wl.d, wl.dtype)
    do = W.make_dout(T, wl.hq, wl.d, wl.dtype)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    res = {}
    for sched in ("allgather", "fused"):
        out, lse = ra.ring_attn_fwd(qd, kd, vd, cu, wl.cp, wl.zz_mode, True, wl.scale, sched)
        grads = ra.ring_attn_bwd(qd, kd, vd, out, lse, dod, cu, wl.cp, wl.zz_mode, True, wl.scale, sched,
                                 grad_dtype=torch.float32)
        torch.cuda.synchronize()
        assert ra.device_status() == 0
        res[sched] = [x.float() for x in (out, lse) + tuple(grads)]
    rows = W.sample_rows(T, 48, 12, list(cu[:-1]) + list(np.maximum(cu[1:] - 1, 0)))
    seg = orc.doc_ids(cu)
    ro, rl = orc.partial_fwd(q[torch.from_numpy(rows)], k, v, seg[rows], seg, rows, np.arange(T), True, wl.scale)
    idx = torch.from_numpy(rows).cuda()
    assert np.abs(res["allgather"][0][idx].cpu().numpy() - ro).max() <= 2e-2
    assert np.abs(res["allgather"][1][:, idx].cpu().numpy().T - rl).max() <= 1e-3
    for a, b in zip(res["allgather"], res["fused"]):
        scale = max(1.0, float(b.abs().max()))
        assert float((a - b).abs().max()) / scale <= 2e-2
