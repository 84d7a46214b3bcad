"""GPU parity of the ring backward (dQ, dK, dV from the saved LSE) against the
fp64 oracle.  bf16 inputs: gradients to max-abs 2e-2 * max(1, max|ref|)
(the gradient rule of _rel), and the full-size packed workload's gradients
of every document to plain max-abs 2e-2; fp32 inputs: 1e-5 plain.  Each
failure message carries the plain error and max|ref|."""
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
    """Plain max-abs error."""
    return float(np.abs(np.asarray(got, dtype=np.float64) - ref).max())


def _rel(got, ref):
    """Max-abs error over max(1, max|ref|), the gradient rule: a gradient of
    a KV head sums the products of its G query heads, formed from bf16
    operands (P, dS) that carry a relative rounding of 2^-9 each, so its
    error grows with its magnitude (which grows with G and the document
    length); a gradient returned in bf16 adds its own rounding of up to
    m * 2^-9 at magnitude m."""
    return _err(got, ref) / max(1.0, float(np.abs(ref).max()))


def _run(ra, q, k, v, do, cu, cp, mode, causal, sched, grad_dtype=torch.float32):
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    out, lse = ra.ring_attn_fwd(qd, kd, vd, cu, cp, mode, causal, None, sched)
    dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, out, lse, dod, cu, cp, mode, causal, None, sched, grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    return out, lse, dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()


@pytest.mark.parametrize("sched", ["fused", "stepwise"])
def test_bwd_c0_fp32(ra, orc, sched):
    wl = W.C0
    cu = wl.cu_seqlens()
    q, k, v = W.make_qkv(wl.T, wl.hq, wl.hkv, wl.d, wl.dtype)
    do = W.make_dout(wl.T, wl.hq, wl.d, wl.dtype)
    _, _, dq, dk, dv = _run(ra, q, k, v, do, cu, wl.cp, wl.zz_mode, True, sched)
    ro, rl = orc.attn_fwd(q, k, v, cu, True, wl.scale)
    rdq, rdk, rdv = orc.attn_bwd(q, k, v, ro, rl, do, cu, True, wl.scale)
    for g, r in ((dq, rdq), (dk, rdk), (dv, rdv)):
        assert _err(g, r) <= 1e-5


@pytest.mark.parametrize("sched", ["fused", "stepwise"])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_bwd_small_bf16(ra, orc, sched, mode, G):
    rng = np.random.default_rng(300 + 10 * G + mode)
    for trial in range(2):
        docs = W.random_doc_lens(rng, 1400, 1, 600)
        cu = W.cu_seqlens(docs)
        T = int(cu[-1])
        cp = [2, 3, 4, 8, 1][(trial + G) % 5]
        hkv = 2
        causal = trial == 0 or G != 2
        q, k, v = W.make_qkv(T, hkv * G, hkv, 128, torch.bfloat16, seed_offset=trial)
        do = W.make_dout(T, hkv * G, 128, torch.bfloat16, seed_offset=trial)
        _, _, dq, dk, dv = _run(ra, q, k, v, do, cu, cp, mode, causal, sched)
        scale = 1 / math.sqrt(128)
        ro, rl = orc.attn_fwd(q, k, v, cu, causal, scale)
        rdq, rdk, rdv = orc.attn_bwd(q, k, v, ro, rl, do, cu, causal, scale)
        for name, g, r in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
            assert _rel(g, r) <= 2e-2, (name, docs, cp, _err(g, r), float(np.abs(r).max()))


def test_bwd_bf16_grad_output(ra, orc):
    """Gradients returned in bf16 (accumulated in fp32, cast at the end)."""
    cu = W.cu_seqlens((300, 41, 500))
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, 16, 4, 128, torch.bfloat16)
    do = W.make_dout(T, 16, 128, torch.bfloat16)
    _, _, dq, dk, dv = _run(ra, q, k, v, do, cu, 4, 1, True, "fused", grad_dtype=torch.bfloat16)
    ro, rl = orc.attn_fwd(q, k, v, cu, True, 1 / math.sqrt(128))
    rdq, rdk, rdv = orc.attn_bwd(q, k, v, ro, rl, do, cu, True, 1 / math.sqrt(128))
    for g, r in ((dq, rdq), (dk, rdk), (dv, rdv)):
        mx = float(np.abs(r).max())
        print(f"bf16 gradient: max-abs {_err(g, r):.4g}, max|ref| {mx:.4g}, relative {_rel(g, r):.4g}")
        assert _rel(g, r) <= 2e-2, (_err(g, r), mx)


def test_bwd_c4_full_size(ra, orc):
    """The packed 32768-token workload at full size, in the launch
    configuration the benchmark times (fused ring, CP=8, per-document
    zigzag): for every document, two KV heads with their G query heads are
    compared element by element with the oracle -- O and LSE of the forward,
    dQ, dK and dV of the backward (fp32 gradients; the bf16 gradients the
    benchmark writes are checked to be exactly those rounded) -- at the
    plain max-abs tolerances (2e-2 on outputs and gradients, 1e-3 on LSE).  Documents do
    not attend to each other, so each is its own oracle problem.  The KV
    heads rotate over the documents so that all eight are covered."""
    wl = W.C4
    cu = wl.cu_seqlens()
    T = wl.T
    G = wl.hq // wl.hkv
    q, k, v = W.make_qkv(T, wl.hq, wl.hkv, wl.d, wl.dtype)
    do = W.make_dout(T, wl.hq, wl.d, wl.dtype)
    out, lse, dq, dk, dv = _run(ra, q, k, v, do, cu, wl.cp, wl.zz_mode, True, "fused")
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    # the benchmark's launch writes bf16 gradients: the same kernels with the
    # bf16 epilogue give exactly the fp32 gradients rounded to bf16 (round to
    # nearest even), so the parity below holds for that launch as well
    _, _, dq16, dk16, dv16 = _run(ra, q, k, v, do, cu, wl.cp, wl.zz_mode, True, "fused", grad_dtype=torch.bfloat16)
    for name, got, f32 in (("dq", dq16, dq), ("dk", dk16, dk), ("dv", dv16, dv)):
        ref16 = torch.from_numpy(np.ascontiguousarray(f32)).to(torch.bfloat16).float().numpy()
        assert np.array_equal(got, ref16), name
    report = []
    for bdoc in range(len(cu) - 1):
        a, e = int(cu[bdoc]), int(cu[bdoc + 1])
        sub = np.array([0, e - a])
        for g in sorted({bdoc % wl.hkv, (bdoc + 3) % wl.hkv}):
            hs = slice(g * G, (g + 1) * G)
            qs, ks, vs, ds = (x.contiguous() for x in (q[a:e, hs], k[a:e, g:g + 1], v[a:e, g:g + 1], do[a:e, hs]))
            ro, rl = orc.attn_fwd(qs, ks, vs, sub, True, wl.scale)
            rdq, rdk, rdv = orc.attn_bwd(qs, ks, vs, ro, rl, ds, sub, True, wl.scale)
            _err_lse = np.abs(lse[hs, a:e].T - rl).max()
            assert _err_lse <= 1e-3, (bdoc, g, _err_lse)
            for name, got, ref in (("o", out[a:e, hs], ro), ("dq", dq[a:e, hs], rdq), ("dk", dk[a:e, g:g + 1], rdk),
                                   ("dv", dv[a:e, g:g + 1], rdv)):
                err = float(np.abs(np.asarray(got, dtype=np.float64) - ref).max())
                mx = float(np.abs(ref).max())
                report.append((name, bdoc, e - a, g, err, mx))
                assert err <= 2e-2, (name, bdoc, e - a, g, err, mx)
    worst = {}
    for name, bdoc, L_, g, err, mx in report:
        if err > worst.get(name, (0.0,))[0]:
            worst[name] = (err, mx, bdoc, L_, g)
    print("worst max-abs error (error, max|ref| of that block, doc, length, KV head):", worst)


@pytest.mark.parametrize("sched", ["fused", "stepwise"])
def test_bwd_reuse_forward_workspace(ra, sched):
    """RA_BWD_FWD_RESERVE: reusing the forward's rank-ordered Q, K, V and
    tables gives exactly the gradients of the full backward; with other
    tensors than the forward's the library ignores the flag."""
    cu = W.cu_seqlens((300, 41, 500, 77))
    T = int(cu[-1])
    q, k, v = (x.cuda() for x in W.make_qkv(T, 16, 4, 128, torch.bfloat16))
    do = W.make_dout(T, 16, 128, torch.bfloat16).cuda()
    nb = max(ra.ring_workspace_bytes(T, 16, 4, 128, 0, cu, 4, 1, sched, bwd=b) for b in (False, True))
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    out, lse = ra.ring_attn_fwd(q, k, v, cu, 4, 1, True, None, sched, workspace=ws)
    ref = ra.ring_attn_bwd(q, k, v, out, lse, do, cu, 4, 1, True, None, sched, workspace=ws)
    ref = [x.clone() for x in ref]
    out, lse = ra.ring_attn_fwd(q, k, v, cu, 4, 1, True, None, sched, workspace=ws)
    got = ra.ring_attn_bwd(q, k, v, out, lse, do, cu, 4, 1, True, None, sched, workspace=ws,
                           reuse_fwd_workspace=True)
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    # a second backward on the same tables and reserve space gives the same
    # gradients (nothing a launch leaves in the workspace changes the next)
    got = [x.clone() for x in got]
    again = ra.ring_attn_bwd(q, k, v, out, lse, do, cu, 4, 1, True, None, sched, workspace=ws,
                             reuse_fwd_workspace=True)
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    for a, b in zip(got, again):
        assert torch.equal(a, b)
    # a different q than the forward saw: the flag must be ignored
    q2 = q.flip(0).contiguous()
    out2, lse2 = ra.ring_attn_fwd(q2, k, v, cu, 4, 1, True, None, sched)
    ref2 = [x.clone() for x in ra.ring_attn_bwd(q2, k, v, out2, lse2, do, cu, 4, 1, True, None, sched)]
    ra.ring_attn_fwd(q, k, v, cu, 4, 1, True, None, sched, workspace=ws)
    got2 = ra.ring_attn_bwd(q2, k, v, out2, lse2, do, cu, 4, 1, True, None, sched, workspace=ws,
                            reuse_fwd_workspace=True)
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    for a, b in zip(ref2, got2):
        assert torch.equal(a, b)


def test_ring_step_cuda_graph(ra):
    """The fused forward and backward (the backward forks its key-side kernel
    onto a second stream and joins it) captured once in a CUDA graph: each
    replay gives bit-identical results to eager calls on the same inputs, and
    a replay after the inputs change follows them."""
    cu = W.cu_seqlens((700, 33, 1200, 129, 300))
    T = int(cu[-1])
    q, k, v = (x.cuda() for x in W.make_qkv(T, 16, 4, 128, torch.bfloat16))
    do = W.make_dout(T, 16, 128, torch.bfloat16).cuda()
    nb = max(ra.ring_workspace_bytes(T, 16, 4, 128, 0, cu, 4, 1, "fused", bwd=b) for b in (False, True))
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    out, dq = torch.empty_like(q), torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    lse = torch.empty((16, T), dtype=torch.float32, device="cuda")

    def step():
        ra.ring_attn_fwd(q, k, v, cu, 4, 1, True, None, "fused", out=out, lse=lse, workspace=ws)
        ra.ring_attn_bwd(q, k, v, out, lse, do, cu, 4, 1, True, None, "fused", dq=dq, dk=dk, dv=dv,
                         workspace=ws, reuse_fwd_workspace=True)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # outside capture: plan, page-locked tables, second stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = [x.clone() for x in (out, lse, dq, dk, dv)]
    for x in (out, lse, dq, dk, dv):
        x.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for x in (out, lse, dq, dk, dv):
            x.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert ra.device_status() == 0
        for a, b in zip(ref, (out, lse, dq, dk, dv)):
            assert torch.equal(a, b)
    # new input values, same shapes: the replay reads them
    q.mul_(0.5)
    do.mul_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    got = [x.clone() for x in (out, lse, dq, dk, dv)]
    step()
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    for a, b in zip(got, (out, lse, dq, dk, dv)):
        assert torch.equal(a, b)
    assert not torch.equal(got[2], ref[2])
