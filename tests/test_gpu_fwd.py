"""GPU parity of the forward path (permute, partial, merge, ring) against the
fp64 oracle.  Tolerances: bf16 inputs -> max-abs 2e-2 on outputs and 1e-3 on
LSE; fp32 inputs -> 1e-5 on both; permutations bit-exact."""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: (2e-2, 1e-3), torch.float32: (1e-5, 1e-5)}


@pytest.fixture(scope="module")
def ra():
    assert torch.cuda.is_available()
    from context_varlen_ring_gb300 import build as b
    b.build()
    import context_varlen_ring_gb300 as m
    m.lib()
    torch.cuda.set_device(0)
    return m


def _cmp_lse(got, ref, tol):
    """got [Hq, T] vs ref [T, Hq]; -inf must match exactly."""
    g = got.T
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(g), fin), "finite/-inf pattern differs"
    assert np.all(g[~fin] == -np.inf)
    if fin.any():
        err = np.abs(g[fin] - ref[fin]).max()
        assert err <= tol, err
        return err
    return 0.0


def _check_status(ra):
    torch.cuda.synchronize()
    assert ra.device_status() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.int8])
def test_permute_unpermute_bit_exact(ra, orc, dtype):
    rng = np.random.default_rng(1)
    for mode in (0, 1):
        cu = W.cu_seqlens(W.random_doc_lens(rng, 3000, 1, 700))
        T = int(cu[-1])
        perm, _, _ = orc.zigzag_plan(cu, 4, mode)
        for shape in ((T, 3, 40), (T, 8, 128), (T, 5)):
            if dtype == torch.int8:
                x = torch.randint(-128, 127, shape, dtype=torch.int8)
            else:
                x = W.randn(shape, 7, dtype)
            y = ra.zigzag_permute(x.cuda(), perm)
            ref = x.numpy() if dtype != torch.bfloat16 else x.view(torch.int16).numpy()
            got = y.cpu()
            got = got.numpy() if dtype != torch.bfloat16 else got.view(torch.int16).numpy()
            assert np.array_equal(got, ref[perm])
            back = ra.zigzag_unpermute(y, perm).cpu()
            back = back.numpy() if dtype != torch.bfloat16 else back.view(torch.int16).numpy()
            assert np.array_equal(back, ref)
    _check_status(ra)


def _positions_two_runs(rng, n):
    """Positions made of two increasing runs (like a zigzag shard)."""
    a = int(rng.integers(0, n + 1))
    s0, s1 = int(rng.integers(0, 1000)), int(rng.integers(2000, 5000))
    return np.concatenate([np.arange(s0, s0 + a), np.arange(s1, s1 + n - a)]).astype(np.int32)


@pytest.mark.parametrize("dtype,d,hq,hkv", [(torch.bfloat16, 128, 8, 2), (torch.bfloat16, 128, 4, 4),
                                           (torch.bfloat16, 128, 16, 1), (torch.float32, 64, 4, 2),
                                           (torch.bfloat16, 64, 4, 2)])
@pytest.mark.parametrize("causal", [True, False])
def test_partial_vs_oracle(ra, orc, dtype, d, hq, hkv, causal):
    rng = np.random.default_rng(2 + d + hq)
    lq = [int(x) for x in rng.integers(0, 400, size=4)]
    lk = [int(x) for x in rng.integers(0, 400, size=4)]
    lq[1], lk[2] = 0, 0            # empty segments on either side
    cuq, cuk = W.cu_seqlens(lq), W.cu_seqlens(lk)
    Tq, Tk = int(cuq[-1]), int(cuk[-1])
    qpos = np.concatenate([_positions_two_runs(rng, L) for L in lq]) if Tq else np.zeros(0, np.int32)
    kpos = np.concatenate([_positions_two_runs(rng, L) for L in lk]) if Tk else np.zeros(0, np.int32)
    q = W.randn((Tq, hq, d), 11, dtype)
    k = W.randn((Tk, hkv, d), 12, dtype)
    v = W.randn((Tk, hkv, d), 13, dtype)
    scale = 1 / math.sqrt(d)
    out, lse = ra.varlen_attn_partial(q.cuda(), k.cuda(), v.cuda(), cuq, cuk, qpos, kpos, causal, scale)
    _check_status(ra)
    ro, rl = orc.partial_fwd(q, k, v, orc.doc_ids(cuq), orc.doc_ids(cuk), qpos, kpos, causal, scale)
    to, tl = TOL[dtype]
    assert np.abs(out.cpu().numpy() - ro).max() <= to
    _cmp_lse(lse.cpu().numpy(), rl, tl)


@pytest.mark.parametrize("d,n", [(128, 5), (64, 3), (160, 33), (4, 64), (256, 8)])
def test_merge_vs_oracle(ra, orc, d, n):
    """Head dims that are not a multiple of 128 leave some lanes without
    elements in the last 128-column pass (d=64: lanes 16-31; d=160: lanes
    8-31 of the second pass), and n > 32 puts part weights in both halves."""
    rng = np.random.default_rng(3 + d + n)
    T, H = 777, 6
    outs, lses = [], []
    for p in range(n):
        o = rng.standard_normal((T, H, d)).astype(np.float32)
        l = (rng.standard_normal((T, H)) * 3).astype(np.float32)
        l[rng.random((T, H)) < 0.2] = -np.inf
        o[np.isneginf(l)] = 0.0
        outs.append(o)
        lses.append(l)
    lses[0][5] = -np.inf  # make some rows fully empty
    for l in lses:
        l[5] = -np.inf
    for o in outs:
        o[5] = 0
    go = [torch.from_numpy(o).cuda() for o in outs]
    gl = [torch.from_numpy(np.ascontiguousarray(l.T)).cuda() for l in lses]
    for dt, tol in ((torch.float32, 1e-5), (torch.bfloat16, 2e-2)):
        mo, ml = ra.lse_merge(go, gl, dt)
        ro, rl = orc.lse_merge(outs, lses)
        assert np.abs(mo.float().cpu().numpy() - ro).max() <= tol
        _cmp_lse(ml.cpu().numpy(), rl, 1e-5)
    _check_status(ra)


@pytest.mark.parametrize("sched", ["fused", "stepwise"])
def test_ring_c0_fp32(ra, orc, sched):
    wl = W.C0
    cu = wl.cu_seqlens()
    q, k, v = W.make_qkv(wl.T, wl.hq, wl.hkv, wl.d, wl.dtype)
    out, lse = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), cu, wl.cp, wl.zz_mode, True, wl.scale, sched)
    _check_status(ra)
    ro, rl = orc.attn_fwd(q, k, v, cu, True, wl.scale)
    assert np.abs(out.cpu().numpy() - ro).max() <= 1e-5
    _cmp_lse(lse.cpu().numpy(), rl, 1e-5)


@pytest.mark.parametrize("sched", ["fused", "stepwise"])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_ring_small_bf16(ra, orc, sched, mode, G):
    rng = np.random.default_rng(100 + 10 * G + mode)
    for trial in range(3):
        docs = W.random_doc_lens(rng, 1800, 1, 700)
        cu = W.cu_seqlens(docs)
        T = int(cu[-1])
        cp = [1, 2, 3, 4, 8][(trial + G) % 5]
        hkv = 2
        q, k, v = W.make_qkv(T, hkv * G, hkv, 128, torch.bfloat16, seed_offset=trial)
        causal = trial != 2
        out, lse = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), cu, cp, mode, causal, None, sched)
        _check_status(ra)
        ro, rl = orc.attn_fwd(q, k, v, cu, causal, 1 / math.sqrt(128))
        err = np.abs(out.float().cpu().numpy() - ro).max()
        assert err <= 2e-2, (docs, cp, err)
        _cmp_lse(lse.cpu().numpy(), rl, 1e-3)


def _sampled_check(ra, orc, wl, nrows, seed, sched="fused"):
    cu = wl.cu_seqlens()
    T = wl.T
    q, k, v = W.make_qkv(T, wl.hq, wl.hkv, wl.d, wl.dtype)
    out, lse = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), cu, wl.cp, wl.zz_mode, True, wl.scale, sched)
    _check_status(ra)
    perm, off, _ = ra.zigzag_plan(cu, wl.cp, wl.zz_mode)
    # rows at every rank boundary, every doc boundary, plus seeded random rows
    must = list(perm[np.minimum(off[:-1], T - 1)]) + list(cu[:-1]) + list(np.maximum(cu[1:] - 1, 0))
    rows = W.sample_rows(T, nrows, seed, must)
    seg = orc.doc_ids(cu)
    ro, rl = orc.partial_fwd(q[torch.from_numpy(rows)], k, v, seg[rows], seg, rows, np.arange(T), True, wl.scale)
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    err = np.abs(got - ro).max()
    assert err <= 2e-2, err
    lerr = np.abs(lse[:, torch.from_numpy(rows).cuda()].cpu().numpy().T - rl).max()
    assert lerr <= 1e-3, lerr
    return err, lerr


def test_ring_c1_sampled(ra, orc):
    _sampled_check(ra, orc, W.C1, 96, 1)


def test_ring_c2_sampled(ra, orc):
    _sampled_check(ra, orc, W.C2, 128, 2)


def test_ring_c2_stepwise_sampled(ra, orc):
    _sampled_check(ra, orc, W.C2, 48, 5, sched="stepwise")


def test_ring_c3_sampled(ra, orc):
    """The 131072-token sequence (CP 16): 256 query rows of all 64 heads,
    every zigzag rank boundary among them."""
    _sampled_check(ra, orc, W.C3, 256, 3)


@pytest.mark.parametrize("name", ["C1", "C2"])
def test_ring_whole_output(ra, orc, name):
    """The 8192-token sequence (CP 4, zigzag over the stream) and the packed
    32768-token workload (CP 8, per-document zigzag) in the bench's
    configuration (fused ring): every output element and every LSE against
    the oracle's forward of the whole workload."""
    wl = W.ALL[name]
    cu = wl.cu_seqlens()
    q, k, v = W.make_qkv(wl.T, wl.hq, wl.hkv, wl.d, wl.dtype)
    out, lse = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), cu, wl.cp, wl.zz_mode, True, wl.scale)
    _check_status(ra)
    ro, rl = orc.attn_fwd(q, k, v, cu, True, wl.scale)
    err = np.abs(out.float().cpu().numpy() - ro).max()
    assert err <= 2e-2, err
    _cmp_lse(lse.cpu().numpy(), rl, 1e-3)


def test_wait_guard_selftest(ra):
    from context_varlen_ring_gb300 import _lib
    _check_status(ra)
    ra.selftest_wait_timeout(2000)
    torch.cuda.synchronize()
    assert ra.device_status() == _lib.RA_ERR_TIMEOUT
    assert ra.device_status() == 0


def test_partial_refuses_stream_capture(ra):
    """The partial call plans on the host and uploads its tables from host
    memory each call, so on a capturing stream it returns
    RA_ERR_UNSUPPORTED before doing any work; eager calls are unaffected."""
    cu = np.array([0, 200], np.int32)
    q, k, v = (x.cuda() for x in W.make_qkv(200, 8, 2, 128, torch.bfloat16))
    out = torch.empty((200, 8, 128), device="cuda")
    lse = torch.empty((8, 200), device="cuda")
    ra.varlen_attn_partial(q, k, v, cu, cu, out=out, lse=lse)
    torch.cuda.synchronize()
    ref = (out.clone(), lse.clone())
    g = torch.cuda.CUDAGraph()
    err = None
    with torch.cuda.graph(g):
        try:
            ra.varlen_attn_partial(q, k, v, cu, cu, out=out, lse=lse)
        except ra.RaError as e:
            err = e
    assert err is not None and err.status == 2, err
    del g
    out.zero_()
    ra.varlen_attn_partial(q, k, v, cu, cu, out=out, lse=lse)
    torch.cuda.synchronize()
    _check_status(ra)
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])


def test_readme_usage_example(ra):
    """The README's Python example runs as written: the whole ring (8 ranks,
    per-document zigzag) and one partial over the whole packed buffer (local
    row index as position, so each document's causal attention) merged alone
    give the same attention, within the bf16 output tolerance, and the
    backward returns finite gradients of the inputs' shapes."""
    cu = [0, 1809, 2202, 2353]
    g = torch.Generator(device="cuda").manual_seed(3)
    q = torch.randn(2353, 32, 128, device="cuda", dtype=torch.bfloat16, generator=g)
    k = torch.randn(2353, 8, 128, device="cuda", dtype=torch.bfloat16, generator=g)
    v = torch.randn(2353, 8, 128, device="cuda", dtype=torch.bfloat16, generator=g)
    out, lse = ra.ring_attn_fwd(q, k, v, cu, 8, ra.RA_ZZ_PER_DOC)
    do = torch.randn(2353, 32, 128, device="cuda", dtype=torch.bfloat16, generator=g)
    dq, dk, dv = ra.ring_attn_bwd(q, k, v, out, lse, do, cu, 8, ra.RA_ZZ_PER_DOC)
    o1, l1 = ra.varlen_attn_partial(q, k, v, cu, cu)
    o, l = ra.lse_merge([o1], [l1], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    assert (out.float() - o.float()).abs().max().item() <= TOL[torch.bfloat16][0]
    assert (lse - l).abs().max().item() <= TOL[torch.bfloat16][1]
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    assert all(torch.isfinite(t.float()).all().item() for t in (dq, dk, dv))
