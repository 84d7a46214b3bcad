"""The partial-attention step with DEVICE segment boundaries and positions
(ra_varlen_attn_partial_dev): its tile tables are built on the GPU with the
host planner's tiling, so on the same inputs its results are bit-identical
to ra_varlen_attn_partial's (whose parity against the oracle is tested in
test_gpu_fwd.py); it is checked against the oracle directly as well, under
CUDA-graph capture, and on malformed device boundaries (which the tile
builder's own checks turn into RA_ERR_DEVICE_BOUNDS)."""
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


def _positions(rng, lens, kind):
    """Per-segment positions: one run, two runs (a zigzag shard), or random
    strides (many runs, so many short tiles)."""
    out = []
    for L in lens:
        base = int(rng.integers(0, 500))
        if kind == "one":
            p = base + np.arange(L)
        elif kind == "two":
            a = L // 2
            p = np.concatenate([base + np.arange(a), base + a + int(rng.integers(1, 300)) + np.arange(L - a)])
        else:
            p = base + np.cumsum(rng.integers(1, 3, L))
        out.append(p)
    return np.concatenate(out).astype(np.int32) if out else np.zeros(0, np.int32)


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("kind", ["one", "two", "random"])
def test_device_arrays_match_host_arrays(ra, G, kind):
    rng = np.random.default_rng(1000 + 7 * G + len(kind))
    hkv = 2 if G < 16 else 1
    for trial in range(3):
        nseg = int(rng.integers(1, 6))
        lq = [int(x) for x in rng.integers(0, 400, nseg)]
        lk = [int(x) for x in rng.integers(0, 500, nseg)]
        if sum(lq) == 0:
            lq[0] = 5
        cuq, cuk = W.cu_seqlens(lq), W.cu_seqlens(lk)
        qp, kp = _positions(rng, lq, kind), _positions(rng, lk, kind)
        causal = bool(trial != 1)
        window = [-1, 50, -1][trial]
        Tq, Tk = int(cuq[-1]), int(cuk[-1])
        q = W.randn((Tq, hkv * G, 128), 11 + trial, torch.bfloat16).cuda()
        k = W.randn((max(Tk, 1), hkv, 128), 12 + trial, torch.bfloat16).cuda()[:Tk]
        v = W.randn((max(Tk, 1), hkv, 128), 13 + trial, torch.bfloat16).cuda()[:Tk]
        if Tk == 0:
            k = torch.empty((0, hkv, 128), dtype=torch.bfloat16, device="cuda")
            v = torch.empty((0, hkv, 128), dtype=torch.bfloat16, device="cuda")
        ro, rl = ra.varlen_attn_partial(q, k, v, cuq, cuk, qp, kp, causal=causal, window=window)
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
        o, l = ra.varlen_attn_partial_dev(q, k, v, dev(cuq), dev(cuk), dev(qp), dev(kp), causal=causal, window=window)
        torch.cuda.synchronize()
        assert ra.device_status() == 0
        assert torch.equal(o, ro) and torch.equal(l, rl), (kind, G, trial, lq, lk)


def test_device_arrays_against_oracle_and_null_positions(ra, orc):
    """A zigzag-like shard against the oracle; NULL positions mean row indices."""
    rng = np.random.default_rng(5)
    lq, lk = [300, 129, 0, 517], [450, 120, 260, 333]
    cuq, cuk = W.cu_seqlens(lq), W.cu_seqlens(lk)
    qp, kp = _positions(rng, lq, "two"), _positions(rng, lk, "two")
    Tq, Tk = int(cuq[-1]), int(cuk[-1])
    q = W.randn((Tq, 16, 128), 21, torch.bfloat16)
    k = W.randn((Tk, 4, 128), 22, torch.bfloat16)
    v = W.randn((Tk, 4, 128), 23, torch.bfloat16)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    o, l = ra.varlen_attn_partial_dev(q.cuda(), k.cuda(), v.cuda(), dev(cuq), dev(cuk), dev(qp), dev(kp))
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    ro, rl = orc.partial_fwd(q, k, v, orc.doc_ids(cuq), orc.doc_ids(cuk), qp, kp, True, 1 / math.sqrt(128))
    assert np.abs(o.cpu().numpy() - ro).max() <= 2e-2
    g, r = l.cpu().numpy().T, rl
    fin = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), fin) and np.abs(g[fin] - r[fin]).max() <= 1e-3
    # NULL positions: the row indices
    o2, l2 = ra.varlen_attn_partial_dev(q.cuda(), k.cuda(), v.cuda(), dev(cuq), dev(cuk))
    ro2, rl2 = ra.varlen_attn_partial(q.cuda(), k.cuda(), v.cuda(), cuq, cuk)
    torch.cuda.synchronize()
    assert torch.equal(o2, ro2) and torch.equal(l2, rl2)


def test_device_arrays_capture_in_cuda_graph(ra):
    """No host round trip: the call captures into a CUDA graph, replays give
    the eager results, and a replay follows changed device arrays."""
    rng = np.random.default_rng(6)
    lq = lk = [200, 333, 91]
    cuq = torch.from_numpy(W.cu_seqlens(lq)).cuda()
    cuk = torch.from_numpy(W.cu_seqlens(lk)).cuda()
    qp = torch.from_numpy(_positions(rng, lq, "two")).cuda()
    kp = qp.clone()
    T = int(sum(lq))
    q, k, v = (x.cuda() for x in W.make_qkv(T, 8, 2, 128, torch.bfloat16))
    out = torch.empty((T, 8, 128), device="cuda")
    lse = torch.empty((8, T), device="cuda")
    ws = torch.empty(ra.lib().ra_partial_workspace_bytes(T, T, 3, 8, 2, 128, 0), dtype=torch.uint8, device="cuda")
    call = lambda: ra.varlen_attn_partial_dev(q, k, v, cuq, cuk, qp, kp, out=out, lse=lse, workspace=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()  # first call outside capture (kernel attributes, tensor-map encoder)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = (out.clone(), lse.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
    # shift the key positions by 50: the causal mask moves, the replay follows
    kp.add_(50)
    g.replay()
    torch.cuda.synchronize()
    got = (out.clone(), lse.clone())
    call()
    torch.cuda.synchronize()
    assert torch.equal(got[0], out) and torch.equal(got[1], lse)
    assert not torch.equal(got[1], ref[1])


def test_device_arrays_malformed_boundaries_are_reported(ra):
    """Segment boundaries that do not end at Tq are caught by the tile
    builder's own check: RA_ERR_DEVICE_BOUNDS in the status word, no work."""
    T = 256
    q, k, v = (x.cuda() for x in W.make_qkv(T, 8, 2, 128, torch.bfloat16))
    bad = torch.tensor([0, 100, 300], dtype=torch.int32, device="cuda")  # 300 != 256
    good = torch.tensor([0, 100, 256], dtype=torch.int32, device="cuda")
    ra.varlen_attn_partial_dev(q, k, v, bad, good)
    torch.cuda.synchronize()
    assert ra.device_status() == 6  # RA_ERR_DEVICE_BOUNDS
    o, l = ra.varlen_attn_partial_dev(q, k, v, good, good)  # the next call runs normally
    torch.cuda.synchronize()
    assert ra.device_status() == 0 and torch.isfinite(o).all()
