"""ra_varlen_attn_partial_noalloc: the partial-attention entry point for
callers that cannot allocate device memory (its scratch is a static device
array inside the library).  Called through the C ABI and compared with the
workspace-taking ra_varlen_attn_partial on the same inputs, on two calls in
a row (the second call must not see anything left over by the first); both
run the same kernel on the same tables, so the results must be
bit-identical.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test."""
import ctypes
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available()
    from context_varlen_ring_gb300 import build as b
    b.build()
    from context_varlen_ring_gb300 import _lib
    torch.cuda.set_device(0)
    return _lib.lib()


def _p(x):
    if isinstance(x, np.ndarray):
        return x.ctypes.data_as(ctypes.c_void_p)
    return ctypes.c_void_p(x.data_ptr())


def _case(seed, lens_q, lens_k, hq, hkv):
    rng = np.random.default_rng(seed)
    cuq, cuk = W.cu_seqlens(lens_q), W.cu_seqlens(lens_k)
    Tq, Tk = int(cuq[-1]), int(cuk[-1])
    qpos = np.concatenate([np.arange(L) + int(rng.integers(200, 400)) for L in lens_q]).astype(np.int32)
    kpos = np.concatenate([np.arange(L) + int(rng.integers(0, 300)) for L in lens_k]).astype(np.int32)
    q = W.randn((Tq, hq, 128), seed + 1, torch.bfloat16).cuda()
    k = W.randn((Tk, hkv, 128), seed + 2, torch.bfloat16).cuda()
    v = W.randn((Tk, hkv, 128), seed + 3, torch.bfloat16).cuda()
    return cuq, cuk, qpos, kpos, q, k, v


def _run_both(L, cuq, cuk, qpos, kpos, q, k, v):
    Tq, hq, d = q.shape
    Tk, hkv, _ = k.shape
    nseg = len(cuq) - 1
    scale = 1.0 / math.sqrt(d)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref_o = torch.empty((Tq, hq, d), dtype=torch.float32, device="cuda")
    ref_l = torch.empty((hq, Tq), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.ra_partial_workspace_bytes(Tq, Tk, nseg, hq, hkv, d, 0), dtype=torch.uint8, device="cuda")
    rc = L.ra_varlen_attn_partial(_p(q), _p(k), _p(v), 0, Tq, Tk, hq, hkv, d, _p(cuq), _p(cuk), nseg, _p(qpos),
                                  _p(kpos), 1, -1, scale, _p(ref_o), _p(ref_l), _p(ws), ws.numel(), stream)
    assert rc == 0, L.ra_last_error()
    # fill the outputs with garbage first: the entry point must write them in full
    out = torch.full((Tq, hq, d), float("nan"), device="cuda")
    lse = torch.full((hq, Tq), float("nan"), device="cuda")
    rc = L.ra_varlen_attn_partial_noalloc(_p(q), _p(k), _p(v), 0, Tq, Tk, hq, hkv, d, _p(cuq), _p(cuk), nseg,
                                          _p(qpos), _p(kpos), 1, -1, scale, _p(out), _p(lse), stream)
    assert rc == 0, L.ra_last_error()
    torch.cuda.synchronize()
    assert L.ra_get_device_status(stream) == 0
    return ref_o.cpu().numpy(), ref_l.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_two_calls(L):
    cases = [
        _case(10, [300, 0, 517], [450, 120, 260], 32, 8),
        _case(20, [64, 1000], [700, 1333], 16, 2),   # different sizes: stale tables must not leak
    ]
    for cuq, cuk, qpos, kpos, q, k, v in cases:
        ro, rl, o, l = _run_both(L, cuq, cuk, qpos, kpos, q, k, v)
        # the same kernel on the same inputs and tables: bit-identical
        # (every row is computed by one work item in a fixed order)
        assert np.array_equal(o, ro)
        assert np.array_equal(l, rl)


def test_noalloc_rejects_oversize_problem(L):
    big = 1 << 21   # needs far more than the static scratch
    cu = np.array([0, big], np.int32)
    need = L.ra_partial_workspace_bytes(big, big, 1, 32, 8, 128, 0)
    assert need > (8 << 20)
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    rc = L.ra_varlen_attn_partial_noalloc(fake, fake, fake, 0, big, big, 32, 8, 128, _p(cu), _p(cu), 1, None, None,
                                          1, -1, 0.1, fake, fake, None)
    assert rc == 4  # RA_ERR_WORKSPACE
    assert b"static" in L.ra_last_error()
