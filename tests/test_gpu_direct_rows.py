"""The tensor-core kernels read a query tile of one position run straight
from the caller's Q (and dO) and take only the rows of two-run tiles from
the rank-ordered copies, which the permutes fill for those rows alone.
These tests fill the workspace with NaN bytes first, so any read of a row
the permutes skipped would turn the results into NaN, and compare with the
fp64 oracle (bf16: max-abs 2e-2 relative to max(1, max|ref|), LSE 1e-3)."""
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


@pytest.mark.parametrize("sched", ["fused", "stepwise"])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("reuse", [False, True])
def test_nan_filled_workspace(ra, orc, sched, G, reuse):
    """Documents whose zigzag chunks are not multiples of a tile, so most
    (rank, document) shares hold a two-run tile, and tails shorter than a
    tile; the backward either reuses the forward's rank-ordered copies or
    makes its own in a freshly NaN-filled workspace."""
    rng = np.random.default_rng(700 + G + 10 * reuse)
    docs = [int(x) for x in rng.integers(50, 700, size=5)] + [129, 31]
    cu = W.cu_seqlens(docs)
    T = int(cu[-1])
    hkv, cp, mode = 2, 4, 1
    q, k, v = W.make_qkv(T, hkv * G, hkv, 128, torch.bfloat16, seed_offset=G)
    do = W.make_dout(T, hkv * G, 128, torch.bfloat16, seed_offset=G)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    nb = max(ra.ring_workspace_bytes(T, hkv * G, hkv, 128, 0, cu, cp, mode, sched, bwd=b) for b in (False, True))
    ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda")
    out, lse = ra.ring_attn_fwd(qd, kd, vd, cu, cp, mode, True, None, sched, workspace=ws)
    if not reuse:
        ws.fill_(0xFF)
    dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, out, lse, dod, cu, cp, mode, True, None, sched,
                                  grad_dtype=torch.float32, workspace=ws, reuse_fwd_workspace=reuse)
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    scale = 1 / math.sqrt(128)
    ro, rl = orc.attn_fwd(q, k, v, cu, True, scale)
    assert _err(out.float().cpu().numpy(), ro) <= 2e-2
    assert _lse_err(lse.cpu().numpy(), rl) <= 1e-3
    rdq, rdk, rdv = orc.attn_bwd(q, k, v, ro, rl, do, cu, True, scale)
    for g, r in ((dq, rdq), (dk, rdk), (dv, rdv)):
        a = g.cpu().numpy()
        assert np.isfinite(a).all()
        assert _gerr(a, r) <= 2e-2, (_err(a, r), float(np.abs(r).max()))
