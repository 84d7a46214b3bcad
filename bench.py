"""Benchmark: packed causal varlen ring attention, fwd+bwd, on GB300.

One step = the whole hot path on the packed 32768-token workload (GQA 32/8,
d=128, bf16, per-document zigzag over 8 simulated CP ranks): zigzag
permute (rank-ordered copies of the rows of tiles that straddle two zigzag
chunks; the kernels read every other tile in place), ring forward with
on-chip merge (O and LSE written in the original order), backward
preprocess (the same copies of dO, D = rowsum(dO*O), per-tile LSE/D), ring
backward with fp32 dK/dV (the backward reuses the forward's copies and tile
tables from the shared workspace, its saved activations).  --sched
allgather times the all-gather form instead (each rank's queries against
every rank's K/V, read in original order).  FLOPs count allowed (causal, same-document) pairs only:
4*d*Hq per pair forward, 10*d*Hq backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU
oracle on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "packed causal varlen attention TFLOP/s (fwd, fwd+bwd) and % bf16 TC peak"
L2_BYTES = 129 * 2**20


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def pairs_of(cu, window: int = -1) -> int:
    """Allowed causal (query, key) pairs of a packing; with a sliding window
    a query sees at most window + 1 keys (itself included)."""
    L = np.diff(np.asarray(cu, dtype=np.int64))
    if window < 0:
        return int((L * (L + 1) // 2).sum())
    w1 = window + 1
    short = L <= w1
    return int((L[short] * (L[short] + 1) // 2).sum() +
               (w1 * (w1 + 1) // 2 + (L[~short] - w1) * w1).sum())


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_sample_docs(lens, pair_budget=15_000_000):
    """A bounded sample of the workload for the CPU oracle: the smaller
    documents up to `pair_budget` causal pairs (15M: about 10-30 s of fp64
    fwd+bwd work on 16 cores)."""
    order = sorted(range(len(lens)), key=lambda i: lens[i])
    pick, pairs = [], 0
    for i in order:
        p = lens[i] * (lens[i] + 1) // 2
        if pairs + p > pair_budget and pick:
            break
        pick.append(i)
        pairs += p
    return sorted(pick)


def run_cpu_oracle(wl, steps=1, window=-1, pair_budget=15_000_000, threads=None):
    """fwd+bwd of the sampled documents with the fp64 oracle; returns
    (TFLOP/s, seconds per step, cores, sample description, sample pairs)."""
    import oracle
    oracle.build()
    cores = oracle.set_threads(threads or os.cpu_count() or 1)
    pick = cpu_sample_docs(list(wl.doc_lens), pair_budget)
    lens = [wl.doc_lens[i] for i in pick]
    cu = W.cu_seqlens(lens)
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, wl.hq, wl.hkv, wl.d, wl.dtype)
    do = W.make_dout(T, wl.hq, wl.d, wl.dtype)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        o, l = oracle.attn_fwd(q, k, v, cu, True, wl.scale, window=window)
        oracle.attn_bwd(q, k, v, o, l, do, cu, True, wl.scale, window=window)
        times.append(time.perf_counter() - t0)
    sec = statistics.median(times)
    if threads:
        oracle.set_threads(os.cpu_count() or 1)
    sp = pairs_of(cu, window)
    flops = 14 * wl.d * wl.hq * sp
    sample = (f"fp64 fwd+bwd of {len(lens)} of the {wl.B} documents ({T} of {wl.T} tokens, "
              f"{sp} of {pairs_of(wl.cu_seqlens(), window)} allowed pairs), all {wl.hq} heads")
    return flops / sec / 1e12, sec, cores, sample, sp


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = W.C4
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state; warm-up steps are not repeated
    # each step a bounded sample sized so that the whole run ends within a
    # few minutes: about 120 s of fp64 work over the K steps (15M pairs take
    # about 18 s on 16 host cores)
    budget = int(min(15_000_000, max(1_000_000, 15_000_000 * 120 / (18 * max(1, args.steps)))))
    tf, sec, cores, sample, _ = run_cpu_oracle(wl, steps=max(1, args.steps), pair_budget=budget)
    line = {"impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "Hq": wl.hq, "Hkv": wl.hkv, "d": wl.d, "cp": wl.cp,
                       "zigzag": "per-doc", "parallelism": "host cores"},
            "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(x, world, device):
    """The largest of every rank's `x` (each rank's own timing); x itself when
    world == 1.  Collective on the default process group."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_step, steps, max_ms):
    """Whole-job throughput: every rank runs `steps` steps of `flops_per_step`
    (replicas, weak scaling) within the slowest rank's `max_ms`."""
    return world * flops_per_step * steps / (max_ms / 1e3) / 1e12


# Work of each timed scope per launch (fused schedule: one launch covers all
# ring steps), in products of 2*d FLOPs per (query head, allowed pair).
# ALGORITHMIC counts what the method needs: the forward's S and PV, the
# backward's recomputed S, dV, dP, dK and dQ (10*d*Hq per pair).  EXECUTED
# counts what the kernels form: the backward runs as two concurrent passes
# (key side: S^T, dP^T, dV, dK; query side: S, dP, dQ), so S and dP are
# formed twice; the difference is implementation overhead and is reported
# beside the roofline, never in it.
ALGORITHMIC_PRODUCTS = {"ra_tc_fwd": 2, "ra_simt_fwd": 2, "ra_tc_bwd": 5, "ra_simt_bwd": 5}
EXECUTED_PRODUCTS = {"ra_tc_fwd": 2, "ra_tc_bwd": 7, "ra_tc_bwd_dkdv": 4, "ra_tc_bwd_dq": 3}
KERNELS_PER_SCOPE = {"ra_tc_bwd": 2}
E2E_REPS = 5  # timed repetitions of the end-to-end loop (median reported)


def kernel_traffic(name):
    """DRAM bytes per launch of `name` from the committed ncu summary, or None
    when there is none or a source of the kernel changed since it was captured.
    An entry lists every source file it depends on with its sha256 (the
    concurrent backward pair lists both kernels' files and sums their bytes)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            tab = json.load(f)
    except (OSError, ValueError):
        return None
    ent = tab.get(name)
    if not ent or not ent.get("sources"):
        return None
    for src, want in ent["sources"].items():
        try:
            with open(os.path.join(ROOT, "context_varlen_ring_gb300", "csrc", src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != want:
                    return None
        except OSError:
            return None
    return ent["dram_bytes_per_launch"]


# Timing scope -> (kernels whose DRAM bytes it sums, source files it depends on).
TRAFFIC_SCOPES = {
    "ra_tc_fwd": (["tc_fwd_kernel"], ["ra_tc_fwd.cu", "ra_dev.cuh", "ra_plan.cpp", "ra_api.cpp"]),
    "ra_tc_bwd": (["tc_dq_kernel", "tc_dkdv_kernel"], ["ra_tc_bwd.cu", "ra_tc_dq.cu", "ra_api.cpp", "ra_dev.cuh",
                                                       "ra_plan.cpp"]),
    "ra_tc_bwd_dkdv": (["tc_dkdv_kernel"], ["ra_tc_bwd.cu", "ra_dev.cuh", "ra_plan.cpp"]),
    "ra_tc_bwd_dq": (["tc_dq_kernel"], ["ra_tc_dq.cu", "ra_dev.cuh", "ra_plan.cpp"]),
    "ra_permute_fwd": (["permute_kernel"], ["ra_misc.cu", "ra_dev.cuh", "ra_plan.cpp", "ra_api.cpp"]),
    "ra_permute_rowdot": (["permute_rowdot_kernel"], ["ra_misc.cu", "ra_dev.cuh", "ra_plan.cpp", "ra_api.cpp"]),
}


def traffic_table(source, profile="profiles/launches_c4_fwd_bwd.md"):
    """The per-scope DRAM bytes table (profiles/traffic.json) from an ncu
    launch list of one fwd+bwd step in CSV form (--metrics
    dram__bytes_read.sum,dram__bytes_write.sum,... --csv; a path, or its
    lines): per scope, the
    read + write bytes of its kernels' launches in the list, with the
    sha256 of every source file the scope depends on at the time of the
    call.  A launch's kernel is the identifier that its argument list (and
    template arguments) follow in the demangled name ncu prints."""
    import csv
    import hashlib
    import re
    src_lines = open(source).read().splitlines() if isinstance(source, str) else list(source)
    lines = [ln for ln in src_lines if not ln.startswith("==")]
    rows = list(csv.reader(lines))
    hdr = rows[0]
    ident = re.compile(r"([A-Za-z_]\w*)\s*(?:<[^()]*>)?\s*\(")
    per = {}
    for r in rows[1:]:
        d = dict(zip(hdr, r))
        m = ident.search(d["Kernel Name"])
        key = (d.get("ID", ""), m.group(1) if m else d["Kernel Name"])
        per.setdefault(key, {})[d["Metric Name"]] = float(d["Metric Value"].replace(",", ""))

    def bytes_of(kernel):
        hits = [m for (i, n), m in per.items() if n == kernel]
        if len(hits) != 1:
            raise ValueError(f"{kernel}: {len(hits)} launches in the list, expected one")
        return int(hits[0]["dram__bytes_read.sum"] + hits[0]["dram__bytes_write.sum"])

    csrc = os.path.join(ROOT, "context_varlen_ring_gb300", "csrc")
    tab = {}
    for scope, (kernels, files) in TRAFFIC_SCOPES.items():
        srcs = {}
        for f in files:
            with open(os.path.join(csrc, f), "rb") as fh:
                srcs[f] = hashlib.sha256(fh.read()).hexdigest()
        tab[scope] = {"sources": srcs, "dram_bytes_per_launch": sum(bytes_of(k) for k in kernels),
                      "profile": profile}
    return tab


def tensor_roofline(name, ms_per_launch, d, hq, pairs, peak, peak_src):
    """Roofline entry of a tensor-core scope: the method's algorithmic FLOPs
    per launch over the launch's CUDA-event time, against the burst bf16
    peak (the scopes are timed inside a loop well under a second long).
    The FLOPs the kernels execute (the backward forms S and dP twice) are
    reported beside it as executed_*."""
    sec = ms_per_launch / 1e3
    n_alg = ALGORITHMIC_PRODUCTS.get(name)
    if n_alg is None:
        return {"kernel": name, "bound": "hbm", "achieved": None, "peak": None, "unit": "GB/s", "frac": None,
                "traffic": kernel_traffic(name)}
    flops = n_alg * 2 * d * hq * pairs
    ach = flops / sec / 1e12
    n_exe = EXECUTED_PRODUCTS.get(name, n_alg)
    exe = n_exe * 2 * d * hq * pairs / sec / 1e12
    return {"kernel": name, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
            "frac": ach / peak, "traffic": kernel_traffic(name),
            "peak_kind": f"{peak_src} dense bf16 burst (the scope is timed inside a loop of well under a second)",
            "ms_per_launch": ms_per_launch,
            "algorithmic_per_launch": flops, "algorithmic_unit": "FLOP",
            "algorithmic_rule": f"{n_alg} products x 2*d FLOPs per (query head, allowed pair)",
            "executed_tflops": exe, "executed_frac": exe / peak,
            "executed_rule": f"{n_exe} products formed by the kernels"}


def time_calls(fn, steps, warmup, stream, torch):
    """Milliseconds per call of fn(): `warmup` untimed calls, then `steps`
    calls between two CUDA events on the launching stream."""
    for _ in range(max(warmup, 3)):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def bandwidth_kernels(ra, torch, dev, wl, steps, warmup, hbm, merge_parts=None):
    """The HBM-bound kernels of the path at full size on the packed
    32768-token workload, each as algorithmic bytes (every byte the
    operation must read and write once) over its CUDA-event time:
      permute   ra_zigzag_permute of Q, K and V into rank order (3 calls a rep)
      unpermute ra_zigzag_unpermute of O back to original order
      merge     ra_lse_merge of cp fp32 partials [T, Hq, d] (+ LSEs), bf16 out
    Each rep moves more than the 129 MB L2 (merge: 4.6 GB, permute 805 MB,
    unpermute 537 MB), so no flush is needed between reps."""
    L = ra.lib()
    cu = wl.cu_seqlens()
    T, hq, hkv, d = wl.T, wl.hq, wl.hkv, wl.d
    perm_h, _, _ = ra.zigzag_plan(cu, wl.cp, wl.zz_mode)
    perm = torch.from_numpy(perm_h.astype(np.int32)).to(dev)
    q, k, v = (x.to(dev) for x in W.make_qkv(T, hq, hkv, d, wl.dtype))
    yq, yk, yv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rb = lambda t: t[0].numel() * t.element_size()

    def permute3():
        for x, y in ((q, yq), (k, yk), (v, yv)):
            assert L.ra_zigzag_permute(P(x), P(y), P(perm), T, rb(x), sp) == 0

    def unpermute_o():
        assert L.ra_zigzag_unpermute(P(yq), P(q), P(perm), T, rb(yq), sp) == 0

    res = {}
    ms = time_calls(permute3, steps, warmup, stream, torch)
    nb = 2 * sum(x.numel() * x.element_size() for x in (q, k, v))
    res["permute_qkv"] = {"ms": ms, "bytes": nb, "gbs": nb / ms / 1e6, "frac": nb / ms / 1e6 / hbm}
    ms = time_calls(unpermute_o, steps, warmup, stream, torch)
    nb = 2 * q.numel() * q.element_size()
    res["unpermute_o"] = {"ms": ms, "bytes": nb, "gbs": nb / ms / 1e6, "frac": nb / ms / 1e6 / hbm}
    del yk, yv
    n = merge_parts or wl.cp
    g = torch.Generator(device=dev).manual_seed(5)
    parts = [torch.randn((T, hq, d), generator=g, device=dev, dtype=torch.float32) for _ in range(n)]
    lses = [torch.randn((hq, T), generator=g, device=dev, dtype=torch.float32) * 3 for _ in range(n)]
    po = (ctypes.c_void_p * n)(*[x.data_ptr() for x in parts])
    pl = (ctypes.c_void_p * n)(*[x.data_ptr() for x in lses])
    mo = torch.empty((T, hq, d), dtype=torch.bfloat16, device=dev)
    ml = torch.empty((hq, T), dtype=torch.float32, device=dev)

    def merge():
        assert L.ra_lse_merge(n, po, pl, T, hq, d, P(mo), 0, P(ml), sp) == 0

    ms = time_calls(merge, steps, warmup, stream, torch)
    nb = sum(x.numel() * 4 for x in parts + lses) + mo.numel() * 2 + ml.numel() * 4
    res["lse_merge"] = {"ms": ms, "bytes": nb, "gbs": nb / ms / 1e6, "frac": nb / ms / 1e6 / hbm, "parts": n,
                        "note": "every partial finite (all parts read)"}
    assert ra.device_status() == 0
    del parts, lses, mo, ml, q, k, v, yq
    torch.cuda.empty_cache()
    return {"peak_gbs": hbm, "rule": "algorithmic bytes (read once + written once) / CUDA-event time", **res}


def fwd_lines(ra, torch, dev, names, steps, warmup, peak, sched="fused"):
    """Forward-only calls of the named workloads (whole call: table upload,
    permute of two-run tile rows, fused forward): ms and TFLOP/s."""
    out = {}
    for name in names:
        wl = W.ALL[name]
        cu = wl.cu_seqlens()
        T, hq, hkv, d = wl.T, wl.hq, wl.hkv, wl.d
        pairs = pairs_of(cu)
        q, k, v = (x.to(dev) for x in W.make_qkv(T, hq, hkv, d, wl.dtype))
        o = torch.empty_like(q)
        lse = torch.empty((hq, T), dtype=torch.float32, device=dev)
        ws = torch.empty(ra.ring_workspace_bytes(T, hq, hkv, d, 0, cu, wl.cp, wl.zz_mode, sched, bwd=False),
                         dtype=torch.uint8, device=dev)
        f = lambda: ra.ring_attn_fwd(q, k, v, cu, wl.cp, wl.zz_mode, True, wl.scale, sched, out=o, lse=lse,
                                     workspace=ws)
        ms = time_calls(f, steps, warmup, torch.cuda.current_stream(dev), torch)
        assert ra.device_status() == 0
        tf = 4 * d * hq * pairs / (ms / 1e3) / 1e12
        out[name] = {"ms": ms, "tflops": tf, "frac_of_peak": tf / peak, "allowed_pairs_per_head": pairs,
                     "T": T, "Hq": hq, "Hkv": hkv, "cp": wl.cp, "sched": sched}
        del q, k, v, o, lse, ws
        torch.cuda.empty_cache()
    return out


def _numa_node_of(addr):
    """NUMA node holding the pages of the mapping that contains `addr`
    (from /proc/self/maps and /proc/self/numa_maps), or None."""
    try:
        start = None
        for line in open("/proc/self/maps"):
            a, b = line.split()[0].split("-")
            if int(a, 16) <= addr < int(b, 16):
                start = a.lstrip("0") or "0"
                break
        if start is None:
            return None
        for line in open("/proc/self/numa_maps"):
            f = line.split()
            if f and (f[0].lstrip("0") or "0") == start:
                nodes = {int(x[1:x.index("=")]): int(x[x.index("=") + 1:]) for x in f if x.startswith("N")}
                return max(nodes, key=nodes.get) if nodes else None
    except (OSError, ValueError):
        return None
    return None


def host_copy_rates(torch, dev, tensors_in, tensors_out, stream):
    """Standalone page-locked copies of one step's inputs (host to device)
    and results (device to host), alone and both directions at once, in
    GB/s, with where the page-locked buffers and the GPU sit."""
    h_in = [x.cpu().pin_memory() for x in tensors_in]
    d_in = [torch.empty_like(x) for x in tensors_in]
    h_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in tensors_out]
    nin = sum(x.numel() * x.element_size() for x in h_in)
    nout = sum(x.numel() * x.element_size() for x in h_out)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, reps=5):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            for a, b in zip(d_in, h_in):
                a.copy_(b, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            for a, b in zip(h_out, tensors_out):
                a.copy_(b, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_in, t_out, t_both = timed(h2d), timed(d2h), timed(both)
    info = {"h2d_gbs": nin / t_in / 1e9, "d2h_gbs": nout / t_out / 1e9,
            "concurrent_gbs_each_way": {"h2d": nin / t_both / 1e9, "d2h": nout / t_both / 1e9},
            "bytes_each_way": [nin, nout], "rule": "best of 5 wall-clock runs of one step's copies"}
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = f"{props.pci_domain_id:04x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        info["gpu_pci"] = bus
        info["gpu_numa_node"] = int(open(f"/sys/bus/pci/devices/{bus}/numa_node").read().strip())
    except Exception:
        pass
    info["pinned_numa_node"] = _numa_node_of(h_in[0].data_ptr())
    try:
        cpus = sorted(os.sched_getaffinity(0))
        info["process_cpus"] = f"{cpus[0]}-{cpus[-1]} ({len(cpus)})" if cpus else None
    except Exception:
        pass
    del h_in, d_in, h_out
    return info



def stepwise_lines(ra, torch, dev, wl, steps, warmup, peak, q, k, v, do):
    """The literal per-step structure (one partial launch per ring step into
    fp32 partials, the LSE merge, the unpermutes; backward per step with
    fp32 dK/dV accumulated in global memory) on the same data as the fused
    step: whole-step and forward times and the per-kernel split."""
    sched = "stepwise"
    cu = wl.cu_seqlens()
    T, hq, hkv, d = wl.T, wl.hq, wl.hkv, wl.d
    pairs = pairs_of(cu)
    nb = max(ra.ring_workspace_bytes(T, hq, hkv, d, 0, cu, wl.cp, wl.zz_mode, sched, bwd=b) for b in (False, True))
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    out, lse = torch.empty_like(q), torch.empty((hq, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def fwd():
        ra.ring_attn_fwd(q, k, v, cu, wl.cp, wl.zz_mode, True, wl.scale, sched, out=out, lse=lse, workspace=ws)

    def step():
        fwd()
        ra.ring_attn_bwd(q, k, v, out, lse, do, cu, wl.cp, wl.zz_mode, True, wl.scale, sched, dq=dq, dk=dk, dv=dv,
                         workspace=ws, reuse_fwd_workspace=True)

    stream = torch.cuda.current_stream(dev)
    ms_step = time_calls(step, steps, warmup, stream, torch)
    ms_fwd = time_calls(fwd, steps, warmup, stream, torch)
    L = ra.lib()
    L.ra_profile_enable(1)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    names = ctypes.create_string_buffer(64 * 32)
    kms = (ctypes.c_double * 32)()
    kn = (ctypes.c_int64 * 32)()
    nk = L.ra_profile_read(32, names, kms, kn)
    L.ra_profile_enable(0)
    per = {}
    for i in range(max(nk, 0)):
        nm = names.raw[64 * i:64 * i + 64].split(b"\0")[0].decode()
        per[nm] = {"ms_per_step": kms[i] / steps, "launches_per_step": int(kn[i]) // steps}
    assert ra.device_status() == 0
    del ws, out, lse, dq, dk, dv
    torch.cuda.empty_cache()
    tf = 14 * d * hq * pairs / (ms_step / 1e3) / 1e12
    tff = 4 * d * hq * pairs / (ms_fwd / 1e3) / 1e12
    return {"ms_per_step": ms_step, "tflops": tf, "frac_of_peak": tf / peak,
            "fwd": {"ms": ms_fwd, "tflops": tff, "frac_of_peak": tff / peak}, "kernels_per_step": per}



def masked_lines(ra, torch, dev, wl, steps, warmup, peak, q, k, v, do, specs):
    """Interval masks (per-token key bounds, workloads.interval_bounds) on
    the same data: the fused ring's fwd+bwd step and forward, TFLOP/s over
    the mask's allowed pairs."""
    cu = wl.cu_seqlens()
    T, hq, hkv, d = wl.T, wl.hq, wl.hkv, wl.d
    res = {}
    for spec in specs:
        kind, _, par = spec.partition(":")
        lo, hi = W.interval_bounds(cu, kind, int(par or 0))
        pairs = W.interval_pairs(cu, lo, hi)
        kw = dict(key_lo=lo, key_hi=hi)
        nb = max(ra.ring_workspace_bytes(T, hq, hkv, d, 0, cu, wl.cp, wl.zz_mode, "fused", bwd=b, **kw)
                 for b in (False, True))
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        out, lse = torch.empty_like(q), torch.empty((hq, T), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def fwd():
            ra.ring_attn_fwd(q, k, v, cu, wl.cp, wl.zz_mode, scale=wl.scale, out=out, lse=lse, workspace=ws, **kw)

        def step():
            fwd()
            ra.ring_attn_bwd(q, k, v, out, lse, do, cu, wl.cp, wl.zz_mode, scale=wl.scale, dq=dq, dk=dk, dv=dv,
                             workspace=ws, reuse_fwd_workspace=True, **kw)

        stream = torch.cuda.current_stream(dev)
        ms_step = time_calls(step, steps, warmup, stream, torch)
        ms_fwd = time_calls(fwd, steps, warmup, stream, torch)
        assert ra.device_status() == 0
        tf = 14 * d * hq * pairs / (ms_step / 1e3) / 1e12
        tff = 4 * d * hq * pairs / (ms_fwd / 1e3) / 1e12
        res[spec] = {"allowed_pairs_per_head": pairs, "ms_per_step": ms_step, "tflops": tf, "frac_of_peak": tf / peak,
                     "fwd": {"ms": ms_fwd, "tflops": tff, "frac_of_peak": tff / peak}}
        del ws, out, lse, dq, dk, dv
        torch.cuda.empty_cache()
    return res



def schedule_lines(ra, torch, dev, wl, steps, warmup, peak, q, k, v, do):
    """The same data under the all-gather KV schedule and, on the fused ring,
    with a 1024-token sliding window: fwd+bwd step and forward, TFLOP/s over
    each case's allowed pairs."""
    cu = wl.cu_seqlens()
    T, hq, hkv, d = wl.T, wl.hq, wl.hkv, wl.d
    res = {}
    for name, sched, window in (("allgather", "allgather", -1), ("window:1024", "fused", 1024)):
        pairs = pairs_of(cu, window)
        nb = max(ra.ring_workspace_bytes(T, hq, hkv, d, 0, cu, wl.cp, wl.zz_mode, sched, bwd=b) for b in (False, True))
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        out, lse = torch.empty_like(q), torch.empty((hq, T), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def fwd():
            ra.ring_attn_fwd(q, k, v, cu, wl.cp, wl.zz_mode, True, wl.scale, sched, out=out, lse=lse, workspace=ws,
                             window=window)

        def step():
            fwd()
            ra.ring_attn_bwd(q, k, v, out, lse, do, cu, wl.cp, wl.zz_mode, True, wl.scale, sched, dq=dq, dk=dk,
                             dv=dv, workspace=ws, reuse_fwd_workspace=True, window=window)

        stream = torch.cuda.current_stream(dev)
        ms_step = time_calls(step, steps, warmup, stream, torch)
        ms_fwd = time_calls(fwd, steps, warmup, stream, torch)
        assert ra.device_status() == 0
        tf = 14 * d * hq * pairs / (ms_step / 1e3) / 1e12
        tff = 4 * d * hq * pairs / (ms_fwd / 1e3) / 1e12
        res[name] = {"sched": sched, "window": window, "allowed_pairs_per_head": pairs, "ms_per_step": ms_step,
                     "tflops": tf, "frac_of_peak": tf / peak,
                     "fwd": {"ms": ms_fwd, "tflops": tff, "frac_of_peak": tff / peak}}
        del ws, out, lse, dq, dk, dv
        torch.cuda.empty_cache()
    return res


def host_planning(ra, torch, dev, wl, q, k, v, n=8):
    """Host cost of a ring forward on a packing the library has not seen (as
    in training on a new varlen batch every step): the wall time of the
    workspace size query plus the forward call, which plans (zigzag split,
    tiles, work items, table image) and enqueues its kernels; packings of
    the same total drawn with the same length distribution (seeds 1..n),
    the device synchronised between calls, outside the timed span."""
    T, hq, hkv, d = wl.T, wl.hq, wl.hkv, wl.d
    out = torch.empty_like(q)
    lse = torch.empty((hq, T), dtype=torch.float32, device=dev)
    ms = []
    for seed in range(1, n + 1):
        cu = W.cu_seqlens(W.loguniform_doc_lens(T, 128, 8192, seed))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        nb = ra.ring_workspace_bytes(T, hq, hkv, d, 0, cu, wl.cp, wl.zz_mode, "fused", bwd=False)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        ra.ring_attn_fwd(q, k, v, cu, wl.cp, wl.zz_mode, True, wl.scale, "fused", out=out, lse=lse, workspace=ws)
        ms.append((time.perf_counter() - t0) * 1e3)
        torch.cuda.synchronize()
        del ws
    assert ra.device_status() == 0
    return {"ms_median": float(np.median(ms)), "ms": ms, "packings": n,
            "rule": "size query + forward call on a new packing (planning and kernel enqueue), host wall time"}


def cpu_configs(args):
    """The fp64 oracle on the host cores, per workload: the 128-token fp32
    batch, the forward of the 8192-token sequence and of the packed
    32768-token workload, and the fwd+bwd of the packed workload, in full;
    the 131072-token sequence on a fixed sample of 2048 query rows (every
    chunk boundary row of its zigzag split plus seeded random rows, all 64
    heads; the whole run extrapolated by allowed pairs and labelled so).
    Each on all cores, and on one core on a smaller sample (extrapolated).
    One JSON line per measurement; host only (several minutes)."""
    import oracle
    oracle.build()
    ncores = os.cpu_count() or 1

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    def line(name, threads, sec, flops, sample, full_flops):
        rate = flops / sec / 1e12
        print(json.dumps({"cpu_config": name, "cores": threads, "sec": sec, "tflops": rate, "sample": sample,
                          "full_sec_extrapolated": None if flops == full_flops else sec * full_flops / flops}),
              flush=True)

    oracle.set_threads(ncores)
    wl = W.C0
    cu = wl.cu_seqlens()
    q, k, v = W.make_qkv(wl.T, wl.hq, wl.hkv, wl.d, wl.dtype)
    full = 4 * wl.d * wl.hq * pairs_of(cu)
    line("C0 fwd", ncores, timed(lambda: oracle.attn_fwd(q, k, v, cu, True, wl.scale)), full, "whole workload", full)
    for name in ("C1", "C2"):
        wl = W.ALL[name]
        cu = wl.cu_seqlens()
        q, k, v = W.make_qkv(wl.T, wl.hq, wl.hkv, wl.d, wl.dtype)
        full = 4 * wl.d * wl.hq * pairs_of(cu)
        seg = oracle.doc_ids(cu)
        pos = np.arange(wl.T)

        def row_pairs(rows):
            return int(sum(r - cu[np.searchsorted(cu, r, side="right") - 1] + 1 for r in rows))

        oracle.set_threads(ncores)
        sec = timed(lambda: oracle.attn_fwd(q, k, v, cu, True, wl.scale))
        line(name + " fwd", ncores, sec, full, "whole workload", full)
        # one core: a fixed sample of 64 query rows of all heads
        rows = W.sample_rows(wl.T, 64, 5, list(cu[:-1]))
        oracle.set_threads(1)
        sec1 = timed(lambda: oracle.partial_fwd(q[torch_index(rows)], k, v, seg[rows], seg, rows, pos, True, wl.scale))
        oracle.set_threads(ncores)
        line(name + " fwd", 1, sec1, 4 * wl.d * wl.hq * row_pairs(rows),
             f"{len(rows)} query rows of {wl.T} (all {wl.hq} heads)", full)
    # fwd+bwd of the packed workload: every document on all cores; the
    # smallest documents up to 1M allowed pairs on one core
    wl = W.C4
    full = 14 * wl.d * wl.hq * pairs_of(wl.cu_seqlens())
    tf, sec, cores, sample, sp = run_cpu_oracle(wl, steps=1, pair_budget=pairs_of(wl.cu_seqlens()))
    line("C4 fwd+bwd", cores, sec, 14 * wl.d * wl.hq * sp, sample, full)
    tf, sec, _, sample, sp = run_cpu_oracle(wl, steps=1, pair_budget=1_000_000, threads=1)
    line("C4 fwd+bwd", 1, sec, 14 * wl.d * wl.hq * sp, sample, full)
    wl = W.C3
    cu = wl.cu_seqlens()
    q, k, v = W.make_qkv(wl.T, wl.hq, wl.hkv, wl.d, wl.dtype)
    n = 2 * wl.cp
    bounds = [c * wl.T // n for c in range(1, n)]
    rows = W.sample_rows(wl.T, 2048, 6, bounds + [b - 1 for b in bounds] + [0, wl.T - 1])
    seg = oracle.doc_ids(cu)
    pos = np.arange(wl.T)
    full = 4 * wl.d * wl.hq * pairs_of(cu)
    for threads, rr in ((ncores, rows), (1, rows[::128])):
        oracle.set_threads(threads)
        rp = int((rr + 1).sum())
        sec = timed(lambda: oracle.partial_fwd(q[torch_index(rr)], k, v, seg[rr], seg, rr, pos, True, wl.scale))
        line("C3 fwd", threads, sec, 4 * wl.d * wl.hq * rp,
             f"{len(rr)} query rows of {wl.T} (zigzag chunk boundaries and seeded rows, all {wl.hq} heads)", full)
    oracle.set_threads(ncores)


def torch_index(rows):
    import torch
    return torch.from_numpy(np.asarray(rows, dtype=np.int64))



def fwd_configs(args, ra, torch):
    """Forward-only TFLOP/s of the named workloads on one GPU (CUDA events on
    the launching stream, W warm-up calls, K timed calls; every input is far
    above L2 except C1's K/V)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak_burst, peak_sust, _, peak_src = peaks()
    for name in [x.strip() for x in args.fwd_configs.split(",") if x.strip()]:
        wl = W.ALL[name]
        cu = wl.cu_seqlens()
        T, hq, hkv, d = wl.T, wl.hq, wl.hkv, wl.d
        pairs = pairs_of(cu, args.window)
        flops = 4 * d * hq * pairs
        q, k, v = (x.to(dev) for x in W.make_qkv(T, hq, hkv, d, wl.dtype))
        out = torch.empty_like(q)
        lse = torch.empty((hq, T), dtype=torch.float32, device=dev)
        ws = torch.empty(ra.ring_workspace_bytes(T, hq, hkv, d, 0 if wl.dtype == torch.bfloat16 else 1, cu, wl.cp,
                                                 wl.zz_mode, args.sched, bwd=False), dtype=torch.uint8, device=dev)
        f = lambda: ra.ring_attn_fwd(q, k, v, cu, wl.cp, wl.zz_mode, True, wl.scale, args.sched, out=out, lse=lse,
                                     workspace=ws, window=args.window)
        for _ in range(max(args.warmup, 3)):
            f()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(args.steps):
            f()
        e1.record(st)
        torch.cuda.synchronize()
        assert ra.device_status() == 0
        ms = e0.elapsed_time(e1) / args.steps
        tf = flops / (ms / 1e3) / 1e12
        print(json.dumps({"fwd_config": wl.name, "T": T, "Hq": hq, "Hkv": hkv, "d": d, "cp": wl.cp,
                          "window": args.window, "sched": args.sched,
                          "allowed_pairs_per_head": pairs, "ms": ms, "tflops": tf,
                          "frac_of_peak": tf / peak_burst, "peak_tflops": peak_burst, "peak_source": peak_src,
                          "steps": args.steps, "warmup": args.warmup}), flush=True)
        del q, k, v, out, lse, ws
        torch.cuda.empty_cache()


def balance_study(args):
    """Per-rank causal load of CP sharding policies on synthetic packings
    (the packing/balance question of "Question about varlen ring attention",
    MiniMax-01 #6): allowed (query, key) pairs each simulated rank computes
    over the whole ring, for per-document zigzag, whole-stream zigzag and
    plain contiguous sharding, with documents in drawn order or sorted by
    length.  The ring's step time follows the busiest rank, so the figure
    of merit is max / mean.  Host only (the library's ra_ring_rank_pairs;
    contiguous sharding is counted here)."""
    import context_varlen_ring_gb300 as ra
    cp = 8

    def contiguous(cu, window):
        T = int(cu[-1])
        counts = np.zeros(cp, dtype=np.int64)
        for b in range(len(cu) - 1):
            i = np.arange(cu[b], cu[b + 1], dtype=np.int64)
            keys = i - cu[b] + 1 if window < 0 else np.minimum(i - cu[b] + 1, window + 1)
            owner = np.minimum(i * cp // T, cp - 1)
            np.add.at(counts, owner, keys)
        return counts

    for seed in range(6):
        lens = W.loguniform_doc_lens(32768, 128, 8192, seed)
        for order in ("drawn", "sorted"):
            ll = sorted(lens, reverse=True) if order == "sorted" else lens
            cu = W.cu_seqlens(ll)
            for window in (-1, 1024):
                res = {}
                for name, f in (("per_doc_zigzag", lambda c, w: ra.ring_rank_pairs(c, cp, W.ZZ_PER_DOC, True, w)),
                                ("stream_zigzag", lambda c, w: ra.ring_rank_pairs(c, cp, W.ZZ_GLOBAL, True, w)),
                                ("contiguous", contiguous)):
                    c = np.asarray(f(cu, window), dtype=np.float64)
                    res[name] = round(float(c.max() / c.mean()), 4)
                print(json.dumps({"balance": "max/mean per-rank allowed pairs", "cp": cp, "T": 32768,
                                  "docs_seed": seed, "doc_order": order, "n_docs": len(ll), "window": window,
                                  **res}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sched", default="fused", choices=["fused", "stepwise", "allgather"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--probe", action="store_true",
                    help="only W+K plain steps (for profilers): no e2e, per-kernel or CPU passes")
    ap.add_argument("--balance", action="store_true",
                    help="host-only study of per-rank causal load under CP sharding policies (JSON lines)")
    ap.add_argument("--window", type=int, default=-1,
                    help="sliding window (a key at most this many positions behind its query); -1: none")
    ap.add_argument("--cpu-configs", action="store_true",
                    help="host only: the fp64 oracle's time per workload on all cores and on one core (JSON lines)")
    ap.add_argument("--bandwidth", action="store_true",
                    help="only the HBM-bound kernels at full size (permute, unpermute, LSE merge): one JSON line")
    ap.add_argument("--merge-parts", type=int, default=0,
                    help="partials merged by --bandwidth (default: the workload's CP size)")
    ap.add_argument("--traffic-from", default="", metavar="CSV",
                    help="write profiles/traffic.json from an ncu launch list of one fwd+bwd step (CSV) and "
                         "exit (host only)")
    ap.add_argument("--fwd-configs", default="",
                    help="comma list of forward-only workloads (e.g. C1,C2,C3) to time instead of the "
                         "fwd+bwd step; one JSON line each (not the headline line)")
    args = ap.parse_args()
    if args.traffic_from:
        tab = traffic_table(args.traffic_from)
        with open(os.path.join(ROOT, "profiles", "traffic.json"), "w") as f:
            json.dump(tab, f, indent=1)
        print(json.dumps({k: v["dram_bytes_per_launch"] for k, v in tab.items()}))
        return
    if args.balance:
        balance_study(args)
        return
    if args.cpu_configs:
        cpu_configs(args)
        return
    if args.impl == "reference":
        reference_arm(args)
        return

    import torch
    import torch.distributed as dist

    import context_varlen_ring_gb300 as ra

    if args.fwd_configs:
        fwd_configs(args, ra, torch)
        return
    if args.bandwidth:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        res = bandwidth_kernels(ra, torch, dev, W.C2, args.steps, args.warmup, peaks()[2],
                                merge_parts=args.merge_parts or None)
        print(json.dumps({"bandwidth_kernels": res, "workload": W.C2.name, "steps": args.steps,
                          "warmup": args.warmup}), flush=True)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    wl = W.C4
    cu = wl.cu_seqlens()
    T, hq, hkv, d = wl.T, wl.hq, wl.hkv, wl.d
    pairs = pairs_of(cu, args.window)
    win = dict(window=args.window)
    fwd_flops = 4 * d * hq * pairs
    bwd_flops = 10 * d * hq * pairs
    step_flops = fwd_flops + bwd_flops

    q, k, v = (x.to(dev) for x in W.make_qkv(T, hq, hkv, d, wl.dtype))
    do = W.make_dout(T, hq, d, wl.dtype).to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((hq, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = max(ra.ring_workspace_bytes(T, hq, hkv, d, 0, cu, wl.cp, wl.zz_mode, args.sched, bwd=False),
                 ra.ring_workspace_bytes(T, hq, hkv, d, 0, cu, wl.cp, wl.zz_mode, args.sched, bwd=True))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def step():
        ra.ring_attn_fwd(q, k, v, cu, wl.cp, wl.zz_mode, True, wl.scale, args.sched, out=out, lse=lse, workspace=ws,
                         **win)
        ra.ring_attn_bwd(q, k, v, out, lse, do, cu, wl.cp, wl.zz_mode, True, wl.scale, args.sched, dq=dq, dk=dk, **win,
                         dv=dv, workspace=ws, reuse_fwd_workspace=True)

    def fwd_only():
        ra.ring_attn_fwd(q, k, v, cu, wl.cp, wl.zz_mode, True, wl.scale, args.sched, out=out, lse=lse, workspace=ws,
                         **win)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        step()
    barrier()
    assert ra.device_status() == 0
    if args.probe:
        for _ in range(args.steps):
            step()
        barrier()
        assert ra.device_status() == 0
        if rank == 0:
            print(json.dumps({"probe": wl.name, "steps": args.steps, "warmup": args.warmup}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- timed region: K steps, device events on the launching stream
    clocks = Clocks(local)
    clocks.start()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_per_step = ms / args.steps
    value = job_tflops(world, step_flops, args.steps, ms)

    # ---- forward alone (same data), for the forward half of the metric
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        fwd_only()
    f1.record(stream)
    barrier()
    fwd_ms = f0.elapsed_time(f1) / args.steps
    fwd_tflops = fwd_flops / (fwd_ms / 1e3) / 1e12

    # ---- per-kernel times over the same K steps (events around each launch)
    L = ra.lib()
    L.ra_profile_enable(1)
    for _ in range(args.steps):
        step()
    barrier()
    names = ctypes.create_string_buffer(64 * 32)
    kms = (ctypes.c_double * 32)()
    kn = (ctypes.c_int64 * 32)()
    nk = L.ra_profile_read(32, names, kms, kn)
    L.ra_profile_enable(0)
    kernels = {}
    for i in range(max(nk, 0)):
        nm = names.raw[64 * i:64 * i + 64].split(b"\0")[0].decode()
        kernels[nm] = {"ms_total": kms[i], "launches": int(kn[i]), "ms_per_launch": kms[i] / max(kn[i], 1)}
    total_kernel_ms = sum(x["ms_total"] for x in kernels.values()) or 1.0
    for x in kernels.values():
        x["share"] = x["ms_total"] / total_kernel_ms
    # every scope is one launch of the library's kernels (the table upload is
    # a kernel reading the page-locked table copy), except the fused
    # backward's, which covers its two concurrent kernels
    gpu_launches = sum(x["launches"] * KERNELS_PER_SCOPE.get(nm, 1) for nm, x in kernels.items())
    peak_burst, peak_sust, hbm, peak_src = peaks()
    dominant = max(kernels, key=lambda n: kernels[n]["ms_total"]) if kernels else None
    roof = None
    if dominant:
        roof = tensor_roofline(dominant, kernels[dominant]["ms_per_launch"], d, hq, pairs, peak_burst, peak_src)
    all_roof = {}
    for nm, x in kernels.items():
        if nm in ALGORITHMIC_PRODUCTS:
            r = tensor_roofline(nm, x["ms_per_launch"], d, hq, pairs, peak_burst, peak_src)
            all_roof[nm] = {k_: r[k_] for k_ in ("achieved", "frac", "executed_tflops", "executed_frac")}

    extras = {}
    if not args.probe and args.sched == "fused" and args.window < 0:
        # the other forward workloads, the per-step schedule on the same data,
        # and the bandwidth-bound kernels at full size
        extras["fwd_configs"] = fwd_lines(ra, torch, dev, ["C1", "C3"], args.steps, args.warmup, peak_burst)
        extras["stepwise"] = stepwise_lines(ra, torch, dev, wl, args.steps, args.warmup, peak_burst, q, k, v, do)
        extras["bandwidth_kernels"] = bandwidth_kernels(ra, torch, dev, wl, args.steps, args.warmup, hbm)
        extras["interval_masks"] = masked_lines(ra, torch, dev, wl, args.steps, args.warmup, peak_burst, q, k, v, do,
                                                ["prefix:512", "chunked:1024"])
        extras["other_schedules"] = schedule_lines(ra, torch, dev, wl, args.steps, args.warmup, peak_burst,
                                                   q, k, v, do)
        extras["host_planning"] = host_planning(ra, torch, dev, wl, q, k, v)
        barrier()

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs (Q, K, V, dO) in from pinned host memory and its
    # results (O, dQ, dK, dV) back out.  As in a training loop that
    # prefetches, step i runs [copy in step i+1's inputs | compute step i |
    # copy out step i-1's results] on three streams, with device inputs and
    # results double-buffered; each such step is one CUDA graph of the
    # library's public calls (captured once per buffer parity, replayed), so
    # the host issues one launch per step.  The timed region holds every copy
    # of every step: step 0's inputs before the loop, the last step's results
    # after it (the loop also copies one spare input set and one stale
    # result set).
    hq_, hk_, hv_, hd_ = (x.cpu().pin_memory() for x in (q, k, v, do))
    host_out = [[torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (out, dq, dk, dv)] for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in (hq_, hk_, hv_, hd_))
    d2h = sum(x.numel() * x.element_size() for x in host_out[0])
    dev_in = [[torch.empty_like(x) for x in (q, k, v, do)] for _ in range(2)]
    dev_out = [[torch.empty_like(x) for x in (q, dq, k, v)] + [torch.empty_like(lse)] for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def copy_in(b):
        with torch.cuda.stream(s_in):
            for dst, src in zip(dev_in[b], (hq_, hk_, hv_, hd_)):
                dst.copy_(src, non_blocking=True)

    def copy_out(b):
        with torch.cuda.stream(s_out):
            for dst, src in zip(host_out[b], dev_out[b][:4]):
                dst.copy_(src, non_blocking=True)

    def pipelined_step(b, copies=True, compute=True):
        cur = torch.cuda.current_stream()
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        if copies:
            copy_in(1 - b)
            copy_out(1 - b)
        if compute:
            q_, k_, v_, do_ = dev_in[b]
            o_, dq_, dk_, dv_, l_ = dev_out[b]
            ra.ring_attn_fwd(q_, k_, v_, cu, wl.cp, wl.zz_mode, True, wl.scale, args.sched, out=o_, lse=l_, **win,
                             workspace=ws)
            ra.ring_attn_bwd(q_, k_, v_, o_, l_, do_, cu, wl.cp, wl.zz_mode, True, wl.scale, args.sched, dq=dq_,
                             **win, dk=dk_, dv=dv_, workspace=ws, reuse_fwd_workspace=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    for b in (0, 1):  # eager once: plans, page-locked tables, the library's second stream
        copy_in(b)
        stream.wait_stream(s_in)
        pipelined_step(b)
    torch.cuda.synchronize()
    graphs = []
    for b in (0, 1):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            pipelined_step(b)
        graphs.append(g)
    # warm-up replays: a graph's first launch carries a one-off upload cost
    # (tens of ms here, varying from run to run) that is not a step's
    for i in range(2 * max(args.warmup, 1)):
        graphs[i % 2].replay()
    torch.cuda.synchronize()
    barrier()
    # The K-step loop is timed E2E_REPS times and the median reported (every
    # repetition is listed): on this platform host<->device copies stall for
    # 40-100 ms about every half second, whichever way the host waits, so a
    # single window of ~50 ms catches one in about a quarter of runs.
    reps_ms = []
    for _ in range(E2E_REPS):
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        s_in.wait_stream(stream)
        copy_in(0)
        stream.wait_stream(s_in)
        for i in range(args.steps):
            graphs[i % 2].replay()
        s_out.wait_stream(stream)
        copy_out((args.steps - 1) % 2)
        stream.wait_stream(s_out)
        g1.record(stream)
        barrier()
        reps_ms.append(max_over_ranks(g0.elapsed_time(g1), world, dev))
    e2e_ms = sorted(reps_ms)[len(reps_ms) // 2]
    # the pipelined results equal the device-resident run's (bit for bit)
    last = host_out[(args.steps - 1) % 2]
    e2e_match = all(torch.equal(h, x.cpu()) for h, x in zip(last, (out, dq, dk, dv)))
    e2e_value = job_tflops(world, step_flops, args.steps, e2e_ms)
    assert ra.device_status() == 0
    # the same step graph with only its copies and with only its compute, on
    # the same buffers (after the timed region): the pipelined step should
    # take about the longer of the two
    parts = {}
    for name, kw in (("copies_only", {"compute": False}), ("compute_only", {"copies": False})):
        gs = []
        for b in (0, 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                pipelined_step(b, **kw)
            gs.append(g)
        for i in range(2):
            gs[i].replay()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(args.steps):
            gs[i % 2].replay()
        c1.record(stream)
        torch.cuda.synchronize()
        parts[name] = c0.elapsed_time(c1) / args.steps
        del gs
    assert ra.device_status() == 0
    e2e_numa = _numa_node_of(hq_.data_ptr())
    copy_rates = host_copy_rates(torch, dev, (q, k, v, do), (out, dq, dk, dv), stream)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu:
        tf, sec, cores, sample, sp = run_cpu_oracle(wl, steps=1, window=args.window)
        tf1, sec1, _, sample1, sp1 = run_cpu_oracle(wl, steps=1, window=args.window, pair_budget=1_000_000,
                                                     threads=1)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample,
               "sec_per_sample": sec,
               "full_workload_s_extrapolated": sec * pairs / sp,
               "extrapolation": "sample seconds x (allowed pairs of the whole workload / of the sample); labelled "
                                "extrapolated, not run",
               "one_core": {"value": tf1, "unit": "TFLOP/s", "cores": 1, "sample": sample1, "sec_per_sample": sec1,
                            "full_workload_s_extrapolated": sec1 * pairs / sp1}}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name + (f", sliding window {args.window}" if args.window >= 0 else "")
                               + (", all-gather KV schedule" if args.sched == "allgather" else ""),
                   "window": args.window, "T": T, "docs": list(wl.doc_lens), "Hq": hq, "Hkv": hkv, "d": d,
                   "cp": wl.cp, "zigzag": "per-doc", "sched": args.sched, "causal_pairs_per_head": pairs,
                   "l2": "no flush: each step streams ~2.6 GB (Q, dO, O 268 MB each, fp32 dQ 537 MB, permuted "
                         "copies), far above the 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "bwd_reserve": "the backward reuses the forward's tile tables and rank-ordered copies (the rows "
                                  "of tiles that straddle two zigzag chunks; the kernels read every other tile in "
                                  "place) from the shared workspace; every step permutes once"},
        "fwd": {"tflops": fwd_tflops, "ms": fwd_ms, "frac_of_peak": fwd_tflops / peak_burst},
        "fwd_bwd_frac_of_peak": value / world / peak_burst,
        "peak_tflops": {"burst": peak_burst, "sustained": peak_sust, "source": peak_src},
        "roofline": roof,
        "kernel_rooflines": all_roof,
        "kernels": kernels,
        "gpu_launches": gpu_launches,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps,
                "overlap": "step i+1's input copies and step i-1's result copies run on two copy streams beside "
                           "step i's compute (double-buffered device inputs and results); each step is one CUDA "
                           "graph of the public calls; every step's copies are inside the timed region",
                "results_match_device_run": e2e_match,
                "timing": f"median of {E2E_REPS} timed repetitions of the {args.steps}-step loop, each holding "
                          f"every copy of its steps",
                "reps_ms_per_step": [x / args.steps for x in reps_ms],
                "step_graph_parts_ms": parts,
                "pinned_numa_node": e2e_numa,
                "host_copies": copy_rates},
        "cpu_baseline": cpu,
        "clocks": clk,
        **extras,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
