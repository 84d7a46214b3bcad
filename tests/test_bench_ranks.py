"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each with its own
timing, agree on the slowest rank's time and report whole-job throughput of
the replicas (every rank runs the full workload)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 100.0 + 25.0 * rank          # rank 1 is the slow one
        m = bench.max_over_ranks(ms, world, torch.device("cpu"))
        out[rank] = m
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1] == 125.0


def test_single_rank_passthrough():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5


def test_job_tflops_is_whole_job():
    # 2 replicas x 10 steps x 1e12 FLOP in 1 s (slowest rank) = 20 TFLOP/s
    assert bench.job_tflops(2, 1e12, 10, 1000.0) == pytest.approx(20.0)
    assert bench.job_tflops(1, 1e12, 10, 1000.0) == pytest.approx(10.0)


def test_balance_study_lines():
    """bench.py --balance (host only): one JSON line per packing, order and
    window; on the packed 32768-token workload per-document zigzag keeps
    every rank within 0.2 % of the mean causal load, and without zigzag the
    busiest rank carries far more."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.abspath(bench.__file__))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--balance"], capture_output=True,
                         text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr
    lines = [json.loads(x) for x in out.stdout.strip().splitlines()]
    assert len(lines) == 6 * 2 * 2
    c2 = [x for x in lines if x["docs_seed"] == 0 and x["doc_order"] == "drawn" and x["window"] == -1][0]
    assert c2["per_doc_zigzag"] < 1.002
    assert c2["contiguous"] > 1.5 and c2["stream_zigzag"] > 1.5


def test_reference_arm_line(monkeypatch, capsys):
    """bench.py --impl reference (host only): times the fp64 oracle on a
    sample of the packed workload and prints one JSON line with the keys the
    harness reads; here the sample is cut to the smallest document so the
    test stays short."""
    import argparse
    import json
    monkeypatch.setattr(bench, "cpu_sample_docs", lambda lens, *a: [min(range(len(lens)), key=lambda i: lens[i])])
    monkeypatch.delenv("RANK", raising=False)
    bench.reference_arm(argparse.Namespace(gpus=1, steps=1, warmup=3))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["metric"] == bench.METRIC and line["value"] > 0 and line["ms_per_step"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert "1 of the 15 documents" in line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["dtype"] == "f64" and line["data"] == "synthetic"


def test_reference_arm_other_ranks_print_nothing(monkeypatch, capsys):
    import argparse
    monkeypatch.setenv("RANK", "1")
    bench.reference_arm(argparse.Namespace(gpus=2, steps=1, warmup=3))
    assert capsys.readouterr().out == ""


def test_flop_count_matches_oracle_pairs(orc):
    """The allowed-pair count behind every reported TFLOP/s equals the
    oracle's per-rank counts summed over ranks (any CP size, both zigzag
    modes, with and without a window), and gives the per-launch FLOPs the
    roofline uses on the packed 32768-token workload."""
    import numpy as np

    import workloads as W
    rng = np.random.default_rng(17)
    for _ in range(6):
        cu = W.cu_seqlens(W.random_doc_lens(rng, int(rng.integers(100, 4000)), 1, 1500))
        for w in (-1, 0, 1, 33, 700, 10**6):
            ref = int(orc.rank_pairs(cu, int(rng.integers(1, 9)), int(rng.integers(0, 2)), True, window=w).sum())
            assert bench.pairs_of(cu, w) == ref
    cu = W.C4.cu_seqlens()
    assert bench.pairs_of(cu) == 67823768
    d, hq = 128, 32
    # the method's work: 4*d*Hq per pair forward, 10*d*Hq backward
    assert 2 * d * hq * bench.ALGORITHMIC_PRODUCTS["ra_tc_fwd"] * 67823768 == pytest.approx(1.111e12, rel=1e-3)
    assert 2 * d * hq * bench.ALGORITHMIC_PRODUCTS["ra_tc_bwd"] * 67823768 == pytest.approx(2.778e12, rel=1e-3)
    # the two backward passes form S and dP twice: 7 products executed
    ex = bench.EXECUTED_PRODUCTS
    assert ex["ra_tc_bwd"] == ex["ra_tc_bwd_dkdv"] + ex["ra_tc_bwd_dq"] == 7
    r = bench.tensor_roofline("ra_tc_bwd", 3.0, d, hq, 67823768, 1902.4, "measured")
    assert r["frac"] == pytest.approx(2.778e12 / 3.0e-3 / 1e12 / 1902.4, rel=1e-3)
    assert r["executed_frac"] == pytest.approx(r["frac"] * 7 / 5)


def test_traffic_table_from_a_launch_list():
    """bench.py --traffic-from: per timing scope, the DRAM read + write bytes
    of its kernels' launches in an ncu CSV launch list (the backward pair
    sums both kernels), with the sha256 of each source file the scope
    depends on, which kernel_traffic checks before reporting the bytes."""
    import hashlib
    hdr = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"'
    kern = {"copy_from_host_kernel(const uint4 *, uint4 *, long, const uint8_t *, uint8_t *, int)": (1, 0),
            "void ra::permute_kernel<uint4>(ra::PermJobs, const int *, long, int, int *)": (70, 20),
            "void ra::(anonymous namespace)::tc_fwd_kernel<0>(ra::(anonymous namespace)::FwdParams)": (400, 200),
            "void ra::permute_rowdot_kernel(ra::PermJobs, const void *, void *, const void *, float *)": (500, 30),
            "void unnamed>::tc_dq_kernel<0>(unnamed>::DqParams)": (700, 250),
            "void unnamed>::tc_dkdv_kernel<0>(unnamed>::BwdParams)": (800, 120)}
    lines = ["==PROF== Connected to process 1", hdr]
    for i, (name, (rd, wr)) in enumerate(kern.items()):
        lines.append(f'"{i}","{name}","dram__bytes_read.sum","byte","{rd * 1_000_000:,}"')
        lines.append(f'"{i}","{name}","dram__bytes_write.sum","byte","{wr * 1_000_000}"')
        lines.append(f'"{i}","{name}","gpu__time_duration.sum","us","12.5"')
    tab = bench.traffic_table(lines)
    mb = {k: v["dram_bytes_per_launch"] // 1_000_000 for k, v in tab.items()}
    assert mb == {"ra_tc_fwd": 600, "ra_tc_bwd": 950 + 920, "ra_tc_bwd_dkdv": 920, "ra_tc_bwd_dq": 950,
                  "ra_permute_fwd": 90, "ra_permute_rowdot": 530}
    csrc = os.path.join(bench.ROOT, "context_varlen_ring_gb300", "csrc")
    for ent in tab.values():
        for f, h in ent["sources"].items():
            assert h == hashlib.sha256(open(os.path.join(csrc, f), "rb").read()).hexdigest()
    # a kernel missing from the list is an error, not a silent zero
    with pytest.raises(ValueError):
        bench.traffic_table([ln for ln in lines if "tc_dq_kernel" not in ln])
