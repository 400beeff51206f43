"""The multi-rank path of bench.py on CPU: gloo process groups of two ranks.

On a GPU node bench.py runs one independent replica per GPU (no data exchange); the job's
time is the slowest rank's and its throughput the sum over ranks.  These tests exercise that
host logic, and the reference arm's rank handling, without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        rate = bench.whole_job_rate(world, 1_000_000_000, slowest)
        out.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(2))
    # both ranks see the slower rank's 15 ms; two ranks x 1 GB in 15 ms = 133.3 GB/s
    for rank, slowest, rate in got:
        assert slowest == 15.0
        assert rate == pytest.approx(2 * 1.0 / 0.015)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_rate(1, 576_000, 1.0) == pytest.approx(0.576)


def test_reference_arm_under_torchrun_prints_once():
    """Under torchrun with two CPU ranks the oracle arm runs on rank 0 only: one JSON line,
    every rank exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "1",
           "--warmup", "0"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_algorithmic_bytes_count_distinct_rows_under_a_shared_prefix():
    import mla_inputs
    case = mla_inputs.make_custom([300, 410, 257, 1200], q_lens=[1, 2, 1, 3], H=12,
                                  shared_prefix=256, seed=3)
    used = case.kv_indices[:case.total_kv]
    distinct = int(used.unique().numel())
    rows = sum(case.q_lens) * case.H
    rest = rows * (576 + 1024 + 4)
    assert mla_inputs.algorithmic_bytes(case) == 580 * case.total_kv + rest
    assert mla_inputs.algorithmic_bytes(case, 256) == 580 * distinct + rest


def test_roofline_names_the_binding_and_carries_the_tensor_view():
    """bench.roofline_for: the HBM roofline of the scope table (580 B per attended position),
    what binds the call, and the algorithmic FP8 work against the FP8 peak (2 x (576 + 512)
    flops per attended row and position, drafts counted causally)."""
    sys.path.insert(0, ROOT)
    import bench
    import mla_inputs
    case = mla_inputs.make_custom([300, 410], q_lens=[1, 3], H=12, seed=4)
    ms, peak = 0.05, 6785.2
    r = bench.roofline_for(case, "plain", ms, peak, "measured", "c16", 0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["frac"] == pytest.approx(mla_inputs.algorithmic_bytes(case) / (ms * 1e-3) / 1e9 / peak)
    assert r["binds"] and "16-row kernel" in r["binds"]
    t = r["tensor_roofline"]
    attended = 300 + (408 + 409 + 410)            # q_len 3 over kv_len 410: causal counts
    assert t["algorithmic_flops"] == 2 * (576 + 512) * 12 * attended
    assert t["bound"] == "tensor" and t["unit"] == "TFLOP/s"
    assert t["peak"] > 0 and t["frac"] == pytest.approx(t["achieved"] / t["peak"])
    r2 = bench.roofline_for(case, "shared_prefix", ms, peak, "measured", "c16", 0)
    assert "96-row kernel" in r2["binds"]
