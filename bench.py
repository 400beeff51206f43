"""Benchmark of paged latent-MLA decode on GB300.

One step = one mla_decode call (split-KV scheduler + tcgen05 decode + LSE merge) over
one synthetic decode batch whose inputs are resident in HBM.  L2 is flushed (a 512 MB
write) before every step, outside the timed region.  Metric: effective KV-cache GB/s
(576 bytes per attended position / time) and microseconds per call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c16] [--impl reference]

--impl reference times the FP64 CPU oracle on a bounded sample of the same workload
(the reference arm); under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import glob
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

import mla_inputs

METRIC = "MLA decode effective KV-cache GB/s (% of GB300 HBM peak) and µs per decode call"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
WORKLOAD_TEXT = {
    "tiny": "tiny decode: batch 2, 12 heads, q_len 1, kv_lens {256, 300}, 1,024-row fp8 pool",
    "c16": "concurrency-16 decode: batch 16, 12 heads, q_len 1, 63,911 shared-prefix + 4,089 "
           "unique + U[0,350) positions per request (~68.2K), 5,283,840-row fp8 pool",
    "c24": "concurrency-24 decode: batch 24, otherwise as c16",
    "long": "long single request: batch 1, 12 heads, kv_len 142,000, 2^18-row fp8 pool",
    "long96": "long single request, 96 heads (context-shard reference shape), kv_len 142,000",
    "mtp": "multi-token verification: batch 64, 12 heads, q_len 4 causal, kv_len "
           "log-uniform [2,048, 65,536], 2^22-row fp8 pool",
    "c16p128": "concurrency-16 decode on 128-token pages: c16's lengths, the shared "
               "prefix's 499 whole pages shared, 41,280-page fp8 pool",
    "longp128": "long single request on 128-token pages: kv_len 142,000 (1,110 pages), "
                "2,048-page fp8 pool",
}


SOAK_S = 1.0   # shortest span of steps the clock record covers


# Sources of other operations, which the decode call never runs: left out of the hash
# that keys the decode kernels' recorded counters.
NOT_DECODE_SOURCES = {"mla_vproj.cu", "mla_selftest.cu", "mla_rope_cache.cu", "mla_noalloc.cu",
                      "mla_prefix_expand.cu"}

# What binds each call, from its ncu capture (profiles/): the roofline's denominator is the
# HBM copy peak, but not every call is HBM-bound.
LIMITER = {
    "c16+shared_prefix": "the 96-row tile pipeline: 34 MMAs per 64-position tile (~0.9-1 us "
                         "of tensor pipe, each bound by the shared-memory bytes it reads) "
                         "issued from a QK and a PV warp, the period (~1.2 us) set by the single "
                         "S buffer's hand-off; the 12-row own units pay a full tile's MMAs; the "
                         "epilogue of 96-row fp32 partials (~6.4 us) and the cascade merge; "
                         "DRAM ~25 % busy (profiles/mla_decode_c16.md)",
    "c24+shared_prefix": "as c16+shared_prefix",
    "c16": "the 16-row tile pipeline while every request gathers the shared prefix (L2 "
           "serves it after the first reads): ~1.44 us per 128-position tile, the row "
           "copies' issue (~0.86 us a tile) and the ring's round trip",
    "c24": "as c16",
    "long": "fixed per-call latencies (launch, first rows ~4 us after launch, epilogue, "
            "the slowest CTA, merge) around 8 tiles per CTA streamed at ~4.7 TB/s "
            "(profiles/mla_decode_long.md)",
    "mtp": "one ring stage's round trip (row copies, QK, softmax, PV) at three stages in "
           "flight; DRAM 65 % busy (profiles/mla_decode_mtp.md)",
    "long96": "the 96-row tile pipeline (one pass over the cache for all 96 heads): 34 MMAs "
              "per 64-position tile from a QK and a PV warp, ~15 tiles per CTA; the epilogue "
              "of 96-row fp32 partials (~6.4 us) and the merge (profiles/mla_decode_long96.md)",
}


def kernel_source_hash() -> str:
    """Hash of the sources the decode call (decode and merge kernels, host side) is built
    from: recorded DRAM counters apply only while it is unchanged."""
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "paged_mla_latent_gb300", "csrc", "*"))):
        if os.path.basename(p) in NOT_DECODE_SOURCES:
            continue
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(config: str, entry: str):
    """dram bytes per decode launch from a committed ncu summary, if it matches this kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(config if entry == "plain" else f"{config}+{entry}")
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_call")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while the GPU runs the steps."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x (the job is as slow as its slowest rank)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, bytes_per_rank: int, ms: float) -> float:
    """GB/s of the whole job: every rank processes its own batch of bytes_per_rank in ms."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return world, rank, local, dist
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local, None


def oracle_sample(case, n_requests: int, n_heads: int):
    """Host copies of a bounded sample: the first n_requests requests, n_heads heads each."""
    reqs = list(range(min(n_requests, case.B)))
    rows, idx, kvp, qop, q = [], [], [0], [0], []
    off = 0
    for b in reqs:
        s, e = int(case.kv_indptr[b]), int(case.kv_indptr[b + 1])
        ps = int(case.meta.get("page_size", 1))
        ids = case.kv_indices[s:e].long()
        if ps > 1:   # token rows of the request's pages, in position order
            ids = (ids[:, None] * ps + torch.arange(ps, device=ids.device)[None, :]).reshape(-1)
            ids = ids[:case.kv_lens[b]]
        r = case.kv.reshape(-1, 576).index_select(0, ids).cpu().numpy()
        rows.append(r)
        idx.append(np.arange(off, off + r.shape[0], dtype=np.int32))
        off += r.shape[0]
        kvp.append(off)
        t0, t1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        q.append(case.q[t0:t1, :n_heads].cpu().numpy())
        qop.append(qop[-1] + (t1 - t0))
    return (np.concatenate(q), np.concatenate(rows), np.array(qop, np.int32),
            np.array(kvp, np.int32), np.concatenate(idx), off)


def time_oracle(case, n_requests, n_heads):
    import oracle
    q, kv, qop, kvp, idx, positions = oracle_sample(case, n_requests, n_heads)
    sm, qs, ks = case.scales()
    t0 = time.perf_counter()
    oracle.decode(q, kv, qop, kvp, idx, sm, qs, ks)
    dt = time.perf_counter() - t0
    # bytes of cache the oracle consumed, scaled to the GPU call's head count
    sample_bytes = 576 * positions * n_heads / case.H
    return dt, sample_bytes, oracle.max_threads(), positions


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return os.uname().machine


def run_reference(args, world, rank):
    """Reference arm: the FP64 CPU oracle, bounded sample per step, on the host cores."""
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = mla_inputs.make_case(args.config, seed=args.seed, device=dev)
    n_req, n_heads = args.ref_requests, args.ref_heads
    for _ in range(args.warmup):
        time_oracle(case, n_req, n_heads)
    times, sb = [], 0.0
    cores = 1
    for _ in range(args.steps):
        dt, sb, cores, pos = time_oracle(case, n_req, n_heads)
        times.append(dt)
    mean = sum(times) / len(times)
    value = sb / mean / 1e9
    sample = (f"first {n_req} request(s) x {n_heads} of {case.H} heads of the {args.config} "
              f"workload per step ({pos} positions); GB/s scaled to all {case.H} heads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config, "seed": args.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_graph(call, steps, warmup, flush, no_flush, stream, dev, eager, salt=0):
    """Mean device time (ms) of `call` per step: W warm-up steps, then the call captured in a
    CUDA graph and replayed K times, each step bracketed by CUDA events on the launching
    stream, with an L2 flush (512 MB write) before every step outside the events."""
    for i in range(warmup):
        if not no_flush:
            flush.fill_((i + salt) & 0xFF)
        call()
    torch.cuda.synchronize(dev)
    graph = None
    if not eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        torch.cuda.synchronize(dev)
        for i in range(2):
            if not no_flush:
                flush.fill_((i + salt) & 0xFF)
            graph.replay()
        torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        if not no_flush:
            flush.fill_((i + 7 + salt) & 0xFF)
        ev[i][0].record(stream)
        graph.replay() if graph is not None else call()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in ev) / steps, graph


# What binds each call's decode kernel, from its timeline and ncu captures (profiles/): the
# HBM roofline below is the contract's, but not every call is HBM-bound.
BINDS = {
    "c16+shared_prefix": "tensor-core MMA stream (96-row kernel: 34 MMAs a 64-position tile, "
                         "each bound by the shared-memory operand bytes it reads)",
    "c24+shared_prefix": "tensor-core MMA stream (96-row kernel)",
    "c16p128+shared_prefix": "tensor-core MMA stream (96-row kernel)",
    "long96": "tensor-core MMA stream (96-row kernel)",
    "c16": "row-copy issue and the ring's refill (16-row kernel; the shared rows from L2)",
    "c24": "row-copy issue and the ring's refill (16-row kernel; the shared rows from L2)",
    "c16p128": "row-copy issue and the ring's refill (16-row kernel)",
    "long": "fixed per-call latencies around ~8 streamed tiles per CTA",
    "longp128": "fixed per-call latencies around ~8 streamed tiles per CTA",
    "mtp": "the 48-row ring's round trip, DRAM 66 % busy",
}
# FP8 dense tensor peak: the measured bf16 cuBLAS burst times the nominal fp8 : bf16 ratio
# (4.5 : 2.25 PFLOP/s).
FP8_OVER_BF16 = 2.0


def measured_fp8_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]) * FP8_OVER_BF16, "measured bf16 burst x 2"
    return FALLBACK_BF16_TFLOPS * FP8_OVER_BF16, "fallback bf16 burst x 2"


def roofline_for(case, entry, ms, peak, peak_kind, config, shared):
    """Roofline of one decode call: algorithmic bytes / device time against the HBM copy
    peak.  A shared-prefix call (and any call on pages, whose shared pages are the same
    memory) counts the shared rows once; the plain call on a shared-prefix batch is given
    both readings.  Beside it, the same call's algorithmic FP8 work (2 x (576 + 512) flops
    per attended row and position) against the FP8 tensor peak, and what binds the call."""
    paged = int(case.meta.get("page_size", 1)) > 1
    distinct = mla_inputs.algorithmic_bytes(case, shared if (entry == "shared_prefix" or paged) else 0)
    r = {"bound": "hbm", "achieved": distinct / (ms * 1e-3) / 1e9, "peak": peak,
         "unit": "GB/s", "peak_kind": f"{peak_kind} copy bandwidth",
         "traffic": recorded_traffic(config, entry),
         "algorithmic_bytes": distinct}
    r["frac"] = r["achieved"] / peak
    key = f"{config}+{entry}" if entry == "shared_prefix" else config
    r["binds"] = BINDS.get(key)
    flops = mla_inputs.useful_flops(case.kv_lens, case.q_lens, case.H)
    tpeak, tkind = measured_fp8_tflops()
    ach = flops / (ms * 1e-3) / 1e12
    r["tensor_roofline"] = {"bound": "tensor", "achieved": ach, "peak": tpeak, "unit": "TFLOP/s",
                            "peak_kind": tkind, "frac": ach / tpeak, "algorithmic_flops": flops}
    if entry == "shared_prefix":
        r["kernel"] = ("mla_decode_shared_prefix call (one cascade decode launch: prefix units "
                       "then per-request units, then the cascade merge)")
        r["bytes_counted"] = ("each distinct cache row once (the shared prefix's rows once for "
                              "the whole batch), 580 B per row with its index (on pages: 576 B "
                              "per distinct row and 4 B per page id of every request), plus q, "
                              "o and lse")
    else:
        r["kernel"] = "mla_decode call (decode + merge kernels)"
        r["bytes_counted"] = ("580 B per attended position (row + index), plus q, o and lse"
                              if not paged else
                              "576 B per distinct cache row, 4 B per page id, plus q, o and lse")
        if shared > 0 and not paged:
            # every request names the shared rows: gathered once per request, but the
            # distinct rows are what DRAM must deliver at least once
            d2 = mla_inputs.algorithmic_bytes(case, shared)
            r["distinct_bytes"] = d2
            r["frac_distinct"] = d2 / (ms * 1e-3) / 1e9 / peak
            r["bytes_counted"] += ("; frac counts the shared prefix once per request (all of "
                                   "it gathered), frac_distinct once per batch")
    return r


def time_adjacent(pm, dev, stream, flush, steps, warmup, seed):
    """The steps around the decode, each on its own (L2 flushed before every call): the
    q-rope + concat + fp8 cache write at the c16 and mtp token counts, and the latent ->
    v_head_dim matmul on the decode's o at the same shapes."""
    out = {}

    def timed(fn):
        for _ in range(warmup):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i in range(steps):
            flush.fill_((i + 41) & 0xFF)
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(b) for a, b in ev) / steps

    peak, _ = measured_peaks()
    # the floor of this timing harness: one launch of a trivial kernel (a 16-element add)
    # between the same events after the same flush; small kernels sit just above it
    x = torch.zeros(16, device=dev)
    out["event_floor_us"] = timed(lambda: x.add_(1.0)) * 1e3
    for name, T in (("c16", 16), ("mtp", 256)):
        H = 12
        inp = mla_inputs.make_rope_inputs(T, H, seed=seed + T, device=dev)
        # the entries land at random slots of a 2^20-row pool (604 MB: larger than L2, small
        # enough for a profiler's replay)
        kv = torch.zeros((1 << 20, 576), dtype=torch.uint8, device=dev)
        g = torch.Generator(device=dev).manual_seed(seed + T)
        slots = torch.randperm(kv.shape[0], generator=g, device=dev)[:T].to(torch.int32)
        q_out = torch.empty((T, H, 576), dtype=torch.uint8, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        qs = torch.tensor(mla_inputs.DEFAULT_Q_SCALE, device=dev)
        ks = torch.tensor(mla_inputs.DEFAULT_KV_SCALE, device=dev)
        ms = timed(lambda: pm.mla_qk_rope_concat_and_cache(
            inp["q_nope"], inp["q_pe"], inp["kv_c"], inp["k_pe"], inp["positions"],
            inp["cos_sin"], 0, slots, qs, ks, q_out, kv, err))
        if int(err.item()) != 0:
            raise RuntimeError("device error in the rope/cache-write timing")
        nbytes = T * (2 * H * 576 + 2 * 576 + 8 + 256 + H * 576 + 576)
        out[f"rope_cache_{name}"] = {
            "op": "mla_qk_rope_concat_and_cache", "tokens": T, "heads": H,
            "us_per_call": ms * 1e3, "bytes": nbytes, "GB/s": nbytes / (ms * 1e-3) / 1e9,
            "frac_of_hbm_peak": nbytes / (ms * 1e-3) / 1e9 / peak,
            "bytes_counted": "bf16 q (latent + rope), new latent + rope key, position, slot, "
                             "table row in; fp8 q and one 576-B cache entry out, per token",
            "launches": 1}
        del kv
        o, w_uv = mla_inputs.make_vproj(T, H, seed=seed + 17, device=dev, o_scale=0.05)
        v = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
        ms = timed(lambda: pm.mla_latent_to_v(o, w_uv, v))
        nbytes = (o.numel() + w_uv.numel() + v.numel()) * 2
        out[f"latent_to_v_{name}"] = {
            "op": "mla_latent_to_v", "tokens": T, "heads": H, "us_per_call": ms * 1e3,
            "bytes": nbytes, "GB/s": nbytes / (ms * 1e-3) / 1e9,
            "frac_of_hbm_peak": nbytes / (ms * 1e-3) / 1e9 / peak,
            "bytes_counted": "o in, every head's 512 x 128 bf16 matrix, v out", "launches": 1}
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="c16", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--num-kv-splits", type=int, default=0)
    ap.add_argument("--entry", default="auto", choices=["auto", "plain", "shared_prefix"],
                    help="auto: mla_decode_shared_prefix for workloads whose requests share a "
                         "prefix by construction (c16, c24), else mla_decode")
    ap.add_argument("--q-scale", type=float, default=mla_inputs.DEFAULT_Q_SCALE)
    ap.add_argument("--kv-scale", type=float, default=mla_inputs.DEFAULT_KV_SCALE)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-l2-flush", action="store_true")
    ap.add_argument("--clock-soak-s", type=float, default=SOAK_S,
                    help="shortest span of steps the nvidia-smi clock record covers")
    ap.add_argument("--eager", action="store_true",
                    help="time eager calls instead of a CUDA-graph replay of the call")
    ap.add_argument("--ref-requests", type=int, default=2)
    ap.add_argument("--ref-heads", type=int, default=12)
    ap.add_argument("--v-proj", action="store_true",
                    help="also time mla_latent_to_v (the latent o mapped to v_head_dim 128) on "
                         "this workload's o, L2 flushed before each call; reported under "
                         "'v_proj', outside the decode's timed region")
    ap.add_argument("--no-adjacent", action="store_true",
                    help="skip timing the steps around the decode (rope/cache write, latent "
                         "-> v_head_dim), reported under 'adjacent_steps'")
    ap.add_argument("--extra-configs", default="default",
                    help="comma-separated workloads also timed in this run (same process, same "
                         "clock record) and reported under 'configs'; 'default': c24 (shared-"
                         "prefix and plain), long, mtp and long96 when the main workload is "
                         "c16; 'none': no others")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    world, rank, local, dist = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        if dist is not None:
            dist.destroy_process_group()
        return

    import paged_mla_latent_gb300 as pm
    dev = torch.device("cuda", local)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = measured_peaks()

    def setup(config, entry_arg):
        case = mla_inputs.make_case(config, seed=args.seed + rank, device=dev,
                                    q_scale=args.q_scale, kv_scale=args.kv_scale)
        n_tok, H = case.q.shape[0], case.q.shape[1]
        o = torch.empty((n_tok, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((n_tok, H), dtype=torch.float32, device=dev)
        shared = int(case.meta.get("shared_prefix", 0))
        entry = entry_arg
        if entry == "auto":
            entry = "shared_prefix" if shared > 0 and args.num_kv_splits <= 0 else "plain"
        # (a shared-prefix workspace also serves the plain call on the same batch)
        ws = pm.make_workspace(case.B, H, case.max_seqlen_q, args.num_kv_splits, dev,
                               shared_prefix=(shared > 0 and args.num_kv_splits <= 0))

        def call(which=None, q=case.q, qo=case.qo_indptr, kvp=case.kv_indptr,
                 idx=case.kv_indices, last=case.kv_last_page_lens, out=o, l=lse):
            # on the current stream (capturable)
            if (which or entry) == "shared_prefix":
                pm.mla_decode_shared_prefix(q, case.kv, out, qo, kvp, idx, last,
                                            case.max_seqlen_q, case.sm_scale, case.q_scale,
                                            case.kv_scale, shared, lse_out=l, workspace=ws)
            else:
                pm.mla_decode(q, case.kv, out, qo, kvp, idx, last, case.max_seqlen_q,
                              case.sm_scale, case.q_scale, case.kv_scale,
                              num_kv_splits=args.num_kv_splits, lse_out=l, workspace=ws)
        return case, entry, shared, ws, o, lse, call

    def check(ws, what):
        st = pm.mla_check_error(ws)
        if st != 0:
            raise RuntimeError(f"device error in {what}: {pm.mla_status_string(st)}")

    case, entry, shared, ws, o, lse, call = setup(args.config, args.entry)
    n_tok, H = case.q.shape[0], case.q.shape[1]
    paged = int(case.meta.get("page_size", 1)) > 1

    for i in range(args.warmup):
        if not args.no_l2_flush:
            flush.fill_(i & 0xFF)
        call()
    torch.cuda.synchronize(dev)
    check(ws, "warm-up")

    # The timed call is a CUDA-graph replay of one mla_decode call (its two kernel launches),
    # so host-side argument marshalling does not leak into the device time.
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        torch.cuda.synchronize(dev)
        for i in range(2):
            if not args.no_l2_flush:
                flush.fill_(i & 0xFF)
            graph.replay()
        torch.cuda.synchronize(dev)
    t_host0 = time.perf_counter()
    for _ in range(20):
        call()
    t_host = (time.perf_counter() - t_host0) / 20
    torch.cuda.synchronize(dev)

    # The other measured workloads (c24, long, mtp, long96), timed in the same process and
    # clock record; their inputs are built before the record starts.
    extra_list = []
    if args.extra_configs == "default":
        if args.config == "c16":
            extra_list = [("c24", "shared_prefix"), ("c24", "plain"), ("long", "plain"),
                          ("mtp", "plain"), ("long96", "plain")]
    elif args.extra_configs != "none":
        extra_list = [(c, "auto") for c in args.extra_configs.split(",") if c]
    built = {}
    extra_setups = []
    for cfg, ent in extra_list:
        if cfg not in built:
            built[cfg] = setup(cfg, ent)
        c2, e2, sh2, ws2, o2, l2, call2 = built[cfg]
        e2 = ent if ent != "auto" else e2
        extra_setups.append((cfg, c2, e2, sh2, ws2,
                             (lambda call2=call2, e2=e2: call2(which=e2))))
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    extras = {}
    with ClockSampler(local) as clocks:
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            if not args.no_l2_flush:
                flush.fill_((i + 7) & 0xFF)
            starts[i].record(stream)
            if graph is not None:
                graph.replay()
            else:
                call()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        # nvidia-smi samples every 100 ms: when the K timed steps take less than a second,
        # the same steps keep running (untimed) until a second has passed, so the clock
        # record covers this load.
        soak = 0
        while time.perf_counter() - t_wall0 < args.clock_soak_s:
            for i in range(64):
                if not args.no_l2_flush:
                    flush.fill_((i + 3) & 0xFF)
                if graph is not None:
                    graph.replay()
                else:
                    call()
            soak += 64
            torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        check(ws, "the timed region")
        step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
        mean_ms = max_over_ranks(sum(step_ms) / len(step_ms), dist, dev)

        # Workloads with a shared prefix: the plain mla_decode on the same inputs, timed the
        # same way, reported beside the shared-prefix call.
        plain = None
        if entry == "shared_prefix":
            p_ms, _ = time_graph(lambda: call(which="plain"), args.steps, max(args.warmup, 3),
                                 flush, args.no_l2_flush, stream, dev, args.eager, salt=11)
            p_ms = max_over_ranks(p_ms, dist, dev)
            gb = mla_inputs.gathered_kv_bytes(case.kv_lens)
            plain = {"entry": "mla_decode", "us_per_call": p_ms * 1e3,
                     "value": whole_job_rate(world, gb, p_ms), "unit": UNIT,
                     "gathered_rate_over_peak_measured": 100.0 * gb / (p_ms * 1e-3) / 1e9 / peak,
                     "roofline": roofline_for(case, "plain", p_ms, peak, peak_kind,
                                              args.config, shared)}
            check(ws, "the plain timing")

        for cfg, c2, e2, sh2, ws2, call2 in extra_setups:
            ms2, _ = time_graph(call2, args.steps, max(args.warmup, 3), flush, args.no_l2_flush,
                                stream, dev, args.eager, salt=23)
            ms2 = max_over_ranks(ms2, dist, dev)
            check(ws2, f"the {cfg} timing")
            gb2 = mla_inputs.gathered_kv_bytes(c2.kv_lens)
            key = cfg if e2 == "plain" and sh2 == 0 else f"{cfg}+{e2}"
            extras[key] = {
                "workload": WORKLOAD_TEXT[cfg],
                "entry": "mla_decode_shared_prefix" if e2 == "shared_prefix" else "mla_decode",
                "us_per_call": ms2 * 1e3, "value": whole_job_rate(world, gb2, ms2), "unit": UNIT,
                "gathered_rate_over_peak_measured": 100.0 * gb2 / (ms2 * 1e-3) / 1e9 / peak,
                "positions": c2.total_kv, "gathered_kv_bytes": gb2,
                "roofline": roofline_for(c2, e2, ms2, peak, peak_kind, cfg, sh2),
            }
            extras[key]["roofline"]["limiter"] = LIMITER.get(key, LIMITER.get(cfg))
    del built, extra_setups

    v_proj = None
    if args.v_proj:
        _, w_uv = mla_inputs.make_vproj(1, H, seed=args.seed + 17, device=dev)
        v_out = torch.empty((n_tok, H, 128), dtype=torch.bfloat16, device=dev)
        for i in range(max(args.warmup, 3)):
            pm.mla_latent_to_v(o, w_uv, v_out)
        vev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_((i + 29) & 0xFF)
            vev[i][0].record(stream)
            pm.mla_latent_to_v(o, w_uv, v_out)
            vev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        v_ms = max_over_ranks(sum(a_.elapsed_time(b_) for a_, b_ in vev) / args.steps, dist, dev)
        v_bytes = (o.numel() + w_uv.numel() + v_out.numel()) * 2
        v_proj = {"op": "mla_latent_to_v", "us_per_call": v_ms * 1e3, "bytes": v_bytes,
                  "GB/s": v_bytes / (v_ms * 1e-3) / 1e9, "launches": 1,
                  "bytes_counted": "o in, every head's 512 x 128 bf16 matrix, v out",
                  "l2": "flushed before every call"}

    adjacent = None
    if not args.no_adjacent:
        adjacent = time_adjacent(pm, dev, stream, flush, args.steps, max(args.warmup, 3),
                                 args.seed)

    gathered = mla_inputs.gathered_kv_bytes(case.kv_lens)
    value = whole_job_rate(world, gathered, mean_ms)
    roof = roofline_for(case, entry, mean_ms, peak, peak_kind, args.config, shared)
    roof["limiter"] = LIMITER.get(f"{args.config}+{entry}", LIMITER.get(args.config))

    # ---- end to end through the C ABI with host buffers (pinned), copies in the timed region
    e2e = None
    if not args.no_e2e:
        # The step's inputs sit in one pinned host buffer and go over in one copy; o and
        # lse are written into one device buffer and come back in one copy (the used part
        # of kv_indices only).
        used = int(case.kv_indptr[-1])
        parts = [("q", case.q), ("qo", case.qo_indptr), ("kvp", case.kv_indptr),
                 ("idx", case.kv_indices[:used]), ("last", case.kv_last_page_lens)]
        # The shared-prefix call's page table goes over as a prefix cache keeps it: the
        # shared pages once, then each request's own pages; mla_expand_shared_prefix_indices
        # builds the full table on the device inside the timed step.
        compact = None
        if entry == "shared_prefix":
            ps = int(case.meta.get("page_size", 1))
            n_sh = shared // ps
            kvp_h = [int(x) for x in case.kv_indptr.cpu()]
            idx_h = case.kv_indices.cpu()
            sh_ids = idx_h[kvp_h[0]:kvp_h[0] + n_sh].clone()
            if all(torch.equal(idx_h[kvp_h[b]:kvp_h[b] + n_sh], sh_ids) for b in range(case.B)):
                owns = [idx_h[kvp_h[b] + n_sh:kvp_h[b + 1]] for b in range(case.B)]
                own_ptr = [0]
                for x in owns:
                    own_ptr.append(own_ptr[-1] + x.numel())
                compact = (n_sh, own_ptr[-1])
                parts = [("q", case.q), ("qo", case.qo_indptr), ("shared", sh_ids),
                         ("optr", torch.tensor(own_ptr, dtype=torch.int32)),
                         ("own", torch.cat(owns)), ("last", case.kv_last_page_lens)]
        offs, tot = {}, 0
        for k, t in parts:
            offs[k] = tot
            tot += (t.numel() * t.element_size() + 255) // 256 * 256
        h_in = torch.empty(tot, dtype=torch.uint8).pin_memory()
        d_in_buf = torch.empty(tot, dtype=torch.uint8, device=dev)
        d_in = {}
        for k, t in parts:
            nb = t.numel() * t.element_size()
            h_in[offs[k]:offs[k] + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
            d_in[k] = d_in_buf[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
        o_bytes = o.numel() * o.element_size()
        lse_off = (o_bytes + 255) // 256 * 256
        d_out = torch.empty(lse_off + lse.numel() * lse.element_size(), dtype=torch.uint8,
                            device=dev)
        o_e = d_out[:o_bytes].view(o.dtype).view(o.shape)
        lse_e = d_out[lse_off:].view(lse.dtype).view(lse.shape)
        h_out = torch.empty(d_out.numel(), dtype=torch.uint8).pin_memory()
        h2d = sum(t.numel() * t.element_size() for _, t in parts)
        d2h = o_bytes + lse.numel() * lse.element_size()
        if compact is not None:
            kvp_dev = torch.empty(case.B + 1, dtype=torch.int32, device=dev)
            idx_dev = torch.empty(case.B * compact[0] + compact[1], dtype=torch.int32, device=dev)
        else:
            kvp_dev, idx_dev = d_in["kvp"], d_in["idx"]
        # the public call prepared once for these buffers (PreparedDecode), run each step
        prep = pm.PreparedDecode(d_in["q"], case.kv, o_e, d_in["qo"], kvp_dev, idx_dev,
                                 d_in["last"], case.max_seqlen_q, case.sm_scale, case.q_scale,
                                 case.kv_scale, num_kv_splits=args.num_kv_splits, lse_out=lse_e,
                                 workspace=ws,
                                 shared_prefix_len=shared if entry == "shared_prefix" else None,
                                 stream=stream,
                                 compact_page_table=(None if compact is None else
                                                     (d_in["shared"], d_in["optr"], d_in["own"])))
        e_ms = []
        n_e2e = max(5, min(args.steps, 20))
        for i in range(n_e2e + 2):
            if not args.no_l2_flush:
                flush.fill_(i & 0xFF)
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            d_in_buf.copy_(h_in, non_blocking=True)
            prep.run()
            h_out.copy_(d_out, non_blocking=True)
            torch.cuda.synchronize(dev)
            if i >= 2:
                e_ms.append((time.perf_counter() - t0) * 1e3)
        check(ws, "the end-to-end timing")
        # (o was last written by the device-timed calls, or by the plain call timed for
        # comparison: the same attention, so equal within the method's tolerance)
        if not torch.allclose(h_out[:o_bytes].view(o.dtype).view(o.shape).float(),
                              o.float().cpu(), rtol=1e-2, atol=1e-2):
            raise RuntimeError("end-to-end output differs from the device-timed call's")
        e_mean = max_over_ranks(sum(e_ms) / len(e_ms), dist, dev)
        e2e = {"value": whole_job_rate(world, gathered, e_mean), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_mean,
               "page_table": ("shared pages once + each request's own pages, expanded on the "
                              "device (mla_expand_shared_prefix_indices, run by "
                              "PreparedDecode) inside the step"
                              if compact is not None else "full CSR uploaded every step")}

    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        dt, sb, cores, pos = time_oracle(case, args.ref_requests, args.ref_heads)
        cpu_base = {"value": sb / dt / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
                    "sample": f"first {args.ref_requests} request(s) x {args.ref_heads} heads of "
                              f"this workload ({pos} positions), GB/s scaled to all {H} heads",
                    "cpu": cpu_model()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "us_per_call": mean_ms * 1e3,
            # 576 B per attended position over the copy peak: a rate, not a DRAM fraction
            # (shared rows served once per group, or from L2, push it past 100 %)
            "gathered_rate_over_peak_measured": 100.0 * value / world / peak,
            "gathered_rate_over_nominal_8tbs": 100.0 * value / world / NOMINAL_HBM_GBS,
            # the DRAM fraction: algorithmic bytes (distinct rows) over the copy peak
            "pct_of_hbm_peak_measured": 100.0 * roof["frac"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8_e4m3 (fp32 accumulate)", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config,
                       "seed": args.seed, "requests": case.B, "heads": H,
                       "q_len": case.max_seqlen_q, "positions": case.total_kv,
                       "gathered_kv_bytes": gathered,
                       "algorithmic_bytes": roof["algorithmic_bytes"],
                       "num_kv_splits": args.num_kv_splits,
                       "entry": ("mla_decode_shared_prefix (shared prefix of %d positions, "
                                 "known to the caller)" % shared) if entry == "shared_prefix"
                                else "mla_decode",
                       "l2": "flushed before every step (512 MB write, outside the timed region)"
                             if not args.no_l2_flush else "not flushed",
                       "parallelism": f"{world} independent replicas (one batch per GPU)"},
            "roofline": roof,
            "cpu_baseline": cpu_base,
            "e2e": e2e,
            "gpu_launches": 2 * args.steps,
            "plain_call": plain,
            "configs": extras,
            "adjacent_steps": adjacent,
            **({"v_proj": v_proj} if v_proj is not None else {}),
            "clocks": dict(clocks.summary(),
                           window=("the timed region" if soak == 0 else
                                   f"the timed region and {soak} identical untimed steps "
                                   f"right after it ({args.clock_soak_s:g} s in all)")
                           + (", then the plain call and the other workloads"
                              if (plain or extras) else "")),
            "wall_s_timed_region": t_wall,
            "timing": "CUDA graph replay of one call per step" if graph is not None else "eager calls",
            "host_us_per_eager_call": t_host * 1e6,
            "kernel_source_hash": kernel_source_hash(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
